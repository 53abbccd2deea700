"""Pins of the oracle's Muon optimizer.

"Teaching Mario to speedrun", sec. 8 and "puff-rs" (PufferLib 5.0 uses Muon,
five Newton-Schulz iterations per weight matrix).  The definition is Muon's
published write-up (quintic iteration with (a, b, c) = (3.4445, -4.7750,
2.0315) on the Frobenius-normalised matrix, Nesterov momentum, update scaled
by sqrt(max(1, rows/cols)); Adam for non-matrix parameters).
Pinned against:
- numpy's SVD: the iteration maps G = U S V^T to U phi^5(S / ||G||) V^T with
  phi(x) = a x + b x^3 + c x^5 (a scalar polynomial on the singular values),
  for wide, tall, square and one-row matrices;
- scale invariance and the transpose symmetry of that map;
- the Muon step's first two steps written out from the write-up's momentum
  rule, and Adam (the pinned orc_adam) on the vector parameters;
- the whole update with Muon equals the composition of its pinned steps.
"""
import math

import numpy as np
import pytest

import oracle

A, B, C = 3.4445, -4.7750, 2.0315


def _phi5(x):
    for _ in range(5):
        x = A * x + B * x ** 3 + C * x ** 5
    return x


def _svd_ns(G):
    U, s, Vt = np.linalg.svd(G, full_matrices=False)
    nrm = math.sqrt(float((G * G).sum()))
    return (U * _phi5(s / (nrm + 1e-7))) @ Vt


@pytest.mark.parametrize("shape", [(3, 7), (7, 3), (16, 16), (1, 9), (9, 1), (64, 256), (16, 256)])
def test_newton_schulz_equals_polynomial_of_singular_values(shape):
    G = np.random.default_rng(sum(shape)).normal(size=shape)
    np.testing.assert_allclose(oracle.newton_schulz5(G), _svd_ns(G), rtol=1e-10, atol=1e-12)


def test_newton_schulz_invariances():
    rng = np.random.default_rng(1)
    G = rng.normal(size=(6, 10))
    X = oracle.newton_schulz5(G)
    # up to the 1e-7 in the normaliser, amplified by at most a^5 ~ 480 (the
    # iteration's slope at 0)
    np.testing.assert_allclose(oracle.newton_schulz5(37.5 * G), X, rtol=1e-5, atol=1e-7)
    np.testing.assert_allclose(oracle.newton_schulz5(G.T), X.T, rtol=1e-12, atol=1e-14)
    # singular values land in the iteration's band around 1 (never exactly 1)
    s = np.linalg.svd(X, compute_uv=False)
    assert np.all((s > 0.6) & (s < 1.2))


NET = oracle.Net(obs_dim=5, h1=8, h2=6, act=0, heads=(3, 2), n_gauss=1)


def _regions(net):
    D, H1, H2, Cc = net.obs_dim, net.h1, net.h2, net.out_cols
    o = 0
    out = {}
    for name, n, shape in [("W1", H1 * D, (H1, D)), ("b1", H1, None), ("W2", H2 * H1, (H2, H1)),
                           ("b2", H2, None), ("W3", Cc * H2, (Cc, H2)), ("b3", Cc, None),
                           ("logstd", net.n_gauss, None)]:
        out[name] = (slice(o, o + n), shape)
        o += n
    return out


def test_muon_first_two_steps_from_the_definition():
    rng = np.random.default_rng(2)
    P = NET.num_params
    p = rng.normal(size=P)
    g1, g2 = rng.normal(size=P), rng.normal(size=P)
    z = np.zeros(P)
    lr_m, beta, lr = 0.02, 0.95, 1e-3
    p1, mom1, m1, v1 = oracle.muon(NET, p, g1, z, z, z, 1, lr_m, beta, lr)
    p2, mom2, m2, v2 = oracle.muon(NET, p1, g2, mom1, m1, v1, 2, lr_m, beta, lr)
    # Adam on the vector parameters: the pinned orc_adam on those entries
    pa1, ma1, va1 = oracle.adam(p, g1, z, z, 1, lr)
    pa2, _, _ = oracle.adam(pa1, g2, ma1, va1, 2, lr)
    for name, (sl, shape) in _regions(NET).items():
        if shape is None:
            np.testing.assert_allclose(p2[sl], pa2[sl], rtol=1e-14, atol=1e-15)
            continue
        rows, cols = shape
        scale = math.sqrt(max(1.0, rows / cols))
        # step 1: mom = g1, u = g1 + beta g1
        mo1 = g1[sl]
        u1 = g1[sl] + beta * mo1
        q1 = p[sl] - lr_m * scale * _svd_ns(u1.reshape(shape)).ravel()
        # step 2: mom = beta mom + g2, u = g2 + beta mom
        mo2 = beta * mo1 + g2[sl]
        u2 = g2[sl] + beta * mo2
        q2 = q1 - lr_m * scale * _svd_ns(u2.reshape(shape)).ravel()
        np.testing.assert_allclose(mom2[sl], mo2, rtol=1e-14)
        np.testing.assert_allclose(p2[sl], q2, rtol=1e-9, atol=1e-11)


def test_update_with_muon_is_the_composition():
    rng = np.random.default_rng(3)
    T, N, E, M = 4, 8, 2, 2
    B = T * N
    P = NET.num_params
    p0 = rng.normal(0, 0.5, P)
    obs = rng.normal(size=(B, NET.obs_dim)).astype(np.float32)
    act = np.stack([rng.integers(0, n, B) for n in NET.heads], 1).astype(np.int32)
    actc = rng.normal(size=(B, NET.n_gauss)).astype(np.float32)
    lp = rng.normal(-2, 0.3, B).astype(np.float32)
    val = rng.normal(size=(T, N)).astype(np.float32)
    rew = rng.normal(size=(T, N)).astype(np.float32)
    done = (rng.random((T, N)) < 0.2).astype(np.float32)
    boot = rng.normal(size=N).astype(np.float32)
    hp = oracle.Hyper(lr=1e-3, seed=9, optimizer=1, muon_lr=0.01, muon_beta=0.9)
    res = oracle.update(NET, hp, T, N, E, M, obs, act, actc, lp, val, rew, done, boot, p0)
    adv, ret = oracle.gae(rew, val, done, boot, hp.gamma, hp.lam)
    mean, sd = oracle.moments(adv)
    q, m, v, mo = p0.copy(), np.zeros(P), np.zeros(P), np.zeros(P)
    step = 0
    mb = B // M
    for e in range(E):
        perm = oracle.perm(hp.seed, e, B)
        for k in range(M):
            _, g, _, _ = oracle.loss_grad(NET, q, perm[k * mb:(k + 1) * mb], obs, act, actc, lp,
                                          adv.ravel(), ret.ravel(), normalize=True, adv_mean=mean,
                                          adv_std=sd)
            _, g = oracle.clip_grad_norm(g, hp.max_grad_norm)
            step += 1
            q, mo, m, v = oracle.muon(NET, q, g, mo, m, v, step, hp.muon_lr, hp.muon_beta, hp.lr)
    np.testing.assert_allclose(res.params, q, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(res.mom, mo, rtol=1e-12, atol=1e-13)
    assert res.step == step


# ---- bf16 Newton-Schulz (the write-up's precision) --------------------------------
@pytest.mark.parametrize("shape", [(64, 256), (256, 256), (16, 256), (512, 1397)])
def test_newton_schulz_bf16_is_close_to_fp64_and_rounds(shape):
    rng = np.random.default_rng(sum(shape))
    G = rng.standard_normal(shape)
    x64 = oracle.newton_schulz5(G)
    x16 = oracle.newton_schulz5(G, bf16=True)
    err = np.linalg.norm(x16 - x64) / np.linalg.norm(x64)
    assert err < 2e-2, err
    assert err > 0
    # every entry of the result is a bf16 value
    assert all(oracle.round_bf16(v) == v for v in x16.ravel()[:2000])


def test_newton_schulz_bf16_transposes_exactly_and_keeps_singular_values_in_band():
    rng = np.random.default_rng(3)
    G = rng.standard_normal((48, 200))
    x = oracle.newton_schulz5(G, bf16=True)
    np.testing.assert_array_equal(oracle.newton_schulz5(G.T.copy(), bf16=True), x.T)
    s = np.linalg.svd(x, compute_uv=False)
    # the quintic's five iterations take every singular value into a band
    # around 1 (the write-up's (a, b, c) do not converge to exactly 1)
    assert s.min() > 0.5 and s.max() < 1.3, (s.min(), s.max())
