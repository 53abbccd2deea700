"""Pins of the oracle's per-minibatch advantages from fresh values.

"Teaching Mario to speedrun", sec. 8 "The Puffer net, and the trainer"
(PufferLib 5.0: advantages computed per minibatch from fresh values, by GAE or
V-trace).  V-trace itself is not on the pages; its definition is Espeholt et
al. 2018 ("IMPALA", sec. 4.1, eq. 1 with the lambda-weighted traces of its
remarks).  The oracle's backward recursion is checked against:
- the definition's sum of trace products, evaluated term by term, over every
  done pattern of short horizons (a wrong index, a dropped clip or a wrong
  trace factor changes at least one pattern);
- its on-policy reduction to GAE (the already pinned oracle.gae), and with
  lambda = 1 to the discounted return-to-go;
- the degenerate clips (rho_bar = 0: no correction; c_bar = 0: one-step
  importance-weighted TD);
- for the whole minibatch step: the ordinary loss of the same rows when the
  stored values equal the fresh ones (so the two advantage routes coincide).
"""
import itertools

import numpy as np
import pytest

import oracle


def _seg_data(T, N, seed, p_done=0.2):
    rng = np.random.default_rng(seed)
    r = rng.normal(size=(T, N)).astype(np.float32)
    d = (rng.random((T, N)) < p_done).astype(np.float32)
    b = rng.normal(size=N).astype(np.float32)
    return rng, r, d, b


def _direct_vtrace(r, d, b, v, rho, gamma, lam, rho_bar, c_bar):
    """v_s - V_s = sum_{t>=s} gamma^{t-s} (prod_{i=s}^{t-1} c_i alive_i) rho_t delta_t
    with rho_t = min(rho_bar, ratio_t), c_i = lam min(c_bar, ratio_i),
    delta_t = r_t + gamma alive_t V_{t+1} - V_t, V_T = boot, alive = 1 - done.
    One segment (1-D arrays over t)."""
    T = r.size
    r, d, v, rho = (np.asarray(x, np.float64) for x in (r, d, v, rho))
    alive = 1.0 - d
    vn = np.append(v[1:], float(b))
    delta = r + gamma * alive * vn - v
    rw = np.minimum(rho_bar, rho)
    c = lam * np.minimum(c_bar, rho)
    out = np.zeros(T)
    for s in range(T):
        acc = 0.0
        for t in range(s, T):
            trace = np.prod(c[s:t] * alive[s:t]) if t > s else 1.0
            acc += gamma ** (t - s) * trace * rw[t] * delta[t]
        out[s] = acc
    return out


@pytest.mark.parametrize("clips", [(1.0, 1.0), (0.7, 1.3), (2.0, 0.5)])
def test_vtrace_recursion_equals_definition_all_done_patterns(clips):
    T, gamma, lam = 4, 0.9, 0.8
    rho_bar, c_bar = clips
    rng = np.random.default_rng(5)
    for pat in itertools.product([0.0, 1.0], repeat=T):
        d = np.array(pat, np.float32)[:, None]
        r = rng.normal(size=(T, 1)).astype(np.float32)
        b = rng.normal(size=1).astype(np.float32)
        v = rng.normal(size=(T, 1))
        ratio = np.exp(rng.normal(0, 0.5, size=(T, 1)))
        adv, ret = oracle.segment_advantage(r, d, b, [0], v, ratio, gamma, lam, rho_bar, c_bar)
        ref = _direct_vtrace(r[:, 0], d[:, 0], b[0], v[:, 0], ratio[:, 0], gamma, lam, rho_bar,
                             c_bar)
        np.testing.assert_allclose(adv[:, 0], ref, rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(ret[:, 0], ref + v[:, 0], rtol=1e-12, atol=1e-12)


def test_on_policy_reduces_to_gae_on_the_selected_segments():
    T, N = 37, 12
    rng, r, d, b = _seg_data(T, N, 1)
    envs = np.array([7, 2, 11, 0, 5], np.int32)
    v = rng.normal(size=(T, envs.size)).astype(np.float32)
    g_adv, g_ret = oracle.gae(r[:, envs], v, d[:, envs], b[envs], 0.97, 0.9)
    a0, r0 = oracle.segment_advantage(r, d, b, envs, v, None, 0.97, 0.9)
    ones = np.ones((T, envs.size))
    a1, r1 = oracle.segment_advantage(r, d, b, envs, v, ones, 0.97, 0.9, 1.0, 1.0)
    a2, r2 = oracle.segment_advantage(r, d, b, envs, v, ones, 0.97, 0.9, 3.0, 2.0)
    for a, rt in ((a0, r0), (a1, r1), (a2, r2)):
        np.testing.assert_allclose(a, g_adv, rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(rt, g_ret, rtol=1e-12, atol=1e-12)


def test_lambda_one_on_policy_is_return_to_go():
    T, N, gamma = 20, 3, 0.95
    rng, r, d, b = _seg_data(T, N, 2)
    v = rng.normal(size=(T, N))
    _, ret = oracle.segment_advantage(r, d, b, np.arange(N), v, np.ones((T, N)), gamma, 1.0)
    G = np.zeros((T, N))
    nxt = b.astype(np.float64)
    r64, d64 = r.astype(np.float64), d.astype(np.float64)
    for t in range(T - 1, -1, -1):
        nxt = r64[t] + gamma * (1.0 - d64[t]) * nxt
        G[t] = nxt
    np.testing.assert_allclose(ret, G, rtol=1e-12, atol=1e-12)


def test_degenerate_clips():
    T, N, gamma, lam = 16, 4, 0.99, 0.95
    rng, r, d, b = _seg_data(T, N, 3)
    v = rng.normal(size=(T, N))
    ratio = np.exp(rng.normal(0, 0.4, size=(T, N)))
    # rho_bar = 0: no correction at all -> v_s = V(x_s)
    adv, ret = oracle.segment_advantage(r, d, b, np.arange(N), v, ratio, gamma, lam, 0.0, 1.0)
    assert np.all(adv == 0.0)
    np.testing.assert_array_equal(ret, v)
    # c_bar = 0: no traces -> adv_t = min(rho_bar, ratio_t) delta_t
    adv, _ = oracle.segment_advantage(r, d, b, np.arange(N), v, ratio, gamma, lam, 1.2, 0.0)
    vn = np.vstack([v[1:], b[None, :].astype(np.float64)])
    delta = r.astype(np.float64) + gamma * (1.0 - d.astype(np.float64)) * vn - v
    np.testing.assert_allclose(adv, np.minimum(1.2, ratio) * delta, rtol=1e-12, atol=1e-12)


NET = oracle.Net(obs_dim=3, h1=4, h2=5, act=0, heads=(3, 2), n_gauss=1)


def _rollout(net, T, N, seed):
    rng = np.random.default_rng(seed)
    p = rng.normal(0, 0.5, net.num_params)
    B = T * N
    obs = rng.normal(size=(B, net.obs_dim)).astype(np.float32)
    act = np.stack([rng.integers(0, n, B) for n in net.heads], 1).astype(np.int32)
    actc = rng.normal(size=(B, net.n_gauss)).astype(np.float32)
    lp = rng.normal(-2.0, 0.3, B).astype(np.float32)
    r = rng.normal(size=(T, N)).astype(np.float32)
    d = (rng.random((T, N)) < 0.15).astype(np.float32)
    b = rng.normal(size=N).astype(np.float32)
    return p, obs, act, actc, lp, r, d, b


def test_fresh_values_are_the_forward_value_and_policy_ratio():
    T, N = 3, 4
    p, obs, act, actc, lp, *_ = _rollout(NET, T, N, 4)
    idx = np.array([5, 0, 11, 7], np.int32)
    val, ratio = oracle.fresh_values(NET, p, idx, obs, act, actc, lp)
    z = oracle.forward(NET, p, obs[idx])
    np.testing.assert_allclose(val, z[:, -1], rtol=1e-13, atol=1e-13)
    logp, _ = oracle.policy_logp(NET, p, obs[idx], act[idx], actc[idx])
    np.testing.assert_allclose(ratio, np.exp(logp - lp[idx].astype(np.float64)), rtol=1e-12)


def test_segment_rows_order():
    rows = oracle.segment_rows(3, 10, [4, 1])
    np.testing.assert_array_equal(rows, [4, 1, 14, 11, 24, 21])


@pytest.mark.parametrize("bf16", [False, True])
def test_fresh_gae_step_equals_ordinary_step_with_fresh_stored_values(bf16):
    """When the rollout's stored values are the current network's values, the
    per-minibatch GAE route and the ordinary route (GAE over the whole
    rollout, then the minibatch's rows, normalised over the minibatch) are the
    same computation."""
    T, N = 6, 8
    p, obs, act, actc, lp, r, d, b = _rollout(NET, T, N, 6)
    envs = np.array([3, 6, 0], np.int32)
    rows = oracle.segment_rows(T, N, envs)
    v_all, _ = oracle.fresh_values(NET, p, np.arange(T * N, dtype=np.int32), obs, act, actc, lp,
                                   bf16_operands=bf16, with_ratio=False)
    val = v_all.reshape(T, N)
    adv, ret = oracle.gae(r, val, d, b, 0.97, 0.9)
    # stored values are fp32; use the fp32-rounded fresh values on both sides
    assert np.allclose(val, val.astype(np.float32), rtol=1e-6)
    mean, sd = oracle.moments(adv.ravel()[rows])
    loss_o, g_o, st_o, _ = oracle.loss_grad(NET, p, rows, obs, act, actc, lp, adv.ravel(),
                                            ret.ravel(), normalize=True, adv_mean=mean,
                                            adv_std=sd, bf16_operands=bf16)
    loss_f, g_f, st_f, _, an, rt = oracle.loss_grad_fresh(
        NET, p, T, N, envs, obs, act, actc, lp, r, d, b, vtrace=False, gamma=0.97, lam=0.9,
        bf16_operands=bf16)
    # oracle.gae reads fp32 values; the fresh route keeps them in fp64
    tol = 1e-6
    np.testing.assert_allclose(rt, ret.ravel()[rows], rtol=tol, atol=tol)
    np.testing.assert_allclose(an, (adv.ravel()[rows] - mean) / (sd + 1e-8), rtol=tol, atol=tol)
    np.testing.assert_allclose(g_f, g_o, rtol=10 * tol, atol=10 * tol)
    np.testing.assert_allclose(st_f, st_o, rtol=10 * tol, atol=10 * tol)


def test_fresh_vtrace_on_policy_equals_fresh_gae():
    T, N = 7, 6
    p, obs, act, actc, lp, r, d, b = _rollout(NET, T, N, 7)
    # logp_old := the current log-probabilities, so every ratio is 1 (up to
    # the fp32 rounding of logp_old)
    logp, _ = oracle.policy_logp(NET, p, obs, act, actc)
    lp = logp.astype(np.float32)
    envs = np.array([5, 1], np.int32)
    a = oracle.loss_grad_fresh(NET, p, T, N, envs, obs, act, actc, lp, r, d, b, vtrace=False)
    v = oracle.loss_grad_fresh(NET, p, T, N, envs, obs, act, actc, lp, r, d, b, vtrace=True,
                               rho_clip=1.0, c_clip=1.0)
    # ratios differ from 1 by the fp32 rounding of logp_old (<= 1e-7 relative)
    for x, y in zip(a[:2] + a[4:], v[:2] + v[4:]):
        np.testing.assert_allclose(x, y, rtol=2e-6, atol=2e-6)


def test_fresh_vtrace_advantages_compose():
    """adv_norm of the V-trace step = normalise(segment_advantage(fresh V,
    fresh ratio)) with the minibatch's own moments."""
    T, N = 5, 6
    p, obs, act, actc, lp, r, d, b = _rollout(NET, T, N, 8)
    envs = np.array([2, 4, 0], np.int32)
    rows = oracle.segment_rows(T, N, envs)
    val, ratio = oracle.fresh_values(NET, p, rows, obs, act, actc, lp)
    adv, ret = oracle.segment_advantage(r, d, b, envs, val, ratio, 0.99, 0.95, 1.0, 1.0)
    mean = adv.mean()
    sd = adv.std(ddof=1)
    *_, an, rt = oracle.loss_grad_fresh(NET, p, T, N, envs, obs, act, actc, lp, r, d, b,
                                        vtrace=True, gamma=0.99, lam=0.95)
    np.testing.assert_allclose(rt, ret.ravel(), rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(an, ((adv - mean) / (sd + 1e-8)).ravel(), rtol=1e-10, atol=1e-10)
    assert np.any(np.abs(ratio - 1.0) > 0.1)   # genuinely off-policy


@pytest.mark.parametrize("mode", [1, 2])
def test_fresh_update_is_the_sequence_of_fresh_steps(mode):
    T, N, E, M = 4, 8, 2, 2
    p, obs, act, actc, lp, r, d, b = _rollout(NET, T, N, 9)
    val = np.zeros((T, N), np.float32)   # unused by the fresh modes
    hp = oracle.Hyper(gamma=0.97, lam=0.9, lr=1e-2, seed=123, adv_mode=mode, rho_clip=1.1,
                      c_clip=0.9)
    res = oracle.update(NET, hp, T, N, E, M, obs, act, actc, lp, val, r, d, b, p)
    q = p.copy()
    m = np.zeros_like(q)
    v = np.zeros_like(q)
    ns = N // M
    step = 0
    for e in range(E):
        perm = oracle.perm(hp.seed, e, N)
        for k in range(M):
            _, g, st, *_ = oracle.loss_grad_fresh(
                NET, q, T, N, perm[k * ns:(k + 1) * ns], obs, act, actc, lp, r, d, b,
                vtrace=(mode == 2), gamma=hp.gamma, lam=hp.lam, rho_clip=hp.rho_clip,
                c_clip=hp.c_clip)
            np.testing.assert_allclose(res.stats[e * M + k], st, rtol=1e-12, atol=1e-12)
            _, g = oracle.clip_grad_norm(g, hp.max_grad_norm)
            step += 1
            q, m, v = oracle.adam(q, g, m, v, step, hp.lr)
    assert res.step == step
    np.testing.assert_allclose(res.params, q, rtol=1e-12, atol=1e-12)
    # a fresh update differs from the once-per-update route on the same data
    assert not np.allclose(res.params, p)
