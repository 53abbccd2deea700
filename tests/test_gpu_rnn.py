"""Recurrent (MinGRU) policy loss and gradient (ppo_rnn_loss_grad) vs the oracle.

"Teaching Mario to speedrun", sec. 8 (bias-free encoder, MinGRU layers with
episode resets, decoder); MinGRU per Feng et al. 2024.
- precision 0 (fp32 CUDA-core kernels) against the fp64 oracle: gradient
  normwise per parameter tensor within 1e-4, loss statistics within 1e-4 of
  max(|y|, mean |term|);
- precision 1 (bf16 tensor-core products) against the oracle's bf16-operand
  mode (the same operands rounded, fp64 sums): 2e-2 on the same measures;
  tanh-free gates make no integer decision, so the pages' shape is also held
  to the plain fp64 oracle at 2e-2;
- cases: a tiny net with a Gaussian dim, the pages' shape (encoder to 128,
  four layers) on a Mario-like head layout, terminals inside segments, a
  carried-in state, normalised advantages, the clipped branch, hidden 256
  with Gaussian dims and a ragged row count, and in bf16 the full Mario-like
  recurrent minibatch (256 segments x T=128 = 32,768 rows).
"""
import math

import numpy as np
import pytest

import oracle
from tests._gpu import dev, host, normwise

pytestmark = pytest.mark.gpu


def _regions(rnn):
    D, H, L, C, G = rnn.obs_dim, rnn.hidden, rnn.layers, rnn.out_cols, rnn.n_gauss
    out, o = {"W_enc": slice(0, H * D)}, H * D
    for l in range(L):
        for name, n in (("W_z", H * H), ("b_z", H), ("W_h", H * H), ("b_h", H)):
            out[f"{name}{l}"] = slice(o, o + n)
            o += n
    out["W_dec"] = slice(o, o + C * H)
    o += C * H
    out["logstd"] = slice(o, o + G)
    return out


def _data(rnn, T, N, seed, wscale=0.5, clip_safe=False):
    rng = np.random.default_rng(seed)
    p = rng.normal(0, wscale, rnn.num_params)
    B = T * N
    obs = rng.normal(size=(B, rnn.obs_dim)).astype(np.float32)
    act = np.stack([rng.integers(0, n, B) for n in rnn.heads], 1).astype(np.int32)
    actc = rng.normal(size=(B, max(rnn.n_gauss, 1))).astype(np.float32)[:, :rnn.n_gauss]
    if clip_safe:
        # near-uniform heads (small weights): logp ~ -sum ln n_h; offsets keep every
        # ratio >= 0.03 in log space from the clip boundaries log(0.8), log(1.2)
        off = np.array([-0.5, -0.1, 0.0, 0.1, 0.5])[np.arange(B) % 5]
        lp = (-sum(math.log(n) for n in rnn.heads) - off).astype(np.float32)
    else:
        lp = rng.normal(-2.0, 0.3, B).astype(np.float32)
    adv = rng.normal(size=B).astype(np.float32)
    ret = rng.normal(size=B).astype(np.float32)
    done = (rng.random((T, N)) < 0.1).astype(np.float32)
    h0 = rng.normal(0, 0.5, size=(N, rnn.layers, rnn.hidden)).astype(np.float32)
    return p, obs, act, actc, lp, adv, ret, done, h0


CASES = [
    # name, rnn, T, N, ns, clip, normalise, wscale
    ("tiny_gauss", oracle.Rnn(obs_dim=3, hidden=4, layers=2, heads=(3, 2), n_gauss=1),
     6, 3, 2, 10.0, False, 0.5),
    ("pages_shape", oracle.Rnn(obs_dim=32, hidden=128, layers=4, heads=(9, 2, 2, 2)),
     32, 64, 16, 10.0, True, 0.1),
    ("two_gauss", oracle.Rnn(obs_dim=10, hidden=64, layers=4, heads=(3, 2, 2), n_gauss=2),
     20, 10, 5, 10.0, False, 0.2),
    ("clipped", oracle.Rnn(obs_dim=8, hidden=32, layers=3, heads=(4, 3)),
     16, 12, 6, 0.2, True, 0.02),
]


@pytest.mark.parametrize("name,rnn,T,N,ns,clip,norm,wscale", CASES, ids=[c[0] for c in CASES])
def test_rnn_loss_grad_matches_oracle(name, rnn, T, N, ns, clip, norm, wscale):
    import torch
    import policy_rl_gb300 as P
    p, obs, act, actc, lp, adv, ret, done, h0 = _data(rnn, T, N, 3, wscale, clip_safe=clip < 1)
    envs = np.random.default_rng(4).permutation(N)[:ns].astype(np.int32)
    cfg = P.make_rnn_config(rnn.obs_dim, rnn.hidden, rnn.layers, rnn.heads, rnn.n_gauss,
                            clip=clip)
    assert P.ppo_rnn_param_count(cfg) == rnn.num_params
    rows = oracle.segment_rows(T, N, envs)
    mean, sd = (float(adv[rows].mean()), float(adv[rows].std())) if norm else (0.0, 1.0)
    stats_in = dev(np.array([mean, sd, 0, 0], np.float32)) if norm else None
    grad = torch.empty(rnn.num_params, device="cuda")
    st6 = torch.zeros(8, device="cuda")
    work = torch.empty(P.ppo_rnn_workspace_bytes(cfg, T, ns), dtype=torch.uint8, device="cuda")
    P.ppo_rnn_loss_grad(cfg, dev(p.astype(np.float32)), dev(envs), dev(obs), dev(act),
                        dev(actc) if rnn.n_gauss else None, dev(lp), dev(adv), dev(ret),
                        dev(done), dev(h0), grad, adv_stats=stats_in, stats6=st6, work=work)
    torch.cuda.synchronize()
    g = host(grad).astype(np.float64)
    s6 = host(st6)[:6]
    _, gref, sref, scale = oracle.rnn_loss_grad(
        rnn, p.astype(np.float32).astype(np.float64), envs, obs, act,
        actc if rnn.n_gauss else None, lp, adv.astype(np.float64), ret.astype(np.float64), done,
        h0.astype(np.float64), clip=clip, normalize=norm, adv_mean=float(np.float32(mean)),
        adv_std=float(np.float32(sd)))
    for nm, sl in _regions(rnn).items():
        if sl.stop > sl.start:
            e = normwise(g[sl], gref[sl])
            assert e <= 1e-4, f"{nm}: normwise error {e:.3e}"
    for k in range(6):
        assert abs(s6[k] - sref[k]) <= 1e-4 * max(abs(sref[k]), scale[k]) + 1e-7, (k, s6, sref)


def test_rnn_loss_grad_is_deterministic():
    import torch
    import policy_rl_gb300 as P
    rnn = oracle.Rnn(obs_dim=16, hidden=64, layers=4, heads=(3, 2))
    T, N, ns = 24, 8, 4
    p, obs, act, actc, lp, adv, ret, done, h0 = _data(rnn, T, N, 5, 0.2)
    cfg = P.make_rnn_config(16, 64, 4, (3, 2))
    envs = dev(np.arange(ns, dtype=np.int32))
    work = torch.empty(P.ppo_rnn_workspace_bytes(cfg, T, ns), dtype=torch.uint8, device="cuda")
    outs = []
    for _ in range(2):
        grad = torch.empty(rnn.num_params, device="cuda")
        P.ppo_rnn_loss_grad(cfg, dev(p.astype(np.float32)), envs, dev(obs), dev(act), None,
                            dev(lp), dev(adv), dev(ret), dev(done), dev(h0), grad, work=work)
        torch.cuda.synchronize()
        outs.append(host(grad).copy())
    assert np.array_equal(outs[0], outs[1])


BF16_CASES = [
    # name, rnn, T, N, ns, clip, normalise, wscale
    ("pages_bf16", oracle.Rnn(obs_dim=64, hidden=128, layers=4, heads=(9, 2, 2, 2)),
     32, 64, 16, 10.0, True, 0.1),
    ("h256_gauss_ragged", oracle.Rnn(obs_dim=20, hidden=256, layers=2, heads=(3, 2, 2),
                                     n_gauss=2), 37, 12, 5, 10.0, False, 0.08),
    ("clipped_bf16", oracle.Rnn(obs_dim=8, hidden=128, layers=3, heads=(4, 3)),
     16, 24, 12, 0.2, True, 0.02),
    ("mario_full_bf16", oracle.Rnn(obs_dim=64, hidden=128, layers=4, heads=(9, 2, 2, 2)),
     128, 2048, 256, 10.0, True, 0.1),
]


def _run_gpu(rnn, cfg, p, envs, obs, act, actc, lp, adv, ret, done, h0, stats_in):
    import torch
    import policy_rl_gb300 as P
    T, N = done.shape
    ns = envs.size
    grad = torch.empty(rnn.num_params, device="cuda")
    st6 = torch.zeros(8, device="cuda")
    work = torch.empty(P.ppo_rnn_workspace_bytes(cfg, T, ns), dtype=torch.uint8, device="cuda")
    P.ppo_rnn_loss_grad(cfg, dev(p.astype(np.float32)), dev(envs), dev(obs), dev(act),
                        dev(actc) if rnn.n_gauss else None, dev(lp), dev(adv), dev(ret),
                        dev(done), dev(h0), grad, adv_stats=stats_in, stats6=st6, work=work)
    torch.cuda.synchronize()
    assert int(work[:4].view(torch.int32).item()) == 0   # no bounded wait gave up
    return host(grad).astype(np.float64), host(st6)[:6].copy()


@pytest.mark.parametrize("name,rnn,T,N,ns,clip,norm,wscale", BF16_CASES,
                         ids=[c[0] for c in BF16_CASES])
def test_rnn_loss_grad_bf16_matches_oracle(name, rnn, T, N, ns, clip, norm, wscale):
    import policy_rl_gb300 as P
    p, obs, act, actc, lp, adv, ret, done, h0 = _data(rnn, T, N, 7, wscale, clip_safe=clip < 1)
    envs = np.random.default_rng(8).permutation(N)[:ns].astype(np.int32)
    cfg = P.make_rnn_config(rnn.obs_dim, rnn.hidden, rnn.layers, rnn.heads, rnn.n_gauss,
                            clip=clip, precision=1)
    rows = oracle.segment_rows(T, N, envs)
    mean, sd = (float(adv[rows].mean()), float(adv[rows].std())) if norm else (0.0, 1.0)
    stats_in = dev(np.array([mean, sd, 0, 0], np.float32)) if norm else None
    g, s6 = _run_gpu(rnn, cfg, p, envs, obs, act, actc, lp, adv, ret, done, h0, stats_in)
    refs = [True] + ([False] if name == "pages_bf16" else [])
    for bf in refs:
        _, gref, sref, scale = oracle.rnn_loss_grad(
            rnn, p.astype(np.float32).astype(np.float64), envs, obs, act,
            actc if rnn.n_gauss else None, lp, adv.astype(np.float64), ret.astype(np.float64),
            done, h0.astype(np.float64), clip=clip, normalize=norm,
            adv_mean=float(np.float32(mean)), adv_std=float(np.float32(sd)), bf16_operands=bf)
        for nm, sl in _regions(rnn).items():
            if sl.stop > sl.start:
                e = normwise(g[sl], gref[sl])
                assert e <= 2e-2, f"{nm} vs {'bf16-operand' if bf else 'fp64'} oracle: {e:.3e}"
        for k in range(6):
            assert abs(s6[k] - sref[k]) <= 2e-2 * max(abs(sref[k]), scale[k]) + 1e-7, \
                (k, s6, sref)


def test_rnn_loss_grad_bf16_is_deterministic():
    import policy_rl_gb300 as P
    rnn = oracle.Rnn(obs_dim=16, hidden=128, layers=2, heads=(3, 2))
    T, N, ns = 24, 40, 20
    p, obs, act, actc, lp, adv, ret, done, h0 = _data(rnn, T, N, 5, 0.1)
    cfg = P.make_rnn_config(16, 128, 2, (3, 2), precision=1)
    envs = np.arange(ns, dtype=np.int32)
    a = _run_gpu(rnn, cfg, p, envs, obs, act, actc, lp, adv, ret, done, h0, None)
    b = _run_gpu(rnn, cfg, p, envs, obs, act, actc, lp, adv, ret, done, h0, None)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


# ---- the recurrent update (ppo_rnn_update) ---------------------------------------
def _rollout(rnn, T, N, seed, wscale):
    p, obs, act, actc, lp, adv, ret, done, h0 = _data(rnn, T, N, seed, wscale, clip_safe=True)
    rng = np.random.default_rng(seed + 1)
    val = rng.normal(size=(T, N)).astype(np.float32)
    rew = np.where(rng.random((T, N)) < 0.9, 0.0, rng.random((T, N))).astype(np.float32)
    boot = rng.normal(size=N).astype(np.float32)
    return p, obs, act, actc, lp, val, rew, done, boot, h0


@pytest.mark.parametrize("prec", [0, 1])
def test_rnn_update_matches_oracle(prec):
    """One update (GAE, global statistics, env permutations, BPTT minibatches,
    clip, Adam).  The first step's gradient is compared directly (the
    update's gradient buffer after a one-step update, 1e-4 fp32 / 2e-2 bf16
    against the fp64 / bf16-operand oracle); the whole trajectory of 2 x 4
    steps by its parameter change (1e-3 fp32, as the MLP update tests; 0.1
    in bf16, two independent trajectories) and every step's statistics."""
    import torch
    import policy_rl_gb300 as P
    H = 32 if prec == 0 else 128
    rnn = oracle.Rnn(obs_dim=24, hidden=H, layers=3, heads=(9, 2, 2), n_gauss=1)
    T, N, E, M = 16, 32, 2, 4
    p, obs, act, actc, lp, val, rew, done, boot, h0 = _rollout(rnn, T, N, 11, 0.1)
    p32 = p.astype(np.float32)
    cfg = P.make_rnn_config(rnn.obs_dim, H, rnn.layers, rnn.heads, rnn.n_gauss,
                            precision=prec)
    hp = oracle.Hyper(gamma=0.99, lam=0.95, clip=0.2, vf_coef=0.5, ent_coef=0.01, lr=2.5e-4,
                      max_grad_norm=0.5, seed=31, bf16_operands=prec == 1)
    args = [dev(obs), dev(act), dev(actc), dev(lp), dev(val), dev(rew), dev(done), dev(boot),
            dev(h0)]
    # one step: the gradient of minibatch 0 of epoch 0 at the initial weights
    ctx = P.RnnContext(cfg, p32, max_T=T, max_N=N, max_epochs=E)
    ctx.update(*args, 1, 1, hp.gamma, hp.lam, hp.lr, hp.seed)
    ctx.sync_status()
    g = host(ctx.grad).astype(np.float64)
    ctx.close()
    adv, ret = oracle.gae(rew, val, done, boot, hp.gamma, hp.lam)
    mean, sd = oracle.moments(adv)
    envs = oracle.perm(hp.seed, 0, N)
    _, gref, _, _ = oracle.rnn_loss_grad(rnn, p32.astype(np.float64), envs, obs, act, actc, lp,
                                         adv.ravel(), ret.ravel(), done, h0.astype(np.float64),
                                         normalize=True, adv_mean=mean, adv_std=sd,
                                         bf16_operands=prec == 1)
    tol = 1e-4 if prec == 0 else 2e-2
    for nm, sl in _regions(rnn).items():
        e = normwise(g[sl], gref[sl])
        assert e <= tol, f"{nm}: {e:.3e}"
    # the whole update
    ctx = P.RnnContext(cfg, p32, max_T=T, max_N=N, max_epochs=E)
    st = torch.zeros(E * M, 6, device="cuda")
    ctx.update(*args, E, M, hp.gamma, hp.lam, hp.lr, hp.seed, stats=st)
    ctx.sync_status()
    pg = host(ctx.params).astype(np.float64)
    sg = host(st)
    ctx.close()
    p_ref, _, _, step, s_ref = oracle.rnn_update(rnn, hp, T, N, E, M, obs, act, actc, lp, val,
                                                 rew, done, boot, h0.astype(np.float64), p32)
    assert step == E * M
    p0 = p32.astype(np.float64)
    e = normwise(pg - p0, p_ref - p0)
    assert e <= (1e-3 if prec == 0 else 0.1), e
    np.testing.assert_allclose(sg[:, 2:4], s_ref[:, 2:4], rtol=1e-3 if prec == 0 else 2e-2)
