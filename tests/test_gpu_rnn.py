"""Recurrent (MinGRU) policy loss and gradient (ppo_rnn_loss_grad) vs the oracle.

"Teaching Mario to speedrun", sec. 8 (bias-free encoder, MinGRU layers with
episode resets, decoder); MinGRU per Feng et al. 2024.  fp32 CUDA-core
kernels against the fp64 oracle (backpropagation through time):
- gradient normwise per parameter tensor within 1e-4;
- loss statistics within 1e-4 of max(|y|, mean |term|);
- cases: a tiny net with a Gaussian dim, the pages' shape (encoder to 128,
  four layers) on a Mario-like head layout, terminals inside segments, a
  carried-in state, normalised advantages, and the clipped branch.
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
