"""Rollout-side policy step (ppo_policy_act) through the C ABI vs the oracle.

"Teaching Mario to speedrun", sec. 6 step 1 and sec. 7; sampling rule and
draw numbering as in ppo.h / the oracle.  Both sides draw the same mulberry32
uniforms (bit-exact), so the sampled category is unique except where u lies
within the logits' error of a category boundary; there the GPU's choice
must be one of the two categories that meet at that boundary.
- actions: equal to the oracle's, or within delta of a boundary (fp32 mode
  delta 1e-5, bf16 2e-2); at most 1 % of rows near a boundary;
- Gaussian actions within 1e-4 (fp32) / 3e-2 (bf16) of (1 + |a|);
- value elementwise 1e-5 / 2e-2 of (|y| + rms(y));
- log-probability against the oracle's at the GPU's own actions, same bars;
- counter property and determinism bit-exact; the empirical distribution of
  16,384 draws of one row matches the softmax (chi-square).
"""
import dataclasses

import numpy as np
import pytest
import scipy.special
import scipy.stats

import oracle
from policy_rl_gb300 import synth
from tests._gpu import assert_elementwise, dev, host

pytestmark = pytest.mark.gpu


def _net(w):
    return oracle.Net(w.obs_dim, w.h1, w.h2, w.act, w.heads, w.n_gauss)


def _gpu_act(ctx, w, obs, seed, draw0):
    import torch
    n = obs.shape[0]
    act = torch.empty(n, max(len(w.heads), 1), dtype=torch.int32, device="cuda")
    actc = torch.empty(n, max(w.n_gauss, 1), device="cuda")
    logp = torch.empty(n, device="cuda")
    val = torch.empty(n, device="cuda")
    ctx.policy_act(dev(obs), seed, draw0, act, actc if w.n_gauss else None, logp, val)
    ctx.sync_status()
    return (host(act)[:, :len(w.heads)], host(actc)[:, :w.n_gauss], host(logp), host(val))


def _check(w, obs, p0, got, seed, draw0):
    bf16 = w.precision == "bf16"
    net = _net(w)
    act, actc, logp, val = got
    ra, rc, rl, rv = oracle.policy_act(net, p0.astype(np.float64), obs, seed, draw0,
                                       bf16_operands=bf16)
    tol = 2e-2 if bf16 else 1e-5
    assert_elementwise(val, rv, tol)
    # categories: exact, or a boundary case within delta
    z = oracle.forward(net, p0.astype(np.float64), obs)
    K = len(w.heads) + 2 * w.n_gauss
    near = 0
    off = 0
    for h, nh in enumerate(w.heads):
        bad = np.flatnonzero(act[:, h] != ra[:, h])
        for i in bad:
            u = oracle.uniform24(oracle.mulberry32_at(seed, draw0 + i * K + h))
            cdf = np.cumsum(scipy.special.softmax(z[i, off:off + nh]))
            lo = min(act[i, h], ra[i, h])
            assert abs(act[i, h] - ra[i, h]) == 1 and abs(cdf[lo] - u) <= tol, \
                (i, h, act[i, h], ra[i, h], u, cdf)
        near += bad.size
        assert np.all((act[:, h] >= 0) & (act[:, h] < nh))
        off += nh
    assert near <= max(1, obs.shape[0] * len(w.heads) // 100), near
    if w.n_gauss:
        ctol = 3e-2 if bf16 else 1e-4
        assert np.all(np.abs(actc - rc) <= ctol * (1 + np.abs(rc))), np.max(np.abs(actc - rc))
    lp_ref, _ = oracle.policy_logp(net, p0.astype(np.float64), obs, act, actc.astype(np.float32))
    ltol = 2e-2 if bf16 else 1e-4
    assert np.all(np.abs(logp - lp_ref) <= ltol * (1 + np.abs(lp_ref))), \
        np.max(np.abs(logp - lp_ref))


CASES = [
    # workload, N agents
    ("tiny", 64),            # fp32, heads [3,2,2]
    ("tiny", 1),
    ("mario", 2048),         # one full Mario-like environment step, bf16
    ("mario", 1000),         # ragged: not a whole number of 128-row tiles
    ("ddnet", 1500),         # one full DDNet-like step: ReLU, D=1397, 2 Gaussian dims
]


@pytest.mark.parametrize("wname,N", CASES)
def test_policy_act_matches_oracle(wname, N):
    import policy_rl_gb300 as P
    w = synth.WORKLOADS[wname]
    ws = w.scaled(T=1, N=N, minibatches=1, epochs=1)
    ro = synth.rollout(ws, seed=4)
    p0 = synth.init_params(w, seed=4)
    ctx = P.Context(P.config_from_workload(ws, max_minibatch=N, max_batch=N), p0)
    seed, draw0 = 2024, 7 * N
    got = _gpu_act(ctx, w, ro.obs, seed, draw0)
    ctx.close()
    _check(w, ro.obs, p0, got, seed, draw0)


def test_policy_act_counter_and_determinism():
    import policy_rl_gb300 as P
    w = synth.WORKLOADS["mario"]
    ws = w.scaled(T=1, N=512, minibatches=1, epochs=1)
    ro = synth.rollout(ws, seed=5)
    ctx = P.Context(P.config_from_workload(ws, max_minibatch=512, max_batch=512),
                    synth.init_params(w, seed=5))
    K = len(w.heads) + 2 * w.n_gauss
    a = _gpu_act(ctx, w, ro.obs, 9, 0)
    b = _gpu_act(ctx, w, ro.obs, 9, 0)
    for x, y in zip(a, b):
        assert np.array_equal(x, y)
    # rows 100.. at counter 100 K are the same agents as rows 100.. at counter 0
    c = _gpu_act(ctx, w, np.ascontiguousarray(ro.obs[100:]), 9, 100 * K)
    assert np.array_equal(c[0], a[0][100:])
    assert np.array_equal(c[3], a[3][100:])
    d = _gpu_act(ctx, w, ro.obs, 10, 0)
    assert not np.array_equal(d[0], a[0])
    ctx.close()


def test_policy_act_empirical_distribution():
    import policy_rl_gb300 as P
    w = dataclasses.replace(synth.WORKLOADS["ddnet"], obs_dim=64)   # bf16, 2 Gaussian dims
    reps = 16384
    ws = w.scaled(T=1, N=reps, minibatches=1, epochs=1)
    p0 = synth.init_params(w, seed=6)
    rng = np.random.default_rng(6)
    obs = np.repeat(rng.normal(size=(1, w.obs_dim)).astype(np.float32), reps, axis=0)
    ctx = P.Context(P.config_from_workload(ws, max_minibatch=reps, max_batch=reps), p0)
    act, actc, logp, val = _gpu_act(ctx, w, obs, 77, 0)
    ctx.close()
    assert np.all(val == val[0]) and np.all(np.isfinite(logp))
    z = oracle.forward(_net(w), p0.astype(np.float64), obs[:1])[0]
    off = 0
    for h, nh in enumerate(w.heads):
        prob = scipy.special.softmax(z[off:off + nh])
        counts = np.bincount(act[:, h], minlength=nh)
        assert scipy.stats.chisquare(counts, prob * reps).pvalue > 1e-4, (h, counts, prob)
        off += nh
    logstd = p0[-w.n_gauss:]
    for g in range(w.n_gauss):
        mu, sd = z[off + g], np.exp(logstd[g])
        assert abs(actc[:, g].mean() - mu) < 5 * sd / np.sqrt(reps) + 2e-2 * (1 + abs(mu))
        assert abs(actc[:, g].std() / sd - 1) < 0.03


def test_policy_act_argument_errors():
    import torch
    import policy_rl_gb300 as P
    w = synth.WORKLOADS["tiny"]
    ctx = P.Context(P.config_from_workload(w.scaled(T=1, N=64, minibatches=1, epochs=1),
                                           max_minibatch=64, max_batch=64), synth.init_params(w))
    obs = torch.zeros(65, w.obs_dim, device="cuda")
    act = torch.zeros(65, 3, dtype=torch.int32, device="cuda")
    with pytest.raises(P.PpoError) as ei:
        ctx.policy_act(obs, 0, 0, act)          # N > max_minibatch
    assert ei.value.status == 1
    with pytest.raises(P.PpoError) as ei:
        ctx.policy_act(obs[:8], 0, 0, None)     # no action buffer for the discrete heads
    assert ei.value.status == 1
    ctx.close()
    cfg = P.make_config(8, 16, 640, heads=(2,), precision=0, max_batch=8, max_minibatch=8)
    ctx = P.Context(cfg)
    with pytest.raises(P.PpoError) as ei:
        ctx.policy_act(torch.zeros(8, 8, device="cuda"), 0, 0,
                       torch.zeros(8, 1, dtype=torch.int32, device="cuda"))
    assert ei.value.status == 4                 # hidden width above 512
    ctx.close()
