"""Minibatch loss/gradient at the workloads' full minibatch sizes, in the launch
configuration the benchmark times.

- Mario-like: one full minibatch (32,768 rows of the T=128 x N=2048 rollout)
  against the oracle (bf16-operand mode), normwise 2e-2 per parameter tensor.
- Large batch: one full minibatch of 262,144 rows.  The oracle would take
  minutes here, so the check is a property that holds at any size: the loss
  is a mean over rows, so |S| g(S) is additive over a split of the rows,
  g(A u B) = (|A| g(A) + |B| g(B)) / (|A| + |B|), up to rounding.
  The oracle comparison of the same network runs at 2,048 rows in
  test_gpu_loss.py.
"""
import numpy as np
import pytest

import oracle
from policy_rl_gb300 import synth
from tests._gpu import LOG_RATIO_OFFSETS, dev, host, normwise, param_slices

pytestmark = pytest.mark.gpu


def _grad(ctx, ro, adv, ret, idx):
    import torch
    st6 = torch.zeros(8, device="cuda")
    ctx.minibatch_loss_grad(dev(ro.obs), dev(ro.act_disc), dev(ro.act_cont), dev(ro.logp_old),
                            dev(adv), dev(ret), dev(np.asarray(idx, np.int32)), stats6=st6)
    ctx.sync_status()
    return host(ctx.grad).copy(), host(st6)[:6].copy()


def test_mario_full_minibatch_matches_oracle():
    import policy_rl_gb300 as P
    w = synth.WORKLOADS["mario"]
    ro = synth.rollout(w, seed=7)
    p0 = synth.init_params(w, seed=7)
    mb = w.B // w.minibatches
    idx = oracle.perm(13, 0, w.B)[:mb]
    net = oracle.Net(w.obs_dim, w.h1, w.h2, w.act, w.heads, w.n_gauss)
    # logp_old of the minibatch rows: oracle log-probability minus the offsets
    lp, _ = oracle.policy_logp(net, p0.astype(np.float64), ro.obs[idx], ro.act_disc[idx],
                               ro.act_cont[idx])
    off = np.array(LOG_RATIO_OFFSETS)[np.arange(mb) % len(LOG_RATIO_OFFSETS)]
    ro.logp_old[idx] = (lp - off).astype(np.float32)
    adv, ret = oracle.gae(ro.rew, ro.val, ro.done, ro.boot, w.gamma, w.lam)
    adv = adv.ravel().astype(np.float32)
    ret = ret.ravel().astype(np.float32)
    ctx = P.Context(P.config_from_workload(w), p0)
    g, s6 = _grad(ctx, ro, adv, ret, idx)
    ctx.close()
    _, gref, sref, scale = oracle.loss_grad(net, p0.astype(np.float64), idx, ro.obs, ro.act_disc,
                                            ro.act_cont, ro.logp_old, adv, ret, clip=w.clip,
                                            vf_coef=w.vf_coef, ent_coef=w.ent_coef,
                                            bf16_operands=True)
    for name, sl in param_slices(w).items():
        if sl.stop > sl.start:
            e = normwise(g[sl], gref[sl])
            assert e <= 2e-2, f"{name}: normwise error {e:.3e}"
    for k in range(6):
        assert abs(s6[k] - sref[k]) <= 2e-2 * max(abs(sref[k]), scale[k]) + 1e-7, (k, s6, sref)


@pytest.mark.parametrize("na,tol", [(131_072, 1e-4), (100_003, 4e-3)])
def test_large_full_minibatch_is_additive_over_rows(na, tol):
    """Two splits of the 262,144 rows.  Halves: dz = dloss/dz / |S| differs
    between the runs by an exact factor of 2, so every bf16 rounding of dz, dP2
    and dP1 scales exactly and only the fp32 summation order differs (1e-4).
    Ragged split (100,003 rows, not a whole number of tiles): the 1/|S| scales
    are not powers of two, so the bf16 roundings of the backpropagated values
    differ by up to 2^-9 relative per element (4e-3)."""
    import policy_rl_gb300 as P
    w = synth.WORKLOADS["large"].scaled(T=4, N=65536, minibatches=1)   # 262,144 rows
    mb = w.B
    ro = synth.rollout(w, seed=3)
    p0 = synth.init_params(w, seed=3)
    rng = np.random.default_rng(0)
    adv = rng.standard_normal(mb).astype(np.float32)
    ret = rng.standard_normal(mb).astype(np.float32)
    idx = oracle.perm(21, 0, mb)
    ctx = P.Context(P.config_from_workload(w, max_minibatch=mb), p0)
    g_all, s_all = _grad(ctx, ro, adv, ret, idx)
    g_a, s_a = _grad(ctx, ro, adv, ret, idx[:na])
    g_b, s_b = _grad(ctx, ro, adv, ret, idx[na:])
    ctx.close()
    comb = (na * g_a.astype(np.float64) + (mb - na) * g_b.astype(np.float64)) / mb
    for name, sl in param_slices(w).items():
        if sl.stop > sl.start:
            e = normwise(g_all[sl], comb[sl])
            assert e <= tol, f"{name}: normwise error {e:.3e}"
    # the loss statistics are means over rows too (fp32 terms, no bf16 step)
    s_comb = (na * s_a.astype(np.float64) + (mb - na) * s_b.astype(np.float64)) / mb
    np.testing.assert_allclose(s_all, s_comb, rtol=1e-4, atol=1e-6)
    assert np.all(np.isfinite(g_all))
