"""Failure detection on the GPU without a GPU fault.

- A bounded device wait that runs out: the cooperative kernels' grid
  barriers (gradient assembly + Adam inside the fp32 update, the
  fresh-advantage kernel) wait at most the context's wait limit.  The test sets that limit
  to 1 ns, so the first block to arrive gives up before the others come in;
  the kernel latches PPO_ERR_TIMEOUT and returns (these kernels hold no
  asynchronous copies or tensor memory, so nothing is left in flight).  The
  next ppo_sync_status must report it once, and the context must stay
  usable: with the default limit restored the next update runs clean and a
  minibatch gradient at the context's current weights matches the oracle.
- A device allocation that fails: a context whose epoch buffers would need
  terabytes returns PPO_ERR_NOMEM from ppo_create and leaves nothing behind.
"""
import numpy as np
import pytest

import oracle
from policy_rl_gb300 import synth
from tests._gpu import conditioned_logp_old, dev, host, normwise

pytestmark = pytest.mark.gpu


def _rollout(w):
    ro = synth.rollout(w, seed=4)
    args = [dev(x) for x in (ro.obs, ro.act_disc, ro.act_cont, ro.logp_old, ro.val, ro.rew,
                             ro.done, ro.boot)]
    return ro, args


@pytest.mark.parametrize("prec,adv_mode", [("fp32", 0), ("bf16", 1)])
def test_grid_barrier_timeout_is_latched_and_context_recovers(prec, adv_mode):
    """fp32 mode, advantages once per update: the grid barrier of the
    cooperative gradient-assembly + Adam kernel.  bf16 mode, fresh
    advantages: the fresh-advantage kernel's grid barriers (and the
    weight-gradient kernel's per-tile waits)."""
    import dataclasses
    import policy_rl_gb300 as P
    w = dataclasses.replace(synth.WORKLOADS["mario"].scaled(T=16, N=256, epochs=1,
                                                            minibatches=4), precision=prec)
    ro, args = _rollout(w)
    p0 = synth.init_params(w, seed=4)
    ctx = P.Context(P.config_from_workload(w, adv_mode=adv_mode), p0)
    hp = (w.epochs, w.minibatches, w.gamma, w.lam, w.lr, 5)
    ctx.update(*args, *hp)
    ctx.sync_status()                         # clean with the default limit
    ctx.set_wait_limit(1)                     # 1 ns: the barrier waits run out
    ctx.update(*args, *hp)
    with pytest.raises(P.PpoError) as ei:
        ctx.sync_status()
    assert ei.value.status == 5, ei.value     # PPO_ERR_TIMEOUT
    ctx.sync_status()                         # reported once, then cleared
    ctx.set_wait_limit(0)                     # back to the default
    ctx.update(*args, *hp)
    ctx.sync_status()
    p = host(ctx.params).astype(np.float64)
    assert np.all(np.isfinite(p))
    # the context still computes correct gradients at its current weights
    # (old log-probabilities conditioned at those weights, so that no ratio
    # lies near a clip boundary)
    import torch
    mb = 1024
    idx = oracle.perm(9, 0, w.B)[:mb]
    rng = np.random.default_rng(1)
    adv = rng.standard_normal(w.B).astype(np.float32)
    ret = rng.standard_normal(w.B).astype(np.float32)
    ro.logp_old = conditioned_logp_old(w, ro, p)
    ctx.minibatch_loss_grad(args[0], args[1], args[2], dev(ro.logp_old), dev(adv), dev(ret),
                            dev(idx.astype(np.int32)), stats6=torch.zeros(8, device="cuda"))
    ctx.sync_status()
    g = host(ctx.grad).copy()
    ctx.close()
    net = oracle.Net(w.obs_dim, w.h1, w.h2, w.act, w.heads, w.n_gauss)
    _, gref, _, _ = oracle.loss_grad(net, p, idx, ro.obs, ro.act_disc, ro.act_cont, ro.logp_old,
                                     adv, ret, clip=w.clip, vf_coef=w.vf_coef,
                                     ent_coef=w.ent_coef, bf16_operands=prec == "bf16")
    assert normwise(g, gref) <= (2e-2 if prec == "bf16" else 1e-4)


def test_create_reports_nomem_for_an_impossible_context():
    import policy_rl_gb300 as P
    w = synth.WORKLOADS["ddnet"]
    # epoch buffers of (2^31 - 1) rows x 1408 bf16 features: about 6 TB
    cfg = P.config_from_workload(w, max_batch=(1 << 31) - 1, max_minibatch=1024)
    with pytest.raises(P.PpoError) as ei:
        P.Context(cfg)
    assert ei.value.status == 6, ei.value     # PPO_ERR_NOMEM
    # the device is still usable
    ctx = P.Context(P.config_from_workload(synth.WORKLOADS["tiny"]))
    ctx.sync_status()
    ctx.close()
