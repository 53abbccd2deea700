"""The whole update (ppo_update), checked step by step against the oracle.

"Teaching Mario to speedrun", sec. 6 "The whole algorithm": GAE, the batch's
advantage statistics, then per epoch a shuffle and per minibatch one backward
pass and one optimizer step.  Two trajectories drift apart (every step feeds
its rounding into the next one), so each step is compared from the GPU's own
state: the update runs with a step trace (ppo_set_step_trace) that copies the
parameters and Adam's m, v before every minibatch step and the assembled
gradient after it.  For step j the oracle then takes the GPU's pre-step
parameters and computes, from its own GAE, statistics and permutation:

- the minibatch gradient, normwise per parameter tensor: 2e-2 in bf16 mode
  (against the oracle's bf16-operand mode at every step; tanh nets also
  against plain fp64 at step 0, where the conditioned old log-probabilities
  keep every ratio away from the clip boundaries) and 1e-4 in fp32 mode;
- the loss statistics of the step (as in the minibatch tests);
- the optimizer: clip + Adam applied by the oracle to the GPU's pre-step
  state and the GPU's gradient gives the GPU's parameter change within 1e-4
  normwise (fp32 parameters round each update at about 2e-5 of the change);
- the parameter change with the oracle's own gradient, from the second step
  on, within the gradient bar.  At Adam's first step the change is
  lr * g / (|g| + eps), lr * sign(g) per element, so a gradient entry near
  zero may flip its sign between the two sides; there the change is not
  a continuous function of the gradient and only the gradient is compared.

Workloads: the Mario-like update at its full size (T=128 x N=2048, 4 epochs x
8 minibatches of 32,768 rows); the large-batch network with full 262,144-row
minibatches (T=4 x N=65536, 2 epochs x 1); the DDNet-like network (ReLU,
1397-d observations, discrete + Gaussian heads) with full 48,000-row
minibatches (T=256 x N=375, 1 epoch x 2); the tiny workload in fp32 mode.
"""
import numpy as np
import pytest

import oracle
from policy_rl_gb300 import synth
from tests._gpu import conditioned_logp_old, dev, host, normwise, param_slices

pytestmark = pytest.mark.gpu

SEED = 29


def _net(w):
    return oracle.Net(w.obs_dim, w.h1, w.h2, w.act, w.heads, w.n_gauss)


def _traced_update(w, seed):
    """Runs ppo_update once with a step trace; returns the rollout, the
    initial parameters, the trace [S][4][P], the final parameters and the
    per-step statistics."""
    import torch
    import policy_rl_gb300 as P
    ro = synth.rollout(w, seed=seed)
    p0 = synth.init_params(w, seed=seed)
    ro.logp_old = conditioned_logp_old(w, ro, p0)
    ctx = P.Context(P.config_from_workload(w), p0)
    S, Pn = w.epochs * w.minibatches, ctx.n_params
    trace = torch.zeros(S * 4 * Pn, device="cuda")
    ctx.set_step_trace(trace, S)
    st = torch.zeros(S, 6, device="cuda")
    ctx.update(dev(ro.obs), dev(ro.act_disc), dev(ro.act_cont), dev(ro.logp_old), dev(ro.val),
               dev(ro.rew), dev(ro.done), dev(ro.boot), w.epochs, w.minibatches, w.gamma,
               w.lam, w.lr, SEED, stats=st)
    ctx.sync_status()
    assert ctx.step() == S
    tr = host(trace).reshape(S, 4, Pn).copy()
    final = host(ctx.params).copy()
    stats = host(st).copy()
    ctx.set_step_trace(None, 0)
    ctx.close()
    return ro, p0, tr, final, stats


def _check_update(w, steps, fp64_step0, grad_tol, dp_tol=None):
    dp_tol = grad_tol if dp_tol is None else dp_tol
    ro, p0, tr, final, stats = _traced_update(w, SEED)
    assert np.array_equal(tr[0, 0], p0.astype(np.float32)), "trace step 0 != initial params"
    net = _net(w)
    bf16 = w.precision == "bf16"
    B, M = w.B, w.minibatches
    mb = B // M
    adv, ret = oracle.gae(ro.rew, ro.val, ro.done, ro.boot, w.gamma, w.lam)
    adv, ret = adv.ravel(), ret.ravel()
    mean, std = oracle.moments(adv)
    S = w.epochs * M
    sl = {k: v for k, v in param_slices(w).items() if v.stop > v.start}
    for j in steps:
        e, k = divmod(j, M)
        idx = oracle.perm(SEED, e, B)[k * mb:(k + 1) * mb]
        p_j, m_j, v_j, g_gpu = (tr[j, i].astype(np.float64) for i in range(4))
        p_next = (tr[j + 1, 0] if j + 1 < S else final).astype(np.float64)
        refs = [("bf16-operand" if bf16 else "fp64", bf16)]
        if j == 0 and fp64_step0 and bf16:
            refs.append(("fp64", False))
        for label, bf in refs:
            _, g_ref, s_ref, scale = oracle.loss_grad(
                net, p_j, idx, ro.obs, ro.act_disc, ro.act_cont, ro.logp_old, adv, ret,
                clip=w.clip, vf_coef=w.vf_coef, ent_coef=w.ent_coef, normalize=True,
                adv_mean=mean, adv_std=std, bf16_operands=bf)
            for name, s in sl.items():
                err = normwise(g_gpu[s], g_ref[s])
                assert err <= grad_tol, f"step {j} {name} vs {label} oracle: {err:.3e}"
            for q in range(6):
                assert abs(stats[j, q] - s_ref[q]) <= grad_tol * max(abs(s_ref[q]), scale[q]) \
                    + 1e-7, (j, q, stats[j], s_ref)
        # the optimizer step on the GPU's own state and gradient
        _, gc = oracle.clip_grad_norm(g_gpu, w.max_grad_norm)
        p_o, _, _ = oracle.adam(p_j, gc, m_j, v_j, j + 1, w.lr)
        err = normwise(p_next - p_j, p_o - p_j)
        assert err <= 1e-4, f"step {j}: Adam on the GPU's gradient differs: {err:.3e}"
        # the whole step with the oracle's gradient (from Adam's second step on)
        if j >= 1:
            _, gc = oracle.clip_grad_norm(g_ref, w.max_grad_norm)
            p_o, _, _ = oracle.adam(p_j, gc, m_j, v_j, j + 1, w.lr)
            err = normwise(p_next - p_j, p_o - p_j)
            assert err <= dp_tol, f"step {j}: parameter change differs: {err:.3e}"


def test_mario_full_update_stepwise():
    """Every one of the 32 steps of the full Mario-like update (T=128 x N=2048,
    4 x 8 minibatches of 32,768 rows, bf16)."""
    w = synth.WORKLOADS["mario"]
    _check_update(w, range(w.epochs * w.minibatches), fp64_step0=True, grad_tol=2e-2)


def test_large_batch_update_stepwise():
    """The large-batch network (128-512-512 tanh) with full 262,144-row
    minibatches: T=4 x N=65536, 2 epochs x 1 minibatch, both steps."""
    w = synth.WORKLOADS["large"].scaled(T=4, N=65536, epochs=2, minibatches=1)
    _check_update(w, range(2), fp64_step0=True, grad_tol=2e-2)


def test_ddnet_update_stepwise():
    """The DDNet-like network (1397-512-512 ReLU, heads [3,2,2] + 2 Gaussian
    dims with a learned log-std) with full 48,000-row minibatches: T=256 x
    N=375, 1 epoch x 2 minibatches, both steps.  ReLU' is a decision taken on
    rounded values, so the reference is the bf16-operand oracle (the rounded
    operands the tensor cores read)."""
    w = synth.WORKLOADS["ddnet"].scaled(T=256, N=375, epochs=1, minibatches=2)
    _check_update(w, range(2), fp64_step0=False, grad_tol=2e-2)


def test_tiny_update_stepwise_fp32():
    """The tiny workload in fp32 mode (CUDA-core FFMA GEMMs): 4 steps at 1e-4."""
    w = synth.WORKLOADS["tiny"]
    _check_update(w, range(w.epochs * w.minibatches), fp64_step0=False, grad_tol=1e-4,
                  dp_tol=1e-3)
