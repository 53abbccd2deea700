"""One minibatch's loss and gradient through the C ABI vs the oracle.

"Teaching Mario to speedrun", sec. 6 (loss_pi, loss_V, entropy; backward).
Tolerances (normwise per parameter tensor, ||g - g_ref|| / ||g_ref||):
  fp32 mode (CUDA-core FFMA, fp32 accumulate)              1e-4
  bf16 mode (tcgen05 bf16 operands, fp32 accumulate)       2e-2
Loss statistics: |x - y| <= tol * max(|y|, mean |per-row term|) -- the
policy term is a mean of signed terms that cancel, so a purely relative test
is ill-posed there.
The clip decision is discontinuous, so the inputs keep every ratio well away
from 1 +- eps (tests/_gpu.py: LOG_RATIO_OFFSETS) -- both sides then take the
same branch on every row.  The ReLU derivative 1[pre > 0] is a decision too:
bf16-mode results are compared with the oracle's bf16-operand mode, which
rounds exactly the GEMM operands the bf16 path rounds, so pre-activations
agree to fp32 accumulation error and every unit takes the same branch.  For
tanh nets the bf16 path is also held to the plain fp64 oracle at 2e-2.
"""
import numpy as np
import pytest

import oracle
from policy_rl_gb300 import synth
from tests._gpu import (MODES, conditioned_logp_old, dev, fused_applies, host, mode_kwargs,
                        normwise, param_slices)

pytestmark = pytest.mark.gpu


def _inputs(w, seed=0):
    ro = synth.rollout(w, seed=seed)
    p0 = synth.init_params(w, seed=seed)
    ro.logp_old = conditioned_logp_old(w, ro, p0)
    adv, ret = oracle.gae(ro.rew, ro.val, ro.done, ro.boot, w.gamma, w.lam)
    adv = adv.ravel().astype(np.float32)
    ret = ret.ravel().astype(np.float32)
    return ro, p0, adv, ret


def _gpu_grad(w, ro, p0, adv, ret, idx, adv_stats=None, repeat=1, mode="per_stage"):
    import torch
    import policy_rl_gb300 as P
    cfg = P.config_from_workload(w, max_minibatch=max(len(idx), 1), **mode_kwargs(mode))
    ctx = P.Context(cfg, p0)
    st6 = torch.zeros(8, device="cuda")
    args = [dev(ro.obs), dev(ro.act_disc), dev(ro.act_cont), dev(ro.logp_old), dev(adv),
            dev(ret), dev(np.asarray(idx, np.int32))]
    stats_t = dev(np.asarray(adv_stats, np.float32)) if adv_stats is not None else None
    grads = []
    for _ in range(repeat):
        ctx.minibatch_loss_grad(*args, adv_stats=stats_t, stats6=st6)
        ctx.sync_status()
        grads.append(host(ctx.grad).copy())
    s6 = host(st6)[:6].copy()
    ctx.close()
    return grads, s6


def _oracle(w, ro, p0, adv, ret, idx, adv_stats=None, bf16_operands=None):
    net = oracle.Net(w.obs_dim, w.h1, w.h2, w.act, w.heads, w.n_gauss)
    if bf16_operands is None:
        bf16_operands = w.precision == "bf16"
    kw = dict(bf16_operands=bf16_operands)
    if adv_stats is not None:
        kw.update(normalize=True, adv_mean=float(adv_stats[0]), adv_std=float(adv_stats[1]))
    return oracle.loss_grad(net, p0.astype(np.float64), idx, ro.obs, ro.act_disc, ro.act_cont,
                            ro.logp_old, adv, ret, clip=w.clip, vf_coef=w.vf_coef,
                            ent_coef=w.ent_coef, **kw)


def _check(w, g, s6, ref, tol):
    _, gref, sref, scale = ref
    for name, sl in param_slices(w).items():
        if sl.stop == sl.start:
            continue
        e = normwise(g[sl], gref[sl])
        assert e <= tol, f"{name}: normwise error {e:.3e} > {tol}"
    for k in range(6):
        assert abs(s6[k] - sref[k]) <= tol * max(abs(sref[k]), scale[k]) + 1e-7, (k, s6, sref)


CASES = [
    # name, workload, rows of the minibatch, tolerance
    ("tiny_fp32", synth.WORKLOADS["tiny"], 2048, 1e-4),
    ("tiny_fp32_ragged", synth.WORKLOADS["tiny"], 1000, 1e-4),
    ("mario_bf16", synth.WORKLOADS["mario"].scaled(T=32, N=256), 4096, 2e-2),
    ("mario_bf16_ragged", synth.WORKLOADS["mario"].scaled(T=32, N=256), 1000, 2e-2),
    ("ddnet_bf16", synth.WORKLOADS["ddnet"].scaled(T=8, N=128), 512, 2e-2),
    ("large_bf16", synth.WORKLOADS["large"].scaled(T=8, N=512), 2048, 2e-2),
    ("mario_fp32", synth.WORKLOADS["mario"].scaled(T=8, N=256), 1024, 1e-4),
]


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("name,w,mb,tol", CASES, ids=[c[0] for c in CASES])
def test_minibatch_grad_matches_oracle(name, w, mb, tol, mode):
    """bf16 cases run every minibatch path: the fused forward/loss/backward-data
    kernel (where the network fits it), one kernel per GEMM stage, and the
    persistent minibatch kernel (fp32 mode has a single path)."""
    if name == "mario_fp32":
        import dataclasses
        w = dataclasses.replace(w, precision="fp32")
    if w.precision == "fp32" and mode != "per_stage":
        pytest.skip("fp32 mode has one path")
    if w.precision == "bf16" and mode == "fused" and not fused_applies(w):
        pytest.skip("the fused kernel does not take this network (per-stage path)")
    ro, p0, adv, ret = _inputs(w)
    idx = oracle.perm(5, 0, w.B)[:mb]
    (g,), s6 = _gpu_grad(w, ro, p0, adv, ret, idx, mode=mode)
    _check(w, g, s6, _oracle(w, ro, p0, adv, ret, idx), tol)


@pytest.mark.parametrize("wname,other", [("large", "persistent"), ("mario", "persistent"),
                                         ("mario", "fused"), ("large", "fused_loss"),
                                         ("mario", "fused_loss")])
def test_minibatch_paths_agree(wname, other):
    """Every path computes the same gradient up to fp32 summation order."""
    w = synth.WORKLOADS[wname].scaled(T=8, N=512)
    ro, p0, adv, ret = _inputs(w, seed=4)
    idx = oracle.perm(6, 0, w.B)[:4096]
    (g0,), s0 = _gpu_grad(w, ro, p0, adv, ret, idx, mode="per_stage")
    (g1,), s1 = _gpu_grad(w, ro, p0, adv, ret, idx, mode=other)
    for name, sl in param_slices(w).items():
        if sl.stop > sl.start:
            assert normwise(g0[sl], g1[sl]) < 1e-5, name
    np.testing.assert_allclose(s0, s1, rtol=1e-5, atol=1e-6)


@pytest.mark.parametrize("prec", ["fp32", "bf16"])
def test_normalised_advantages(prec):
    import dataclasses
    w = dataclasses.replace(synth.WORKLOADS["mario"].scaled(T=16, N=128), precision=prec)
    ro, p0, adv, ret = _inputs(w, seed=1)
    m, s = oracle.moments(adv.astype(np.float64))
    st = np.array([m, s], np.float32)
    idx = oracle.perm(9, 1, w.B)[:1024]
    (g,), s6 = _gpu_grad(w, ro, p0, adv, ret, idx, adv_stats=st)
    _check(w, g, s6, _oracle(w, ro, p0, adv, ret, idx, adv_stats=st),
           1e-4 if prec == "fp32" else 2e-2)


@pytest.mark.parametrize("wname", ["mario", "large"])
def test_bf16_close_to_fp64_definition(wname):
    w = synth.WORKLOADS[wname].scaled(T=16, N=256)
    ro, p0, adv, ret = _inputs(w, seed=3)
    idx = oracle.perm(2, 0, w.B)[:2048]
    (g,), s6 = _gpu_grad(w, ro, p0, adv, ret, idx)
    _check(w, g, s6, _oracle(w, ro, p0, adv, ret, idx, bf16_operands=False), 2e-2)


@pytest.mark.parametrize("mode", MODES)
def test_gradient_is_deterministic(mode):
    w = synth.WORKLOADS["mario"].scaled(T=32, N=256)
    ro, p0, adv, ret = _inputs(w)
    idx = oracle.perm(5, 0, w.B)[:4096]
    grads, _ = _gpu_grad(w, ro, p0, adv, ret, idx, repeat=3, mode=mode)
    assert np.array_equal(grads[0], grads[1]) and np.array_equal(grads[0], grads[2])


def test_ratio_one_first_epoch():
    """logp_old equal to the current policy's log-prob (r = 1): no sample is
    clipped and the policy gradient is the vanilla one."""
    import dataclasses
    w = dataclasses.replace(synth.WORKLOADS["tiny"].scaled(T=16, N=64), precision="fp32")
    ro, p0, adv, ret = _inputs(w, seed=2)
    net = oracle.Net(w.obs_dim, w.h1, w.h2, w.act, w.heads, w.n_gauss)
    z = oracle.forward(net, p0.astype(np.float64), ro.obs)
    from scipy.special import log_softmax
    lp = np.zeros(w.B)
    off = 0
    for h, n in enumerate(w.heads):
        lp += log_softmax(z[:, off:off + n], axis=1)[np.arange(w.B), ro.act_disc[:, h]]
        off += n
    ro.logp_old = lp.astype(np.float32)
    idx = np.arange(w.B, dtype=np.int32)
    (g,), s6 = _gpu_grad(w, ro, p0, adv, ret, idx)
    ref = _oracle(w, ro, p0, adv, ret, idx)
    _check(w, g, s6, ref, 1e-4)
    assert s6[4] == 0.0                     # clipfrac
    assert abs(s6[5]) < 1e-6                # approx_kl at r = 1
