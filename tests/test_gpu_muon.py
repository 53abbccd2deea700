"""Muon optimizer step (ppo_muon_step) and the update with optimizer 1, vs the oracle.

"Teaching Mario to speedrun", sec. 8 and "puff-rs" (Muon, five Newton-Schulz
iterations per weight matrix); definition from Muon's published write-up.
- one to three steps on identical gradients: the parameter change of the
  weight matrices normwise within 1e-4 of the fp64 oracle in fp32 contexts
  (fp32 CUDA-core products; the quintic iteration amplifies rounding by at
  most a^5 ~ 480 on the smallest singular directions), and within 2e-2 of
  the oracle's bf16 Newton-Schulz in bf16 contexts (tensor-core products
  with X, A, B stored as bf16, as in the write-up); momentum buffers within
  1e-6, Adam on the biases / log-std as in test_gpu_update (1e-6), gradient
  norm 1e-5;
- shapes: wide, tall (transposed) and square matrices up to 512 x 1397;
- whole update with Muon: parameter change against the oracle's trajectory
  (fp32 1e-3, bf16 0.1 as for Adam), bit-identical replays.
"""
import dataclasses

import numpy as np
import pytest

import oracle
from policy_rl_gb300 import synth
from tests._gpu import conditioned_logp_old, dev, host, normwise, param_slices

pytestmark = pytest.mark.gpu


def _net(w):
    return oracle.Net(w.obs_dim, w.h1, w.h2, w.act, w.heads, w.n_gauss)


@pytest.mark.parametrize("wname,prec", [("mario", "fp32"), ("mario", "bf16"), ("ddnet", "bf16"),
                                        ("tiny", "fp32")])
def test_muon_steps_match_oracle(wname, prec):
    import torch
    import policy_rl_gb300 as P
    w = dataclasses.replace(synth.WORKLOADS[wname].scaled(T=4, N=64), precision=prec)
    p0 = synth.init_params(w, seed=1)
    cfg = P.config_from_workload(w, max_minibatch=64, optimizer=1, muon_lr=0.02, muon_beta=0.95)
    ctx = P.Context(cfg, p0)
    net = _net(w)
    rng = np.random.default_rng(0)
    p, m, v, mom = (p0.astype(np.float64), np.zeros(p0.size), np.zeros(p0.size),
                    np.zeros(p0.size))
    lr = 2.5e-4
    for step in range(1, 4):
        g = (rng.normal(size=p0.size) * 0.05).astype(np.float32)
        ctx.grad.copy_(dev(g))
        gn = torch.zeros(4, device="cuda")
        ctx.muon_step(lr, grad_norm=gn)
        ctx.sync_status()
        norm, gc = oracle.clip_grad_norm(g.astype(np.float64), w.max_grad_norm)
        p, mom, m, v = oracle.muon(net, p, gc, mom, m, v, step, 0.02, 0.95, lr,
                                   bf16=prec == "bf16")
        assert abs(host(gn)[0] - norm) <= 1e-5 * norm
    assert ctx.step() == 3
    got = host(ctx.params).astype(np.float64)
    tol = 1e-4 if prec == "fp32" else 2e-2
    for name, sl in param_slices(w).items():
        if sl.stop == sl.start:
            continue
        if name.startswith("W"):
            e = normwise(got[sl] - p0[sl], p[sl] - p0[sl])
            assert e <= tol, (name, e)
        else:
            np.testing.assert_allclose(got[sl], p[sl], rtol=1e-6, atol=1e-7)
    ctx.close()


def _update(w, seed=0, reps=1):
    import torch
    import policy_rl_gb300 as P
    ro = synth.rollout(w, seed=seed)
    p0 = synth.init_params(w, seed=seed)
    ro.logp_old = conditioned_logp_old(w, ro, p0)
    ctx = P.Context(P.config_from_workload(w, optimizer=1, muon_lr=0.01, muon_beta=0.9), p0)
    E, M = w.epochs, w.minibatches
    st = torch.zeros(E * M, 6, device="cuda")
    args = [dev(x) for x in (ro.obs, ro.act_disc, ro.act_cont, ro.logp_old, ro.val, ro.rew,
                             ro.done, ro.boot)]
    for _ in range(reps):
        ctx.update(*args, E, M, w.gamma, w.lam, w.lr, 11, stats=st)
    ctx.sync_status()
    out = host(ctx.params).copy(), host(st).copy(), ctx.step()
    ctx.close()
    return ro, p0, out


@pytest.mark.parametrize("wname", ["tiny", "mario_small"])
def test_update_with_muon_matches_oracle(wname):
    if wname == "tiny":
        w = synth.WORKLOADS["tiny"]
        tol = 1e-3
    else:
        w = synth.WORKLOADS["mario"].scaled(T=16, N=256, epochs=2, minibatches=4)
        tol = 0.1
    ro, p0, (p, stats, step) = _update(w)
    assert step == w.epochs * w.minibatches
    hp = oracle.Hyper(gamma=w.gamma, lam=w.lam, clip=w.clip, vf_coef=w.vf_coef,
                      ent_coef=w.ent_coef, lr=w.lr, max_grad_norm=w.max_grad_norm, seed=11,
                      bf16_operands=w.precision == "bf16", optimizer=1, muon_lr=0.01,
                      muon_beta=0.9)
    ref = oracle.update(_net(w), hp, w.T, w.N, w.epochs, w.minibatches, ro.obs, ro.act_disc,
                        ro.act_cont, ro.logp_old, ro.val, ro.rew, ro.done, ro.boot, p0)
    e = normwise(p - p0, ref.params - p0)
    assert e <= tol, e
    rtol = 2e-2 if w.precision == "bf16" else 1e-4
    np.testing.assert_allclose(stats[:, 2:4], ref.stats[:, 2:4], rtol=rtol)


def test_update_with_muon_is_deterministic():
    w = synth.WORKLOADS["mario"].scaled(T=16, N=256, epochs=2, minibatches=4)
    a = _update(w, reps=2)[2]
    b = _update(w, reps=2)[2]
    assert a[2] == 16 and np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_muon_step_needs_a_muon_context():
    import policy_rl_gb300 as P
    w = synth.WORKLOADS["tiny"]
    ctx = P.Context(P.config_from_workload(w), synth.init_params(w))
    with pytest.raises(P.PpoError) as ei:
        ctx.muon_step(1e-3)
    assert ei.value.status == 1
    ctx.close()
