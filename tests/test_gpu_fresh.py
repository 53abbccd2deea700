"""Per-minibatch advantages from fresh values through the C ABI vs the oracle.

"Teaching Mario to speedrun", sec. 8 "The Puffer net, and the trainer"
(advantages per minibatch from fresh values, GAE or V-trace); V-trace as
defined by Espeholt et al. 2018 ("IMPALA", sec. 4.1).

- ppo_segment_advantage on given values/ratios: advantages, targets and the
  normalised advantages elementwise within 1e-5 (|y| + rms(y)) of the fp64
  oracle; moments within 1e-5.  Cases span several scan windows with a ragged
  last one, one segment, one step, all-done segments and the degenerate clips.
- ppo_minibatch_loss_grad_fresh: gradients normwise per parameter tensor
  (1e-4 fp32, 2e-2 bf16), loss statistics, and the fresh advantages/targets.
- ppo_update in the fresh modes: the parameter change against the oracle's
  trajectory (as in test_gpu_update), and bit-identical replays.
"""

import numpy as np
import pytest

import oracle
from policy_rl_gb300 import synth
from tests._gpu import (LOG_RATIO_OFFSETS, assert_elementwise, dev, host, normwise,
                        param_slices)

pytestmark = pytest.mark.gpu


def _seg_inputs(T, N, ns, seed, p_done=0.02, vtrace=False):
    rng = np.random.default_rng(seed)
    rew = rng.normal(size=(T, N)).astype(np.float32)
    done = (rng.random((T, N)) < p_done).astype(np.float32)
    boot = rng.normal(size=N).astype(np.float32)
    envs = rng.permutation(N)[:ns].astype(np.int32)
    val = rng.normal(size=(T, ns)).astype(np.float32)
    ratio = np.exp(rng.normal(0, 0.3, size=(T, ns))).astype(np.float32) if vtrace else None
    return rew, done, boot, envs, val, ratio


def _gpu_segment(rew, done, boot, envs, val, ratio, gamma, lam, rho_clip, c_clip):
    import torch
    import policy_rl_gb300 as P
    T, ns = val.shape
    adv = torch.empty(T, ns, device="cuda")
    ret = torch.empty(T, ns, device="cuda")
    an = torch.empty(T, ns, device="cuda")
    st = torch.zeros(4, device="cuda")
    work = torch.empty(P.ppo_segment_advantage_workspace_bytes(), dtype=torch.uint8,
                       device="cuda")
    P.ppo_segment_advantage(dev(rew), dev(done), dev(boot), dev(envs), dev(val),
                            None if ratio is None else dev(ratio), gamma, lam, adv, ret,
                            rho_clip=rho_clip, c_clip=c_clip, adv_norm=an, stats=st, work=work)
    torch.cuda.synchronize()
    assert host(work[4:8]).view(np.int32)[0] == 0   # no bounded wait gave up
    return host(adv), host(ret), host(an), host(st)[:2]


CASES = [
    # T, N, ns, vtrace, clips, p_done
    (128, 2048, 256, False, (1.0, 1.0), 0.004),   # one Mario-like minibatch of segments
    (128, 2048, 256, True, (1.0, 1.0), 0.004),
    (300, 64, 64, True, (0.8, 1.2), 0.02),        # windows 128 + 128 + 44
    (37, 1000, 1, False, (1.0, 1.0), 0.05),       # one segment, one partial window
    (1, 5, 3, True, (1.0, 1.0), 0.3),             # one step
    (200, 40, 17, True, (2.0, 0.5), 1.0),         # every step terminal
    (129, 33, 33, True, (1.0, 1.0), 0.0),         # a window of a single step
    (64, 32768, 32768, True, (1.0, 1.0), 0.01),   # thread-per-segment scan (>= 16,384)
    (37, 20000, 16384, False, (1.0, 1.0), 0.05),  # its threshold, ragged T
]


@pytest.mark.parametrize("T,N,ns,vtrace,clips,p_done", CASES)
def test_segment_advantage_matches_oracle(T, N, ns, vtrace, clips, p_done):
    rew, done, boot, envs, val, ratio = _seg_inputs(T, N, ns, 3, p_done, vtrace)
    gamma, lam = 0.99, 0.95
    a, r, an, st = _gpu_segment(rew, done, boot, envs, val, ratio, gamma, lam, *clips)
    ra, rr = oracle.segment_advantage(rew, done, boot, envs, val.astype(np.float64),
                                      None if ratio is None else ratio.astype(np.float64),
                                      gamma, lam, *clips)
    assert_elementwise(a, ra, 1e-5)
    assert_elementwise(r, rr, 1e-5)
    mean, sd = oracle.moments(ra)
    assert abs(st[0] - mean) <= 1e-5 * (abs(mean) + sd) + 1e-7
    assert abs(st[1] - sd) <= 1e-5 * sd + 1e-7
    assert_elementwise(an, (ra - mean) / (sd + 1e-8), 1e-5)


def test_segment_advantage_degenerate():
    T, N, ns = 50, 20, 20
    rew, done, boot, envs, val, ratio = _seg_inputs(T, N, ns, 4, 0.05, True)
    # rho_bar = 0: no correction, the targets are the values themselves
    a, r, an, st = _gpu_segment(rew, done, boot, envs, val, ratio, 0.99, 0.95, 0.0, 1.0)
    assert np.all(a == 0.0) and np.array_equal(r, val)
    assert np.all(an == 0.0) and st[1] == 0.0
    # constant advantages (every step terminal, r = V + c, all exact in fp32):
    # A = c, normalised 0
    val = (np.random.default_rng(5).integers(-16, 16, size=val.shape) / 4).astype(np.float32)
    done1 = np.ones((T, N), np.float32)
    rew1 = np.zeros((T, N), np.float32)
    rew1[:, envs] = val + 0.25
    a, r, an, st = _gpu_segment(rew1, done1, boot, envs, val, None, 0.99, 0.95, 1.0, 1.0)
    assert np.all(a == np.float32(0.25)) and np.all(an == 0.0)


def _fresh_setup(w, ns, seed):
    ro = synth.rollout(w, seed=seed)
    p0 = synth.init_params(w, seed=seed)
    net = oracle.Net(w.obs_dim, w.h1, w.h2, w.act, w.heads, w.n_gauss)
    # behaviour log-probabilities: the oracle's at p0 minus row offsets, so
    # that ratios spread over both clipped and unclipped sides
    lp, _ = oracle.policy_logp(net, p0.astype(np.float64), ro.obs, ro.act_disc, ro.act_cont)
    off = np.array(LOG_RATIO_OFFSETS)[np.arange(lp.size) % len(LOG_RATIO_OFFSETS)]
    ro.logp_old = (lp - off).astype(np.float32)
    envs = oracle.perm(5, 0, w.N)[:ns]
    return ro, p0, net, envs


@pytest.mark.parametrize("wname,ns,adv_mode", [("tiny", 16, 1), ("tiny", 16, 2),
                                              ("mario", 64, 1), ("mario", 64, 2)])
def test_fresh_minibatch_matches_oracle(wname, ns, adv_mode):
    import torch
    import policy_rl_gb300 as P
    w = synth.WORKLOADS[wname]
    ro, p0, net, envs = _fresh_setup(w, ns, 9)
    mb = w.T * ns
    ctx = P.Context(P.config_from_workload(w, max_minibatch=mb), p0)
    st6 = torch.zeros(8, device="cuda")
    a_out = torch.empty(mb, device="cuda")
    r_out = torch.empty(mb, device="cuda")
    ctx.minibatch_loss_grad_fresh(dev(ro.obs), dev(ro.act_disc), dev(ro.act_cont),
                                  dev(ro.logp_old), dev(ro.rew), dev(ro.done), dev(ro.boot),
                                  dev(envs), adv_mode, w.gamma, w.lam, stats6=st6,
                                  adv_out=a_out, ret_out=r_out)
    ctx.sync_status()
    g = host(ctx.grad).copy()
    s6 = host(st6)[:6]
    an, rt = host(a_out), host(r_out)
    ctx.close()
    bf16 = w.precision == "bf16"
    _, gref, sref, scale, an_ref, rt_ref = oracle.loss_grad_fresh(
        net, p0.astype(np.float64), w.T, w.N, envs, ro.obs, ro.act_disc, ro.act_cont,
        ro.logp_old, ro.rew, ro.done, ro.boot, vtrace=adv_mode == 2, gamma=w.gamma, lam=w.lam,
        clip=w.clip, vf_coef=w.vf_coef, ent_coef=w.ent_coef, bf16_operands=bf16)
    tol = 2e-2 if bf16 else 1e-4
    if bf16:
        assert normwise(an, an_ref) <= 1e-2
        assert normwise(rt, rt_ref) <= 1e-2
    else:
        assert_elementwise(an, an_ref, 1e-4)
        assert_elementwise(rt, rt_ref, 1e-4)
    for name, sl in param_slices(w).items():
        if sl.stop > sl.start:
            e = normwise(g[sl], gref[sl])
            assert e <= tol, f"{name}: normwise error {e:.3e}"
    for k in range(6):
        assert abs(s6[k] - sref[k]) <= tol * max(abs(sref[k]), scale[k]) + 1e-7, (k, s6, sref)


def _fresh_update(w, adv_mode, seed=0, reps=1):
    import torch
    import policy_rl_gb300 as P
    ro, p0, net, _ = _fresh_setup(w, 1, seed)
    ctx = P.Context(P.config_from_workload(w, adv_mode=adv_mode, vtrace_rho_clip=1.0,
                                           vtrace_c_clip=0.9), p0)
    E, M = w.epochs, w.minibatches
    st = torch.zeros(E * M, 6, device="cuda")
    args = [dev(x) for x in (ro.obs, ro.act_disc, ro.act_cont, ro.logp_old, ro.val, ro.rew,
                             ro.done, ro.boot)]
    for _ in range(reps):
        ctx.update(*args, E, M, w.gamma, w.lam, w.lr, 11, stats=st)
    ctx.sync_status()
    out = (host(ctx.params).copy(), host(st).copy(), ctx.step())
    ctx.close()
    return ro, p0, net, out


@pytest.mark.parametrize("adv_mode", [1, 2])
def test_tiny_fresh_update_fp32(adv_mode):
    w = synth.WORKLOADS["tiny"]                   # T=128, N=64, 1 epoch x 4 minibatches
    ro, p0, net, (p, stats, step) = _fresh_update(w, adv_mode)
    assert step == w.epochs * w.minibatches
    hp = oracle.Hyper(gamma=w.gamma, lam=w.lam, clip=w.clip, vf_coef=w.vf_coef,
                      ent_coef=w.ent_coef, lr=w.lr, max_grad_norm=w.max_grad_norm, seed=11,
                      adv_mode=adv_mode, rho_clip=1.0, c_clip=0.9)
    ref = oracle.update(net, hp, w.T, w.N, w.epochs, w.minibatches, ro.obs, ro.act_disc,
                        ro.act_cont, ro.logp_old, ro.val, ro.rew, ro.done, ro.boot, p0)
    e = normwise(p - p0, ref.params - p0)
    assert e <= 1e-3, e
    np.testing.assert_allclose(stats[:, 0], ref.stats[:, 0], rtol=1e-4, atol=1e-6)
    np.testing.assert_allclose(stats[:, 2:4], ref.stats[:, 2:4], rtol=1e-4)


@pytest.mark.parametrize("adv_mode", [1, 2])
def test_small_fresh_update_bf16(adv_mode):
    w = synth.WORKLOADS["mario"].scaled(T=16, N=256, epochs=2, minibatches=4)
    ro, p0, net, (p, stats, step) = _fresh_update(w, adv_mode)
    assert step == 8
    hp = oracle.Hyper(gamma=w.gamma, lam=w.lam, clip=w.clip, vf_coef=w.vf_coef,
                      ent_coef=w.ent_coef, lr=w.lr, max_grad_norm=w.max_grad_norm, seed=11,
                      bf16_operands=True, adv_mode=adv_mode, rho_clip=1.0, c_clip=0.9)
    ref = oracle.update(net, hp, w.T, w.N, w.epochs, w.minibatches, ro.obs, ro.act_disc,
                        ro.act_cont, ro.logp_old, ro.val, ro.rew, ro.done, ro.boot, p0)
    e = normwise(p - p0, ref.params - p0)
    assert e <= 0.1, e
    np.testing.assert_allclose(stats[:, 2:4], ref.stats[:, 2:4], rtol=2e-2)


def test_fresh_update_replays_and_is_deterministic():
    w = synth.WORKLOADS["mario"].scaled(T=16, N=256, epochs=2, minibatches=4)
    finals = [_fresh_update(w, 2, reps=2)[3] for _ in range(2)]
    assert finals[0][2] == 16
    assert np.array_equal(finals[0][0], finals[1][0])
    assert np.array_equal(finals[0][1], finals[1][1])


def test_fresh_update_rejects_ragged_segments():
    import policy_rl_gb300 as P
    w = synth.WORKLOADS["tiny"].scaled(N=60, minibatches=8)   # 60 % 8 != 0, B % 8 == 0
    ro = synth.rollout(w)
    ctx = P.Context(P.config_from_workload(w, adv_mode=1), synth.init_params(w))
    args = [dev(x) for x in (ro.obs, ro.act_disc, ro.act_cont, ro.logp_old, ro.val, ro.rew,
                             ro.done, ro.boot)]
    with pytest.raises(P.PpoError) as ei:
        ctx.update(*args, 1, 8, w.gamma, w.lam, w.lr, 0)
    assert ei.value.status == 1
    ctx.close()
