"""Adam step and the whole update through the C ABI vs the oracle.

"PlayTrain", Table 8 (Adam, grad-norm clip 0.5); "Teaching Mario to
speedrun", sec. 6 "The whole algorithm".
Adam on identical gradients: params/moments normwise within 1e-5 (fp32 Adam
against fp64).  Whole update: each side runs its own trajectory from the same
initial weights; the parameter change p - p0 is compared normwise (1e-3 in
fp32 mode: per-step gradient agreement ~1e-6 relative, amplified only where
Adam divides a near-zero gradient by its own magnitude), and the per-minibatch
statistics as in the minibatch test.
"""
import dataclasses

import numpy as np
import pytest

import oracle
from policy_rl_gb300 import synth
from tests._gpu import MODES, conditioned_logp_old, dev, host, mode_kwargs, normwise

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("prec", ["fp32", "bf16"])
@pytest.mark.parametrize("max_norm", [0.5, 0.0, 1e6])
def test_adam_step_matches_oracle(prec, max_norm):
    import torch
    import policy_rl_gb300 as P
    w = dataclasses.replace(synth.WORKLOADS["mario"].scaled(T=4, N=64), precision=prec,
                            max_grad_norm=max_norm)
    p0 = synth.init_params(w)
    cfg = P.config_from_workload(w, max_minibatch=64)
    ctx = P.Context(cfg, p0)
    rng = np.random.default_rng(0)
    p, m, v = p0.astype(np.float64), np.zeros(p0.size), np.zeros(p0.size)
    for step in range(1, 4):
        g = (rng.normal(size=p0.size) * 0.05).astype(np.float32)
        ctx.grad.copy_(dev(g))
        gn = torch.zeros(4, device="cuda")
        ctx.adam_step(2.5e-4, grad_norm=gn)
        ctx.sync_status()
        norm, gc = oracle.clip_grad_norm(g.astype(np.float64), max_norm)
        p, m, v = oracle.adam(p, gc, m, v, step, 2.5e-4)
        assert abs(host(gn)[0] - norm) <= 1e-5 * norm
    assert ctx.step() == 3
    assert normwise(host(ctx.params), p) <= 1e-6
    assert normwise(host(ctx.adam_m), m) <= 1e-5
    assert normwise(host(ctx.adam_v), v) <= 1e-5
    ctx.close()


def _update(w, seed=0, host_api=False, mode="per_stage"):
    import torch
    import policy_rl_gb300 as P
    ro = synth.rollout(w, seed=seed)
    p0 = synth.init_params(w, seed=seed)
    ro.logp_old = conditioned_logp_old(w, ro, p0)
    ctx = P.Context(P.config_from_workload(w, **mode_kwargs(mode)), p0)
    E, M = w.epochs, w.minibatches
    if host_api:
        stats = np.zeros((E * M, 6), np.float32)
        ctx.update_host(ro.obs, ro.act_disc, ro.act_cont, ro.logp_old, ro.val, ro.rew, ro.done,
                        ro.boot, E, M, w.gamma, w.lam, w.lr, 11, stats=stats)
    else:
        st = torch.zeros(E * M, 6, device="cuda")
        ctx.update(dev(ro.obs), dev(ro.act_disc), dev(ro.act_cont), dev(ro.logp_old),
                   dev(ro.val), dev(ro.rew), dev(ro.done), dev(ro.boot), E, M, w.gamma, w.lam,
                   w.lr, 11, stats=st)
        ctx.sync_status()
        stats = host(st)
    params = host(ctx.params).copy()
    step = ctx.step()
    ctx.close()
    net = oracle.Net(w.obs_dim, w.h1, w.h2, w.act, w.heads, w.n_gauss)
    hp = oracle.Hyper(gamma=w.gamma, lam=w.lam, clip=w.clip, vf_coef=w.vf_coef,
                      ent_coef=w.ent_coef, lr=w.lr, max_grad_norm=w.max_grad_norm, seed=11,
                      bf16_operands=w.precision == "bf16")
    ref = oracle.update(net, hp, w.T, w.N, E, M, ro.obs, ro.act_disc, ro.act_cont, ro.logp_old,
                        ro.val, ro.rew, ro.done, ro.boot, p0)
    return p0, params, stats, step, ref


@pytest.mark.parametrize("host_api", [False, True])
def test_tiny_update_fp32(host_api):
    w = synth.WORKLOADS["tiny"]                   # T=128, N=64, 1 epoch x 4 minibatches
    p0, p, stats, step, ref = _update(w, host_api=host_api)
    assert step == w.epochs * w.minibatches
    e = normwise(p - p0, ref.params - p0)
    assert e <= 1e-3, e
    np.testing.assert_allclose(stats[:, 0], ref.stats[:, 0], rtol=1e-4, atol=1e-6)
    np.testing.assert_allclose(stats[:, 2:4], ref.stats[:, 2:4], rtol=1e-4)


@pytest.mark.parametrize("mode", MODES)
def test_small_update_bf16(mode):
    w = synth.WORKLOADS["mario"].scaled(T=16, N=256, epochs=2, minibatches=4)
    p0, p, stats, step, ref = _update(w, mode=mode)
    assert step == 8
    e = normwise(p - p0, ref.params - p0)
    assert e <= 0.1, e
    np.testing.assert_allclose(stats[:, 2:4], ref.stats[:, 2:4], rtol=2e-2)


def test_update_replays_graph_and_is_deterministic():
    import torch
    import policy_rl_gb300 as P
    w = synth.WORKLOADS["mario"].scaled(T=16, N=256, epochs=2, minibatches=4)
    ro = synth.rollout(w)
    p0 = synth.init_params(w)
    finals = []
    for _ in range(2):
        ctx = P.Context(P.config_from_workload(w), p0)
        args = [dev(x) for x in (ro.obs, ro.act_disc, ro.act_cont, ro.logp_old, ro.val, ro.rew,
                                 ro.done, ro.boot)]
        for _ in range(2):       # second call replays the captured graph
            ctx.update(*args, w.epochs, w.minibatches, w.gamma, w.lam, w.lr, 3)
        ctx.sync_status()
        assert ctx.step() == 16
        finals.append(host(ctx.params).copy())
        ctx.close()
    assert np.array_equal(finals[0], finals[1])


@pytest.mark.parametrize("prec", ["fp32", "bf16"])
def test_pipelined_host_updates_match_synchronous(prec):
    """ppo_update_host_async over five distinct pinned rollouts (both staging
    slots used more than once) gives the same bits as five ppo_update_host
    calls: parameters, optimizer step count and every call's statistics.  On
    return from call k the statistics of call k-2 are already on the host."""
    import torch
    import policy_rl_gb300 as P
    w = dataclasses.replace(synth.WORKLOADS["mario"].scaled(T=16, N=256, epochs=2,
                                                            minibatches=4), precision=prec)
    p0 = synth.init_params(w, seed=2)
    E, M, K = w.epochs, w.minibatches, 5
    pin = lambda x: torch.from_numpy(np.ascontiguousarray(x)).pin_memory()
    rolls = []
    for k in range(K):
        ro = synth.rollout(w, seed=20 + k)
        rolls.append([pin(x) for x in (ro.obs, ro.act_disc, ro.act_cont, ro.logp_old, ro.val,
                                       ro.rew, ro.done, ro.boot)])
    hp = (E, M, w.gamma, w.lam, w.lr)
    stream = torch.cuda.Stream()
    ref = P.Context(P.config_from_workload(w), p0)
    ref_stats = []
    for k in range(K):
        st = torch.zeros(E * M, 6).pin_memory()
        ref.update_host(*rolls[k], *hp, 100 + k, stats=st, stream=stream)
        ref_stats.append(st.numpy().copy())
    ref_p = host(ref.params).copy()
    ref.close()
    assert np.all(np.isfinite(ref_p)) and np.all(np.isfinite(np.stack(ref_stats)))

    ctx = P.Context(P.config_from_workload(w), p0)
    stats = [torch.full((E * M, 6), float("nan")).pin_memory() for _ in range(K)]
    for k in range(K):
        ctx.update_host_async(*rolls[k], *hp, 100 + k, stats=stats[k], stream=stream)
        if k >= 2:
            np.testing.assert_array_equal(stats[k - 2].numpy(), ref_stats[k - 2])
    ctx.host_wait()
    for k in range(K):
        np.testing.assert_array_equal(stats[k].numpy(), ref_stats[k])
    np.testing.assert_array_equal(host(ctx.params), ref_p)
    assert ctx.step() == K * E * M
    # a synchronous call after pipelined ones, and a call on another stream,
    # continue the same trajectory
    ctx.update_host_async(*rolls[0], *hp, 7, stream=torch.cuda.Stream())
    ctx.update_host(*rolls[1], *hp, 8, stream=stream)
    ctx.sync_status()
    assert ctx.step() == (K + 2) * E * M
    ctx.close()
