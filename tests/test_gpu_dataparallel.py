"""The data-parallel update path of the library (ppo_set_collective) on one GPU.

A run with two ranks needs two GPUs; here rank 0 of a two-rank job runs
alone with a collective that stands for a second rank holding an identical
shard: the sum all-reduce doubles the buffer, the all-gather copies rank 0's
values into rank 1's slot.  That is exactly what two ranks with the same
environments would compute, so rank 0's update must equal the oracle's
emulated two-rank update ("PlayTrain", App. C.3, data-parallel learner) on
the rollout made of the shard twice.  The statistics differ from the
single-rank update of the shard (the unbiased std of the doubled set), so
the test also sees the gathered moments take effect.
Bars: fp32 mode 1e-4 on the parameter change per step from the trace's
gradients, and the whole update's parameter change 1e-3 (as the single-rank
whole-update tests); bf16 mode 2e-2 on step 0's gradient against the
bf16-operand oracle and 0.1 on the trajectory.
"""
import ctypes

import numpy as np
import pytest

import oracle
from policy_rl_gb300 import synth
from tests._gpu import conditioned_logp_old, dev, host, normwise

pytestmark = pytest.mark.gpu


class _TwinRank:
    """Collective of a two-rank job whose other rank holds the same shard."""

    def __init__(self):
        from policy_rl_gb300 import _abi
        self.fn = _abi.COLLECTIVE_FN(self._call)
        self.calls = []

    def _call(self, user, op, buf, count, stream):
        import torch
        from policy_rl_gb300 import _DevArray
        self.calls.append(op)
        # the library's stream (the legacy default stream arrives as NULL)
        s = torch.cuda.ExternalStream(stream) if stream else torch.cuda.default_stream()
        with torch.cuda.stream(s):
            if op == 0:
                torch.as_tensor(_DevArray(buf, count, "<f4"), device="cuda").mul_(2.0)
            else:
                t = torch.as_tensor(_DevArray(buf, 2 * count, "<f8"), device="cuda")
                t[count:].copy_(t[:count])
        return 0


def _twice(x, T, N):
    """[T*N, ...] rows (or [T, N]) -> the rollout of the shard twice, [T, 2N]."""
    if x.ndim == 2 and x.shape == (T, N):
        return np.concatenate([x, x], axis=1)
    y = x.reshape(T, N, *x.shape[1:])
    return np.concatenate([y, y], axis=1).reshape(T * 2 * N, *x.shape[1:])


@pytest.mark.parametrize("prec", ["fp32", "bf16"])
def test_data_parallel_update_with_a_twin_rank(prec):
    import dataclasses
    import torch
    import policy_rl_gb300 as P
    base = synth.WORKLOADS["tiny"] if prec == "fp32" else \
        synth.WORKLOADS["mario"].scaled(T=16, N=128, epochs=2, minibatches=4)
    w = dataclasses.replace(base, precision=prec)
    ro = synth.rollout(w, seed=6)
    p0 = synth.init_params(w, seed=6)
    ro.logp_old = conditioned_logp_old(w, ro, p0)
    ctx = P.Context(P.config_from_workload(w), p0)
    twin = _TwinRank()
    ctx.set_collective(2, 0, twin)
    S, Pn = w.epochs * w.minibatches, ctx.n_params
    trace = torch.zeros(S * 4 * Pn, device="cuda")
    ctx.set_step_trace(trace, S)
    st = torch.zeros(S, 6, device="cuda")
    ctx.update(dev(ro.obs), dev(ro.act_disc), dev(ro.act_cont), dev(ro.logp_old), dev(ro.val),
               dev(ro.rew), dev(ro.done), dev(ro.boot), w.epochs, w.minibatches, w.gamma, w.lam,
               w.lr, 23, stats=st)
    ctx.sync_status()
    # one gather of the moments, then per step the gradient and the statistics
    assert twin.calls == [1] + [0, 0] * S
    tr = host(trace).reshape(S, 4, Pn).copy()
    final = host(ctx.params).astype(np.float64)
    stats = host(st)
    ctx.close()

    net = oracle.Net(w.obs_dim, w.h1, w.h2, w.act, w.heads, w.n_gauss)
    hp = oracle.Hyper(gamma=w.gamma, lam=w.lam, clip=w.clip, vf_coef=w.vf_coef,
                      ent_coef=w.ent_coef, lr=w.lr, max_grad_norm=w.max_grad_norm, seed=23,
                      bf16_operands=prec == "bf16")
    T, N = w.T, w.N
    two = dict(obs=_twice(ro.obs, T, N), act=_twice(ro.act_disc, T, N),
               actc=_twice(ro.act_cont, T, N), logp=_twice(ro.logp_old, T, N),
               val=_twice(ro.val, T, N), rew=_twice(ro.rew, T, N), done=_twice(ro.done, T, N),
               boot=np.concatenate([ro.boot, ro.boot]))
    ref = oracle.update_sharded(net, hp, 2, T, 2 * N, w.epochs, w.minibatches, two["obs"],
                                two["act"], two["actc"], two["logp"], two["val"], two["rew"],
                                two["done"], two["boot"], p0)
    single = oracle.update(net, hp, T, N, w.epochs, w.minibatches, ro.obs, ro.act_disc,
                           ro.act_cont, ro.logp_old, ro.val, ro.rew, ro.done, ro.boot, p0)
    assert not np.array_equal(ref.params, single.params)   # the merged moments matter

    # step 0: the GPU's gradient against the union loss of the two ranks' slices
    adv, ret = oracle.gae(two["rew"], two["val"], two["done"], two["boot"], w.gamma, w.lam)
    mean, sd = oracle.moments(adv)
    Br, M = T * N, w.minibatches
    mbr = Br // M
    loc = oracle.perm(23, 0, Br)[:mbr]
    idx = np.concatenate([(loc // N) * (2 * N) + r * N + loc % N for r in range(2)])
    _, g_ref, s_ref, scale = oracle.loss_grad(
        net, p0.astype(np.float64), idx.astype(np.int32), two["obs"], two["act"], two["actc"],
        two["logp"], adv.ravel(), ret.ravel(), clip=w.clip, vf_coef=w.vf_coef,
        ent_coef=w.ent_coef, normalize=True, adv_mean=mean, adv_std=sd,
        bf16_operands=prec == "bf16")
    tol = 1e-4 if prec == "fp32" else 2e-2
    assert normwise(tr[0, 3], g_ref) <= tol
    for q in range(6):
        assert abs(stats[0, q] - s_ref[q]) <= tol * max(abs(s_ref[q]), scale[q]) + 1e-7
    # every step's optimizer: clip + Adam of the all-reduced gradient
    for j in range(S):
        p_j, m_j, v_j, g_j = (tr[j, i].astype(np.float64) for i in range(4))
        p_next = tr[j + 1, 0].astype(np.float64) if j + 1 < S else final
        _, gc = oracle.clip_grad_norm(g_j, w.max_grad_norm)
        p_o, _, _ = oracle.adam(p_j, gc, m_j, v_j, j + 1, w.lr)
        assert normwise(p_next - p_j, p_o - p_j) <= 1e-4, j
    # the whole trajectory
    e = normwise(final - p0, ref.params - p0)
    assert e <= (1e-3 if prec == "fp32" else 0.1), e
