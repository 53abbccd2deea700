"""World-size-2 checks on the CPU (gloo), no GPU.

1. Data-parallel decomposition of the learner step ("Teaching Mario to
   speedrun", sec. 6: the loss is a mean over the minibatch): with the
   minibatch rows split across two ranks, the sum all-reduce of each rank's
   row-count-weighted oracle gradient equals the single-rank oracle gradient.
   That single all-reduce is the one exchange a multi-GPU learner needs
   (between gradient assembly and Adam).
2. The bench's multi-rank timing: barrier and max over ranks.
3. Per-minibatch fresh advantages (GAE and V-trace) with the minibatch's
   environment segments split across ranks: one all-gather of (n, mean, M2)
   per rank plus the gradient all-reduce reproduce the single-rank step.
"""
import os
import socket

import numpy as np
import pytest

torch = pytest.importorskip("torch")


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, out):
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    sys.path.insert(0, root)
    import torch.distributed as dist
    import oracle
    import bench
    from policy_rl_gb300 import synth
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w = synth.WORKLOADS["tiny"].scaled(T=16, N=16)
        ro = synth.rollout(w)
        p0 = synth.init_params(w).astype(np.float64)
        net = oracle.Net(w.obs_dim, w.h1, w.h2, w.act, w.heads, w.n_gauss)
        adv, ret = oracle.gae(ro.rew, ro.val, ro.done, ro.boot, w.gamma, w.lam)
        idx = oracle.perm(4, 0, w.B)[:100]
        mine = np.array_split(idx, world)[rank]
        _, g, _, _ = oracle.loss_grad(net, p0, mine, ro.obs, ro.act_disc, ro.act_cont,
                                      ro.logp_old, adv.ravel(), ret.ravel())
        t = torch.from_numpy(g * (len(mine) / len(idx)))
        dist.all_reduce(t)                       # the data-parallel exchange
        _, gref, _, _ = oracle.loss_grad(net, p0, idx, ro.obs, ro.act_disc, ro.act_cont,
                                         ro.logp_old, adv.ravel(), ret.ravel())
        err = np.linalg.norm(t.numpy() - gref) / np.linalg.norm(gref)
        bench._barrier(world)
        mx = bench._max_over_ranks(float(rank + 1), world)
        out.put((rank, err, mx))
    finally:
        dist.destroy_process_group()


def test_two_rank_gradient_decomposition_and_timing():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, err, mx in res:
        assert err < 1e-12, err
        assert mx == 2.0


def _fresh_worker(rank, world, port, vtrace, out):
    """Per-minibatch fresh advantages ("Teaching Mario to speedrun", sec. 8)
    with the minibatch's environment segments split across ranks: each rank
    computes its segments' fresh values, advantages and (n, mean, M2); one
    all-gather of those three numbers gives the minibatch's moments (Chan's
    merge); each rank normalises its rows and computes its row-weighted
    gradient; the sum all-reduce equals the single-rank fresh step."""
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    sys.path.insert(0, root)
    import torch.distributed as dist
    import oracle
    from policy_rl_gb300 import synth
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w = synth.WORKLOADS["tiny"].scaled(T=12, N=16)
        ro = synth.rollout(w)
        p0 = synth.init_params(w).astype(np.float64)
        net = oracle.Net(w.obs_dim, w.h1, w.h2, w.act, w.heads, w.n_gauss)
        envs = oracle.perm(6, 0, w.N)[:10]              # one minibatch of 10 segments
        mine = np.array_split(envs, world)[rank]
        rows = oracle.segment_rows(w.T, w.N, mine)
        val, ratio = oracle.fresh_values(net, p0, rows, ro.obs, ro.act_disc, ro.act_cont,
                                         ro.logp_old, with_ratio=vtrace)
        adv, ret = oracle.segment_advantage(ro.rew, ro.done, ro.boot, mine, val, ratio, w.gamma,
                                            w.lam)
        a = adv.ravel()
        mom = torch.tensor([[a.size, a.mean(), ((a - a.mean()) ** 2).sum()]], dtype=torch.float64)
        allm = [torch.zeros_like(mom) for _ in range(world)]
        dist.all_gather(allm, mom)                      # the moment exchange
        n, mean, m2 = 0.0, 0.0, 0.0
        for t in allm:                                  # Chan's merge, rank order
            nb, mb, m2b = t[0].tolist()
            d = mb - mean
            tot = n + nb
            mean, m2, n = mean + d * nb / tot, m2 + m2b + d * d * n * nb / tot, tot
        sd = np.sqrt(m2 / (n - 1))
        af = np.zeros(w.B)
        rf = np.zeros(w.B)
        af[rows] = a
        rf[rows] = ret.ravel()
        _, g, _, _ = oracle.loss_grad(net, p0, rows, ro.obs, ro.act_disc, ro.act_cont,
                                      ro.logp_old, af, rf, normalize=True, adv_mean=mean,
                                      adv_std=sd)
        t = torch.from_numpy(g * (rows.size / (w.T * envs.size)))
        dist.all_reduce(t)                              # the gradient exchange
        _, gref, *_ = oracle.loss_grad_fresh(net, p0, w.T, w.N, envs, ro.obs, ro.act_disc,
                                             ro.act_cont, ro.logp_old, ro.rew, ro.done, ro.boot,
                                             vtrace=vtrace, gamma=w.gamma, lam=w.lam)
        out.put((rank, float(np.linalg.norm(t.numpy() - gref) / np.linalg.norm(gref))))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("vtrace", [False, True])
def test_two_rank_fresh_advantage_decomposition(vtrace):
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_fresh_worker, args=(r, 2, port, vtrace, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, err in res:
        assert err < 1e-10, err
