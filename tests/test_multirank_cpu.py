"""World-size-2 checks on the CPU (gloo), no GPU.

1. Data-parallel decomposition of the learner step ("Teaching Mario to
   speedrun", sec. 6: the loss is a mean over the minibatch): with the
   minibatch rows split across two ranks, the sum all-reduce of each rank's
   row-count-weighted oracle gradient equals the single-rank oracle gradient.
   That single all-reduce is the one exchange a multi-GPU learner needs
   (between gradient assembly and Adam).
2. The bench's multi-rank timing: barrier and max over ranks.
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
