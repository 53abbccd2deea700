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
4. The data-parallel update over environment shards ("PlayTrain", App. C.3):
   the oracle's emulated sharded update is pinned to one loss over the union
   of the ranks' slices per step and to the plain update at one rank, the
   (count, mean, M2) merge to the two-pass moments of the union; two gloo
   ranks running the decomposition, with the shard moments gathered through
   the library binding's TorchCollective, reproduce it to 1e-10.
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


# ---- the data-parallel update: env shards, merged moments, gradient all-reduce ----
def _tiny_sharded_setup(N=32):
    import oracle
    from policy_rl_gb300 import synth
    w = synth.WORKLOADS["tiny"].scaled(T=16, N=N, epochs=2, minibatches=4)
    ro = synth.rollout(w, seed=2)
    p0 = synth.init_params(w, seed=2).astype(np.float64)
    net = oracle.Net(w.obs_dim, w.h1, w.h2, w.act, w.heads, w.n_gauss)
    hp = oracle.Hyper(gamma=w.gamma, lam=w.lam, clip=w.clip, vf_coef=w.vf_coef,
                      ent_coef=w.ent_coef, lr=w.lr, max_grad_norm=w.max_grad_norm, seed=17)
    return w, ro, p0, net, hp


def test_moments_merge_equals_two_pass_moments_of_the_union():
    import oracle
    rng = np.random.default_rng(5)
    x = rng.standard_normal(1001) * 3 + 1
    for cut in (1, 17, 500, 1000):
        m = oracle.moments_merge(oracle.moments3(x[:cut]), oracle.moments3(x[cut:]))
        assert m[0] == x.size
        assert abs(m[1] - x.mean()) <= 1e-14 * (1 + abs(x.mean()))
        assert abs(m[2] - x.var() * x.size) <= 1e-12 * x.var() * x.size
    empty = np.zeros(3)
    assert np.array_equal(oracle.moments_merge(empty, oracle.moments3(x)), oracle.moments3(x))


def test_sharded_update_one_rank_is_the_update():
    import oracle
    w, ro, p0, net, hp = _tiny_sharded_setup()
    a = oracle.update_sharded(net, hp, 1, w.T, w.N, w.epochs, w.minibatches, ro.obs,
                              ro.act_disc, ro.act_cont, ro.logp_old, ro.val, ro.rew, ro.done,
                              ro.boot, p0)
    b = oracle.update(net, hp, w.T, w.N, w.epochs, w.minibatches, ro.obs, ro.act_disc,
                      ro.act_cont, ro.logp_old, ro.val, ro.rew, ro.done, ro.boot, p0)
    assert np.array_equal(a.params, b.params) and np.array_equal(a.stats, b.stats)


def test_sharded_update_steps_on_the_union_of_rank_slices():
    """Two shards: every step's gradient is that of one loss over the union
    of the ranks' slices (plain orc_loss_grad on those rows, advantages of
    the whole rollout normalised by the moments of all of them)."""
    import oracle
    w, ro, p0, net, hp = _tiny_sharded_setup()
    world, T, N, M = 2, w.T, w.N, w.minibatches
    Nr = N // world
    Br, mbr = T * Nr, T * Nr // M
    got = oracle.update_sharded(net, hp, world, T, N, w.epochs, M, ro.obs, ro.act_disc,
                                ro.act_cont, ro.logp_old, ro.val, ro.rew, ro.done, ro.boot, p0)
    adv, ret = oracle.gae(ro.rew, ro.val, ro.done, ro.boot, w.gamma, w.lam)
    mean, sd = oracle.moments(adv)
    p, m, v, step = p0.copy(), np.zeros(p0.size), np.zeros(p0.size), 0
    for e in range(w.epochs):
        perm = oracle.perm(hp.seed, e, Br)
        for k in range(M):
            loc = perm[k * mbr:(k + 1) * mbr]
            idx = np.concatenate([(loc // Nr) * N + r * Nr + loc % Nr for r in range(world)])
            _, g, _, _ = oracle.loss_grad(net, p, idx.astype(np.int32), ro.obs, ro.act_disc,
                                          ro.act_cont, ro.logp_old, adv.ravel(), ret.ravel(),
                                          clip=w.clip, vf_coef=w.vf_coef, ent_coef=w.ent_coef,
                                          normalize=True, adv_mean=mean, adv_std=sd)
            _, gc = oracle.clip_grad_norm(g, w.max_grad_norm)
            step += 1
            p, m, v = oracle.adam(p, gc, m, v, step, w.lr)
    err = np.linalg.norm(got.params - p) / np.linalg.norm(p)
    assert err < 1e-12, err


def _dp_worker(rank, world, port, out):
    """One rank of the data-parallel update with the oracle's pieces and
    exchanges over gloo (the moments through the library binding's
    TorchCollective)."""
    import ctypes
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    sys.path.insert(0, root)
    import torch.distributed as dist
    import oracle
    from policy_rl_gb300 import TorchCollective, _abi
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        coll = TorchCollective(device="cpu")
        w, ro, p0, net, hp = _tiny_sharded_setup()
        T, N, M = w.T, w.N, w.minibatches
        Nr = N // world
        cols = np.arange(rank * Nr, (rank + 1) * Nr)
        sh = lambda x: np.ascontiguousarray(x.reshape(T, N, *x.shape[1:])[:, cols]).reshape(
            T * Nr, *x.shape[1:])
        obs, act, logp = sh(ro.obs), sh(ro.act_disc), sh(ro.logp_old)
        rew = np.ascontiguousarray(ro.rew[:, cols])
        val = np.ascontiguousarray(ro.val[:, cols])
        done = np.ascontiguousarray(ro.done[:, cols])
        boot = np.ascontiguousarray(ro.boot[cols])
        adv, ret = oracle.gae(rew, val, done, boot, w.gamma, w.lam)
        mom = np.zeros((world, 3))
        mom[rank] = oracle.moments3(adv)
        assert coll.fn(None, _abi.COLL_ALLGATHER_F64, mom.ctypes.data, 3, None) == 0
        tot = np.zeros(3)
        for r in range(world):            # rank order
            tot = oracle.moments_merge(tot, mom[r])
        mean, sd = tot[1], np.sqrt(tot[2] / (tot[0] - 1))
        Br = T * Nr
        mbr = Br // M
        p, m, v, step = p0.copy(), np.zeros(p0.size), np.zeros(p0.size), 0
        for e in range(w.epochs):
            perm = oracle.perm(hp.seed, e, Br)
            for k in range(M):
                _, g, _, _ = oracle.loss_grad(net, p, perm[k * mbr:(k + 1) * mbr], obs, act,
                                              None, logp, adv.ravel(), ret.ravel(), clip=w.clip,
                                              vf_coef=w.vf_coef, ent_coef=w.ent_coef,
                                              normalize=True, adv_mean=mean, adv_std=sd)
                # the gradient exchange (fp64 here: the oracle's precision)
                t = torch.from_numpy(g / world)
                dist.all_reduce(t)
                _, gc = oracle.clip_grad_norm(t.numpy(), w.max_grad_norm)
                step += 1
                p, m, v = oracle.adam(p, gc, m, v, step, w.lr)
        # the binding's fp32 sum all-reduce, on values whose sums are exact
        buf = (np.arange(1000, dtype=np.float32) * 0.25 + rank).astype(np.float32)
        assert coll.fn(None, _abi.COLL_ALLREDUCE_SUM_F32, buf.ctypes.data, buf.size, None) == 0
        exact = np.array_equal(buf, np.arange(1000, dtype=np.float32) * 0.5 + 1)
        out.put((rank, (p, exact)))
    finally:
        dist.destroy_process_group()


def test_two_rank_sharded_update_through_the_binding_collective():
    """Each rank holds half of the environments; the shard moments are
    all-gathered through TorchCollective (the callback the library calls
    inside ppo_update) and merged in rank order, each rank permutes its own
    rows, and the fp64 gradients are sum-all-reduced.  Both ranks end at the
    oracle's emulated sharded update (1e-10).  The callback's fp32 sum
    all-reduce is checked on values whose sums are exact."""
    import torch.multiprocessing as mp
    import oracle
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_dp_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = dict(q.get(timeout=180) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    w, ro, p0, net, hp = _tiny_sharded_setup()
    ref = oracle.update_sharded(net, hp, 2, w.T, w.N, w.epochs, w.minibatches, ro.obs,
                                ro.act_disc, ro.act_cont, ro.logp_old, ro.val, ro.rew, ro.done,
                                ro.boot, p0)
    for r in (0, 1):
        p, exact = res[r]
        assert exact, r
        err = np.linalg.norm(p - ref.params) / np.linalg.norm(ref.params - p0)
        assert err < 1e-10, (r, err)
