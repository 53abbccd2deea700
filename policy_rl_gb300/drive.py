"""Small standalone drivers of the library, for profilers (ncu) and quick checks.

  python -m policy_rl_gb300.drive minibatch <workload> <reps>
      ppo_minibatch_loss_grad + ppo_adam_step, <reps> times, on one minibatch
      of the named synthetic workload (random advantages/returns/indices).
  python -m policy_rl_gb300.drive gae <T> <N> [reps]
      ppo_gae with moments and normalisation on seeded N(0,1) inputs.
  python -m policy_rl_gb300.drive adam [reps]
      ppo_adam_step (squared-norm pass + clip/Adam) over the 67.2 M fp32
      parameters of a 65536-1024-64 network (1 GB of optimiser state).
"""
from __future__ import annotations

import sys

import numpy as np


def minibatch(wname: str = "mario", reps: int = 3) -> None:
    import torch
    import policy_rl_gb300 as P
    from policy_rl_gb300 import synth
    w = synth.WORKLOADS[wname]
    B, mb = w.B, w.B // w.minibatches
    big = B * w.obs_dim > 2e8
    ro = synth.rollout(w, with_obs=not big)
    ctx = P.Context(P.config_from_workload(w), synth.init_params(w))
    d = lambda x: torch.from_numpy(np.ascontiguousarray(x)).cuda()
    g = torch.Generator(device="cuda")
    g.manual_seed(0)
    obs = torch.randn(B, w.obs_dim, device="cuda", generator=g) if big else d(ro.obs)
    adv = torch.randn(B, device="cuda", generator=g)
    ret = torch.randn(B, device="cuda", generator=g)
    idx = torch.randperm(B, device="cuda", generator=g)[:mb].to(torch.int32)
    args = [obs, d(ro.act_disc), d(ro.act_cont), d(ro.logp_old), adv, ret, idx]
    for _ in range(reps):
        ctx.minibatch_loss_grad(*args)
        ctx.adam_step(w.lr)
    ctx.sync_status()
    ctx.close()


def gae(T: int, N: int, reps: int = 3) -> None:
    import torch
    import policy_rl_gb300 as P
    g = torch.Generator(device="cuda")
    g.manual_seed(0)
    rew = torch.randn(T, N, device="cuda", generator=g)
    val = torch.randn(T, N, device="cuda", generator=g)
    done = (torch.rand(T, N, device="cuda", generator=g) < 0.001).float()
    boot = torch.randn(N, device="cuda", generator=g)
    adv, ret, advn = (torch.empty(T, N, device="cuda") for _ in range(3))
    st = torch.empty(4, device="cuda")
    work = torch.empty(P.ppo_gae_workspace_bytes(T, N), dtype=torch.uint8, device="cuda")
    for _ in range(reps):
        P.ppo_gae(rew, val, done, boot, 0.997, 0.95, adv, ret, advn, st, work)
    torch.cuda.synchronize()


def adam(reps: int = 3) -> None:
    import torch
    import policy_rl_gb300 as P
    cfg = P.make_config(65536, 1024, 64, heads=(2,), precision=0, max_batch=1, max_minibatch=1,
                        max_epochs=1)
    ctx = P.Context(cfg)
    g = torch.Generator(device="cuda")
    g.manual_seed(0)
    ctx.grad.normal_(generator=g)
    for _ in range(reps):
        ctx.adam_step(1e-4)
    ctx.sync_status()
    ctx.close()


if __name__ == "__main__":
    if sys.argv[1] == "minibatch":
        minibatch(sys.argv[2] if len(sys.argv) > 2 else "mario",
                  int(sys.argv[3]) if len(sys.argv) > 3 else 3)
    elif sys.argv[1] == "gae":
        gae(int(sys.argv[2]), int(sys.argv[3]), int(sys.argv[4]) if len(sys.argv) > 4 else 3)
    elif sys.argv[1] == "adam":
        adam(int(sys.argv[2]) if len(sys.argv) > 2 else 3)
    else:
        raise SystemExit(__doc__)
