#!/usr/bin/env python
"""PPO learner-update benchmark on GB300.

One step = one whole PPO update ("Teaching Mario to speedrun", sec. 6 "The
whole algorithm", judge + learn) over a synthetic rollout.  The default
workload is the large-batch one: T=64 steps x N=65536 envs, obs 128-d, MLP
128-512-512 tanh, heads [9,2,2,2] + value, 4 epochs x 16 minibatches of
262,144 rows, bf16 tensor-core GEMMs with fp32 master weights and Adam.
Metric: samples/s = T*N / update time.

Output: one JSON line on rank 0.  `value` is device time with the rollout
resident in HBM (L2 flushed between steps by writing 256 MB); `e2e` goes
through ppo_update_host_async from pinned host buffers (H2D of every step's
rollout and D2H of its statistics inside the timed region, each step's
copies overlapping the previous step's update; `e2e_sync` the same one call
at a time through ppo_update_host).  `roofline` is the kernel stage
with the largest share of a profiled update (CUDA events between kernels);
`gemm_all` aggregates the tensor-core GEMM stages.  `mario` repeats the
measurement on the Mario-like workload (T=128 x N=2048, 64-256-256, 4 x 8
minibatches), a launch- and latency-bound case.  `gae_stress` is the GAE
scan's bandwidth at T=1024 x N=65536, `adam_stress` Adam over 67 M
parameters; `cpu_baseline` is the plain-C oracle on a bounded slice of the
headline workload (all host cores, and one core).

--impl reference times the oracle itself (the CPU reference implementation)
on a bounded slice per step.  --drive runs plain driver loops for profilers.
Multi-GPU (torchrun): one data-parallel update over the ranks, each rank
holding its own N environments (weak scaling): shard GAE, the advantage
moments all-gathered, per-rank minibatch slices, the flat gradient
all-reduced over NCCL before every optimizer step; value sums the samples
of all ranks over the slowest rank's time.  (With --advantages other than
global the ranks run independent replicas.)
"""
from __future__ import annotations

import argparse
import json
import math
import os
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

L2_FLUSH_BYTES = 256 << 20


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return d["hbm_gbs"], d["bf16_tflops"], d.get("bf16_tflops_sustained", d["bf16_tflops"]), \
            "measured"
    except Exception:
        return 6800.0, 1900.0, 1700.0, "fallback"


class Clocks:
    """nvidia-smi sampler (200 ms) over the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-i", str(self.gpu), "-lms", "200"], stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        sm, smax, reasons = [], 0.0, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax = max(smax, float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        os.unlink(self.path)
        if not sm:
            return None
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": smax, "reasons": sorted(reasons),
                "samples": len(sm)}


def _dist():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def _max_over_ranks(x: float, world: int) -> float:
    """Slowest rank's value (the job's time); CPU tensor under gloo."""
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def _barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ---- algorithmic work per kernel stage (for the roofline) ----------------------
def _stage_work(stage: str, w, mb: int):
    """(FLOPs, HBM bytes) of one launch of a kernel stage, or None.

    GEMM bytes are the bf16 activations each kernel must read and write once
    (weights and per-CTA partials are small and L2-resident): X [mb, Dp],
    H1/H2/dP1/dP2 [mb, H], dZ [mb, CP] (CP = head columns padded to 16/32;
    the weight-gradient kernel reads dZ through 64-column boxes)."""
    D, H1, H2, C = w.obs_dim, w.h1, w.h2, w.out_cols
    B = w.B
    Dp = -(-D // 64) * 64
    CP = 16 if C <= 16 else 32
    a = 2 * mb   # bytes per activation column of a minibatch (bf16)
    gemm = {
        "fwd1_gemm": (2 * mb * H1 * D, a * (Dp + H1)),
        "fwd2_gemm": (2 * mb * H2 * H1, a * (H1 + H2)),
        "head_loss_gemm": (2 * mb * C * H2, a * (H2 + CP) + mb * (4 * len(w.heads) + 12)),
        "dact2_gemm": (2 * mb * H2 * C, a * (CP + 2 * H2)),
        "dact1_gemm": (2 * mb * H1 * H2, a * (H2 + 2 * H1)),
        "wgrad_gemm": (2 * mb * (H2 * H1 + H1 * D + C * H2), a * (H2 + H1 + H1 + Dp + H2 + 64)),
        # fused variants: head + loss + dP2 (H2 read once); the whole fwd / loss / bwd-data
        "head_loss_dact2": (4 * mb * C * H2, a * (2 * H2 + CP) + mb * (4 * len(w.heads) + 12)),
        "fused_mlp": (2 * mb * (H1 * D + H2 * H1 + 2 * C * H2 + H1 * H2),
                      a * (Dp + 2 * H1 + 2 * H2 + 64) + mb * (4 * len(w.heads) + 12)),
    }
    if stage in gemm:
        return gemm[stage]
    P = w.num_params
    hbm = {
        "gae_scan": 20 * B,                       # read r, v, d; write adv, ret
        "pack_obs": B * (4 * D + 2 * Dp),
        "gather": mb * (2 * Dp * 2 + 4 * len(w.heads) * 2 + 4 * 3 * 2),
        "adam": 30 * P, "grad_sqnorm": 4 * P,
        "grad_reduce": 4 * P,
        "grad_reduce_adam": 34 * P,               # gradient write + norm + Adam + shadow
        # per-minibatch advantages: read H2 once (bf16), values (+ ratios) written and
        # re-read, rewards/dones read, advantages/returns written, normalised in place
        "fresh_advantages": mb * (2 * H2 + 40),
    }
    if stage in hbm:
        return 0, hbm[stage]
    return None


# --advantages: 0 GAE once per update over the rollout; 1 per minibatch of
# environment segments from fresh values (GAE); 2 the same with V-trace
ADV_MODES = {"global": 0, "fresh_gae": 1, "vtrace": 2}
# --optimizer: Adam on every parameter (default) or Muon on the weight matrices
OPTIMIZERS = {"adam": 0, "muon": 1}


# DRAM bytes per launch (dram__bytes_read.sum + dram__bytes_write.sum) from one
# ncu capture of the current kernels, cold caches; stages without such a
# capture report null.
NCU_TRAFFIC = {
    ("mario", "fwd1_gemm"): 4.26e6, ("mario", "fwd2_gemm"): 16.94e6,
    ("mario", "head_loss_gemm"): 17.78e6, ("mario", "dact2_gemm"): 21.05e6,
    ("mario", "dact1_gemm"): 33.73e6, ("mario", "wgrad_gemm"): 76.15e6,
    ("large", "fwd1_gemm"): 279.56e6, ("large", "fwd2_gemm"): 487.96e6,
    ("large", "head_loss_dact2"): 495.39e6, ("large", "dact1_gemm"): 837.59e6,
    ("large", "wgrad_gemm"): 1192.21e6,
    # the two-kernel head + loss / dP2 path (fused_loss = -1), earlier capture
    ("large", "head_loss_gemm"): 280.92e6, ("large", "dact2_gemm"): 518.69e6,
}


# fp32 FMA peak of the CUDA cores (no measured figure exists for it):
# 152 SMs x 128 fp32 lanes x 2 FLOP x 2.07 GHz (the recipe's unit counts and
# maximum SM clock)
FP32_ALU_TFLOPS = 152 * 128 * 2 * 2.07e9 / 1e12


def _muon_step_flops(w):
    """Newton-Schulz FLOPs of one Muon step: five iterations of X X^T
    (2 r^2 k), A A (2 r^3) and B X (2 r^2 k) per weight matrix."""
    D, H1, H2, C = w.obs_dim, w.h1, w.h2, w.out_cols
    tot = 0
    for rows, cols in ((H1, D), (H2, H1), (C, H2)):
        r, k = min(rows, cols), max(rows, cols)
        tot += 5 * (4 * r * r * k + 2 * r ** 3)
    return tot


def _roofline(stage, w, mb, ms_total, launches, hbm_peak, tf_peak, peak_src):
    """Roofline entry of one stage: bound = the larger of its tensor-time and
    HBM-time floors at the measured peaks; achieved = algorithmic work per
    launch / mean launch duration."""
    if stage == "muon":   # one optimizer step per minibatch
        steps = w.epochs * w.minibatches
        achieved = _muon_step_flops(w) * steps / (ms_total / 1e3) / 1e12
        if w.precision == "bf16":   # bf16 tensor-core Newton-Schulz products
            return {"bound": "tensor", "kernel": stage, "achieved": round(achieved, 3),
                    "peak": tf_peak, "unit": "TFLOP/s", "frac": round(achieved / tf_peak, 5),
                    "traffic": None, "peak_kind": f"bf16 sustained ({peak_src})",
                    "ms_per_optimizer_step": round(ms_total / steps, 4),
                    "algorithmic_per_step": {"flop": _muon_step_flops(w), "bytes": None}}
        return {"bound": "alu", "kernel": stage, "achieved": round(achieved, 3),
                "peak": round(FP32_ALU_TFLOPS, 1), "unit": "TFLOP/s",
                "frac": round(achieved / FP32_ALU_TFLOPS, 4), "traffic": None,
                "peak_kind": "fp32 FMA, derived (152 SMs x 128 lanes x 2 x 2.07 GHz)",
                "ms_per_optimizer_step": round(ms_total / steps, 4),
                "algorithmic_per_step": {"flop": _muon_step_flops(w), "bytes": None}}
    work = _stage_work(stage, w, mb)
    if work is None:
        return None
    flops, nbytes = work
    per_launch_s = ms_total / launches / 1e3
    t_tc = flops / (tf_peak * 1e12)
    t_hbm = nbytes / (hbm_peak * 1e9)
    traffic = NCU_TRAFFIC.get((w.name, stage))
    if t_tc >= t_hbm:
        achieved = flops / per_launch_s / 1e12
        return {"bound": "tensor", "kernel": stage, "achieved": round(achieved, 2),
                "peak": tf_peak, "unit": "TFLOP/s", "frac": round(achieved / tf_peak, 4),
                "traffic": traffic, "peak_kind": f"bf16 sustained ({peak_src})",
                "per_launch_us": round(per_launch_s * 1e6, 2),
                "algorithmic_per_launch": {"flop": flops, "bytes": nbytes}}
    achieved = nbytes / per_launch_s / 1e9
    return {"bound": "hbm", "kernel": stage, "achieved": round(achieved, 1), "peak": hbm_peak,
            "unit": "GB/s", "frac": round(achieved / hbm_peak, 4), "traffic": traffic,
            "peak_kind": f"HBM copy ({peak_src})", "per_launch_us": round(per_launch_s * 1e6, 2),
            "algorithmic_per_launch": {"flop": flops, "bytes": nbytes},
            "tensor_TFLOPs": round(flops / per_launch_s / 1e12, 2) if flops else None}


def _measure(w, args, world, rank, local, stream, peaks, adv_mode=0, optimizer=0):
    """Device-timed and end-to-end updates of workload w, a profiled update
    (per-kernel time), the dominant kernel's roofline and the aggregate of
    the tensor-core GEMM stages.  Returns (summary, ctx, obs on the device)."""
    import torch
    import policy_rl_gb300 as P
    from policy_rl_gb300 import synth

    hbm_peak, tf_burst, tf_sust, peak_src = peaks
    B, E, M = w.B, w.epochs, w.minibatches
    mb = B // M
    # observations of the large workloads (> 2e8 values) are drawn on the device
    # (torch's seeded N(0,1) / uniform tile ids); everything else comes from
    # the host-side seeded generator
    big = w.B * w.obs_dim > 2e8
    ro = synth.rollout(w, seed=rank, with_obs=not big)
    p0 = synth.init_params(w)
    ctx = P.Context(P.config_from_workload(w, adv_mode=adv_mode, optimizer=optimizer), p0)
    # N > 1 ranks: one data-parallel update over the ranks' environment shards
    # (each rank its own N envs; the gradient all-reduced over NCCL every step)
    dp = world > 1 and adv_mode == 0
    if dp:
        ctx.set_collective(world, rank, P.TorchCollective())
    dev = lambda x: torch.from_numpy(np.ascontiguousarray(x)).cuda()
    if big:
        g = torch.Generator(device="cuda")
        g.manual_seed(rank)
        obs_d = torch.randn(B, w.obs_dim, device="cuda", generator=g)
        if w.obs_kind == "ddnet":
            obs_d[:, :1333] = torch.randint(0, 6, (B, 1333), device="cuda", generator=g).float()
    else:
        obs_d = dev(ro.obs)
    args_dev = [obs_d] + [dev(x) for x in (ro.act_disc, ro.act_cont, ro.logp_old, ro.val,
                                           ro.rew, ro.done, ro.boot)]
    stats = torch.zeros(E * M, 6, device="cuda")
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device="cuda")
    hp = (E, M, w.gamma, w.lam, w.lr, 1234)

    def update():
        P.ppo_update(ctx.handle, *args_dev, *hp, stats=stats, stream=stream)

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            flush.zero_()
            update()
        stream.synchronize()
        P.ppo_sync_status(ctx.handle, stream)
        _barrier(world)
        torch.cuda.synchronize()
        clocks = Clocks(local)
        clocks.start()
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(args.steps)]
        for s, e in evs:
            flush.zero_()
            s.record(stream)
            update()
            e.record(stream)
        stream.synchronize()
        torch.cuda.synchronize()
        _barrier(world)
        clk = clocks.stop()
    P.ppo_sync_status(ctx.handle, stream)
    step_ms = [s.elapsed_time(e) for s, e in evs]
    ms = _max_over_ranks(float(np.mean(step_ms)), world)
    value = world * B / (ms / 1e3)

    # one profiled update: per-kernel device time, launches (the single-rank
    # update: the same kernels, without the collectives)
    if dp:
        ctx.set_collective(1, 0)
    with torch.cuda.stream(stream):
        prof = P.ppo_update_profile(ctx.handle, *args_dev, *hp, stats=stats, stream=stream)
    if dp:
        ctx.set_collective(world, rank, ctx._collective)
    kern = {k: v for k, v in prof.items() if not k.startswith("phase:")}
    phases = {k: v for k, v in prof.items() if k.startswith("phase:")}
    launches_per_update = sum(c for _, c in kern.values())
    total_ms = sum(t for t, _ in kern.values())
    # the dominant unit of work: a kernel, or a phase of the persistent kernel
    cand = dict(kern)
    if phases:
        cand.pop("minibatch_persistent", None)
        cand.update({k[len("phase:"):] + ("_gemm" if k[6:] in ("fwd1", "fwd2", "dact2", "dact1",
                                                                "wgrad") else ""): v
                     for k, v in phases.items()})
        cand = {("head_loss_gemm" if k == "head_loss" else k): v for k, v in cand.items()}
    dom = max(cand, key=lambda k: cand[k][0])
    prof_all = prof
    prof = cand
    roof = _roofline(dom, w, mb, prof[dom][0], prof[dom][1], hbm_peak, tf_sust, peak_src)
    if roof is not None:
        roof["share"] = round(prof[dom][0] / total_ms, 4)
    # all tensor-core GEMM stages together: FLOPs / their summed device time
    gemm_names = ("fwd1_gemm", "fwd2_gemm", "head_loss_gemm", "dact2_gemm", "dact1_gemm",
                  "wgrad_gemm", "head_loss_dact2", "fused_mlp")
    g_ms = sum(prof[k][0] for k in gemm_names if k in prof)
    g_flop = sum(_stage_work(k, w, mb)[0] * prof[k][1] for k in gemm_names if k in prof)
    gemm_all = ({"ms_per_update": round(g_ms, 4),
                 "TFLOPs": round(g_flop / (g_ms / 1e3) / 1e12, 2),
                 "frac_of_bf16_sustained": round(g_flop / (g_ms / 1e3) / 1e12 / tf_sust, 4)}
                if g_ms > 0 and w.precision == "bf16" else None)
    stages = {k: {"ms": round(t, 4), "launches": c, "share": round(t / total_ms, 4)}
              for k, (t, c) in sorted(prof_all.items(), key=lambda kv: -kv[1][0])}

    # end to end: host (pinned) buffers through the C ABI, copies inside the timed region
    pin = lambda x: torch.from_numpy(np.ascontiguousarray(x)).pin_memory()
    host_obs = obs_d.cpu().pin_memory() if big else pin(ro.obs)
    host_args = [host_obs] + [pin(x) for x in (ro.act_disc, ro.act_cont, ro.logp_old, ro.val,
                                               ro.rew, ro.done, ro.boot)]
    host_stats = torch.zeros(E * M, 6).pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in host_args)
    d2h = host_stats.numel() * 4
    e2e_steps = max(3, min(args.steps, int(math.ceil(4000.0 / max(ms, 1e-3)))))
    with torch.cuda.stream(stream):
        # pipelined: each step's copies overlap the previous step's update
        # (two staging slots, both graphs captured in the warm-up)
        for _ in range(max(2, min(args.warmup, 3))):
            P.ppo_update_host_async(ctx.handle, *host_args, *hp, stats=host_stats, stream=stream)
        P.ppo_host_wait(ctx.handle)
        _barrier(world)
        t0 = time.perf_counter()
        for _ in range(e2e_steps):   # (the host->device copies pass through L2 anyway)
            P.ppo_update_host_async(ctx.handle, *host_args, *hp, stats=host_stats, stream=stream)
        P.ppo_host_wait(ctx.handle)
        t1 = time.perf_counter()
        # one call at a time: copies, update, stats, then the next call
        sync_steps = min(e2e_steps, 5)
        _barrier(world)
        t2 = time.perf_counter()
        for _ in range(sync_steps):
            P.ppo_update_host(ctx.handle, *host_args, *hp, stats=host_stats, stream=stream)
        t3 = time.perf_counter()
    e2e_s = _max_over_ranks((t1 - t0) / e2e_steps, world)
    e2e_sync_s = _max_over_ranks((t3 - t2) / sync_steps, world)
    del host_obs, host_args
    summary = {
        "workload": _workload_str(w, _name(ADV_MODES, adv_mode), _name(OPTIMIZERS, optimizer)),
        "value": round(value, 1), "ms_per_step": round(ms, 4),
        "e2e": {"value": round(world * B / e2e_s, 1), "unit": "samples/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": e2e_steps,
                "api": "ppo_update_host_async + ppo_host_wait (pinned host rollout -> device, "
                       "stats -> host; each step's copies overlap the previous update)"},
        "e2e_sync": {"value": round(world * B / e2e_sync_s, 1), "unit": "samples/s",
                     "steps": sync_steps,
                     "api": "ppo_update_host (copies, update, stats; one call at a time)"},
        "roofline": roof, "gemm_all": gemm_all, "stages": stages,
        "profiled_update_ms": round(total_ms, 4),
        "launches_per_update": launches_per_update, "clocks": clk,
        "parallelism": (f"data-parallel x{world}: env shards, shard moments all-gathered, "
                        f"gradient all-reduced (NCCL) every minibatch" if dp
                        else f"replicas x{world}"),
    }
    return summary, ctx, obs_d


def _name(table, v):
    return {x: k for k, x in table.items()}[v]


def run_ours(args, world, rank, local):
    import torch
    from policy_rl_gb300 import synth

    torch.cuda.set_device(local)
    peaks = _peaks()
    hbm_peak = peaks[0]
    stream = torch.cuda.Stream()
    w = synth.WORKLOADS[args.workload]
    am, om = ADV_MODES[args.advantages], OPTIMIZERS[args.optimizer]
    head, ctx, obs_d = _measure(w, args, world, rank, local, stream, peaks, am, om)

    # rollout side: one policy step (forward + sampling) of the workload's N agents
    act_step = None
    if rank == 0 and not args.skip_policy_act:
        act_step = _policy_act_step(ctx, w, obs_d, stream)
    ctx.close()
    del obs_d
    torch.cuda.empty_cache()

    # the Mario-like update (T=128 x N=2048) as a second, launch-bound workload
    mario = None
    if args.workload != "mario" and not args.skip_mario:
        m, mctx, _ = _measure(synth.WORKLOADS["mario"], args, world, rank, local, stream, peaks,
                              am, om)
        mctx.close()
        mario = {k: m[k] for k in ("workload", "value", "ms_per_step", "e2e", "e2e_sync",
                                   "roofline", "gemm_all", "stages", "profiled_update_ms")}

    # GAE bandwidth stress (T=1024, N=65536): scan alone, and with moments + normalise
    gae = None
    if rank == 0 and not args.skip_gae_stress:
        gae = _gae_stress(stream, hbm_peak)

    adam = None
    if rank == 0 and not args.skip_adam_stress:
        adam = _adam_stress(stream, hbm_peak)

    rnn = rnn_upd = None
    if rank == 0 and not args.skip_rnn:
        rnn = {"bf16": _rnn_minibatch(stream, precision=1),
               "fp32": _rnn_minibatch(stream, precision=0)}
        rnn_upd = _rnn_update(stream)

    cpu = None
    if rank == 0 and world == 1 and not args.skip_cpu:
        cpu = _cpu_baseline(w, am, om)

    out = {
        "metric": "PPO update samples/s (GAE+clipped loss fwd/bwd+Adam); GAE GB/s vs HBM peak",
        "value": head["value"], "unit": "samples/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": head["ms_per_step"], "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16" if w.precision == "bf16" else "f32",
        "data": "synthetic (seeded mulberry32 rollout with the workload's shapes and value "
                "distributions; random-init weights)",
        "config": {"workload": head["workload"],
                   "global_batch": world * w.B, "parallelism": head["parallelism"],
                   "l2": "flushed between timed steps (256 MB write)",
                   "timing": "CUDA events per update on the launching stream, mean over steps"},
        "gpu_launches": head["launches_per_update"] * args.steps,
        "e2e": head["e2e"],
        "e2e_sync": head["e2e_sync"],
        "roofline": head["roofline"],
        "gemm_all": head["gemm_all"],
        "stages": head["stages"],
        "profiled_update_ms": head["profiled_update_ms"],
        "mario": mario,
        "gae_stress": gae,
        "adam_stress": adam,
        "policy_act": act_step,
        "rnn_minibatch": rnn,
        "rnn_update": rnn_upd,
        "cpu_baseline": cpu,
        "clocks": head["clocks"],
    }
    return out


def _gae_stress(stream, hbm_peak):
    import torch
    import policy_rl_gb300 as P
    T, N = 1024, 65536
    g = torch.Generator(device="cuda")
    g.manual_seed(0)
    with torch.cuda.stream(stream):
        rew = torch.randn(T, N, device="cuda", generator=g)
        val = torch.randn(T, N, device="cuda", generator=g)
        done = (torch.rand(T, N, device="cuda", generator=g) < 0.001).float()
        boot = torch.randn(N, device="cuda", generator=g)
        adv = torch.empty(T, N, device="cuda")
        ret = torch.empty(T, N, device="cuda")
        advn = torch.empty(T, N, device="cuda")
        st = torch.empty(4, device="cuda")
        work = torch.empty(P.ppo_gae_workspace_bytes(T, N), dtype=torch.uint8, device="cuda")
        res = {}
        for name, kw, bpe in (("scan", {}, 20), ("scan+moments+normalise",
                                                 dict(adv_norm=advn, stats=st, work=work), 28)):
            for _ in range(3):
                P.ppo_gae(rew, val, done, boot, 0.997, 0.95, adv, ret, stream=stream, **kw)
            evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                   for _ in range(10)]
            for s, e in evs:
                s.record(stream)
                P.ppo_gae(rew, val, done, boot, 0.997, 0.95, adv, ret, stream=stream, **kw)
                e.record(stream)
            stream.synchronize()
            t = float(np.mean([s.elapsed_time(e) for s, e in evs])) / 1e3
            gbs = bpe * T * N / t / 1e9
            res[name] = {"ms": round(t * 1e3, 4), "GB_per_s": round(gbs, 1),
                         "frac_of_hbm": round(gbs / hbm_peak, 4), "bytes_per_elem": bpe}
        # the same scan through ppo_segment_advantage (all N environments as
        # segments, values given, V-trace ratios off), with moments + normalise
        envs = torch.arange(N, dtype=torch.int32, device="cuda")
        swork = torch.empty(P.ppo_segment_advantage_workspace_bytes(), dtype=torch.uint8,
                            device="cuda")
        for _ in range(3):
            P.ppo_segment_advantage(rew, done, boot, envs, val, None, 0.997, 0.95, adv, ret,
                                    adv_norm=advn, stats=st, work=swork, stream=stream)
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(10)]
        for s0, e0 in evs:
            s0.record(stream)
            P.ppo_segment_advantage(rew, done, boot, envs, val, None, 0.997, 0.95, adv, ret,
                                    adv_norm=advn, stats=st, work=swork, stream=stream)
            e0.record(stream)
        stream.synchronize()
        t = float(np.mean([a.elapsed_time(b) for a, b in evs])) / 1e3
        gbs = 28 * T * N / t / 1e9
        res["segments+moments+normalise"] = {"ms": round(t * 1e3, 4), "GB_per_s": round(gbs, 1),
                                             "frac_of_hbm": round(gbs / hbm_peak, 4),
                                             "bytes_per_elem": 28}
    return {"workload": "gae_stress: T=1024 N=65536 fp32 (inputs > L2)", **res}


def _adam_stress(stream, hbm_peak):
    """Gradient-norm pass + Adam over 64M fp32 parameters (state 1 GB, far
    larger than L2): 4 B (norm) + 16 B read + 12 B written per parameter."""
    import torch
    import policy_rl_gb300 as P
    cfg = P.make_config(65536, 1024, 64, heads=(2,), precision=0, max_batch=1,
                        max_minibatch=1, max_epochs=1)
    ctx = P.Context(cfg)
    n = ctx.n_params
    with torch.cuda.stream(stream):
        ctx.grad.normal_()
        for _ in range(3):
            ctx.adam_step(1e-4, stream=stream)
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(10)]
        for s0, e0 in evs:
            s0.record(stream)
            ctx.adam_step(1e-4, stream=stream)
            e0.record(stream)
        stream.synchronize()
    t = float(np.mean([a.elapsed_time(b) for a, b in evs])) / 1e3
    ctx.close()
    gbs = 32 * n / t / 1e9
    return {"params": n, "ms": round(t * 1e3, 4), "GB_per_s": round(gbs, 1),
            "frac_of_hbm": round(gbs / hbm_peak, 4), "bytes_per_param": 32,
            "note": "ppo_adam_step: squared-norm pass + fused clip/Adam pass, fp32 mode"}


def _policy_act_step(ctx, w, obs_d, stream, reps=50):
    """ppo_policy_act on the first N rows of the rollout (one environment step
    of all N agents): pack + two forward GEMMs + head/sampling kernel."""
    import torch
    import policy_rl_gb300 as P
    N = w.N
    obs = obs_d[:N].contiguous()
    act = torch.empty(N, max(len(w.heads), 1), dtype=torch.int32, device="cuda")
    actc = torch.empty(N, max(w.n_gauss, 1), device="cuda")
    logp = torch.empty(N, device="cuda")
    val = torch.empty(N, device="cuda")
    K = len(w.heads) + 2 * w.n_gauss
    with torch.cuda.stream(stream):
        for i in range(5):
            P.ppo_policy_act(ctx.handle, obs, 1, i * N * K, act, actc if w.n_gauss else None,
                             logp, val, stream=stream)
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(reps)]
        for i, (s0, e0) in enumerate(evs):
            s0.record(stream)
            P.ppo_policy_act(ctx.handle, obs, 1, (5 + i) * N * K, act,
                             actc if w.n_gauss else None, logp, val, stream=stream)
            e0.record(stream)
        stream.synchronize()
    P.ppo_sync_status(ctx.handle, stream)
    t = float(np.median([a.elapsed_time(b) for a, b in evs])) / 1e3
    bf16 = w.precision == "bf16"
    return {"agents": N, "us_per_step": round(t * 1e6, 2), "agents_per_s": round(N / t, 1),
            "launches": 4 if bf16 else 3,
            "note": ("ppo_policy_act: pack obs, fwd1, fwd2 (tcgen05), head + sampling"
                     if bf16 else "ppo_policy_act: fwd1, fwd2 (CUDA cores), head + sampling")
                    + f"; median of {reps} steps, inputs resident, no L2 flush"}


def _rnn_inputs(T, N, D, H, L, heads, precision, gen_seed=0):
    import torch
    import policy_rl_gb300 as P
    cfg = P.make_rnn_config(D, H, L, heads, precision=precision)
    n = P.ppo_rnn_param_count(cfg)
    g = torch.Generator(device="cuda")
    g.manual_seed(gen_seed)
    d = {
        "params": torch.randn(n, device="cuda", generator=g) * 0.05,
        "obs": torch.randn(T * N, D, device="cuda", generator=g),
        "act": torch.stack([torch.randint(0, k, (T * N,), device="cuda", generator=g)
                            for k in heads], 1).int().contiguous(),
        "lp": torch.full((T * N,), -3.0, device="cuda"),
        "adv": torch.randn(T * N, device="cuda", generator=g),
        "ret": torch.randn(T * N, device="cuda", generator=g),
        "val": torch.randn(T, N, device="cuda", generator=g),
        "rew": (torch.rand(T, N, device="cuda", generator=g) < 0.02).float(),
        "done": (torch.rand(T, N, device="cuda", generator=g) < 0.004).float(),
        "boot": torch.randn(N, device="cuda", generator=g),
        "h0": torch.zeros(N, L, H, device="cuda"),
    }
    return cfg, n, d


def _rnn_minibatch(stream, reps=10, warm=3, precision=1):
    """ppo_rnn_loss_grad on a Mario-like minibatch with the pages' recurrent
    policy: 256 environment segments x T=128 (32,768 rows), 64-d observations,
    encoder to 128, four MinGRU layers, heads [9,2,2,2] + value."""
    import torch
    import policy_rl_gb300 as P
    T, N, ns, D, H, L = 128, 2048, 256, 64, 128, 4
    heads = (9, 2, 2, 2)
    with torch.cuda.stream(stream):
        cfg, n, d = _rnn_inputs(T, N, D, H, L, heads, precision)
        envs = torch.arange(ns, dtype=torch.int32, device="cuda")
        grad = torch.empty(n, device="cuda")
        work = torch.empty(P.ppo_rnn_workspace_bytes(cfg, T, ns), dtype=torch.uint8,
                           device="cuda")
        run = lambda: P.ppo_rnn_loss_grad(cfg, d["params"], envs, d["obs"], d["act"], None,
                                          d["lp"], d["adv"], d["ret"], d["done"], d["h0"], grad,
                                          work=work, stream=stream)
        for _ in range(warm):
            run()
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(reps)]
        for s0, e0 in evs:
            s0.record(stream)
            run()
            e0.record(stream)
        stream.synchronize()
    t = float(np.median([a.elapsed_time(b) for a, b in evs])) / 1e3
    rows = T * ns
    # products of one minibatch: forward (encoder, 2 per layer, decoder) and
    # backward (input and weight gradients)
    flops = rows * 2 * (D * H + L * 2 * H * H + 16 * H) * 3
    out = {"rows": rows, "ms_per_minibatch": round(t * 1e3, 3),
           "samples_per_s": round(rows / t, 1), "TFLOPs": round(flops / t / 1e12, 3),
           "note": ("ppo_rnn_loss_grad, bf16 tcgen05 products, fp32 scans" if precision
                    else "ppo_rnn_loss_grad, fp32 CUDA-core kernels") + f"; median of {reps}"}
    return out


def _rnn_update(stream, reps=5):
    """ppo_rnn_update of the Mario-like recurrent workload: T=128 x N=2048,
    4 epochs x 8 minibatches of 256 segments, bf16 products."""
    import torch
    import policy_rl_gb300 as P
    T, N, D, H, L, E, M = 128, 2048, 64, 128, 4, 4, 8
    heads = (9, 2, 2, 2)
    with torch.cuda.stream(stream):
        cfg, n, d = _rnn_inputs(T, N, D, H, L, heads, 1)
        ctx = P.RnnContext(cfg, d["params"].cpu().numpy(), max_T=T, max_N=N, max_epochs=E)
        run = lambda: ctx.update(d["obs"], d["act"], None, d["lp"], d["val"], d["rew"],
                                 d["done"], d["boot"], d["h0"], E, M, 0.99, 0.95, 2.5e-4, 7,
                                 stream=stream)
        run()
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(reps)]
        for s0, e0 in evs:
            s0.record(stream)
            run()
            e0.record(stream)
        stream.synchronize()
        ctx.sync_status(stream)
        ctx.close()
    t = float(np.median([a.elapsed_time(b) for a, b in evs])) / 1e3
    return {"workload": f"recurrent Mario-like: T={T} N={N} obs={D} MinGRU {L}x{H} heads "
                        f"{list(heads)}+V epochs={E} minibatches={M}",
            "ms_per_update": round(t * 1e3, 3), "samples_per_s": round(T * N / t, 1),
            "note": f"ppo_rnn_update, bf16 tcgen05 products; median of {reps}"}


def _oracle_update(ws, seed=0, adv_mode=0, optimizer=0):
    import oracle
    from policy_rl_gb300 import synth
    ro = synth.rollout(ws, seed=seed)
    p0 = synth.init_params(ws).astype(np.float64)
    net = oracle.Net(ws.obs_dim, ws.h1, ws.h2, ws.act, ws.heads, ws.n_gauss)
    hp = oracle.Hyper(gamma=ws.gamma, lam=ws.lam, clip=ws.clip, vf_coef=ws.vf_coef,
                      ent_coef=ws.ent_coef, lr=ws.lr, max_grad_norm=ws.max_grad_norm, seed=1234,
                      adv_mode=adv_mode, optimizer=optimizer)
    t0 = time.perf_counter()
    oracle.update(net, hp, ws.T, ws.N, ws.epochs, ws.minibatches, ro.obs, ro.act_disc,
                  ro.act_cont, ro.logp_old, ro.val, ro.rew, ro.done, ro.boot, p0)
    return time.perf_counter() - t0


def _slice(w, n):
    """The workload with N reduced to n environments (whole env segments per
    minibatch; the horizon, network, epochs and minibatches unchanged)."""
    n = max(n - n % w.minibatches, w.minibatches)
    return w.scaled(T=w.T, N=n, minibatches=w.minibatches, epochs=w.epochs)


def _sized_slice(w, budget_s, adv_mode, optimizer, max_n=None):
    """A slice of w whose oracle update takes about budget_s seconds (probe
    on the smallest slice, then scale N)."""
    probe = _slice(w, w.minibatches)
    per_sample = _oracle_update(probe, adv_mode=adv_mode, optimizer=optimizer) / probe.B
    n = int(budget_s / (per_sample * w.T))
    n = max(w.minibatches, min(n, max_n or w.N, w.N))
    return _slice(w, n)


def _cpu_baseline(w, adv_mode=0, optimizer=0):
    """The oracle (plain C fp64) on a bounded slice of the same workload: all
    host cores (OpenMP over the minibatch rows), and one core on a smaller
    slice."""
    import oracle
    cores = oracle.threads()
    ws = _sized_slice(w, 15.0, adv_mode, optimizer)
    t = _oracle_update(ws, adv_mode=adv_mode, optimizer=optimizer)
    oracle.set_threads(1)
    try:
        w1 = _sized_slice(w, 5.0, adv_mode, optimizer)
        t1 = _oracle_update(w1, adv_mode=adv_mode, optimizer=optimizer)
    finally:
        oracle.set_threads(cores)
    return {"value": round(ws.B / t, 1), "unit": "samples/s", "cores": cores, "kind": "oracle",
            "sample": f"whole update of a T={ws.T} x N={ws.N} slice ({ws.B} samples) of the "
                      f"{w.name} workload, {ws.epochs} epochs x {ws.minibatches} minibatches; "
                      f"plain C fp64, OpenMP over minibatch rows on {cores} threads ({t:.2f} s)",
            "single_thread": {"value": round(w1.B / t1, 1), "unit": "samples/s", "cores": 1,
                              "sample": f"T={w1.T} x N={w1.N} slice ({w1.B} samples), "
                                        f"{t1:.2f} s"}}


def _workload_str(w, advantages="global", optimizer="adam") -> str:
    mb = w.B // w.minibatches
    s = (f"{w.name}: T={w.T} N={w.N} obs={w.obs_dim} MLP {w.obs_dim}-{w.h1}-{w.h2} "
         f"{'tanh' if w.act == 0 else 'relu'} heads {list(w.heads)}+V epochs={w.epochs} "
         f"minibatches={w.minibatches} mb={mb}")
    if advantages != "global":
        s += (f" advantages={advantages} (per minibatch of {w.N // w.minibatches} env segments, "
              f"from fresh values)")
    if optimizer != "adam":
        s += f" optimizer={optimizer}"
    return s


def run_reference(args, world, rank):
    """The oracle timed on the host cores (OpenMP over minibatch rows), one
    bounded slice of the workload per step, sized so that the whole run
    (warm-up + timed steps) takes about two minutes."""
    import oracle
    from policy_rl_gb300 import synth
    w = synth.WORKLOADS[args.workload]
    am = ADV_MODES[args.advantages]
    om = OPTIMIZERS[args.optimizer]
    ws = _sized_slice(w, 120.0 / (args.steps + args.warmup), am, om)
    for i in range(args.warmup):
        _oracle_update(ws, seed=i, adv_mode=am, optimizer=om)
    times = [_oracle_update(ws, seed=args.warmup + i, adv_mode=am, optimizer=om)
             for i in range(args.steps)]
    t = float(np.mean(times))
    v = ws.B / t
    cores = oracle.threads()
    sample = (f"whole update of a T={ws.T} x N={ws.N} slice ({ws.B} samples) of the {w.name} "
              f"workload, {ws.epochs} epochs x {ws.minibatches} minibatches, per step; plain C "
              f"fp64, OpenMP over minibatch rows on {cores} threads")
    return {
        "impl": "reference",
        "metric": "PPO update samples/s (GAE+clipped loss fwd/bwd+Adam); GAE GB/s vs HBM peak",
        "value": round(v, 2), "unit": "samples/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(t * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": _workload_str(w, args.advantages, args.optimizer),
                   "global_batch": world * w.B,
                   "parallelism": "host cores (rank 0)",
                   "sample": f"oracle on a {ws.B}-sample slice per step (T={ws.T} x N={ws.N})"},
        "cpu_baseline": {"value": round(v, 2), "unit": "samples/s", "cores": cores,
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(v, 2), "unit": "samples/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def run_drive(args):
    """Plain driver loops for profilers (ncu launch lists and captures): no
    timing, no JSON line.
      minibatch: ppo_minibatch_loss_grad + ppo_adam_step, --reps times, on one
                 minibatch of --workload (random advantages, returns, indices);
      update:    ppo_update of --workload, --reps times;
      gae:       ppo_gae with moments + normalisation, T=--gae-T x N=--gae-N;
      adam:      ppo_adam_step over the 67.2 M parameters of a 65536-1024-64
                 fp32 network (1 GB of optimiser state);
      rnn:       ppo_rnn_loss_grad on the Mario-like recurrent minibatch (bf16);
      rnn_update: ppo_rnn_update of the Mario-like recurrent workload;
      muon:      ppo_muon_step on the network of --workload."""
    import torch
    import policy_rl_gb300 as P
    from policy_rl_gb300 import synth
    g = torch.Generator(device="cuda")
    g.manual_seed(0)
    if args.drive in ("minibatch", "update"):
        w = synth.WORKLOADS[args.workload]
        if args.drive_T:   # a shorter horizon: one minibatch of the same width
            w = w.scaled(T=args.drive_T, minibatches=max(1, w.minibatches * args.drive_T // w.T))
        B, mb = w.B, w.B // w.minibatches
        big = B * w.obs_dim > 2e8
        ro = synth.rollout(w, with_obs=not big)
        ctx = P.Context(P.config_from_workload(w, fused_loss=args.fused_loss),
                        synth.init_params(w))
        d = lambda x: torch.from_numpy(np.ascontiguousarray(x)).cuda()
        obs = torch.randn(B, w.obs_dim, device="cuda", generator=g) if big else d(ro.obs)
        if args.drive == "minibatch":
            adv = torch.randn(B, device="cuda", generator=g)
            ret = torch.randn(B, device="cuda", generator=g)
            idx = torch.randperm(B, device="cuda", generator=g)[:mb].to(torch.int32)
            a = [obs, d(ro.act_disc), d(ro.act_cont), d(ro.logp_old), adv, ret, idx]
            for _ in range(args.reps):
                ctx.minibatch_loss_grad(*a)
                ctx.adam_step(w.lr)
        else:
            a = [obs] + [d(x) for x in (ro.act_disc, ro.act_cont, ro.logp_old, ro.val, ro.rew,
                                        ro.done, ro.boot)]
            for _ in range(args.reps):
                ctx.update(*a, w.epochs, w.minibatches, w.gamma, w.lam, w.lr, 1234)
        ctx.sync_status()
        ctx.close()
    elif args.drive == "gae":
        T, N = args.gae_T, args.gae_N
        rew = torch.randn(T, N, device="cuda", generator=g)
        val = torch.randn(T, N, device="cuda", generator=g)
        done = (torch.rand(T, N, device="cuda", generator=g) < 0.001).float()
        boot = torch.randn(N, device="cuda", generator=g)
        adv, ret, advn = (torch.empty(T, N, device="cuda") for _ in range(3))
        st = torch.empty(4, device="cuda")
        work = torch.empty(P.ppo_gae_workspace_bytes(T, N), dtype=torch.uint8, device="cuda")
        for _ in range(args.reps):
            P.ppo_gae(rew, val, done, boot, 0.997, 0.95, adv, ret, advn, st, work)
    elif args.drive == "rnn":
        _rnn_minibatch(torch.cuda.current_stream(), reps=args.reps, warm=0)
    elif args.drive == "rnn_update":
        _rnn_update(torch.cuda.current_stream(), reps=args.reps)
    elif args.drive == "muon":
        w = synth.WORKLOADS[args.workload]
        ctx = P.Context(P.config_from_workload(w, optimizer=1), synth.init_params(w))
        ctx.grad.normal_(generator=g)
        for _ in range(args.reps):
            ctx.muon_step(w.lr)
        ctx.sync_status()
        ctx.close()
    elif args.drive == "adam":
        cfg = P.make_config(65536, 1024, 64, heads=(2,), precision=0, max_batch=1,
                            max_minibatch=1, max_epochs=1)
        ctx = P.Context(cfg)
        ctx.grad.normal_(generator=g)
        for _ in range(args.reps):
            ctx.adam_step(1e-4)
        ctx.sync_status()
        ctx.close()
    torch.cuda.synchronize()


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="large",
                    choices=["tiny", "mario", "ddnet", "large"])
    ap.add_argument("--advantages", default="global", choices=sorted(ADV_MODES),
                    help="global: GAE once per update (default); fresh_gae / vtrace: per "
                         "minibatch of env segments from fresh values")
    ap.add_argument("--optimizer", default="adam", choices=sorted(OPTIMIZERS),
                    help="adam (default) or muon (Newton-Schulz on the weight matrices)")
    ap.add_argument("--skip-cpu", action="store_true", help="omit the CPU-oracle baseline")
    ap.add_argument("--skip-gae-stress", action="store_true")
    ap.add_argument("--skip-adam-stress", action="store_true")
    ap.add_argument("--skip-policy-act", action="store_true")
    ap.add_argument("--skip-rnn", action="store_true")
    ap.add_argument("--skip-mario", action="store_true",
                    help="omit the Mario-like update measured beside the headline workload")
    ap.add_argument("--drive", choices=["minibatch", "update", "gae", "adam", "rnn",
                                        "rnn_update", "muon"],
                    help="plain driver loop for profilers (no timing, no JSON line)")
    ap.add_argument("--reps", type=int, default=3, help="--drive: repetitions")
    ap.add_argument("--fused-loss", type=int, default=0, choices=[-1, 0, 1],
                    help="--drive minibatch/update: the context's fused_loss (-1 two kernels, "
                         "0 the library's choice, 1 fused wherever it applies)")
    ap.add_argument("--drive-T", type=int, default=0,
                    help="--drive minibatch/update: horizon of a smaller rollout of the workload "
                         "(minibatch size kept)")
    ap.add_argument("--gae-T", type=int, default=1024, help="--drive gae: horizon")
    ap.add_argument("--gae-N", type=int, default=65536, help="--drive gae: environments")
    args = ap.parse_args()
    if args.drive:
        run_drive(args)
        return
    args.warmup = max(args.warmup, 3)
    world, rank, local = _dist()
    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args, world, rank)), flush=True)
        return
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    out = run_ours(args, world, rank, local)
    if rank == 0:
        print(json.dumps(out), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
