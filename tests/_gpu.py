"""Shared helpers of the GPU parity tests (marshalling only)."""
import numpy as np


def dev(x):
    import torch
    return torch.from_numpy(np.ascontiguousarray(x)).cuda()


def host(t):
    return t.detach().cpu().numpy()


def normwise(x, ref):
    """||x - ref||_2 / ||ref||_2 (0 when both vanish)."""
    x = np.asarray(x, np.float64).ravel()
    ref = np.asarray(ref, np.float64).ravel()
    d = np.linalg.norm(x - ref)
    n = np.linalg.norm(ref)
    return 0.0 if d == 0 else d / max(n, 1e-300)


def assert_elementwise(x, ref, rtol):
    """|x - ref| <= rtol * (|ref| + rms(ref)) element by element."""
    x = np.asarray(x, np.float64)
    ref = np.asarray(ref, np.float64)
    rms = float(np.sqrt(np.mean(ref * ref))) if ref.size else 0.0
    bad = np.abs(x - ref) > rtol * (np.abs(ref) + rms)
    if bad.any():
        i = np.flatnonzero(bad.ravel())[0]
        raise AssertionError(f"{bad.sum()} of {bad.size} elements differ; first at {i}: "
                             f"{x.ravel()[i]!r} vs {ref.ravel()[i]!r} (rms {rms:.3g})")


def param_slices(w):
    """name -> slice of the flat parameter vector."""
    D, H1, H2, C, G = w.obs_dim, w.h1, w.h2, w.out_cols, w.n_gauss
    sizes = [("W1", H1 * D), ("b1", H1), ("W2", H2 * H1), ("b2", H2), ("W3", C * H2),
             ("b3", C), ("logstd", G)]
    out, o = {}, 0
    for n, s in sizes:
        out[n] = slice(o, o + s)
        o += s
    return out


# log-ratio offsets given to the rows in turn: both clipped branches (-0.5,
# +0.5), both unclipped sides (-0.1, +0.1) and r = 1; every one lies at least
# 0.08 in log space from the clip boundaries log(0.8) and log(1.2), far more
# than the bf16 path's log-probability error (~1e-3), so the GPU and the
# oracle take the same clip branch on every row.
LOG_RATIO_OFFSETS = (-0.5, -0.1, 0.0, 0.1, 0.5)


def conditioned_logp_old(w, ro, params):
    """logp_old = (oracle log-probability at params) - offset, per row."""
    import oracle
    net = oracle.Net(w.obs_dim, w.h1, w.h2, w.act, w.heads, w.n_gauss)
    lp, _ = oracle.policy_logp(net, np.asarray(params, np.float64), ro.obs, ro.act_disc,
                               ro.act_cont)
    off = np.array(LOG_RATIO_OFFSETS)[np.arange(lp.size) % len(LOG_RATIO_OFFSETS)]
    return (lp - off).astype(np.float32)


MODES = ("fused", "per_stage", "fused_loss", "persistent")


def mode_kwargs(mode):
    """Context options of the bf16 minibatch paths: forward, loss and
    backward-data fused in one kernel (where the network fits it); one kernel
    per GEMM stage; the same with head + loss and layer-2 backward-data in one
    kernel (the default where H2 = 256 or 512 with 16 head columns); and the
    persistent cooperative kernel."""
    return {"fused": {"fused_mlp": 1}, "per_stage": {"fused_loss": -1},
            "fused_loss": {"fused_loss": 1},
            "persistent": {"persistent_minibatch": 1}}[mode]


def fused_applies(w):
    Dp = -(-w.obs_dim // 64) * 64
    return (w.precision == "bf16" and Dp == 64 and w.h1 in (128, 256) and w.h2 in (128, 256)
            and w.out_cols <= 32 and w.n_gauss <= 4)
