"""GB300 (sm_103a) PPO learner step: Python binding of ``include/ppo.h``.

The functions here carry the C ABI's names and only marshal arguments: torch
tensors supply device memory (``data_ptr()``) and the current CUDA stream;
every step of the computation runs in the library's CUDA kernels.  There is
no CPU fallback -- without the built library (``policy_rl_gb300.build``) or
an sm_103a device every call raises.
"""
from __future__ import annotations

import ctypes
from dataclasses import dataclass

from . import _abi
from ._abi import PpoConfig, PpoError, RnnConfig

__all__ = [
    "PpoConfig", "PpoError", "Context", "make_config", "ppo_param_count", "ppo_gae",
    "ppo_gae_workspace_bytes", "ppo_gae_noalloc", "ppo_minibatch_perm", "ppo_perm_workspace_bytes",
    "ppo_segment_advantage", "ppo_segment_advantage_workspace_bytes",
    "ppo_minibatch_loss_grad_fresh", "ppo_policy_act", "ppo_muon_step", "RnnConfig",
    "make_rnn_config", "ppo_rnn_param_count", "ppo_rnn_workspace_bytes", "ppo_rnn_loss_grad",
    "ppo_create", "ppo_destroy", "ppo_buffers", "ppo_params_changed", "ppo_get_step",
    "ppo_minibatch_loss_grad", "ppo_adam_step", "ppo_update", "ppo_update_host",
    "ppo_update_host_async", "ppo_host_wait",
    "ppo_sync_status", "ppo_stage_name", "ppo_update_profile", "ppo_set_step_trace",
    "ppo_set_wait_limit", "ppo_set_collective", "TorchCollective", "RnnContext",
    "library_path",
]


def library_path() -> str:
    return _abi.LIB_PATH


def _lib():
    return _abi.load()


def _ptr(t):
    """Device (or host) address of a tensor / numpy array, None for None."""
    if t is None:
        return None
    if hasattr(t, "data_ptr"):
        if not t.is_contiguous():
            raise ValueError("tensor must be contiguous")
        return ctypes.c_void_p(t.data_ptr())
    if hasattr(t, "ctypes"):
        return ctypes.c_void_p(t.ctypes.data)
    return ctypes.c_void_p(int(t))


def _stream(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def make_config(obs_dim, h1, h2, act=0, heads=(3, 2, 2), n_gauss=0, precision=1, clip=0.2,
                vf_coef=0.5, ent_coef=0.01, beta1=0.9, beta2=0.999, adam_eps=1e-8,
                max_grad_norm=0.5, max_batch=1, max_minibatch=1, max_epochs=1,
                persistent_minibatch=0, fused_mlp=0, fused_loss=0, adv_mode=0,
                vtrace_rho_clip=1.0, vtrace_c_clip=1.0, optimizer=0, muon_lr=0.02,
                muon_beta=0.95) -> PpoConfig:
    hn = (ctypes.c_int32 * _abi.MAX_HEADS)(*(list(heads) + [0] * (_abi.MAX_HEADS - len(heads))))
    return PpoConfig(obs_dim, h1, h2, act, len(heads), hn, n_gauss, precision, clip, vf_coef,
                     ent_coef, max_grad_norm, beta1, beta2, adam_eps, max_batch, max_minibatch,
                     max_epochs, persistent_minibatch, fused_mlp, fused_loss, adv_mode,
                     vtrace_rho_clip, vtrace_c_clip, optimizer, muon_lr, muon_beta)


def config_from_workload(w, max_batch=None, max_minibatch=None, max_epochs=None,
                         persistent_minibatch=0, fused_mlp=0, fused_loss=0, adv_mode=0,
                         vtrace_rho_clip=1.0, vtrace_c_clip=1.0, optimizer=0, muon_lr=0.02,
                         muon_beta=0.95) -> PpoConfig:
    B = w.T * w.N
    return make_config(w.obs_dim, w.h1, w.h2, w.act, tuple(w.heads), w.n_gauss,
                       1 if w.precision == "bf16" else 0, w.clip, w.vf_coef, w.ent_coef,
                       max_grad_norm=w.max_grad_norm, max_batch=max_batch or B,
                       max_minibatch=max_minibatch or B // w.minibatches,
                       max_epochs=max_epochs or w.epochs,
                       persistent_minibatch=persistent_minibatch,
                       fused_mlp=fused_mlp, fused_loss=fused_loss, adv_mode=adv_mode,
                       vtrace_rho_clip=vtrace_rho_clip, vtrace_c_clip=vtrace_c_clip,
                       optimizer=optimizer, muon_lr=muon_lr, muon_beta=muon_beta)


# ---- free functions -----------------------------------------------------------
def ppo_param_count(cfg: PpoConfig) -> int:
    n = ctypes.c_int64()
    _abi.check(_lib().ppo_param_count(ctypes.byref(cfg), ctypes.byref(n)), "ppo_param_count")
    return n.value


def ppo_gae_workspace_bytes(T: int, N: int) -> int:
    n = ctypes.c_size_t()
    _abi.check(_lib().ppo_gae_workspace_bytes(T, N, ctypes.byref(n)), "ppo_gae_workspace_bytes")
    return n.value


def ppo_gae(rew, val, done, boot, gamma, lam, adv, ret, adv_norm=None, stats=None, work=None,
            stream=None) -> None:
    T, N = rew.shape
    wb = work.numel() * work.element_size() if work is not None else 0
    _abi.check(_lib().ppo_gae(_ptr(rew), _ptr(val), _ptr(done), _ptr(boot), T, N, gamma, lam,
                              _ptr(adv), _ptr(ret), _ptr(adv_norm), _ptr(stats), _ptr(work), wb,
                              _stream(stream)), "ppo_gae")


def ppo_gae_noalloc(rew, val, done, boot, gamma, lam, adv, ret, adv_norm=None, stats=None,
                    stream=None) -> None:
    """ppo_gae for callers that cannot allocate device memory (see ppo.h)."""
    T, N = rew.shape
    _abi.check(_lib().ppo_gae_noalloc(_ptr(rew), _ptr(val), _ptr(done), _ptr(boot), T, N, gamma,
                                      lam, _ptr(adv), _ptr(ret), _ptr(adv_norm), _ptr(stats),
                                      _stream(stream)), "ppo_gae_noalloc")


def ppo_segment_advantage_workspace_bytes() -> int:
    n = ctypes.c_size_t()
    _abi.check(_lib().ppo_segment_advantage_workspace_bytes(ctypes.byref(n)),
               "ppo_segment_advantage_workspace_bytes")
    return n.value


def ppo_segment_advantage(rew, done, boot, envs, val, ratio, gamma, lam, adv, ret,
                          rho_clip=1.0, c_clip=1.0, adv_norm=None, stats=None, work=None,
                          stream=None) -> None:
    """GAE / V-trace advantages of the environment segments ``envs`` (see ppo.h)."""
    T, N = rew.shape
    ns = envs.numel()
    wb = work.numel() * work.element_size() if work is not None else 0
    _abi.check(_lib().ppo_segment_advantage(
        _ptr(rew), _ptr(done), _ptr(boot), T, N, _ptr(envs), ns, _ptr(val), _ptr(ratio), gamma,
        lam, rho_clip, c_clip, _ptr(adv), _ptr(ret), _ptr(adv_norm), _ptr(stats), _ptr(work), wb,
        _stream(stream)), "ppo_segment_advantage")


def ppo_perm_workspace_bytes(B: int) -> int:
    n = ctypes.c_size_t()
    _abi.check(_lib().ppo_perm_workspace_bytes(B, ctypes.byref(n)), "ppo_perm_workspace_bytes")
    return n.value


def ppo_minibatch_perm(seed, epoch, B, perm, work, stream=None) -> None:
    wb = work.numel() * work.element_size()
    _abi.check(_lib().ppo_minibatch_perm(seed & 0xFFFFFFFF, epoch, B, _ptr(perm), _ptr(work), wb,
                                         _stream(stream)), "ppo_minibatch_perm")


def make_rnn_config(obs_dim, hidden=128, layers=4, heads=(3, 2, 2), n_gauss=0, clip=0.2,
                    vf_coef=0.5, ent_coef=0.01, precision=0, max_grad_norm=0.5, beta1=0.9,
                    beta2=0.999, adam_eps=1e-8) -> RnnConfig:
    hn = (ctypes.c_int32 * _abi.MAX_HEADS)(*(list(heads) + [0] * (_abi.MAX_HEADS - len(heads))))
    return RnnConfig(obs_dim, hidden, layers, len(heads), hn, n_gauss, clip, vf_coef, ent_coef,
                     precision, max_grad_norm, beta1, beta2, adam_eps)


def ppo_rnn_param_count(cfg: RnnConfig) -> int:
    n = ctypes.c_int64()
    _abi.check(_lib().ppo_rnn_param_count(ctypes.byref(cfg), ctypes.byref(n)),
               "ppo_rnn_param_count")
    return n.value


def ppo_rnn_workspace_bytes(cfg: RnnConfig, T: int, ns: int) -> int:
    n = ctypes.c_size_t()
    _abi.check(_lib().ppo_rnn_workspace_bytes(ctypes.byref(cfg), T, ns, ctypes.byref(n)),
               "ppo_rnn_workspace_bytes")
    return n.value


def ppo_rnn_loss_grad(cfg: RnnConfig, params, envs, obs, act_disc, act_cont, logp_old, adv, ret,
                      done, h0, grad, adv_stats=None, stats6=None, work=None, stream=None) -> None:
    """Loss and BPTT gradient of the recurrent policy over the segments envs (see ppo.h)."""
    T, N = done.shape
    wb = work.numel() * work.element_size() if work is not None else 0
    _abi.check(_lib().ppo_rnn_loss_grad(
        ctypes.byref(cfg), _ptr(params), T, N, _ptr(envs), envs.numel(), _ptr(obs),
        _ptr(act_disc), _ptr(act_cont), _ptr(logp_old), _ptr(adv), _ptr(ret), _ptr(adv_stats),
        _ptr(done), _ptr(h0), _ptr(grad), _ptr(stats6), _ptr(work), wb, _stream(stream)),
        "ppo_rnn_loss_grad")


class RnnContext:
    """Owns one ppo_rnn_ctx: the recurrent policy's parameters, gradient, Adam
    state and update workspaces (see ppo.h, ppo_rnn_update)."""

    def __init__(self, cfg: RnnConfig, init_params=None, max_T=1, max_N=1, max_epochs=1):
        import numpy as np
        self.cfg = cfg
        self.n_params = ppo_rnn_param_count(cfg)
        h = ctypes.c_void_p()
        ip = None if init_params is None else np.ascontiguousarray(init_params, np.float32)
        _abi.check(_lib().ppo_rnn_create(ctypes.byref(cfg), _ptr(ip), max_T, max_N, max_epochs,
                                         ctypes.byref(h)), "ppo_rnn_create")
        self.handle = h
        ps = [ctypes.c_void_p() for _ in range(4)]
        _abi.check(_lib().ppo_rnn_buffers(h, *[ctypes.byref(p) for p in ps]), "ppo_rnn_buffers")
        import torch
        self.params, self.grad, self.adam_m, self.adam_v = (
            torch.as_tensor(_DevArray(p.value, self.n_params), device="cuda") for p in ps)

    def update(self, obs, act_disc, act_cont, logp_old, val, rew, done, boot, h0, epochs,
               minibatches, gamma, lam, lr, seed, stats=None, stream=None):
        T, N = val.shape
        _abi.check(_lib().ppo_rnn_update(
            self.handle, _ptr(obs), _ptr(act_disc), _ptr(act_cont), _ptr(logp_old), _ptr(val),
            _ptr(rew), _ptr(done), _ptr(boot), _ptr(h0), T, N, epochs, minibatches, gamma, lam,
            lr, seed & 0xFFFFFFFF, _ptr(stats), _stream(stream)), "ppo_rnn_update")

    def sync_status(self, stream=None):
        _abi.check(_lib().ppo_rnn_sync_status(self.handle, _stream(stream)),
                   "ppo_rnn_sync_status")

    def close(self):
        if self.handle is not None:
            _lib().ppo_rnn_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


# ---- context ------------------------------------------------------------------
def ppo_create(cfg: PpoConfig, init_params=None):
    h = ctypes.c_void_p()
    if init_params is not None:
        import numpy as np
        init_params = np.ascontiguousarray(init_params, dtype=np.float32)
    _abi.check(_lib().ppo_create(ctypes.byref(cfg), _ptr(init_params), ctypes.byref(h)),
               "ppo_create")
    return h


def ppo_destroy(ctx) -> None:
    _abi.check(_lib().ppo_destroy(ctx), "ppo_destroy")


class _DevArray:
    """Zero-copy view of library-owned device memory (CUDA array interface)."""

    def __init__(self, ptr: int, n: int, typestr: str = "<f4"):
        self.__cuda_array_interface__ = {"shape": (n,), "typestr": typestr,
                                         "data": (ptr, False), "version": 3, "strides": None}


def ppo_buffers(ctx, n_params: int):
    """Torch views (params, grad, adam_m, adam_v) of the context's buffers."""
    import torch
    ps = [ctypes.c_void_p() for _ in range(4)]
    _abi.check(_lib().ppo_buffers(ctx, *[ctypes.byref(p) for p in ps]), "ppo_buffers")
    return tuple(torch.as_tensor(_DevArray(p.value, n_params), device="cuda") for p in ps)


def ppo_params_changed(ctx, stream=None) -> None:
    _abi.check(_lib().ppo_params_changed(ctx, _stream(stream)), "ppo_params_changed")


def ppo_get_step(ctx) -> int:
    n = ctypes.c_int64()
    _abi.check(_lib().ppo_get_step(ctx, ctypes.byref(n)), "ppo_get_step")
    return n.value


def ppo_minibatch_loss_grad(ctx, obs, act_disc, act_cont, logp_old, adv, ret, idx,
                            adv_stats=None, stats6=None, stream=None) -> None:
    B = obs.shape[0]
    _abi.check(_lib().ppo_minibatch_loss_grad(
        ctx, _ptr(obs), _ptr(act_disc), _ptr(act_cont), _ptr(logp_old), _ptr(adv), _ptr(ret),
        _ptr(idx), B, idx.numel(), _ptr(adv_stats), _ptr(stats6), _stream(stream)),
        "ppo_minibatch_loss_grad")


def ppo_minibatch_loss_grad_fresh(ctx, obs, act_disc, act_cont, logp_old, rew, done, boot, envs,
                                  adv_mode, gamma, lam, stats6=None, adv_out=None, ret_out=None,
                                  stream=None) -> None:
    T, N = rew.shape
    _abi.check(_lib().ppo_minibatch_loss_grad_fresh(
        ctx, _ptr(obs), _ptr(act_disc), _ptr(act_cont), _ptr(logp_old), _ptr(rew), _ptr(done),
        _ptr(boot), T, N, _ptr(envs), envs.numel(), adv_mode, gamma, lam, _ptr(stats6),
        _ptr(adv_out), _ptr(ret_out), _stream(stream)), "ppo_minibatch_loss_grad_fresh")


def ppo_policy_act(ctx, obs, seed, draw0, act_disc, act_cont=None, logp=None, value=None,
                   stream=None) -> None:
    """Sampled actions, their log-probability and the value for the rows of obs."""
    _abi.check(_lib().ppo_policy_act(
        ctx, _ptr(obs), obs.shape[0], seed & 0xFFFFFFFF, int(draw0), _ptr(act_disc),
        _ptr(act_cont), _ptr(logp), _ptr(value), _stream(stream)), "ppo_policy_act")


def ppo_muon_step(ctx, lr, grad_norm=None, stream=None) -> None:
    _abi.check(_lib().ppo_muon_step(ctx, lr, _ptr(grad_norm), _stream(stream)), "ppo_muon_step")


def ppo_adam_step(ctx, lr, grad_norm=None, stream=None) -> None:
    _abi.check(_lib().ppo_adam_step(ctx, lr, _ptr(grad_norm), _stream(stream)), "ppo_adam_step")


def ppo_update(ctx, obs, act_disc, act_cont, logp_old, val, rew, done, boot, epochs,
               minibatches, gamma, lam, lr, seed, stats=None, stream=None) -> None:
    T, N = val.shape
    _abi.check(_lib().ppo_update(
        ctx, _ptr(obs), _ptr(act_disc), _ptr(act_cont), _ptr(logp_old), _ptr(val), _ptr(rew),
        _ptr(done), _ptr(boot), T, N, epochs, minibatches, gamma, lam, lr, seed & 0xFFFFFFFF,
        _ptr(stats), _stream(stream)), "ppo_update")


def ppo_update_host(ctx, obs, act_disc, act_cont, logp_old, val, rew, done, boot, epochs,
                    minibatches, gamma, lam, lr, seed, stats=None, stream=None) -> None:
    T, N = val.shape
    _abi.check(_lib().ppo_update_host(
        ctx, _ptr(obs), _ptr(act_disc), _ptr(act_cont), _ptr(logp_old), _ptr(val), _ptr(rew),
        _ptr(done), _ptr(boot), T, N, epochs, minibatches, gamma, lam, lr, seed & 0xFFFFFFFF,
        _ptr(stats), _stream(stream)), "ppo_update_host")


def ppo_update_host_async(ctx, obs, act_disc, act_cont, logp_old, val, rew, done, boot, epochs,
                          minibatches, gamma, lam, lr, seed, stats=None, stream=None) -> None:
    T, N = val.shape
    _abi.check(_lib().ppo_update_host_async(
        ctx, _ptr(obs), _ptr(act_disc), _ptr(act_cont), _ptr(logp_old), _ptr(val), _ptr(rew),
        _ptr(done), _ptr(boot), T, N, epochs, minibatches, gamma, lam, lr, seed & 0xFFFFFFFF,
        _ptr(stats), _stream(stream)), "ppo_update_host_async")


def ppo_host_wait(ctx) -> None:
    _abi.check(_lib().ppo_host_wait(ctx), "ppo_host_wait")


def ppo_stage_name(stage: int) -> str:
    return _lib().ppo_stage_name(stage).decode()


def ppo_update_profile(ctx, obs, act_disc, act_cont, logp_old, val, rew, done, boot, epochs,
                       minibatches, gamma, lam, lr, seed, stats=None, stream=None):
    """One profiled update; returns {stage name: (total ms, launches)}."""
    T, N = val.shape
    ms = (ctypes.c_float * _abi.NUM_STAGES)()
    cnt = (ctypes.c_int32 * _abi.NUM_STAGES)()
    _abi.check(_lib().ppo_update_profile(
        ctx, _ptr(obs), _ptr(act_disc), _ptr(act_cont), _ptr(logp_old), _ptr(val), _ptr(rew),
        _ptr(done), _ptr(boot), T, N, epochs, minibatches, gamma, lam, lr, seed & 0xFFFFFFFF,
        _ptr(stats), ms, cnt, _stream(stream)), "ppo_update_profile")
    return {ppo_stage_name(i): (ms[i], cnt[i]) for i in range(_abi.NUM_STAGES) if cnt[i]}


def ppo_sync_status(ctx, stream=None) -> None:
    _abi.check(_lib().ppo_sync_status(ctx, _stream(stream)), "ppo_sync_status")


def ppo_set_collective(ctx, world: int, rank: int, fn=None, user=None) -> None:
    """Registers the collective of the data-parallel update (see ppo.h); fn is
    an _abi.COLLECTIVE_FN (e.g. TorchCollective(...).fn)."""
    cfn = fn if fn is not None else ctypes.cast(None, _abi.COLLECTIVE_FN)
    _abi.check(_lib().ppo_set_collective(ctx, world, rank, cfn, user), "ppo_set_collective")


class TorchCollective:
    """The library's collective over torch.distributed: an in-place sum
    all-reduce of fp32 buffers and an all-gather of fp64 buffers, issued on
    the stream the library passes (so that they are ordered with its
    kernels).  device: "cuda" (NCCL; buffers are device pointers) or "cpu"
    (gloo; host pointers).  Keep the object alive while the context uses it."""

    def __init__(self, group=None, device: str = "cuda"):
        self.group = group
        self.device = device
        self.fn = _abi.COLLECTIVE_FN(self._call)
        self.error = None

    def _view(self, ptr: int, n: int, fp64: bool):
        import torch
        if self.device == "cuda":
            return torch.as_tensor(_DevArray(ptr, n, "<f8" if fp64 else "<f4"), device="cuda")
        import numpy as np
        ct = ctypes.c_double if fp64 else ctypes.c_float
        return torch.from_numpy(np.ctypeslib.as_array((ct * n).from_address(ptr)))

    def _call(self, user, op, buf, count, stream):
        try:
            import contextlib
            import torch
            import torch.distributed as dist
            world = dist.get_world_size(self.group)
            rank = dist.get_rank(self.group)
            # the library's stream (the legacy default stream arrives as NULL)
            if self.device != "cuda":
                ctxm = contextlib.nullcontext()
            else:
                ctxm = torch.cuda.stream(torch.cuda.ExternalStream(stream) if stream
                                         else torch.cuda.default_stream())
            with ctxm:
                if op == _abi.COLL_ALLREDUCE_SUM_F32:
                    dist.all_reduce(self._view(buf, count, False), group=self.group)
                elif op == _abi.COLL_ALLGATHER_F64:
                    t = self._view(buf, world * count, True)
                    parts = list(t.split(count))
                    mine = parts[rank].clone()
                    dist.all_gather(parts, mine, group=self.group)
                else:
                    return 1
            return 0
        except Exception as e:   # reported to the library as a failed collective
            self.error = e
            return 1


def ppo_set_step_trace(ctx, trace=None, max_steps: int = 0) -> None:
    """Per-step copies of params, m, v and the gradient inside ppo_update (see ppo.h)."""
    _abi.check(_lib().ppo_set_step_trace(ctx, _ptr(trace), max_steps), "ppo_set_step_trace")


def ppo_set_wait_limit(ctx, limit_ns: int = 0) -> None:
    """Limit of the cooperative kernels' grid-barrier waits (0: the 2 s default)."""
    _abi.check(_lib().ppo_set_wait_limit(ctx, int(limit_ns)), "ppo_set_wait_limit")


class Context:
    """Owns one ppo_ctx (parameters, gradient, Adam state, workspaces)."""

    def __init__(self, cfg: PpoConfig, init_params=None):
        self.cfg = cfg
        self.n_params = ppo_param_count(cfg)
        self.handle = ppo_create(cfg, init_params)
        self.params, self.grad, self.adam_m, self.adam_v = ppo_buffers(self.handle, self.n_params)

    def close(self):
        if self.handle is not None:
            ppo_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def minibatch_loss_grad(self, *a, **k):
        return ppo_minibatch_loss_grad(self.handle, *a, **k)

    def minibatch_loss_grad_fresh(self, *a, **k):
        return ppo_minibatch_loss_grad_fresh(self.handle, *a, **k)

    def policy_act(self, *a, **k):
        return ppo_policy_act(self.handle, *a, **k)

    def muon_step(self, *a, **k):
        return ppo_muon_step(self.handle, *a, **k)

    def adam_step(self, *a, **k):
        return ppo_adam_step(self.handle, *a, **k)

    def update(self, *a, **k):
        return ppo_update(self.handle, *a, **k)

    def update_host(self, *a, **k):
        return ppo_update_host(self.handle, *a, **k)

    def update_host_async(self, *a, **k):
        return ppo_update_host_async(self.handle, *a, **k)

    def host_wait(self):
        return ppo_host_wait(self.handle)

    def update_profile(self, *a, **k):
        return ppo_update_profile(self.handle, *a, **k)

    def sync_status(self, stream=None):
        return ppo_sync_status(self.handle, stream)

    def params_changed(self, stream=None):
        return ppo_params_changed(self.handle, stream)

    def step(self) -> int:
        return ppo_get_step(self.handle)

    def set_step_trace(self, trace=None, max_steps: int = 0):
        return ppo_set_step_trace(self.handle, trace, max_steps)

    def set_wait_limit(self, limit_ns: int = 0):
        return ppo_set_wait_limit(self.handle, limit_ns)

    def set_collective(self, world: int, rank: int, collective=None):
        """Data-parallel update over `world` ranks (collective: a
        TorchCollective, or None with world == 1)."""
        self._collective = collective   # kept alive with the context
        return ppo_set_collective(self.handle, world, rank,
                                  collective.fn if collective is not None else None)
