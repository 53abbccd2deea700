"""ctypes declarations of the C ABI in ``include/ppo.h``.

The shared library is built in-tree (``policy_rl_gb300/_build/libppo_gb300.so``,
see ``policy_rl_gb300.build``).  There is no fallback: if the library is
missing every call raises ``RuntimeError`` naming the build command.
"""
from __future__ import annotations

import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "_build", "libppo_gb300.so")
MAX_HEADS = 8

# exported symbols, in the order ppo.h declares them
SYMBOLS = (
    "ppo_status_string", "ppo_create", "ppo_destroy", "ppo_param_count", "ppo_buffers",
    "ppo_params_changed", "ppo_get_step", "ppo_gae_workspace_bytes", "ppo_gae",
    "ppo_gae_noalloc", "ppo_segment_advantage_workspace_bytes", "ppo_segment_advantage",
    "ppo_perm_workspace_bytes", "ppo_minibatch_perm", "ppo_minibatch_loss_grad",
    "ppo_minibatch_loss_grad_fresh", "ppo_policy_act", "ppo_adam_step", "ppo_muon_step",
    "ppo_rnn_param_count", "ppo_rnn_workspace_bytes", "ppo_rnn_loss_grad", "ppo_rnn_create",
    "ppo_rnn_destroy", "ppo_rnn_buffers", "ppo_rnn_update", "ppo_rnn_sync_status", "ppo_update",
    "ppo_update_host", "ppo_update_host_async", "ppo_host_wait", "ppo_stage_name",
    "ppo_update_profile", "ppo_sync_status", "ppo_set_collective", "ppo_set_step_trace",
    "ppo_set_wait_limit",
)
NUM_STAGES = 34
NUM_KERNEL_STAGES = 25

STATUS = {0: "PPO_OK", 1: "PPO_ERR_INVALID", 2: "PPO_ERR_ALIGN", 3: "PPO_ERR_CUDA",
          4: "PPO_ERR_UNSUPPORTED", 5: "PPO_ERR_TIMEOUT", 6: "PPO_ERR_NOMEM"}


class PpoError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {STATUS.get(status, status)}")


class PpoConfig(ctypes.Structure):
    _fields_ = [
        ("obs_dim", ctypes.c_int32), ("h1", ctypes.c_int32), ("h2", ctypes.c_int32),
        ("act", ctypes.c_int32), ("n_heads", ctypes.c_int32),
        ("head_n", ctypes.c_int32 * MAX_HEADS), ("n_gauss", ctypes.c_int32),
        ("precision", ctypes.c_int32), ("clip", ctypes.c_float), ("vf_coef", ctypes.c_float),
        ("ent_coef", ctypes.c_float), ("max_grad_norm", ctypes.c_float),
        ("beta1", ctypes.c_double), ("beta2", ctypes.c_double), ("adam_eps", ctypes.c_double),
        ("max_batch", ctypes.c_int64), ("max_minibatch", ctypes.c_int64),
        ("max_epochs", ctypes.c_int32), ("persistent_minibatch", ctypes.c_int32),
        ("fused_mlp", ctypes.c_int32), ("fused_loss", ctypes.c_int32),
        ("adv_mode", ctypes.c_int32), ("vtrace_rho_clip", ctypes.c_float),
        ("vtrace_c_clip", ctypes.c_float), ("optimizer", ctypes.c_int32),
        ("muon_lr", ctypes.c_float), ("muon_beta", ctypes.c_float),
    ]


class RnnConfig(ctypes.Structure):
    _fields_ = [
        ("obs_dim", ctypes.c_int32), ("hidden", ctypes.c_int32), ("layers", ctypes.c_int32),
        ("n_heads", ctypes.c_int32), ("head_n", ctypes.c_int32 * MAX_HEADS),
        ("n_gauss", ctypes.c_int32), ("clip", ctypes.c_float), ("vf_coef", ctypes.c_float),
        ("ent_coef", ctypes.c_float), ("precision", ctypes.c_int32),
        ("max_grad_norm", ctypes.c_float), ("beta1", ctypes.c_double),
        ("beta2", ctypes.c_double), ("adam_eps", ctypes.c_double),
    ]


_P = ctypes.c_void_p
_I64 = ctypes.c_int64

# ppo_collective_fn: int (*)(void* user, int32_t op, void* d_buf, int64_t count, cudaStream_t)
COLLECTIVE_FN = ctypes.CFUNCTYPE(ctypes.c_int, ctypes.c_void_p, ctypes.c_int32, ctypes.c_void_p,
                                 ctypes.c_int64, ctypes.c_void_p)
COLL_ALLREDUCE_SUM_F32 = 0
COLL_ALLGATHER_F64 = 1
_F = ctypes.c_float
_SZ = ctypes.c_size_t
_lib = None


def load(path: str = LIB_PATH):
    """Loads the library once and declares every entry point."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(
            f"policy_rl_gb300: CUDA library not built ({path} missing); run "
            "`python -c 'import __graft_entry__ as g; g.build()'` or "
            "`python -m policy_rl_gb300.build`")
    L = ctypes.CDLL(path)
    i32, u32 = ctypes.c_int32, ctypes.c_uint32
    sig = {
        "ppo_status_string": ([ctypes.c_int], ctypes.c_char_p),
        "ppo_create": ([ctypes.POINTER(PpoConfig), _P, ctypes.POINTER(_P)], ctypes.c_int),
        "ppo_destroy": ([_P], ctypes.c_int),
        "ppo_param_count": ([ctypes.POINTER(PpoConfig), ctypes.POINTER(_I64)], ctypes.c_int),
        "ppo_buffers": ([_P, ctypes.POINTER(_P), ctypes.POINTER(_P), ctypes.POINTER(_P),
                         ctypes.POINTER(_P)], ctypes.c_int),
        "ppo_params_changed": ([_P, _P], ctypes.c_int),
        "ppo_get_step": ([_P, ctypes.POINTER(_I64)], ctypes.c_int),
        "ppo_gae_workspace_bytes": ([_I64, _I64, ctypes.POINTER(_SZ)], ctypes.c_int),
        "ppo_gae": ([_P, _P, _P, _P, _I64, _I64, _F, _F, _P, _P, _P, _P, _P, _SZ, _P],
                    ctypes.c_int),
        "ppo_gae_noalloc": ([_P, _P, _P, _P, _I64, _I64, _F, _F, _P, _P, _P, _P, _P],
                            ctypes.c_int),
        "ppo_segment_advantage_workspace_bytes": ([ctypes.POINTER(_SZ)], ctypes.c_int),
        "ppo_segment_advantage": ([_P, _P, _P, _I64, _I64, _P, _I64, _P, _P, _F, _F, _F, _F,
                                   _P, _P, _P, _P, _P, _SZ, _P], ctypes.c_int),
        "ppo_perm_workspace_bytes": ([_I64, ctypes.POINTER(_SZ)], ctypes.c_int),
        "ppo_minibatch_perm": ([u32, _I64, _I64, _P, _P, _SZ, _P], ctypes.c_int),
        "ppo_minibatch_loss_grad": ([_P, _P, _P, _P, _P, _P, _P, _P, _I64, _I64, _P, _P, _P],
                                    ctypes.c_int),
        "ppo_minibatch_loss_grad_fresh": ([_P, _P, _P, _P, _P, _P, _P, _P, _I64, _I64, _P, _I64,
                                           i32, _F, _F, _P, _P, _P, _P], ctypes.c_int),
        "ppo_policy_act": ([_P, _P, _I64, u32, ctypes.c_uint64, _P, _P, _P, _P, _P], ctypes.c_int),
        "ppo_adam_step": ([_P, _F, _P, _P], ctypes.c_int),
        "ppo_muon_step": ([_P, _F, _P, _P], ctypes.c_int),
        "ppo_rnn_param_count": ([ctypes.POINTER(RnnConfig), ctypes.POINTER(_I64)], ctypes.c_int),
        "ppo_rnn_workspace_bytes": ([ctypes.POINTER(RnnConfig), _I64, _I64, ctypes.POINTER(_SZ)],
                                    ctypes.c_int),
        "ppo_rnn_loss_grad": ([ctypes.POINTER(RnnConfig), _P, _I64, _I64, _P, _I64, _P, _P, _P, _P,
                               _P, _P, _P, _P, _P, _P, _P, _P, _SZ, _P], ctypes.c_int),
        "ppo_rnn_create": ([ctypes.POINTER(RnnConfig), _P, _I64, _I64, i32, ctypes.POINTER(_P)],
                           ctypes.c_int),
        "ppo_rnn_destroy": ([_P], ctypes.c_int),
        "ppo_rnn_buffers": ([_P, ctypes.POINTER(_P), ctypes.POINTER(_P), ctypes.POINTER(_P),
                             ctypes.POINTER(_P)], ctypes.c_int),
        "ppo_rnn_update": ([_P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _I64, _I64, i32, i32, _F, _F,
                            _F, u32, _P, _P], ctypes.c_int),
        "ppo_rnn_sync_status": ([_P, _P], ctypes.c_int),
        "ppo_update": ([_P, _P, _P, _P, _P, _P, _P, _P, _P, _I64, _I64, i32, i32, _F, _F, _F,
                        u32, _P, _P], ctypes.c_int),
        "ppo_update_host": ([_P, _P, _P, _P, _P, _P, _P, _P, _P, _I64, _I64, i32, i32, _F, _F,
                             _F, u32, _P, _P], ctypes.c_int),
        "ppo_update_host_async": ([_P, _P, _P, _P, _P, _P, _P, _P, _P, _I64, _I64, i32, i32,
                                   _F, _F, _F, u32, _P, _P], ctypes.c_int),
        "ppo_host_wait": ([_P], ctypes.c_int),
        "ppo_stage_name": ([i32], ctypes.c_char_p),
        "ppo_update_profile": ([_P, _P, _P, _P, _P, _P, _P, _P, _P, _I64, _I64, i32, i32, _F,
                                _F, _F, u32, _P, _P, _P, _P], ctypes.c_int),
        "ppo_sync_status": ([_P, _P], ctypes.c_int),
        "ppo_set_collective": ([_P, i32, i32, COLLECTIVE_FN, _P], ctypes.c_int),
        "ppo_set_step_trace": ([_P, _P, _I64], ctypes.c_int),
        "ppo_set_wait_limit": ([_P, ctypes.c_uint64], ctypes.c_int),
    }
    for name, (args, res) in sig.items():
        fn = getattr(L, name)
        fn.argtypes = args
        fn.restype = res
    _lib = L
    return L


def check(status: int, what: str) -> None:
    if status != 0:
        raise PpoError(status, what)
