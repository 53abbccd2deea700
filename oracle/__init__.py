"""Plain CPU oracle of the PPO learner step (fp64), driven through ctypes.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package.  The CUDA library
(``policy_rl_gb300``) never imports it and shares no code with it.

The arithmetic lives in ``ppo_oracle.c``; this module only compiles it (gcc,
``-ffp-contract=off`` so that no fused multiply-add changes the rounding of the
plain C expressions) and marshals numpy arrays.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass, field

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ppo_oracle.c")
_LIB_DIR = os.path.join(_HERE, "_build")
_LIB = os.path.join(_LIB_DIR, "libppo_oracle.so")

_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle into ``oracle/_build/libppo_oracle.so``."""
    os.makedirs(_LIB_DIR, exist_ok=True)
    hdr = os.path.join(_HERE, "ppo_oracle.h")
    newest = max(os.path.getmtime(_SRC), os.path.getmtime(hdr))
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < newest:
        tmp = _LIB + f".{os.getpid()}.tmp"
        base = ["gcc", "-std=c99", "-O2", "-ffp-contract=off", "-Wall", "-shared", "-fPIC"]
        # OpenMP (row loops of the minibatch gradient) when the compiler has it
        if subprocess.call(base + ["-fopenmp", _SRC, "-o", tmp, "-lm"],
                           stderr=subprocess.DEVNULL) != 0:
            subprocess.check_call(base + [_SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def threads() -> int:
    """Threads of the oracle's OpenMP row loops (1 without OpenMP)."""
    return int(lib().orc_threads())


def set_threads(n: int) -> None:
    """Thread count of the oracle's OpenMP row loops."""
    lib().orc_set_threads(int(n))


class _Net(ctypes.Structure):
    _fields_ = [("obs_dim", ctypes.c_int32), ("h1", ctypes.c_int32), ("h2", ctypes.c_int32),
                ("act", ctypes.c_int32), ("n_heads", ctypes.c_int32),
                ("head_n", ctypes.c_int32 * 8), ("n_gauss", ctypes.c_int32)]


class _Rnn(ctypes.Structure):
    _fields_ = [("obs_dim", ctypes.c_int32), ("hidden", ctypes.c_int32), ("layers", ctypes.c_int32),
                ("n_heads", ctypes.c_int32), ("head_n", ctypes.c_int32 * 8),
                ("n_gauss", ctypes.c_int32)]


class _LossCfg(ctypes.Structure):
    _fields_ = [("clip", ctypes.c_double), ("vf_coef", ctypes.c_double),
                ("ent_coef", ctypes.c_double), ("bf16_operands", ctypes.c_int)]


class _Hyper(ctypes.Structure):
    _fields_ = [("gamma", ctypes.c_double), ("lambda_", ctypes.c_double),
                ("clip", ctypes.c_double), ("vf_coef", ctypes.c_double),
                ("ent_coef", ctypes.c_double), ("lr", ctypes.c_double),
                ("beta1", ctypes.c_double), ("beta2", ctypes.c_double),
                ("adam_eps", ctypes.c_double), ("max_grad_norm", ctypes.c_double),
                ("seed", ctypes.c_uint32), ("bf16_operands", ctypes.c_int),
                ("adv_mode", ctypes.c_int), ("rho_clip", ctypes.c_double),
                ("c_clip", ctypes.c_double), ("optimizer", ctypes.c_int),
                ("muon_lr", ctypes.c_double), ("muon_beta", ctypes.c_double)]


_P = ctypes.c_void_p
_I64 = ctypes.c_int64
_D = ctypes.c_double


def lib():
    global _lib
    if _lib is None:
        _lib = ctypes.CDLL(build())
        L = _lib
        L.orc_mulberry32_next.argtypes = [ctypes.POINTER(ctypes.c_uint32)]
        L.orc_mulberry32_next.restype = ctypes.c_uint32
        L.orc_gae.argtypes = [_I64, _I64, _P, _P, _P, _P, _D, _D, _P, _P]
        L.orc_moments.argtypes = [_I64, _P, ctypes.POINTER(_D), ctypes.POINTER(_D)]
        L.orc_normalize.argtypes = [_I64, _P, _D, _D, _P]
        L.orc_perm.argtypes = [ctypes.c_uint32, _I64, _I64, _P]
        L.orc_out_cols.argtypes = [ctypes.POINTER(_Net)]
        L.orc_out_cols.restype = _I64
        L.orc_num_params.argtypes = [ctypes.POINTER(_Net)]
        L.orc_num_params.restype = _I64
        L.orc_forward.argtypes = [ctypes.POINTER(_Net), _P, _P, _P]
        L.orc_round_bf16.argtypes = [_D]
        L.orc_round_bf16.restype = _D
        L.orc_policy_logp.argtypes = [ctypes.POINTER(_Net), _P, _I64, _P, _P, _P, _P, _P]
        L.orc_loss_grad.argtypes = [ctypes.POINTER(_Net), ctypes.POINTER(_LossCfg), _P, _I64, _P,
                                    _P, _P, _P, _P, _P, _P, ctypes.c_int, _D, _D, _P, _P, _P]
        L.orc_loss_grad.restype = _D
        L.orc_clip_grad_norm.argtypes = [_I64, _P, _D]
        L.orc_clip_grad_norm.restype = _D
        L.orc_adam.argtypes = [_I64, _P, _P, _P, _P, _I64, _D, _D, _D, _D]
        L.orc_segment_advantage.argtypes = [_I64, _I64, _P, _P, _P, _I64, _P, _P, _P, _D, _D,
                                            _D, _D, _P, _P]
        L.orc_fresh_values.argtypes = [ctypes.POINTER(_Net), ctypes.c_int, _P, _I64, _P, _P, _P,
                                       _P, _P, _P, _P]
        L.orc_loss_grad_fresh.argtypes = [ctypes.POINTER(_Net), ctypes.POINTER(_LossCfg), _P,
                                          _I64, _I64, _I64, _P, _P, _P, _P, _P, _P, _P, _P,
                                          ctypes.c_int, _D, _D, _D, _D, _P, _P, _P, _P, _P]
        L.orc_loss_grad_fresh.restype = _D
        L.orc_uniform24.argtypes = [ctypes.c_uint32]
        L.orc_uniform24.restype = _D
        L.orc_mulberry32_at.argtypes = [ctypes.c_uint32, ctypes.c_uint64]
        L.orc_mulberry32_at.restype = ctypes.c_uint32
        L.orc_sample_categorical.argtypes = [_P, ctypes.c_int, _D]
        L.orc_sample_categorical.restype = ctypes.c_int
        L.orc_box_muller.argtypes = [_D, _D]
        L.orc_box_muller.restype = _D
        L.orc_policy_act.argtypes = [ctypes.POINTER(_Net), ctypes.c_int, _P, _I64, _P, ctypes.c_uint32,
                                     ctypes.c_uint64, _P, _P, _P, _P]
        L.orc_newton_schulz5.argtypes = [_I64, _I64, _P, ctypes.c_int, _P]
        L.orc_newton_schulz5_bf16.argtypes = [_I64, _I64, _P, ctypes.c_int, _P]
        L.orc_muon.argtypes = [ctypes.POINTER(_Net), _P, _P, _P, _P, _P, _I64, _D, _D, _D, _D, _D,
                               _D]
        L.orc_muon_bf16.argtypes = L.orc_muon.argtypes
        L.orc_rnn_num_params.argtypes = [ctypes.POINTER(_Rnn)]
        L.orc_rnn_num_params.restype = _I64
        L.orc_rnn_forward.argtypes = [ctypes.POINTER(_Rnn), _P, _I64, _I64, _I64, _P, _P, _P, _P,
                                      _P, _P, _P, _P, _P]
        L.orc_rnn_loss_grad.argtypes = [ctypes.POINTER(_Rnn), ctypes.POINTER(_LossCfg), _P, _I64,
                                        _I64, _I64, _P, _P, _P, _P, _P, _P, _P, ctypes.c_int, _D,
                                        _D, _P, _P, _P, _P, _P]
        L.orc_rnn_loss_grad.restype = _D
        L.orc_rnn_update.restype = ctypes.c_int
        L.orc_rnn_update.argtypes = [ctypes.POINTER(_Rnn), ctypes.POINTER(_Hyper), _I64, _I64, _I64,
                                     _I64, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P,
                                     ctypes.POINTER(_I64), _P]
        L.orc_moments3.argtypes = [_I64, _P, _P]
        L.orc_moments_merge.argtypes = [_P, _P, _P]
        L.orc_update_sharded.restype = ctypes.c_int
        L.orc_update_sharded.argtypes = [ctypes.POINTER(_Net), ctypes.POINTER(_Hyper), _I64, _I64,
                                         _I64, _I64, _I64, _P, _P, _P, _P, _P, _P, _P, _P, _P,
                                         _P, _P, _P, ctypes.POINTER(_I64), _P]
        L.orc_threads.argtypes = []
        L.orc_threads.restype = ctypes.c_int
        L.orc_set_threads.argtypes = [ctypes.c_int]
        L.orc_update.argtypes = [ctypes.POINTER(_Net), ctypes.POINTER(_Hyper), _I64, _I64, _I64, _I64,
                                 _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P,
                                 ctypes.POINTER(_I64), _P, _P, _P]
    return _lib


def _ptr(a: np.ndarray | None):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data


def _as(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


@dataclass
class Net:
    """MLP actor-critic shape.  act: 0 tanh, 1 ReLU."""
    obs_dim: int
    h1: int
    h2: int
    act: int = 0
    heads: tuple = (3, 2, 2)
    n_gauss: int = 0

    def c(self) -> _Net:
        hn = (ctypes.c_int32 * 8)(*(list(self.heads) + [0] * (8 - len(self.heads))))
        return _Net(self.obs_dim, self.h1, self.h2, self.act, len(self.heads), hn, self.n_gauss)

    @property
    def out_cols(self) -> int:
        return int(sum(self.heads)) + self.n_gauss + 1

    @property
    def num_params(self) -> int:
        D, H1, H2, C = self.obs_dim, self.h1, self.h2, self.out_cols
        return H1 * D + H1 + H2 * H1 + H2 + C * H2 + C + self.n_gauss


@dataclass
class Rnn:
    """Recurrent policy: bias-free encoder D -> hidden, `layers` MinGRU layers,
    bias-free decoder to the head columns (logits, Gaussian means, value)."""
    obs_dim: int
    hidden: int = 128
    layers: int = 4
    heads: tuple = (3, 2, 2)
    n_gauss: int = 0

    def c(self) -> _Rnn:
        hn = (ctypes.c_int32 * 8)(*(list(self.heads) + [0] * (8 - len(self.heads))))
        return _Rnn(self.obs_dim, self.hidden, self.layers, len(self.heads), hn, self.n_gauss)

    @property
    def out_cols(self) -> int:
        return int(sum(self.heads)) + self.n_gauss + 1

    @property
    def num_params(self) -> int:
        D, H, L, C = self.obs_dim, self.hidden, self.layers, self.out_cols
        return H * D + L * (2 * H * H + 2 * H) + C * H + self.n_gauss


@dataclass
class Hyper:
    gamma: float = 0.99
    lam: float = 0.95
    clip: float = 0.2
    vf_coef: float = 0.5
    ent_coef: float = 0.01
    lr: float = 2.5e-4
    beta1: float = 0.9
    beta2: float = 0.999
    adam_eps: float = 1e-8
    max_grad_norm: float = 0.5
    seed: int = 0
    bf16_operands: bool = False
    adv_mode: int = 0          # 0 once per update, 1 fresh GAE, 2 fresh V-trace
    rho_clip: float = 1.0
    c_clip: float = 1.0
    optimizer: int = 0         # 0 Adam, 1 Muon (weight matrices) + Adam (vectors)
    muon_lr: float = 0.02
    muon_beta: float = 0.95

    def c(self) -> _Hyper:
        return _Hyper(self.gamma, self.lam, self.clip, self.vf_coef, self.ent_coef, self.lr,
                      self.beta1, self.beta2, self.adam_eps, self.max_grad_norm, self.seed,
                      int(self.bf16_operands), int(self.adv_mode), self.rho_clip, self.c_clip,
                      int(self.optimizer), self.muon_lr, self.muon_beta)


def mulberry32_stream(seed: int, count: int) -> np.ndarray:
    """First ``count`` raw uint32 draws of the stream seeded with ``seed``."""
    L = lib()
    st = ctypes.c_uint32(seed & 0xFFFFFFFF)
    return np.array([L.orc_mulberry32_next(ctypes.byref(st)) for _ in range(count)],
                    dtype=np.uint32)


def gae(rew, val, done, boot, gamma, lam):
    rew, val, done = (_as(x, np.float32) for x in (rew, val, done))
    boot = _as(boot, np.float32)
    T, N = rew.shape
    adv = np.empty((T, N), np.float64)
    ret = np.empty((T, N), np.float64)
    lib().orc_gae(T, N, _ptr(rew), _ptr(val), _ptr(done), _ptr(boot), gamma, lam,
                  _ptr(adv), _ptr(ret))
    return adv, ret


def segment_advantage(rew, done, boot, envs, val, ratio, gamma, lam, rho_clip=1.0, c_clip=1.0):
    """Advantages and value targets of the environment segments ``envs`` from
    the given values ``val`` [T][ns] (and ratios, V-trace; None = GAE).
    Returns (adv, ret), each float64 [T][ns]."""
    rew, done = _as(rew, np.float32), _as(done, np.float32)
    boot = _as(boot, np.float32)
    envs = _as(envs, np.int32)
    T, N = rew.shape
    ns = envs.size
    val = _as(val, np.float64).reshape(T, ns)
    ratio = None if ratio is None else _as(ratio, np.float64).reshape(T, ns)
    adv = np.empty((T, ns), np.float64)
    ret = np.empty((T, ns), np.float64)
    lib().orc_segment_advantage(T, N, _ptr(rew), _ptr(done), _ptr(boot), ns, _ptr(envs),
                                _ptr(val), _ptr(ratio), gamma, lam, rho_clip, c_clip,
                                _ptr(adv), _ptr(ret))
    return adv, ret


def segment_rows(T: int, N: int, envs) -> np.ndarray:
    """Flat batch rows of a segment minibatch, in minibatch order t*ns + j."""
    envs = np.asarray(envs, np.int64)
    return (np.arange(T, dtype=np.int64)[:, None] * N + envs[None, :]).ravel().astype(np.int32)


def fresh_values(net: Net, params, idx, obs, act_disc, act_cont, logp_old, bf16_operands=False,
                 with_ratio=True):
    """(value, ratio) of rows idx at params (ratio None unless with_ratio)."""
    params = _as(params, np.float64)
    idx = _as(idx, np.int32)
    n = idx.size
    val = np.empty(n, np.float64)
    ratio = np.empty(n, np.float64) if with_ratio else None
    act_cont = _as(act_cont if act_cont is not None else np.zeros(1), np.float32)
    cn = net.c()
    lib().orc_fresh_values(ctypes.byref(cn), int(bool(bf16_operands)), _ptr(params), n, _ptr(idx),
                           _ptr(_as(obs, np.float32)), _ptr(_as(act_disc, np.int32)),
                           _ptr(act_cont), _ptr(_as(logp_old, np.float32)), _ptr(val),
                           _ptr(ratio))
    return val, ratio


def loss_grad_fresh(net: Net, params, T, N, envs, obs, act_disc, act_cont, logp_old, rew, done,
                    boot, vtrace=False, gamma=0.99, lam=0.95, rho_clip=1.0, c_clip=1.0,
                    clip=0.2, vf_coef=0.5, ent_coef=0.01, bf16_operands=False):
    """Segment minibatch with fresh advantages.  Returns
    (loss, grad[P], stats6, scale6, adv_norm[T*ns], ret[T*ns])."""
    params = _as(params, np.float64)
    envs = _as(envs, np.int32)
    ns = envs.size
    grad = np.empty(net.num_params, np.float64)
    st = np.empty(6, np.float64)
    sc = np.empty(6, np.float64)
    an = np.empty(T * ns, np.float64)
    rt = np.empty(T * ns, np.float64)
    act_cont = _as(act_cont if act_cont is not None else np.zeros(1), np.float32)
    cfg = _LossCfg(clip, vf_coef, ent_coef, int(bool(bf16_operands)))
    cn = net.c()
    loss = lib().orc_loss_grad_fresh(
        ctypes.byref(cn), ctypes.byref(cfg), _ptr(params), T, N, ns, _ptr(envs),
        _ptr(_as(obs, np.float32)), _ptr(_as(act_disc, np.int32)), _ptr(act_cont),
        _ptr(_as(logp_old, np.float32)), _ptr(_as(rew, np.float32)), _ptr(_as(done, np.float32)),
        _ptr(_as(boot, np.float32)), int(bool(vtrace)), gamma, lam, rho_clip, c_clip,
        _ptr(grad), _ptr(st), _ptr(sc), _ptr(an), _ptr(rt))
    return loss, grad, st, sc, an, rt


def uniform24(x: int) -> float:
    return lib().orc_uniform24(int(x) & 0xFFFFFFFF)


def mulberry32_at(seed: int, draw: int) -> int:
    """Draw number ``draw`` (0-based) of the mulberry32 stream seeded with ``seed``."""
    return lib().orc_mulberry32_at(seed & 0xFFFFFFFF, int(draw))


def sample_categorical(z, u: float) -> int:
    z = _as(z, np.float64)
    return lib().orc_sample_categorical(_ptr(z), z.size, float(u))


def box_muller(u1: float, u2: float) -> float:
    return lib().orc_box_muller(float(u1), float(u2))


def policy_act(net: Net, params, obs, seed: int, draw0: int = 0, bf16_operands=False):
    """Sampled (act_disc [n][NH] int32, act_cont [n][G], logp [n], value [n])."""
    params = _as(params, np.float64)
    obs = _as(obs, np.float32).reshape(-1, net.obs_dim)
    n = obs.shape[0]
    NH, G = len(net.heads), net.n_gauss
    act = np.empty((n, max(NH, 1)), np.int32)
    actc = np.empty((n, max(G, 1)), np.float64)
    logp = np.empty(n, np.float64)
    val = np.empty(n, np.float64)
    cn = net.c()
    lib().orc_policy_act(ctypes.byref(cn), int(bool(bf16_operands)), _ptr(params), n, _ptr(obs),
                         seed & 0xFFFFFFFF, int(draw0), _ptr(act), _ptr(actc), _ptr(logp),
                         _ptr(val))
    return act[:, :NH], actc[:, :G], logp, val


def rnn_forward(rnn: Rnn, params, obs, done, h0, n: int = 0):
    """Head outputs [T][C] of segment n; obs rows t*N + n, done [T][N], h0 [L][H]."""
    done = _as(done, np.float32)
    T, N = done.shape
    out = np.empty((T, rnn.out_cols), np.float64)
    cn = rnn.c()
    lib().orc_rnn_forward(ctypes.byref(cn), _ptr(_as(params, np.float64)), T, N, n,
                          _ptr(_as(obs, np.float32)), _ptr(done), _ptr(_as(h0, np.float64)),
                          _ptr(out), None, None, None, None, None)
    return out


def rnn_loss_grad(rnn: Rnn, params, envs, obs, act_disc, act_cont, logp_old, adv, ret, done, h0,
                  clip=0.2, vf_coef=0.5, ent_coef=0.01, normalize=False, adv_mean=0.0,
                  adv_std=1.0, bf16_operands=False):
    """Loss and BPTT gradient of the segments envs; returns (loss, grad, stats6, scale6).
    obs [T*N][D] (row t*N + n), adv / ret [T*N], done [T][N], h0 [N][L][H]."""
    done = _as(done, np.float32)
    T, N = done.shape
    envs = _as(envs, np.int32)
    grad = np.empty(rnn.num_params, np.float64)
    st = np.empty(6, np.float64)
    sc = np.empty(6, np.float64)
    act_cont = _as(act_cont if act_cont is not None else np.zeros(1), np.float32)
    cfg = _LossCfg(clip, vf_coef, ent_coef, int(bool(bf16_operands)))
    cn = rnn.c()
    loss = lib().orc_rnn_loss_grad(
        ctypes.byref(cn), ctypes.byref(cfg), _ptr(_as(params, np.float64)), T, N, envs.size,
        _ptr(envs), _ptr(_as(obs, np.float32)), _ptr(_as(act_disc, np.int32)), _ptr(act_cont),
        _ptr(_as(logp_old, np.float32)), _ptr(_as(adv, np.float64)), _ptr(_as(ret, np.float64)),
        int(bool(normalize)), adv_mean, adv_std, _ptr(done), _ptr(_as(h0, np.float64)),
        _ptr(grad), _ptr(st), _ptr(sc))
    return loss, grad, st, sc


def rnn_update(rnn: Rnn, hp, T, N, epochs, minibatches, obs, act_disc, act_cont, logp_old, val,
               rew, done, boot, h0, params, m=None, v=None, step=0):
    """One recurrent-policy update; returns (params, m, v, step, stats [E*M][6])."""
    P = rnn.num_params
    params = _as(params, np.float64).copy()
    m = np.zeros(P) if m is None else _as(m, np.float64).copy()
    v = np.zeros(P) if v is None else _as(v, np.float64).copy()
    stats = np.empty((epochs * minibatches, 6), np.float64)
    st = _I64(step)
    arrs = [_as(obs, np.float32), _as(act_disc, np.int32),
            _as(act_cont if act_cont is not None else np.zeros(1), np.float32),
            _as(logp_old, np.float32), _as(val, np.float32), _as(rew, np.float32),
            _as(done, np.float32), _as(boot, np.float32), _as(h0, np.float64)]
    cn, ch = rnn.c(), hp.c()
    if minibatches < 1 or N % minibatches:
        raise ValueError("minibatches must be >= 1 and divide N (whole segments)")
    lib().orc_rnn_update(ctypes.byref(cn), ctypes.byref(ch), T, N, epochs, minibatches,
                         *[_ptr(a) for a in arrs], _ptr(params), _ptr(m), _ptr(v),
                         ctypes.byref(st), _ptr(stats))
    return params, m, v, st.value, stats


def moments(x):
    x = _as(x, np.float64).ravel()
    m, s = _D(), _D()
    lib().orc_moments(x.size, _ptr(x), ctypes.byref(m), ctypes.byref(s))
    return m.value, s.value


def moments3(x):
    """(count, mean, M2) of x (two-pass)."""
    x = _as(x, np.float64).ravel()
    out = np.empty(3, np.float64)
    lib().orc_moments3(x.size, _ptr(x), _ptr(out))
    return out


def moments_merge(a, b):
    """Pairwise merge of two (count, mean, M2) triples."""
    a = _as(a, np.float64)
    b = _as(b, np.float64)
    out = np.empty(3, np.float64)
    lib().orc_moments_merge(_ptr(a), _ptr(b), _ptr(out))
    return out


def normalize(x, mean, std):
    x = _as(x, np.float64)
    out = np.empty_like(x)
    lib().orc_normalize(x.size, _ptr(x), mean, std, _ptr(out))
    return out


def perm(seed: int, epoch: int, B: int) -> np.ndarray:
    out = np.empty(B, np.int32)
    lib().orc_perm(seed & 0xFFFFFFFF, epoch, B, _ptr(out))
    return out


def forward(net: Net, params, x):
    params = _as(params, np.float64)
    x = _as(x, np.float32)
    rows = x.reshape(-1, net.obs_dim)
    out = np.empty((rows.shape[0], net.out_cols), np.float64)
    cn = net.c()
    for i in range(rows.shape[0]):
        r = np.ascontiguousarray(rows[i])
        o = np.empty(net.out_cols, np.float64)
        lib().orc_forward(ctypes.byref(cn), _ptr(params), _ptr(r), _ptr(o))
        out[i] = o
    return out


def round_bf16(x: float) -> float:
    return lib().orc_round_bf16(float(x))


def policy_logp(net: Net, params, obs, act_disc, act_cont=None):
    """Per-row (log-probability of the action, entropy) under params."""
    params = _as(params, np.float64)
    obs = _as(obs, np.float32).reshape(-1, net.obs_dim)
    n = obs.shape[0]
    act_disc = _as(act_disc, np.int32)
    act_cont = _as(act_cont if act_cont is not None and net.n_gauss else np.zeros(1), np.float32)
    lp = np.empty(n, np.float64)
    ent = np.empty(n, np.float64)
    cn = net.c()
    lib().orc_policy_logp(ctypes.byref(cn), _ptr(params), n, _ptr(obs), _ptr(act_disc),
                          _ptr(act_cont), _ptr(lp), _ptr(ent))
    return lp, ent


def loss_grad(net: Net, params, idx, obs, act_disc, act_cont, logp_old, adv, ret,
              clip=0.2, vf_coef=0.5, ent_coef=0.01, normalize=False, adv_mean=0.0,
              adv_std=1.0, bf16_operands=False):
    """Returns (loss, grad[P], stats6[6], scale6[6])."""
    params = _as(params, np.float64)
    idx = _as(idx, np.int32)
    obs = _as(obs, np.float32)
    act_disc = _as(act_disc, np.int32)
    act_cont = _as(act_cont if act_cont is not None else np.zeros((1,), np.float32), np.float32)
    logp_old = _as(logp_old, np.float32)
    adv = _as(adv, np.float64)
    ret = _as(ret, np.float64)
    grad = np.empty(net.num_params, np.float64)
    st = np.empty(6, np.float64)
    sc = np.empty(6, np.float64)
    cfg = _LossCfg(clip, vf_coef, ent_coef, int(bool(bf16_operands)))
    cn = net.c()
    loss = lib().orc_loss_grad(ctypes.byref(cn), ctypes.byref(cfg), _ptr(params), idx.size,
                               _ptr(idx), _ptr(obs), _ptr(act_disc), _ptr(act_cont),
                               _ptr(logp_old), _ptr(adv), _ptr(ret), int(bool(normalize)),
                               adv_mean, adv_std, _ptr(grad), _ptr(st), _ptr(sc))
    return loss, grad, st, sc


def clip_grad_norm(g, max_norm):
    g = _as(g, np.float64).copy()
    n = lib().orc_clip_grad_norm(g.size, _ptr(g), max_norm)
    return n, g


def adam(p, g, m, v, step, lr, beta1=0.9, beta2=0.999, eps=1e-8):
    p = _as(p, np.float64).copy()
    m = _as(m, np.float64).copy()
    v = _as(v, np.float64).copy()
    g = _as(g, np.float64)
    lib().orc_adam(p.size, _ptr(p), _ptr(g), _ptr(m), _ptr(v), step, lr, beta1, beta2, eps)
    return p, m, v


def newton_schulz5(G, steps: int = 5, bf16: bool = False):
    """Muon's quintic Newton-Schulz orthogonalisation of a matrix (fp64; bf16:
    X, A, B stored as bf16)."""
    G = _as(G, np.float64)
    rows, cols = G.shape
    out = np.empty_like(G)
    fn = lib().orc_newton_schulz5_bf16 if bf16 else lib().orc_newton_schulz5
    fn(rows, cols, _ptr(G), steps, _ptr(out))
    return out


def muon(net: Net, p, g, mom, m, v, step, muon_lr=0.02, muon_beta=0.95, lr=2.5e-4,
         beta1=0.9, beta2=0.999, eps=1e-8, bf16=False):
    """One Muon step (matrices) + Adam (vectors); returns (p, mom, m, v)."""
    p, mom, m, v = (_as(x, np.float64).copy() for x in (p, mom, m, v))
    g = _as(g, np.float64)
    cn = net.c()
    (lib().orc_muon_bf16 if bf16 else lib().orc_muon)(ctypes.byref(cn), _ptr(p), _ptr(g), _ptr(mom), _ptr(m), _ptr(v), step, muon_lr,
                   muon_beta, lr, beta1, beta2, eps)
    return p, mom, m, v


@dataclass
class UpdateResult:
    params: np.ndarray
    m: np.ndarray
    v: np.ndarray
    mom: np.ndarray
    step: int
    stats: np.ndarray
    adv: np.ndarray
    ret: np.ndarray


def update(net: Net, hp: Hyper, T, N, epochs, minibatches, obs, act_disc, act_cont, logp_old,
           val, rew, done, boot, params, m=None, v=None, step=0, mom=None) -> UpdateResult:
    P = net.num_params
    params = _as(params, np.float64).copy()
    m = np.zeros(P) if m is None else _as(m, np.float64).copy()
    v = np.zeros(P) if v is None else _as(v, np.float64).copy()
    mom = np.zeros(P) if mom is None else _as(mom, np.float64).copy()
    stats = np.empty((epochs * minibatches, 6), np.float64)
    adv = np.zeros(T * N, np.float64)   # not written in the fresh-advantage modes
    ret = np.zeros(T * N, np.float64)
    st = _I64(step)
    arrs = [_as(obs, np.float32), _as(act_disc, np.int32),
            _as(act_cont if act_cont is not None else np.zeros(1), np.float32),
            _as(logp_old, np.float32), _as(val, np.float32), _as(rew, np.float32),
            _as(done, np.float32), _as(boot, np.float32)]
    cn, ch = net.c(), hp.c()
    lib().orc_update(ctypes.byref(cn), ctypes.byref(ch), T, N, epochs, minibatches,
                     *[_ptr(a) for a in arrs], _ptr(params), _ptr(m), _ptr(v), _ptr(mom),
                     ctypes.byref(st), _ptr(stats), _ptr(adv), _ptr(ret))
    return UpdateResult(params, m, v, mom, st.value, stats, adv.reshape(T, N), ret.reshape(T, N))


def update_sharded(net: Net, hp: Hyper, world, T, N, epochs, minibatches, obs, act_disc,
                   act_cont, logp_old, val, rew, done, boot, params, m=None, v=None, step=0,
                   mom=None) -> UpdateResult:
    """The update data-parallel over `world` env shards of the [T][N] rollout
    (one process; see orc_update_sharded)."""
    P = net.num_params
    params = _as(params, np.float64).copy()
    m = np.zeros(P) if m is None else _as(m, np.float64).copy()
    v = np.zeros(P) if v is None else _as(v, np.float64).copy()
    mom = np.zeros(P) if mom is None else _as(mom, np.float64).copy()
    stats = np.empty((epochs * minibatches, 6), np.float64)
    st = _I64(step)
    arrs = [_as(obs, np.float32), _as(act_disc, np.int32),
            _as(act_cont if act_cont is not None else np.zeros(1), np.float32),
            _as(logp_old, np.float32), _as(val, np.float32), _as(rew, np.float32),
            _as(done, np.float32), _as(boot, np.float32)]
    cn, ch = net.c(), hp.c()
    if lib().orc_update_sharded(ctypes.byref(cn), ctypes.byref(ch), world, T, N, epochs,
                                minibatches, *[_ptr(a) for a in arrs], _ptr(params), _ptr(m),
                                _ptr(v), _ptr(mom), ctypes.byref(st), _ptr(stats)) != 0:
        raise ValueError("world must divide N and minibatches must divide T*N/world")
    return UpdateResult(params, m, v, mom, st.value, stats, None, None)
