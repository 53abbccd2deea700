"""Seeded synthetic rollouts and initial weights for the PPO learner step.

This module only draws random numbers and lays them out; it contains none of
the learner's arithmetic.  Both the CUDA path's tests/bench and the oracle
receive the same host arrays from here, so both sides see identical bits.

Generator: mulberry32 ("PlayTrain", Appendix F.2 "seeded RNG"), used as a
counter-based generator -- draw k of the stream seeded with s is a pure
function of s + (k+1) * 0x6D2B79F5 (mod 2^32).  Every array gets its own
stream, seeded with the first draw of the stream seeded with
``seed + array_id * 0x9E3779B9``.

Distributions:
* U(0,1): draw / 2^32;  N(0,1): Box-Muller on two draws per element;
* Bernoulli(p): u < p;  "0 w.p. q else U(0,1)": u0 < q ? 0 : u1;
* tile ids uniform in 0..5: floor(6 u) as float32;
* discrete actions: floor(n_h u) per head;  Gaussian actions: N(0,1);
* weights U(-1/sqrt(fan_in), +1/sqrt(fan_in)), biases 0, log-std 0;
* logp_old: log-probability of the taken action under a uniform policy for
  the discrete heads and a standard normal for the Gaussian dims, plus
  N(0, 0.1^2) jitter, so that both the clipped and the unclipped branches of
  the surrogate are populated (a freshly initialised MLP policy is close to,
  but not exactly, uniform).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

_INC = np.uint32(0x6D2B79F5)
_GOLD = 0x9E3779B9


def _mix(t: np.ndarray) -> np.ndarray:
    t = t.astype(np.uint32, copy=False)
    n = (t ^ (t >> np.uint32(15))) * (t | np.uint32(1))
    n ^= n + (n ^ (n >> np.uint32(7))) * (n | np.uint32(61))
    return n ^ (n >> np.uint32(14))


def draws(stream_seed: int, start: int, count: int) -> np.ndarray:
    """Raw uint32 draws number start..start+count-1 of a mulberry32 stream."""
    k = np.arange(start + 1, start + count + 1, dtype=np.uint64)
    t = (np.uint64(stream_seed & 0xFFFFFFFF) + k * np.uint64(0x6D2B79F5)) & np.uint64(0xFFFFFFFF)
    return _mix(t.astype(np.uint32))


def stream_seed(seed: int, array_id: int) -> int:
    base = (seed + array_id * _GOLD) & 0xFFFFFFFF
    return int(draws(base, 0, 1)[0])


def uniform(seed: int, array_id: int, count: int, offset: int = 0) -> np.ndarray:
    return draws(stream_seed(seed, array_id), offset, count).astype(np.float64) / 4294967296.0


def normal(seed: int, array_id: int, count: int) -> np.ndarray:
    raw = draws(stream_seed(seed, array_id), 0, 2 * count).astype(np.float64)
    u1 = (raw[0::2] + 0.5) / 4294967296.0
    u2 = raw[1::2] / 4294967296.0
    return np.sqrt(-2.0 * np.log(u1)) * np.cos(2.0 * math.pi * u2)


# array ids (fixed, so that changing one array never moves another)
_ID = dict(obs=1, rew0=2, rew1=3, done=4, val=5, boot=6, act=7, actc=8, jitter=9,
           w1=10, w2=11, w3=12, tiles=13)


@dataclass
class Workload:
    """One synthetic workload: rollout shape, network, hyper-parameters."""
    name: str
    T: int
    N: int
    obs_dim: int
    h1: int = 0
    h2: int = 0
    act: int = 0                      # 0 tanh, 1 ReLU
    heads: tuple = ()
    n_gauss: int = 0
    reward: str = "sparse"            # "sparse" | "normal"
    reward_p0: float = 0.95           # P(reward == 0) for "sparse"
    reward_sigma: float = 1.0         # std for "normal"
    done_p: float = 0.01
    gamma: float = 0.99
    lam: float = 0.95
    clip: float = 0.2
    vf_coef: float = 0.5
    ent_coef: float = 0.01
    epochs: int = 1
    minibatches: int = 1
    precision: str = "fp32"           # "fp32" | "bf16"
    obs_kind: str = "normal"          # "normal" | "ddnet"
    gae_only: bool = False
    lr: float = 2.5e-4
    max_grad_norm: float = 0.5
    seed: int = 0

    @property
    def B(self) -> int:
        return self.T * self.N

    @property
    def out_cols(self) -> int:
        return int(sum(self.heads)) + self.n_gauss + 1

    @property
    def num_params(self) -> int:
        D, H1, H2, C = self.obs_dim, self.h1, self.h2, self.out_cols
        return H1 * D + H1 + H2 * H1 + H2 + C * H2 + C + self.n_gauss

    def flops_per_sample_pass(self) -> int:
        """Forward + backward GEMM flops per sample, without layer-1 dX."""
        D, H1, H2, C = self.obs_dim, self.h1, self.h2, self.out_cols
        fwd = 2 * (D * H1 + H1 * H2 + H2 * C)
        bwd_data = 2 * (C * H2 + H2 * H1)
        bwd_w = 2 * (C * H2 + H2 * H1 + H1 * D)
        return fwd + bwd_data + bwd_w

    def scaled(self, T: int | None = None, N: int | None = None, minibatches=None,
               epochs=None) -> "Workload":
        import dataclasses
        return dataclasses.replace(self, T=T or self.T, N=N or self.N,
                                   minibatches=minibatches or self.minibatches,
                                   epochs=epochs or self.epochs)


# The five workloads: a tiny step, a Mario-like and a DDNet-like learner,
# a large-batch learner and a GAE-only bandwidth stress case.
WORKLOADS = {
    "tiny": Workload("tiny", T=128, N=64, obs_dim=32, h1=64, h2=64, act=0, heads=(3, 2, 2),
                     reward="sparse", reward_p0=0.95, done_p=0.01, gamma=0.99, lam=0.95,
                     epochs=1, minibatches=4, precision="fp32"),
    "mario": Workload("mario", T=128, N=2048, obs_dim=64, h1=256, h2=256, act=0,
                      heads=(9, 2, 2, 2), reward="sparse", reward_p0=0.98, done_p=0.004,
                      gamma=0.99, lam=0.95, epochs=4, minibatches=8, precision="bf16"),
    "ddnet": Workload("ddnet", T=256, N=1500, obs_dim=1397, h1=512, h2=512, act=1,
                      heads=(3, 2, 2), n_gauss=2, reward="normal", reward_sigma=0.1,
                      done_p=0.002, gamma=0.99, lam=0.95, epochs=4, minibatches=8,
                      precision="bf16", obs_kind="ddnet"),
    "large": Workload("large", T=64, N=65536, obs_dim=128, h1=512, h2=512, act=0,
                      heads=(9, 2, 2, 2), reward="sparse", reward_p0=0.95, done_p=0.005,
                      gamma=0.99, lam=0.95, epochs=4, minibatches=16, precision="bf16"),
    "gae_stress": Workload("gae_stress", T=1024, N=65536, obs_dim=0, reward="normal",
                           reward_sigma=1.0, done_p=0.001, gamma=0.997, lam=0.95,
                           gae_only=True),
}


@dataclass
class Rollout:
    obs: np.ndarray | None        # [T*N, D] float32
    act_disc: np.ndarray | None   # [T*N, n_heads] int32
    act_cont: np.ndarray | None   # [T*N, n_gauss] float32
    logp_old: np.ndarray | None   # [T*N] float32
    val: np.ndarray               # [T, N] float32
    rew: np.ndarray               # [T, N] float32
    done: np.ndarray              # [T, N] float32 (0/1)
    boot: np.ndarray              # [N] float32


def rollout(w: Workload, seed: int | None = None, with_obs: bool = True) -> Rollout:
    """Seeded rollout.  with_obs=False leaves obs None (a caller that fills a
    very large observation buffer itself)."""
    s = w.seed if seed is None else seed
    T, N, B = w.T, w.N, w.B
    if w.reward == "sparse":
        zero = uniform(s, _ID["rew0"], B) < w.reward_p0
        rew = np.where(zero, 0.0, uniform(s, _ID["rew1"], B))
    else:
        rew = w.reward_sigma * normal(s, _ID["rew1"], B)
    rew = rew.astype(np.float32).reshape(T, N)
    done = (uniform(s, _ID["done"], B) < w.done_p).astype(np.float32).reshape(T, N)
    val = normal(s, _ID["val"], B).astype(np.float32).reshape(T, N)
    boot = normal(s, _ID["boot"], N).astype(np.float32)
    if w.gae_only:
        return Rollout(None, None, None, None, val, rew, done, boot)

    D = w.obs_dim
    if not with_obs:
        obs = None
    elif w.obs_kind == "ddnet":
        # 43x31 tile grid of integer ids 0..5, 15-d player state x 4 frames,
        # 4-d checkpoint navigation
        tiles = np.floor(6.0 * uniform(s, _ID["tiles"], B * 1333)).astype(np.float32)
        rest = normal(s, _ID["obs"], B * 64).astype(np.float32)
        obs = np.concatenate([tiles.reshape(B, 1333), rest.reshape(B, 64)], axis=1)
    else:
        obs = normal(s, _ID["obs"], B * D).astype(np.float32).reshape(B, D)

    nh = len(w.heads)
    u = uniform(s, _ID["act"], B * nh).reshape(B, nh)
    act_disc = np.floor(u * np.array(w.heads, np.float64)).astype(np.int32)
    act_disc = np.minimum(act_disc, np.array(w.heads, np.int32) - 1)
    if w.n_gauss:
        act_cont = normal(s, _ID["actc"], B * w.n_gauss).astype(np.float32).reshape(B, w.n_gauss)
    else:
        act_cont = np.zeros((B, 0), np.float32)
    lp = -sum(math.log(n) for n in w.heads) * np.ones(B)
    if w.n_gauss:
        lp += (-0.5 * act_cont.astype(np.float64) ** 2 - 0.5 * math.log(2 * math.pi)).sum(1)
    lp += 0.1 * normal(s, _ID["jitter"], B)
    return Rollout(None if obs is None else np.ascontiguousarray(obs), act_disc, act_cont,
                   lp.astype(np.float32), val, rew, done, boot)


def init_params(w: Workload, seed: int | None = None) -> np.ndarray:
    """Flat fp32 parameters: W1[h1][D], b1, W2[h2][h1], b2, W3[C][h2], b3, logstd."""
    s = w.seed if seed is None else seed
    D, H1, H2, C = w.obs_dim, w.h1, w.h2, w.out_cols
    def U(aid, n, fan_in):
        a = 1.0 / math.sqrt(fan_in)
        return (2.0 * uniform(s, aid, n) - 1.0) * a
    parts = [U(_ID["w1"], H1 * D, D), np.zeros(H1), U(_ID["w2"], H2 * H1, H1), np.zeros(H2),
             U(_ID["w3"], C * H2, H2), np.zeros(C), np.zeros(w.n_gauss)]
    return np.concatenate(parts).astype(np.float32)
