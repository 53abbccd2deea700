// common.cuh -- internal declarations shared by the CUDA translation units of
// the PPO learner library.  Nothing here is part of the public C ABI.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

#include "../../include/ppo.h"

namespace ppo {

constexpr int kWarp = 32;

// ---------------------------------------------------------------------------
// error latch: device-side failures (bounded waits that gave up) OR a code
// into this word; the host reads it in ppo_sync_status.
enum DevErr : int { kDevOk = 0, kDevTimeout = 1 };

// ---------------------------------------------------------------------------
// Network shape as the kernels see it.
struct NetShape {
  int D, Dp;        // observation width; padded (bf16: multiple of 64)
  int H1, H2;
  int act;          // 0 tanh, 1 relu
  int NH;           // discrete heads
  int head_n[PPO_MAX_HEADS];
  int G;            // Gaussian dims
  int C;            // output columns = sum(head_n) + G + 1
  int CP;           // C padded to the head GEMM's N (16 or 32)
  // flat parameter offsets
  int64_t oW1, ob1, oW2, ob2, oW3, ob3, ologstd, P;
};

struct LossCoef {
  float clip, vf, ent;
};

// Per-row inputs of the loss epilogue (already gathered to minibatch order).
struct LossRows {
  const int32_t* act;      // [mb][NH]
  const float* actc;       // [mb][G]
  const float* logp_old;   // [mb]
  const float* adv;        // [mb] (normalised)
  const float* ret;        // [mb]
};

// number of per-CTA scalar partials written by the loss epilogue
// (6 stats, then dlogstd[G<=4])
constexpr int kLossPartials = 12;

// ---------------------------------------------------------------------------
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Transposing reduction across a warp: on entry lane l holds v[0..31] (its
// row's 32 column values); on exit lane l returns sum over lanes of v[l].
// 31 shuffles, fixed order (deterministic).
__device__ __forceinline__ float warp_reduce_scatter32(float (&v)[32]) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int half = 16; half >= 1; half >>= 1) {
    const bool upper = (lane & half) != 0;
#pragma unroll
    for (int i = 0; i < half; ++i) {
      // keep v[i + half] if upper, v[i] otherwise; send the other one
      float send = upper ? v[i] : v[i + half];
      float keep = upper ? v[i + half] : v[i];
      float recv = __shfl_xor_sync(0xffffffffu, send, half);
      v[i] = keep + recv;
    }
  }
  return v[0];
}

// Programmatic dependent launch: a kernel launched with the programmatic
// stream-serialization attribute may start while its predecessor finishes;
// pdl_wait() blocks until the predecessor grid has completed and its memory
// is visible (every kernel of a chain calls it before touching data that an
// earlier kernel wrote), pdl_trigger() lets the successor begin launching.
// Both are no-ops for a kernel launched without the attribute.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Launch with the programmatic stream-serialization attribute.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t st, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

__device__ __forceinline__ float tanh_fast(float x) {
  float y;
  asm("tanh.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

__device__ __forceinline__ float2 unpack_bf16x2(uint32_t u) {
  __nv_bfloat162 h = *reinterpret_cast<__nv_bfloat162*>(&u);
  return __bfloat1622float2(h);
}

// ---------------------------------------------------------------------------
// Per-row PPO loss ("Teaching Mario to speedrun", sec. 6 "Don't move too far
// at once"; sec. 5 for d logp / d logits = 1[k==a] - p_k).  z holds the C
// output columns of one row (bias included).  Writes dz (already scaled by
// 1/mb), returns the six per-row terms and the per-row dlogstd contribution.
__device__ __forceinline__ void row_loss(const NetShape& s, const LossCoef& lc, float inv_mb,
                                         const float* z, const int32_t* act, const float* actc,
                                         const float* logstd, float logp_old, float A, float R,
                                         float* dz, float* terms6, float* dlogstd) {
  const float LOG_2PI = 1.8378770664093453f;
  float logp = 0.f, ent = 0.f;
  float head_ent[PPO_MAX_HEADS];
  int off = 0;
#pragma unroll 1
  for (int h = 0; h < s.NH; ++h) {
    const int n = s.head_n[h];
    float zmax = z[off];
    for (int k = 1; k < n; ++k) zmax = fmaxf(zmax, z[off + k]);
    float se = 0.f;
    for (int k = 0; k < n; ++k) se += expf(z[off + k] - zmax);
    const float lse = zmax + logf(se);
    float eh = 0.f;
    for (int k = 0; k < n; ++k) {
      const float lp = z[off + k] - lse;
      eh -= expf(lp) * lp;
    }
    head_ent[h] = eh;
    ent += eh;
    logp += z[off + act[h]] - lse;
    off += n;
  }
  for (int g = 0; g < s.G; ++g) {
    const float mu = z[off + g], ls = logstd[g];
    const float a = actc[g];
    const float inv_var = expf(-2.f * ls);
    logp += -0.5f * (a - mu) * (a - mu) * inv_var - ls - 0.5f * LOG_2PI;
    ent += 0.5f + 0.5f * LOG_2PI + ls;
  }
  const float value = z[s.C - 1];
  const float log_ratio = logp - logp_old;
  const float ratio = expf(log_ratio);
  const float lo = 1.f - lc.clip, hi = 1.f + lc.clip;
  const float clipped = fminf(fmaxf(ratio, lo), hi);
  const float s1 = ratio * A, s2 = clipped * A;
  const float pg = -fminf(s1, s2);
  const float vdiff = value - R;
  const float vl = vdiff * vdiff;
  terms6[0] = pg + lc.vf * vl - lc.ent * ent;
  terms6[1] = pg;
  terms6[2] = vl;
  terms6[3] = ent;
  terms6[4] = fabsf(ratio - 1.f) > lc.clip ? 1.f : 0.f;
  terms6[5] = (ratio - 1.f) - log_ratio;

  const float g_logp = (s1 <= s2) ? -A * ratio * inv_mb : 0.f;
  const float g_ent = -lc.ent * inv_mb;
  off = 0;
#pragma unroll 1
  for (int h = 0; h < s.NH; ++h) {
    const int n = s.head_n[h];
    float zmax = z[off];
    for (int k = 1; k < n; ++k) zmax = fmaxf(zmax, z[off + k]);
    float se = 0.f;
    for (int k = 0; k < n; ++k) se += expf(z[off + k] - zmax);
    const float lse = zmax + logf(se);
    for (int k = 0; k < n; ++k) {
      const float lp = z[off + k] - lse;
      const float p = expf(lp);
      const float dlogp = (k == act[h] ? 1.f : 0.f) - p;
      const float dent = -p * (lp + head_ent[h]);
      dz[off + k] = g_logp * dlogp + g_ent * dent;
    }
    off += n;
  }
  for (int g = 0; g < s.G; ++g) {
    const float mu = z[off + g], ls = logstd[g];
    const float a = actc[g];
    const float inv_var = expf(-2.f * ls);
    dz[off + g] = g_logp * (a - mu) * inv_var;
    dlogstd[g] = g_logp * ((a - mu) * (a - mu) * inv_var - 1.f) + g_ent;
  }
  dz[s.C - 1] = lc.vf * 2.f * vdiff * inv_mb;
}

// ---------------------------------------------------------------------------
// Kernel stages of one update; every stage is exactly one kernel launch.  A
// Trace hook, when set, is called on the launching stream after each launch
// (the profiler records a CUDA event there).
enum Stage : int {
  ST_PACK = 0, ST_GAE, ST_GAE_FINALIZE, ST_GAE_NORMALIZE, ST_PERM_HIST, ST_PERM_SCAN,
  ST_PERM_SCATTER, ST_GATHER, ST_FWD1, ST_FWD2, ST_LOSS, ST_DACT2, ST_DACT1, ST_WGRAD,
  ST_REDUCE, ST_SQNORM, ST_ADAM, ST_SHADOW, ST_MINIBATCH, ST_FUSED_MLP, ST_REDUCE_ADAM,
  ST_LOSS_DACT2, ST_FRESH_ADV, ST_POLICY_ACT, ST_MUON, ST_COUNT
};

struct Trace {
  void (*fn)(void* user, int stage, cudaStream_t st) = nullptr;
  void* user = nullptr;
  void mark(int stage, cudaStream_t st) const {
    if (fn) fn(user, stage, st);
  }
};

// ---------------------------------------------------------------------------
// Host-side launchers (defined in the .cu files).
// Longest horizon the GAE kernels accept: a warp's moment count (at most
// 32 * T) must stay exact in fp32 (below 2^24).
constexpr int64_t kGaeMaxT = 1 << 19;
cudaError_t launch_gae(const float* rew, const float* val, const float* done, const float* boot,
                       int T, int N, float gamma, float lambda, float* adv, float* ret,
                       double* partials, int num_partial_blocks, cudaStream_t st);
int gae_num_blocks(int N);
cudaError_t launch_gae_finalize(const double* partials, int nblocks, float* stats,
                                cudaStream_t st);
// The merged (count, mean, M2) of the per-block moments, fp64 triple[3] (a
// shard's moments, merged with other ranks' by launch_gae_finalize over the
// gathered triples).
cudaError_t launch_gae_moments(const double* partials, int nblocks, double* triple,
                               cudaStream_t st);
cudaError_t launch_normalize(const float* adv, const float* stats, float* out, int64_t n,
                             cudaStream_t st);

size_t perm_workspace_bytes(int64_t B, int epochs);
cudaError_t launch_perm(uint32_t seed, int64_t epoch0, int epochs, int64_t B, int32_t* perm,
                        void* work, cudaStream_t st, const Trace* tr = nullptr);

cudaError_t launch_pack_obs(const float* obs, int64_t B, int D, int Dp, __nv_bfloat16* out,
                            cudaStream_t st);

// Gather one minibatch: X (bf16 [mb][Dp] or fp32 [mb][D]) and per-row side data.
struct GatherArgs {
  const float* obs_f32;            // [B][D] (used when obs_bf16 == nullptr)
  const __nv_bfloat16* obs_bf16;   // [B][Dp] packed, or nullptr
  const int32_t* act;              // [B][NH]
  const float* actc;               // [B][G]
  const float* logp_old;           // [B]
  const float* adv;                // [B]
  const float* ret;                // [B]
  const float* adv_stats;          // [2] mean, std or nullptr
  const int32_t* idx;              // [mb], entries clamped to [0, B); unused with seg_envs
  int64_t mb;
  int64_t B;
  // segment rows instead of idx: row r = (m, t, j) with r = (m*T + t)*ns + j
  // gathers batch row t*seg_N + seg_envs[m*ns + j] (entries clamped to [0, seg_N))
  const int32_t* seg_envs;
  int seg_T, seg_ns;
  int64_t seg_N;
  // outputs
  void* X;                         // bf16 [mb][Dp] or fp32 [mb][D]
  int x_bf16;
  int32_t* act_mb;
  float* actc_mb;
  float* logp_mb;
  float* adv_mb;
  float* ret_mb;
};
cudaError_t launch_gather(const NetShape& s, const GatherArgs& a, cudaStream_t st);

// Advantages of a minibatch of environment segments from fresh values
// (fresh.cu).  Rows are ordered t*ns + j (segment j = environment envs[j]).
constexpr int kFreshMaxGrid = 1024;
struct FreshAdvArgs {
  // phase A (head != 0): value, and with ratio != nullptr the importance
  // ratio, of every row from the last hidden layer
  int head;
  NetShape s;
  const void* H2;          // [rows][H2], bf16 (h2_bf16) or fp32
  int h2_bf16;
  const void* W3;          // bf16 shadow [CP][H2] or fp32 [C][H2]
  const float* b3;
  const float* logstd;
  const int32_t* act;      // [rows][NH]
  const float* actc;       // [rows][G]
  const float* logp_old;   // [rows]
  // phase B
  const float* rew;        // [T][N]
  const float* done;       // [T][N]
  const float* boot;       // [N]
  const int32_t* envs;     // [ns]
  int T, ns;
  int64_t N;
  float* val;              // [rows] (written by phase A, else given)
  float* ratio;            // [rows] or nullptr (GAE)
  float gamma, lambda, rho_clip, c_clip;
  float* adv;              // [rows] advantages
  float* ret;              // [rows] value targets
  float* adv_norm;         // [rows] normalised advantages (may equal adv), or nullptr
  float* stats;            // [2] {mean, unbiased std} of adv, or nullptr
  float* part;             // [kFreshMaxGrid][3] per-block (count, mean, M2)
  unsigned* bar;           // zero on entry; reset to zero by the launch
  int* err;
  uint64_t timeout_ns;
};
cudaError_t fresh_prepare();
cudaError_t launch_fresh_adv(const FreshAdvArgs& a, int num_sms, cudaStream_t st);

// Rollout-side policy step (act.cu): sampled actions, log-probability of the
// stored action and value for n agents, from the last hidden layer.
struct PolicyActArgs {
  NetShape s;
  const void* h;           // [n][H2], bf16 (h_bf16) or fp32
  int h_bf16;
  const void* W3;          // bf16 shadow [CP][H2] or fp32 [C][H2]
  const float* b3;
  const float* logstd;
  int64_t n;
  uint32_t seed;
  uint64_t draw0;
  int32_t* act;            // [n][NH]
  float* actc;             // [n][G]
  float* logp;             // [n] or nullptr
  float* value;            // [n] or nullptr
};
cudaError_t policy_act_prepare();
cudaError_t launch_policy_act(const PolicyActArgs& a, cudaStream_t st);

// Loss and gradient of the recurrent MinGRU policy over a minibatch of
// environment segments (rnn.cu).  params / grad in the recurrent layout:
// W_enc[H][D], per layer W_z[H][H], b_z[H], W_h[H][H], b_h[H], W_dec[C][H],
// logstd[G].  s carries the head layout (NH, head_n, G, C).
struct RnnLaunch {
  NetShape s;
  LossCoef lc;
  int T, ns, D, H, L;
  int64_t N;
  const float* params;
  const int32_t* envs;      // [ns]
  const float* obs;         // [T*N][D]
  const int32_t* act;       // [T*N][NH]
  const float* actc;        // [T*N][G]
  const float* logp_old;    // [T*N]
  const float* adv;         // [T*N]
  const float* ret;         // [T*N]
  const float* adv_stats;   // [2] or nullptr
  const float* done;        // [T][N]
  const float* h0;          // [N][L][H]
  float* grad;
  float* stats6;            // [6] or nullptr
  float* work;              // rnn_workspace_floats(D, H, L, T*ns)
  int* err;                 // tensor-core path: error word of bounded waits (nullptr:
                            // the workspace's own, cleared at the call's start)
};
size_t rnn_workspace_floats(int D, int H, int L, int64_t rows);
cudaError_t launch_rnn_loss_grad(const RnnLaunch& a, cudaStream_t st);

}  // namespace ppo
