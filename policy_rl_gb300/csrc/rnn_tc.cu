// rnn_tc.cu -- loss and BPTT gradient of the recurrent (MinGRU) policy with
// every dense product on the bf16 tensor-core kernels of gemm_tc.cu.
//
// "Teaching Mario to speedrun", sec. 8 "The Puffer net, and the trainer": a
// bias-free encoder, MinGRU layers (Feng et al. 2024: z = sigmoid(W_z u +
// b_z), h~ = W_h u + b_h, h = (1 - z) h_prev + z h~, the state cleared after
// a terminal), one decoder matrix to the heads and the value.  For a
// minibatch of environment segments (rows r = t*ns + j, segment j = env
// envs[j], t < T):
//   X  = obs rows (bf16, padded to Dp)          gather
//   U0 = X W_enc^T                              tcgen05 GEMM (plain epilogue)
//   per layer: PRE = U_l [W_z; W_h]^T + [b_z; b_h]   tcgen05 GEMM, [rows][2H]
//              forward scan -> states H_l (fp32), U_{l+1} = bf16(H_l)
//   z = W_dec U_L, per-row PPO loss, dz (bf16)  CUDA cores (C <= 32 columns)
//   dIn = dz W_dec                              tcgen05 GEMM
//   per layer, top down: backward scan -> dP = [dpz | dph] (bf16) and the
//              bias sums; dU = dP [W_z; W_h]      tcgen05 GEMM;
//              dW_z, dW_h = dP^T U_l            weight-gradient kernel
//   dW_dec, dW_enc                              weight-gradient kernel
// The stored operands are bf16, accumulation fp32; the recurrence and the
// bias gradients stay fp32 (the oracle's bf16-operand reading of the policy).
//
// The scans are chunked affine scans along time (see rnn_fwd_scan_tc_kernel):
// a warp covers 32 consecutive units of one segment and one chunk of steps,
// so every [rows][H] access is coalesced and a chunk's loads are all in
// flight at once.
#include <utility>

#include "common.cuh"
#include "gemm.h"
#include "tc_tile.cuh"

namespace ppo {

namespace {

constexpr int kLossThreads = 128;
constexpr uint64_t kWaitNs = 2000000000ull;

struct Dims {
  int T, ns, D, Dp, H, L, C, G;
  int64_t N, rows;
};

__device__ __forceinline__ int64_t seg_env(const int32_t* envs, int j, int64_t N) {
  int64_t e = __ldg(envs + j);
  return e < 0 ? 0 : (e >= N ? N - 1 : e);
}

__device__ __forceinline__ float bf(float x) { return __bfloat162float(__float2bfloat16_rn(x)); }
__device__ __forceinline__ float sigm(float x) { return 1.f / (1.f + expf(-x)); }

// bf16 operand forms of the weights and the concatenated biases:
//   Wenc_s [H][Dp] (zero beyond D), Wcat_s[l] [2H][H] (rows of W_z, then W_h),
//   WcatT_s[l] [H][2H] (its transpose), WdecT_s [H][64] (W_dec^T, zero beyond C),
//   bcat[l] [2H] fp32 (b_z, then b_h).
__global__ void rnn_shadow_kernel(Dims d, const float* __restrict__ P,
                                  __nv_bfloat16* __restrict__ Wenc_s,
                                  __nv_bfloat16* __restrict__ Wcat_s,
                                  __nv_bfloat16* __restrict__ WcatT_s,
                                  __nv_bfloat16* __restrict__ WdecT_s, float* __restrict__ bcat) {
  const int H = d.H;
  const int64_t per = 2ll * H * H + 2 * H, oL = (int64_t)H * d.D, oDec = oL + d.L * per;
  const int64_t HH2 = 2ll * H * H;
  const int64_t n1 = (int64_t)H * d.Dp, n2 = d.L * HH2, n4 = (int64_t)H * 64,
                n5 = 2ll * H * d.L;
  const int64_t total = n1 + 2 * n2 + n4 + n5;
  auto wcat = [&](int l, int r, int k) {   // [W_z; W_h] row r, column k
    const int64_t b = oL + l * per;
    return r < H ? P[b + (int64_t)r * H + k] : P[b + (int64_t)H * H + H + (int64_t)(r - H) * H + k];
  };
  for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < total;
       e += (int64_t)gridDim.x * blockDim.x) {
    if (e < n1) {
      const int i = (int)(e / d.Dp), k = (int)(e % d.Dp);
      Wenc_s[e] = __float2bfloat16_rn(k < d.D ? P[(int64_t)i * d.D + k] : 0.f);
    } else if (e < n1 + n2) {
      const int64_t q = e - n1;
      const int l = (int)(q / HH2);
      const int64_t rem = q % HH2;
      Wcat_s[q] = __float2bfloat16_rn(wcat(l, (int)(rem / H), (int)(rem % H)));
    } else if (e < n1 + 2 * n2) {
      const int64_t q = e - n1 - n2;
      const int l = (int)(q / HH2);
      const int64_t rem = q % HH2;
      const int i = (int)(rem / (2 * H)), c = (int)(rem % (2 * H));
      WcatT_s[q] = __float2bfloat16_rn(wcat(l, c, i));
    } else if (e < n1 + 2 * n2 + n4) {
      const int64_t q = e - n1 - 2 * n2;
      const int i = (int)(q / 64), c = (int)(q % 64);
      WdecT_s[q] = __float2bfloat16_rn(c < d.C ? P[oDec + (int64_t)c * H + i] : 0.f);
    } else {
      const int64_t q = e - n1 - 2 * n2 - n4;
      const int l = (int)(q / (2 * H)), c = (int)(q % (2 * H));
      const int64_t b = oL + l * per;
      bcat[q] = c < H ? P[b + (int64_t)H * H + c] : P[b + 2ll * H * H + H + (c - H)];
    }
  }
}

// X[r][k] = bf16(obs[(t N + env_j) D + k]) for k < D, 0 up to Dp.
__global__ void rnn_gather_bf16_kernel(Dims d, const float* __restrict__ obs,
                                       const int32_t* __restrict__ envs,
                                       __nv_bfloat16* __restrict__ X) {
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= d.rows * d.Dp) return;
  const int64_t r = i / d.Dp;
  const int k = (int)(i - r * d.Dp);
  const int t = (int)(r / d.ns), j = (int)(r - (int64_t)t * d.ns);
  X[i] = __float2bfloat16_rn(
      k < d.D ? __ldg(obs + ((int64_t)t * d.N + seg_env(envs, j, d.N)) * d.D + k) : 0.f);
}

// The recurrences are affine in the carried value, so the horizon is cut
// into chunks of kCL steps scanned in parallel: a block covers 32 units of
// one segment (blockIdx.y) and kCS chunks (one warp each); a round of kCS
// chunks at a time, carrying the state from round to round.  Each warp loads
// its chunk's inputs at once (all loads in flight), composes the chunk's map
// x_end = A x_start + B, the maps are combined in time order through shared
// memory, and each warp replays its chunk from its exact incoming value.
constexpr int kCL = 16;   // steps per chunk
constexpr int kCS = 8;    // chunks per round (warps per block)

// Forward recurrence of layer l: h_t = a_t h_{t-1} + b_t with a_t = (1 - z_t)
// m_t, b_t = z_t h~_t (m_t = 0 when the episode ended at t - 1).
// PRE [rows][2H] = [pz | ph] (bf16), Hs [rows][H] fp32 states, Un [rows][H]
// bf16 states (the next layer's operand).
__global__ void __launch_bounds__(32 * kCS)
rnn_fwd_scan_tc_kernel(Dims d, int l, const float* __restrict__ done,
                       const int32_t* __restrict__ envs, const float* __restrict__ h0,
                       const __nv_bfloat16* __restrict__ PRE, float* __restrict__ Hs,
                       __nv_bfloat16* __restrict__ Un) {
  __shared__ float mA[kCS][32], mB[kCS][32], carry[32];
  const int lane = threadIdx.x % 32, c = threadIdx.x / 32;
  const int j = blockIdx.y, i = blockIdx.x * 32 + lane;
  const bool on = i < d.H;
  const int H = d.H;
  const int64_t e = seg_env(envs, j, d.N);
  if (c == 0) carry[lane] = on ? __ldg(h0 + (e * d.L + l) * H + i) : 0.f;
  for (int t_r = 0; t_r < d.T; t_r += kCS * kCL) {
    const int t0 = t_r + c * kCL;
    float a[kCL], b[kCL];
#pragma unroll
    for (int u = 0; u < kCL; ++u) {
      const int t = t0 + u;
      float pz = 0.f, ph = 0.f, m = 1.f;
      if (on && t < d.T) {
        const int64_t o = ((int64_t)t * d.ns + j) * 2 * H + i;
        pz = __bfloat162float(PRE[o]);
        ph = __bfloat162float(PRE[o + H]);
        if (t > 0 && __ldg(done + (int64_t)(t - 1) * d.N + e) != 0.f) m = 0.f;
      }
      const float z = sigm(pz);
      a[u] = (t < d.T) ? (1.f - z) * m : 1.f;   // steps past the horizon: identity
      b[u] = (t < d.T) ? z * ph : 0.f;
    }
    float A = 1.f, B = 0.f;
#pragma unroll
    for (int u = 0; u < kCL; ++u) {
      A = a[u] * A;
      B = a[u] * B + b[u];
    }
    mA[c][lane] = A;
    mB[c][lane] = B;
    __syncthreads();
    float h = carry[lane];
    for (int cc = 0; cc < c; ++cc) h = mA[cc][lane] * h + mB[cc][lane];
#pragma unroll
    for (int u = 0; u < kCL; ++u) {
      const int t = t0 + u;
      h = a[u] * h + b[u];
      if (on && t < d.T) {
        const int64_t o = ((int64_t)t * d.ns + j) * H + i;
        Hs[o] = h;
        Un[o] = __float2bfloat16_rn(h);
      }
    }
    __syncthreads();                       // every warp has read carry and the maps
    if (c == kCS - 1) carry[lane] = h;     // the state after this round
    __syncthreads();
  }
}

// Backward recurrence of layer l, reverse time.  With dIn [rows][H] (bf16)
// dL/dh from above and x_t the gradient flowing into h_t from step t + 1:
// dh_t = dIn_t + x_{t+1}, x_t = c_t dh_t with c_t = (1 - z_t) m_t, so
// x_t = c_t x_{t+1} + c_t dIn_t.  dP [rows][2H] receives bf16 [dpz | dph]
// (dpz = dh (h~ - hp) z (1 - z), dph = dh z, hp = m_t h_{t-1}); bsum [ns][2H]
// the per-segment sums of dpz, dph (fp32, for the bias gradients).
__global__ void __launch_bounds__(32 * kCS, 3)
rnn_bwd_scan_tc_kernel(Dims d, int l, const float* __restrict__ done,
                       const int32_t* __restrict__ envs, const float* __restrict__ h0,
                       const __nv_bfloat16* __restrict__ PRE, const float* __restrict__ Hs,
                       const __nv_bfloat16* __restrict__ dIn, __nv_bfloat16* __restrict__ dP,
                       float* __restrict__ bsum) {
  __shared__ float mA[kCS][32], mB[kCS][32], carry[32], ssz[kCS][32], ssh[kCS][32];
  const int lane = threadIdx.x % 32, c = threadIdx.x / 32;
  const int j = blockIdx.y, i = blockIdx.x * 32 + lane;
  const bool on = i < d.H;
  const int H = d.H;
  const int64_t e = seg_env(envs, j, d.N);
  const float hinit = on ? __ldg(h0 + (e * d.L + l) * H + i) : 0.f;
  if (c == 0) carry[lane] = 0.f;
  float sz = 0.f, sh = 0.f;
  const int rounds = (d.T + kCS * kCL - 1) / (kCS * kCL);
  for (int r = rounds - 1; r >= 0; --r) {
    const int t0 = r * kCS * kCL + c * kCL;
    // per step: the gate (from pz), h~, the masked previous state, dIn; the
    // factor c_t = (1 - z_t) m_t is recomputed where it is needed
    float z[kCL], ph[kCL], hp[kCL], di[kCL];
#pragma unroll
    for (int u = 0; u < kCL; ++u) {
      const int t = t0 + u;
      float pz = 0.f, hprev = 0.f;
      ph[u] = di[u] = 0.f;
      if (on && t < d.T) {
        const int64_t o = (int64_t)t * d.ns + j;
        pz = __bfloat162float(PRE[o * 2 * H + i]);
        ph[u] = __bfloat162float(PRE[o * 2 * H + H + i]);
        di[u] = __bfloat162float(dIn[o * H + i]);
        if (t > 0) {
          if (__ldg(done + (int64_t)(t - 1) * d.N + e) == 0.f) hprev = Hs[(o - d.ns) * H + i];
        } else {
          hprev = hinit;
        }
      }
      z[u] = sigm(pz);
      hp[u] = hprev;   // m_t h_{t-1}: zero after a terminal
    }
    // m_t of step t0 + u (1 past the horizon: identity steps)
    auto cfac = [&](int u) {
      const int t = t0 + u;
      if (t >= d.T) return 1.f;
      const bool cut = t > 0 && __ldg(done + (int64_t)(t - 1) * d.N + e) != 0.f;
      return cut ? 0.f : 1.f - z[u];
    };
    float A = 1.f, B = 0.f;   // x_{t0} = A x_{t0 + kCL} + B
#pragma unroll
    for (int u = kCL - 1; u >= 0; --u) {
      const float cf = cfac(u);
      A = cf * A;
      B = cf * (B + di[u]);
    }
    mA[c][lane] = A;
    mB[c][lane] = B;
    __syncthreads();
    float x = carry[lane];
    for (int cc = kCS - 1; cc > c; --cc) x = mA[cc][lane] * x + mB[cc][lane];
#pragma unroll
    for (int u = kCL - 1; u >= 0; --u) {
      const int t = t0 + u;
      if (on && t < d.T) {
        const float dh = di[u] + x;
        const float dpz = dh * (ph[u] - hp[u]) * z[u] * (1.f - z[u]);
        const float dph = dh * z[u];
        x = dh * cfac(u);
        const int64_t o = ((int64_t)t * d.ns + j) * 2 * H + i;
        dP[o] = __float2bfloat16_rn(dpz);
        dP[o + H] = __float2bfloat16_rn(dph);
        sz += dpz;
        sh += dph;
      }
    }
    __syncthreads();                 // every warp has read carry and the maps
    if (c == 0) carry[lane] = x;     // the flow into the step before this round
    __syncthreads();
  }
  ssz[c][lane] = sz;
  ssh[c][lane] = sh;
  __syncthreads();
  if (c == 0 && on) {
    float a0 = 0.f, a1 = 0.f;
    for (int cc = 0; cc < kCS; ++cc) {
      a0 += ssz[cc][lane];
      a1 += ssh[cc][lane];
    }
    bsum[(int64_t)j * 2 * H + i] = a0;
    bsum[(int64_t)j * 2 * H + H + i] = a1;
  }
}

// Decoder z = W_dec u (thread per row; W_dec rounded to bf16 and staged as
// [H][32]), then the per-row PPO loss epilogue of the MLP path: dz [rows][64]
// bf16 (zero beyond C) and per-block partials {6 loss terms, dlogstd[4]}.
__global__ void __launch_bounds__(kLossThreads)
rnn_loss_tc_kernel(Dims d, NetShape s, LossCoef lc, const float* __restrict__ Wdec,
                   const float* __restrict__ logstd, const __nv_bfloat16* __restrict__ Utop,
                   const int32_t* __restrict__ act, const float* __restrict__ actc,
                   const float* __restrict__ logp_old, const float* __restrict__ adv,
                   const float* __restrict__ ret, const float* adv_stats,
                   const int32_t* __restrict__ envs, float inv_mb,
                   __nv_bfloat16* __restrict__ dz, float* __restrict__ part) {
  extern __shared__ float wsm[];   // [H][32]
  for (int e = threadIdx.x; e < d.H * 32; e += kLossThreads) {
    const int k = e / 32, c = e % 32;
    wsm[e] = c < d.C ? bf(Wdec[(int64_t)c * d.H + k]) : 0.f;
  }
  __syncthreads();
  const int64_t r = (int64_t)blockIdx.x * kLossThreads + threadIdx.x;
  float t6[6] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f}, dls[4] = {0.f, 0.f, 0.f, 0.f};
  if (r < d.rows) {
    float z[32];
#pragma unroll
    for (int c = 0; c < 32; ++c) z[c] = 0.f;
    const __nv_bfloat16* h = Utop + r * d.H;
    for (int k = 0; k < d.H; ++k) {
      const float hk = __bfloat162float(h[k]);
#pragma unroll
      for (int c = 0; c < 32; ++c) z[c] = fmaf(wsm[k * 32 + c], hk, z[c]);
    }
    const int t = (int)(r / d.ns), j = (int)(r - (int64_t)t * d.ns);
    const int64_t src = (int64_t)t * d.N + seg_env(envs, j, d.N);
    uint32_t amask = 0u;
    int off = 0;
    for (int hh = 0; hh < s.NH; ++hh) {
      int a = __ldg(act + src * s.NH + hh);
      a = a < 0 ? 0 : (a >= s.head_n[hh] ? s.head_n[hh] - 1 : a);
      amask |= 1u << (off + a);
      off += s.head_n[hh];
    }
    float A = __ldg(adv + src);
    if (adv_stats) A = (A - __ldg(adv_stats)) / (__ldg(adv_stats + 1) + 1e-8f);
    const tc::HeadMasks hm = tc::head_masks(s);
    float dzr[32];
    tc::row_loss_seg<32>(hm, lc, inv_mb, z, amask, actc + src * s.G, logstd,
                         __ldg(logp_old + src), A, __ldg(ret + src), dzr, t6, dls);
    __nv_bfloat16* o = dz + r * 64;
#pragma unroll
    for (int c = 0; c < 64; c += 2) {
      const float a0 = c < d.C ? dzr[c < 32 ? c : 0] : 0.f;
      const float a1 = c + 1 < d.C ? dzr[c + 1 < 32 ? c + 1 : 0] : 0.f;
      *reinterpret_cast<__nv_bfloat162*>(o + c) = __floats2bfloat162_rn(a0, a1);
    }
  }
  // fixed-order block reduction of the 10 partials
  __shared__ float red[kLossThreads / 32][10];
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  float v[10] = {t6[0], t6[1], t6[2], t6[3], t6[4], t6[5], dls[0], dls[1], dls[2], dls[3]};
#pragma unroll
  for (int q = 0; q < 10; ++q) {
    const float x = warp_sum(v[q]);
    if (lane == 0) red[w][q] = x;
  }
  __syncthreads();
  if (threadIdx.x < 10) {
    float x = 0.f;
    for (int ww = 0; ww < kLossThreads / 32; ++ww) x += red[ww][threadIdx.x];
    part[(int64_t)blockIdx.x * 10 + threadIdx.x] = x;
  }
}

// stats6 = mean of the six loss terms and the log-std gradient (blocks in
// order); the bias gradients: one warp per column of [b_z | b_h] of a layer,
// lane l summing segments l, l + 32, ... (eight loads in flight), then a
// fixed xor-shuffle tree.
constexpr int kFinThreads = 256;
__global__ void __launch_bounds__(kFinThreads)
rnn_tc_finalize_kernel(Dims d, int nblocks, const float* __restrict__ part,
                       const float* __restrict__ bsum, float inv_mb, float* stats6, float* G) {
  const int H = d.H;
  const int64_t per = 2ll * H * H + 2 * H, oL = (int64_t)H * d.D;
  const int64_t ologstd = oL + d.L * per + (int64_t)d.C * H;
  const int lane = threadIdx.x % 32;
  const int w = blockIdx.x * (kFinThreads / 32) + threadIdx.x / 32;
  if (w == 0) {
    if (lane < 10) {
      float x = 0.f;
      for (int b = 0; b < nblocks; ++b) x += part[(int64_t)b * 10 + lane];
      if (lane < 6) {
        if (stats6) stats6[lane] = x * inv_mb;
      } else if (lane - 6 < d.G) {
        G[ologstd + (lane - 6)] = x;
      }
    }
    return;
  }
  const int q = w - 1;
  if (q >= d.L * 2 * H) return;
  const int l = q / (2 * H), c = q % (2 * H);
  const float* b = bsum + (int64_t)l * d.ns * 2 * H + c;
  float v = 0.f;
  for (int j0 = lane; j0 < d.ns; j0 += 8 * 32) {
    float x[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int j = j0 + 32 * u;
      x[u] = j < d.ns ? b[(int64_t)j * 2 * H] : 0.f;
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) v += x[u];
  }
  v = warp_sum(v);
  if (lane == 0) G[oL + l * per + (c < H ? (int64_t)H * H + c : 2ll * H * H + H + (c - H))] = v;
}

// Workspace layout (256-byte aligned pieces).
struct Work {
  int* err;
  unsigned* tile_ctr;
  double* sq;
  __nv_bfloat16 *Wenc_s, *Wcat_s, *WcatT_s, *WdecT_s;
  float* bcat;
  __nv_bfloat16 *X, *U, *PRE, *dz, *dIn, *dU, *dP;
  float *Hs, *bsum, *part, *wpart;
  size_t bytes;
};

size_t wpart_floats(int Dp, int H) {
  const size_t layer = 2ull * kMaxWgSplit * H * H;
  const size_t fin = (size_t)kMaxWgSplit * H * 64 + (size_t)kMaxWgSplit * H * Dp;
  return layer > fin ? layer : fin;
}

Work carve(void* base, int D, int H, int L, int64_t T, int64_t ns, int num_sms) {
  const int Dp = (D + 63) / 64 * 64;
  const int64_t rows = T * ns;
  Work w{};
  // the error word at the start, then pieces at 256-byte boundaries
  const uintptr_t p0 = reinterpret_cast<uintptr_t>(base);
  uintptr_t p = p0 + 16;
  auto take = [&](size_t bytes) {
    p = (p + 255) & ~uintptr_t(255);
    const uintptr_t r = p;
    p += bytes;
    return reinterpret_cast<void*>(r);
  };
  const size_t b2 = sizeof(__nv_bfloat16);
  w.err = reinterpret_cast<int*>(p0);
  w.tile_ctr = static_cast<unsigned*>(take(2 * kWgradMaxTiles * sizeof(unsigned)));
  w.sq = static_cast<double*>(take((size_t)(num_sms > 256 ? num_sms : 256) * sizeof(double)));
  w.Wenc_s = static_cast<__nv_bfloat16*>(take((size_t)H * Dp * b2));
  w.Wcat_s = static_cast<__nv_bfloat16*>(take((size_t)L * 2 * H * H * b2));
  w.WcatT_s = static_cast<__nv_bfloat16*>(take((size_t)L * 2 * H * H * b2));
  w.WdecT_s = static_cast<__nv_bfloat16*>(take((size_t)H * 64 * b2));
  w.bcat = static_cast<float*>(take((size_t)L * 2 * H * sizeof(float)));
  w.X = static_cast<__nv_bfloat16*>(take((size_t)rows * Dp * b2));
  w.U = static_cast<__nv_bfloat16*>(take((size_t)(L + 1) * rows * H * b2));
  w.PRE = static_cast<__nv_bfloat16*>(take((size_t)L * rows * 2 * H * b2));
  w.dz = static_cast<__nv_bfloat16*>(take((size_t)rows * 64 * b2));
  w.dIn = static_cast<__nv_bfloat16*>(take((size_t)rows * H * b2));
  w.dU = static_cast<__nv_bfloat16*>(take((size_t)rows * H * b2));
  w.dP = static_cast<__nv_bfloat16*>(take((size_t)rows * 2 * H * b2));
  w.Hs = static_cast<float*>(take((size_t)L * rows * H * sizeof(float)));
  w.bsum = static_cast<float*>(take((size_t)L * ns * 2 * H * sizeof(float)));
  w.part = static_cast<float*>(take((10 * ((rows + kLossThreads - 1) / kLossThreads) + 64) *
                                    sizeof(float)));
  w.wpart = static_cast<float*>(take(wpart_floats(Dp, H) * sizeof(float)));
  w.bytes = (p - p0) + 256;
  return w;
}

}  // namespace

bool rnn_tc_supported(int D, int H) { return (H == 128 || H == 256) && D >= 1; }

size_t rnn_tc_workspace_bytes(int D, int H, int L, int64_t T, int64_t ns, int num_sms) {
  return carve(nullptr, D, H, L, T, ns, num_sms).bytes;
}

cudaError_t launch_rnn_loss_grad_tc(const RnnLaunch& a, int num_sms, cudaStream_t st,
                                    int** err_out) {
  const int D = a.D, H = a.H, L = a.L, C = a.s.C;
  const int Dp = (D + 63) / 64 * 64;
  const int64_t rows = (int64_t)a.T * a.ns;
  if (!rnn_tc_supported(D, H) || rows >= (1ll << 31)) return cudaErrorInvalidValue;
  Dims d{a.T, a.ns, D, Dp, H, L, C, a.s.G, a.N, rows};
  Work w = carve(a.work, D, H, L, a.T, a.ns, num_sms);
  const bool own_err = a.err == nullptr;
  if (!own_err) w.err = a.err;
  if (err_out) *err_out = w.err;
  const float* P = a.params;
  const int64_t per = 2ll * H * H + 2 * H, oL = (int64_t)H * D, oDec = oL + L * per;
  float* G = a.grad;
  const float inv_mb = 1.f / (float)rows;
  cudaError_t e;
#define RTC_TRY(x) do { if ((e = (x)) != cudaSuccess) return e; } while (0)
  if (own_err) RTC_TRY(cudaMemsetAsync(w.err, 0, sizeof(int), st));
  RTC_TRY(cudaMemsetAsync(w.tile_ctr, 0, 2 * kWgradMaxTiles * sizeof(unsigned), st));
  {
    const int64_t tot = (int64_t)H * Dp + 4ll * L * H * H + (int64_t)H * 64 + 2ll * L * H;
    rnn_shadow_kernel<<<(unsigned)((tot + 255) / 256), 256, 0, st>>>(d, P, w.Wenc_s, w.Wcat_s,
                                                                   w.WcatT_s, w.WdecT_s, w.bcat);
    RTC_TRY(cudaGetLastError());
  }
  rnn_gather_bf16_kernel<<<(unsigned)((rows * Dp + 255) / 256), 256, 0, st>>>(d, a.obs, a.envs,
                                                                             w.X);
  RTC_TRY(cudaGetLastError());
  const int M = (int)rows;
  auto Ul = [&](int l) { return w.U + (size_t)l * rows * H; };
  // encoder: U0 = X W_enc^T (a plain product)
  RTC_TRY(tc_gemm_bias_act(GemmOperands{w.X, Dp, w.Wenc_s, Dp, M, H, Dp}, nullptr, 2, Ul(0), H,
                           w.err, kWaitNs, num_sms, st));
  const dim3 sgrid((unsigned)((H + 31) / 32), (unsigned)a.ns);
  for (int l = 0; l < L; ++l) {
    __nv_bfloat16* PRE = w.PRE + (size_t)l * rows * 2 * H;
    RTC_TRY(tc_gemm_bias_act(
        GemmOperands{Ul(l), H, w.Wcat_s + (size_t)l * 2 * H * H, H, M, 2 * H, H},
        w.bcat + (size_t)l * 2 * H, 2, PRE, 2 * H, w.err, kWaitNs, num_sms, st));
    rnn_fwd_scan_tc_kernel<<<sgrid, 32 * kCS, 0, st>>>(d, l, a.done, a.envs, a.h0, PRE,
                                                           w.Hs + (size_t)l * rows * H, Ul(l + 1));
    RTC_TRY(cudaGetLastError());
  }
  // decoder + loss -> dz (bf16)
  const int lblocks = (int)((rows + kLossThreads - 1) / kLossThreads);
  rnn_loss_tc_kernel<<<lblocks, kLossThreads, (size_t)H * 32 * sizeof(float), st>>>(
      d, a.s, a.lc, P + oDec, P + oDec + (int64_t)C * H, Ul(L), a.act, a.actc, a.logp_old,
      a.adv, a.ret, a.adv_stats, a.envs, inv_mb, w.dz, w.part);
  RTC_TRY(cudaGetLastError());
  // dIn = dz W_dec
  RTC_TRY(tc_gemm_bias_act(GemmOperands{w.dz, 64, w.WdecT_s, 64, M, H, 64}, nullptr, 2, w.dIn,
                           H, w.err, kWaitNs, num_sms, st));
  __nv_bfloat16 *din = w.dIn, *dout = w.dU;
  const size_t lp = (size_t)kMaxWgSplit * H * H;   // partials of one layer region
  for (int l = L - 1; l >= 0; --l) {
    const __nv_bfloat16* PRE = w.PRE + (size_t)l * rows * 2 * H;
    rnn_bwd_scan_tc_kernel<<<sgrid, 32 * kCS, 0, st>>>(
        d, l, a.done, a.envs, a.h0, PRE, w.Hs + (size_t)l * rows * H, din, w.dP,
        w.bsum + (size_t)l * a.ns * 2 * H);
    RTC_TRY(cudaGetLastError());
    // dU = dP [W_z; W_h] (the layer below's dL/dh)
    RTC_TRY(tc_gemm_bias_act(
        GemmOperands{w.dP, 2 * H, w.WcatT_s + (size_t)l * 2 * H * H, 2 * H, M, H, 2 * H},
        nullptr, 2, dout, H, w.err, kWaitNs, num_sms, st));
    // dW_z = dpz^T U_l, dW_h = dph^T U_l, assembled into the gradient in-kernel
    const int mn[2][2] = {{H, H}, {H, H}};
    int kt[2];
    tc_wgrad_plan(mn, 2, rows, num_sms, kMaxWgSplit, kt);
    float* gWz = G + oL + l * per;
    float* gWh = gWz + (int64_t)H * H + H;
    WGradRegion regs[2] = {{w.dP, 2 * H, H, Ul(l), H, H, kt[0], w.wpart, {gWz, H, H, H, 1}},
                           {w.dP + H, 2 * H, H, Ul(l), H, H, kt[1], w.wpart + lp,
                            {gWh, H, H, H, 1}}};
    RTC_TRY(tc_wgrad(regs, 2, M, 8192, 1024, w.err, kWaitNs, num_sms, st, w.tile_ctr, w.sq,
                     nullptr, kWaitNs, nullptr));
    std::swap(din, dout);
  }
  // dW_dec (from its transpose: P[k][c] = sum_r U_L[r][k] dz[r][c]) and dW_enc
  {
    const int mn[2][2] = {{H, 64}, {H, Dp}};
    int kt[2];
    tc_wgrad_plan(mn, 2, rows, num_sms, kMaxWgSplit, kt);
    WGradRegion regs[2] = {
        {Ul(L), H, H, w.dz, 64, 64, kt[0], w.wpart, {G + oDec, H, C, 1, H}},
        {din, H, H, w.X, Dp, Dp, kt[1], w.wpart + (size_t)kMaxWgSplit * H * 64,
         {G, H, D, D, 1}}};
    RTC_TRY(tc_wgrad(regs, 2, M, 8192, 1024, w.err, kWaitNs, num_sms, st, w.tile_ctr, w.sq,
                     nullptr, kWaitNs, nullptr));
  }
  {
    const int warps = 1 + 2 * L * H, per_block = kFinThreads / 32;
    rnn_tc_finalize_kernel<<<(unsigned)((warps + per_block - 1) / per_block), kFinThreads, 0,
                             st>>>(d, lblocks, w.part, w.bsum, inv_mb, a.stats6, G);
  }
  RTC_TRY(cudaGetLastError());
#undef RTC_TRY
  return cudaSuccess;
}

}  // namespace ppo
