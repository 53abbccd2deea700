// fresh.cu -- per-minibatch advantages from fresh values.
//
// "Teaching Mario to speedrun", sec. 8 "The Puffer net, and the trainer":
// PufferLib 5.0 recomputes the advantages of every minibatch from fresh
// values, by GAE or by V-trace.  A minibatch here is a set of whole
// environment segments (env e over the horizon t = 0..T-1), its rows ordered
// t*ns + j for segment j.  V-trace follows Espeholt et al. 2018 ("IMPALA",
// sec. 4.1): with rho_t = min(rho_bar, pi/mu) and c_t = lambda min(c_bar, pi/mu),
//   A_t = v_t - V_t = rho_t delta_t + gamma c_t (1 - d_t) A_{t+1},
//   delta_t = r_t + gamma (1 - d_t) V_{t+1} - V_t,   ret_t = A_t + V_t,
// and GAE is the on-policy case (rho = 1, c = lambda).
//
// One cooperative launch, three phases separated by bounded grid barriers:
//  A (optional) fresh values: one warp per row, V = w_V . h2 + b_V from the
//    last hidden layer the forward pass just wrote (and, for V-trace, all
//    head columns -> log-probability of the taken action -> the ratio);
//  B the segment scan: one warp per segment; the recursion is affine in
//    A_{t+1} (A_t = b_t + a_t A_{t+1}), so each lane composes the maps of a
//    run of K steps, a suffix scan over the lanes composes the runs, and each
//    lane then replays its K steps from the exact incoming value.  Windows of
//    32 K steps are chained from the end of the horizon.  Each lane keeps
//    (n, mean, M2) of its advantages in fp64 (Welford; Chan merges upward);
//  C every block merges all blocks' moments in the same fixed order, and the
//    advantages are normalised in place: (A - mean) / (std + 1e-8), std the
//    unbiased estimate.
#include "common.cuh"
#include "tc_ptx.cuh"

namespace ppo {

namespace {

constexpr int kFreshThreads = 256;
constexpr int kFreshWarps = kFreshThreads / 32;
constexpr int kRun = 4;   // steps per lane per window

struct Mom {
  double n, mean, m2;
};

__device__ __forceinline__ Mom mom_merge(Mom a, Mom b) {
  if (a.n == 0.0) return b;
  if (b.n == 0.0) return a;
  const double n = a.n + b.n;
  const double d = b.mean - a.mean;
  Mom r;
  r.n = n;
  r.mean = a.mean + d * (b.n / n);
  r.m2 = a.m2 + b.m2 + d * d * (a.n * b.n / n);
  return r;
}

__device__ __forceinline__ Mom mom_shfl(Mom m, int o) {
  Mom r;
  r.n = __shfl_xor_sync(0xffffffffu, m.n, o);
  r.mean = __shfl_xor_sync(0xffffffffu, m.mean, o);
  r.m2 = __shfl_xor_sync(0xffffffffu, m.m2, o);
  return r;
}

__device__ __forceinline__ Mom mom_warp(Mom m) {
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) m = mom_merge(m, mom_shfl(m, o));
  return m;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

__device__ __forceinline__ unsigned ld_acquire(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Grid barrier number `k` (1-based): every block arrives once per barrier, so
// barrier k is passed when the counter reaches k * gridDim.x.  Bounded: on
// expiry the block latches kDevTimeout and reports failure.
__device__ bool grid_barrier(unsigned* bar, unsigned k, int* err, uint64_t limit_ns,
                             int* s_abort) {
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    atomicAdd(bar, 1u);
    const unsigned target = k * gridDim.x;
    if (ld_acquire(bar) < target) {
      const uint64_t t0 = ptx::globaltimer();
      while (ld_acquire(bar) < target) {
        if (ptx::globaltimer() - t0 > limit_ns) {
          atomicOr(err, kDevTimeout);
          *s_abort = 1;
          break;
        }
      }
    }
    __threadfence();
  }
  __syncthreads();
  return *s_abort == 0;
}

__device__ __forceinline__ float bf_lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf_hi(uint32_t u) { return __uint_as_float(u & 0xffff0000u); }

__device__ __forceinline__ float dot8(uint4 h, uint4 w) {
  float s = bf_lo(h.x) * bf_lo(w.x);
  s = fmaf(bf_hi(h.x), bf_hi(w.x), s);
  s = fmaf(bf_lo(h.y), bf_lo(w.y), s);
  s = fmaf(bf_hi(h.y), bf_hi(w.y), s);
  s = fmaf(bf_lo(h.z), bf_lo(w.z), s);
  s = fmaf(bf_hi(h.z), bf_hi(w.z), s);
  s = fmaf(bf_lo(h.w), bf_lo(w.w), s);
  s = fmaf(bf_hi(h.w), bf_hi(w.w), s);
  return s;
}

// This lane's share of the last hidden layer of a row, bf16 mode: the
// 8-element chunks at lane*8 and lane*8 + 256 (hidden width <= 512).
struct HRow {
  uint4 h[2];
};

__device__ __forceinline__ HRow load_hrow(const FreshAdvArgs& a, int64_t row, int lane) {
  const int H = a.s.H2;
  const __nv_bfloat16* h = static_cast<const __nv_bfloat16*>(a.H2) + row * H;
  HRow r;
  const uint4 z{0u, 0u, 0u, 0u};
  r.h[0] = lane * 8 < H ? *reinterpret_cast<const uint4*>(h + lane * 8) : z;
  r.h[1] = lane * 8 + 256 < H ? *reinterpret_cast<const uint4*>(h + lane * 8 + 256) : z;
  return r;
}

// Partial (over this lane's share of the hidden width) of output column c.
__device__ __forceinline__ float col_partial(const FreshAdvArgs& a, const HRow& hr, int64_t row,
                                             int c, int lane) {
  const int H = a.s.H2;
  if (a.h2_bf16) {
    const __nv_bfloat16* w = static_cast<const __nv_bfloat16*>(a.W3) + (int64_t)c * H;
    float acc = 0.f;
    if (lane * 8 < H) acc = dot8(hr.h[0], __ldg(reinterpret_cast<const uint4*>(w + lane * 8)));
    if (lane * 8 + 256 < H)
      acc += dot8(hr.h[1], __ldg(reinterpret_cast<const uint4*>(w + lane * 8 + 256)));
    return acc;
  }
  const float* h = static_cast<const float*>(a.H2) + row * H;
  const float* w = static_cast<const float*>(a.W3) + (int64_t)c * H;
  float acc = 0.f;
  for (int k = lane; k < H; k += 32) acc = fmaf(h[k], __ldg(w + k), acc);
  return acc;
}

// Phase A for one row: fresh value, and for V-trace the ratio of the taken
// action's probability to the behaviour policy's.
__device__ __forceinline__ void fresh_row(const FreshAdvArgs& a, int64_t row, int lane) {
  const NetShape& s = a.s;
  const int C = s.C;
  HRow hr;
  if (a.h2_bf16) hr = load_hrow(a, row, lane);
  if (a.ratio == nullptr) {
    const float v = warp_sum(col_partial(a, hr, row, C - 1, lane)) + __ldg(a.b3 + C - 1);
    if (lane == 0) a.val[row] = v;
    return;
  }
  // lane c ends with column c (one butterfly sum per column keeps the
  // register footprint small)
  float z = 0.f;
#pragma unroll 4
  for (int c = 0; c < C; ++c) {
    const float col = warp_sum(col_partial(a, hr, row, c, lane));
    if (lane == c) z = col;
  }
  if (lane < C) z += __ldg(a.b3 + lane);
  // log-probability of the action: log-softmax per discrete head, then the
  // diagonal-Gaussian dimensions
  const float neg_inf = -__int_as_float(0x7f800000);
  float contrib = 0.f;
  int off = 0;
  for (int h = 0; h < s.NH; ++h) {
    const int n = s.head_n[h];
    const bool in = lane >= off && lane < off + n;
    const float m = warp_max(in ? z : neg_inf);
    const float se = warp_sum(in ? expf(z - m) : 0.f);
    int act = __ldg(a.act + row * s.NH + h);
    act = act < 0 ? 0 : (act >= n ? n - 1 : act);
    if (lane == off + act) contrib += z - (m + logf(se));
    off += n;
  }
  if (lane >= off && lane < off + s.G) {
    const int g = lane - off;
    const float ls = __ldg(a.logstd + g);
    const float d = __ldg(a.actc + row * s.G + g) - z;
    contrib += -d * d * 0.5f * expf(-2.f * ls) - ls - 0.91893853320467274f;   // ln(2 pi) / 2
  }
  const float logp = warp_sum(contrib);
  const float v = __shfl_sync(0xffffffffu, z, C - 1);
  if (lane == 0) {
    a.val[row] = v;
    a.ratio[row] = expf(logp - __ldg(a.logp_old + row));
  }
}

// Phase B for segment j: the scan over the horizon; returns this lane's
// moments of the advantages it wrote.
__device__ __forceinline__ Mom fresh_segment(const FreshAdvArgs& a, int j, int lane, Mom mom) {
  const int T = a.T, ns = a.ns;
  const int64_t N = a.N;
  int e = __ldg(a.envs + j);
  e = e < 0 ? 0 : (e >= N ? (int)(N - 1) : e);
  const bool vtrace = a.ratio != nullptr;
  float A_in = 0.f;            // advantage at t_hi
  float v_in = __ldg(a.boot + e);   // value at t_hi
  for (int t_hi = T; t_hi > 0; t_hi -= 32 * kRun) {
    const int t_lo = t_hi - 32 * kRun > 0 ? t_hi - 32 * kRun : 0;
    const int start = t_lo + lane * kRun;
    int cnt = t_hi - start;
    cnt = cnt < 0 ? 0 : (cnt > kRun ? kRun : cnt);
    float r[kRun], d[kRun], v[kRun], rho[kRun];
#pragma unroll
    for (int q = 0; q < kRun; ++q) {
      r[q] = d[q] = v[q] = 0.f;
      rho[q] = 1.f;
      if (q < cnt) {
        const int t = start + q;
        const int64_t i = (int64_t)t * N + e;
        const int64_t k = (int64_t)t * ns + j;
        r[q] = __ldg(a.rew + i);
        d[q] = __ldg(a.done + i);
        v[q] = a.val[k];          // written by phase A of this launch: plain load
        if (vtrace) rho[q] = a.ratio[k];
      }
    }
    // value after this lane's run: the next lane's first value, or v_in
    const float v_next_lane = __shfl_down_sync(0xffffffffu, v[0], 1);
    const float v_after = (start + cnt == t_hi || lane == 31) ? v_in : v_next_lane;
    float bq[kRun], aq[kRun];
    float alpha = 1.f, beta = 0.f;
#pragma unroll
    for (int q = kRun - 1; q >= 0; --q) {
      bq[q] = 0.f;
      aq[q] = 1.f;
      if (q < cnt) {
        const float vn = q + 1 < cnt ? v[q + 1 < kRun ? q + 1 : q] : v_after;
        const float alive = d[q] != 0.f ? 0.f : 1.f;
        float w = 1.f, c = a.lambda;
        if (vtrace) {
          w = fminf(a.rho_clip, rho[q]);
          c = a.lambda * fminf(a.c_clip, rho[q]);
        }
        bq[q] = w * (r[q] + a.gamma * alive * vn - v[q]);
        aq[q] = a.gamma * alive * c;
        beta = bq[q] + aq[q] * beta;
        alpha = aq[q] * alpha;
      }
    }
    // suffix composition over lanes: lane L ends with the map from the
    // advantage at t_hi to the advantage at its run's start
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float a2 = __shfl_down_sync(0xffffffffu, alpha, o);
      const float b2 = __shfl_down_sync(0xffffffffu, beta, o);
      if (lane + o < 32) {
        beta = beta + alpha * b2;
        alpha = alpha * a2;
      }
    }
    const float y = beta + alpha * A_in;
    const float y_next = __shfl_down_sync(0xffffffffu, y, 1);
    float A = (start + cnt == t_hi || lane == 31) ? A_in : y_next;
#pragma unroll
    for (int q = kRun - 1; q >= 0; --q) {
      if (q < cnt) {
        A = bq[q] + aq[q] * A;
        const int64_t k = (int64_t)(start + q) * ns + j;
        a.adv[k] = A;
        a.ret[k] = A + v[q];
        // Welford update of this lane's moments
        mom.n += 1.0;
        const double dx = (double)A - mom.mean;
        mom.mean += dx / mom.n;
        mom.m2 += dx * ((double)A - mom.mean);
      }
    }
    A_in = __shfl_sync(0xffffffffu, A, 0);
    v_in = __shfl_sync(0xffffffffu, v[0], 0);
  }
  return mom;
}

__global__ void __launch_bounds__(kFreshThreads, 2)
fresh_adv_kernel(FreshAdvArgs a) {
  __shared__ int s_abort;
  __shared__ Mom s_mom[kFreshWarps];
  __shared__ float s_stats[2];
  pdl_wait();
  if (threadIdx.x == 0) s_abort = 0;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int gwarp = blockIdx.x * kFreshWarps + warp;
  const int nwarps = gridDim.x * kFreshWarps;
  const int64_t rows = (int64_t)a.T * a.ns;
  unsigned k = 0;
  if (a.head) {
    for (int64_t row = gwarp; row < rows; row += nwarps) fresh_row(a, row, lane);
    if (!grid_barrier(a.bar, ++k, a.err, a.timeout_ns, &s_abort)) return;
  }
  Mom mom{0.0, 0.0, 0.0};
  for (int j = gwarp; j < a.ns; j += nwarps) mom = fresh_segment(a, j, lane, mom);
  mom = mom_warp(mom);
  if (lane == 0) s_mom[warp] = mom;
  __syncthreads();
  if (threadIdx.x == 0) {
    Mom b = s_mom[0];
    for (int w = 1; w < kFreshWarps; ++w) b = mom_merge(b, s_mom[w]);
    a.part[3 * blockIdx.x + 0] = b.n;
    a.part[3 * blockIdx.x + 1] = b.mean;
    a.part[3 * blockIdx.x + 2] = b.m2;
  }
  if (!grid_barrier(a.bar, ++k, a.err, a.timeout_ns, &s_abort)) return;
  if (warp == 0) {
    // the same fixed merge order in every block: lane l takes blocks
    // l, l + 32, ... in turn, then the xor tree
    Mom m{0.0, 0.0, 0.0};
    for (int b = lane; b < (int)gridDim.x; b += 32) {
      const Mom p{a.part[3 * b], a.part[3 * b + 1], a.part[3 * b + 2]};
      m = mom_merge(m, p);
    }
    m = mom_warp(m);
    if (lane == 0) {
      const double sd = m.n > 1.0 ? sqrt(m.m2 / (m.n - 1.0)) : 0.0;
      s_stats[0] = (float)m.mean;
      s_stats[1] = (float)sd;
      if (blockIdx.x == 0 && a.stats) {
        a.stats[0] = (float)m.mean;
        a.stats[1] = (float)sd;
      }
    }
  }
  __syncthreads();
  pdl_trigger();
  if (a.adv_norm) {
    const float mean = s_stats[0], inv = 1.f / (s_stats[1] + 1e-8f);
    const int64_t stride = (int64_t)gridDim.x * kFreshThreads;
    for (int64_t i = (int64_t)blockIdx.x * kFreshThreads + threadIdx.x; i < rows; i += stride)
      a.adv_norm[i] = (a.adv[i] - mean) * inv;
  }
  // the last block out resets the barrier counter for the next launch
  if (threadIdx.x == 0) {
    const unsigned total = (k + 1) * gridDim.x;
    if (atomicAdd(a.bar, 1u) == total - 1) atomicExch(a.bar, 0u);
  }
}

int g_fresh_blocks_per_sm = 0;

}  // namespace

cudaError_t fresh_prepare() {
  if (g_fresh_blocks_per_sm > 0) return cudaSuccess;
  int n = 0;
  cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, fresh_adv_kernel,
                                                                kFreshThreads, 0);
  if (e != cudaSuccess) return e;
  g_fresh_blocks_per_sm = n < 1 ? 1 : n;
  return cudaSuccess;
}

int fresh_grid(int64_t rows, int ns, int head, int num_sms) {
  const int bps = g_fresh_blocks_per_sm < 4 ? g_fresh_blocks_per_sm : 4;
  int64_t cap = (int64_t)num_sms * (bps > 0 ? bps : 1);
  if (cap > kFreshMaxGrid) cap = kFreshMaxGrid;
  int64_t want = (ns + kFreshWarps - 1) / kFreshWarps;
  const int64_t per_rows = head ? (rows + 4 * kFreshWarps - 1) / (4 * kFreshWarps)
                                : (rows + 8 * kFreshThreads - 1) / (8 * kFreshThreads);
  if (per_rows > want) want = per_rows;
  if (want > cap) want = cap;
  return want < 1 ? 1 : (int)want;
}

cudaError_t launch_fresh_adv(const FreshAdvArgs& a, int num_sms, cudaStream_t st) {
  if (g_fresh_blocks_per_sm <= 0) return cudaErrorInitializationError;
  const int grid = fresh_grid((int64_t)a.T * a.ns, a.ns, a.head, num_sms);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kFreshThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = st;
  // cooperative: all blocks are resident and meet at the grid barriers
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, fresh_adv_kernel, a);
}

}  // namespace ppo
