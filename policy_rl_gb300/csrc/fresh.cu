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
//  A (optional) fresh values: one thread per row computes the row's
//    head outputs from the last hidden layer the forward pass just wrote
//    (head_rows.cuh; one thread per row measured faster than 2 or 4 lanes
//    per row -- 22.5 against 22.8 / 26.6 us per Mario-like minibatch --
//    because more lanes need more blocks, and the grid barriers and the
//    final merge grow with the block count).  GAE needs only the value column (NCOL = 1); V-trace needs
//    every column to form the log-probability of the taken action and the
//    ratio pi/mu = exp(logp - logp_old).
//  B the segment scan (from 16,384 segments: one thread per segment, a
//    coalesced backward walk like the GAE kernel); otherwise one warp per
//    segment, for latency: the recursion is affine in
//    A_{t+1} (A_t = b_t + a_t A_{t+1}), so each lane composes the maps of a
//    run of kRun steps, a suffix scan over the lanes composes the runs, and
//    each lane then replays its steps from the exact incoming value.  Windows
//    of 32 kRun steps are chained from the end of the horizon.
//  C moments: each lane keeps shifted fp32 sums of its advantages, merged by
//    Chan's formula up the warp and the block into per-block partials; after
//    the barrier every block merges all partials in the same fixed order and
//    normalises its share of the advantages: (A - mean) / (std + 1e-8), std
//    the unbiased estimate.  (fp32 throughout: GB300's fp64 rate is a small
//    fraction of its fp32 rate.)
#include "common.cuh"
#include "head_rows.cuh"
#include "tc_ptx.cuh"

namespace ppo {

namespace {

constexpr int kFreshThreads = 256;
constexpr int kFreshWarps = kFreshThreads / 32;
constexpr int kRun = 4;   // steps per lane per window

struct MomF {
  float n, mean, m2;
};

// Chan et al. pairwise merge of (count, mean, M2).
__device__ __forceinline__ MomF mom_merge(MomF a, MomF b) {
  if (a.n == 0.f) return b;
  if (b.n == 0.f) return a;
  const float n = a.n + b.n;
  const float d = b.mean - a.mean;
  const float fb = b.n / n;
  MomF r;
  r.n = n;
  r.mean = a.mean + d * fb;
  r.m2 = a.m2 + b.m2 + d * d * a.n * fb;
  return r;
}

__device__ __forceinline__ MomF mom_shfl(MomF m, int o) {
  MomF r;
  r.n = __shfl_xor_sync(0xffffffffu, m.n, o);
  r.mean = __shfl_xor_sync(0xffffffffu, m.mean, o);
  r.m2 = __shfl_xor_sync(0xffffffffu, m.m2, o);
  return r;
}

// Butterfly merge; lane 0's result is the one used (the merge is not
// symmetric in rounding, so lanes may differ in the last bits).
__device__ __forceinline__ MomF mom_warp(MomF m) {
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) m = mom_merge(m, mom_shfl(m, o));
  return m;
}

// Shifted sums of one lane: values x are accumulated as e = x - shift with
// shift = the lane's first value, so that constant inputs give M2 = 0 exactly.
struct LaneSums {
  float n, shift, s1, s2;
  __device__ __forceinline__ void add(float x) {
    if (n == 0.f) shift = x;
    const float e = x - shift;
    n += 1.f;
    s1 += e;
    s2 += e * e;
  }
  __device__ __forceinline__ MomF moments() const {
    if (n == 0.f) return MomF{0.f, 0.f, 0.f};
    const float q = s1 / n;
    return MomF{n, shift + q, fmaxf(s2 - s1 * q, 0.f)};
  }
};

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

// Log-probability of the taken action from a row of head outputs z (thread
// = row): log-softmax per discrete head by segmented running max / sum over
// the compile-time-indexed columns, then the diagonal-Gaussian dimensions.
template <int NCOL>
__device__ __forceinline__ float row_logp(const FreshAdvArgs& a, int64_t row,
                                          const float (&z)[NCOL]) {
  const NetShape& s = a.s;
  uint32_t hs = 0u, he = 0u, hd = 0u, amask = 0u;
  int off = 0;
  for (int h = 0; h < s.NH; ++h) {
    const int n = s.head_n[h];
    int act = __ldg(a.act + row * s.NH + h);
    act = act < 0 ? 0 : (act >= n ? n - 1 : act);
    hs |= 1u << off;
    he |= 1u << (off + n - 1);
    hd |= ((1u << n) - 1u) << off;
    amask |= 1u << (off + act);
    off += n;
  }
  float mx[NCOL], se[NCOL];
  float run = 0.f;
#pragma unroll
  for (int k = 0; k < NCOL; ++k) {
    run = ((hs >> k) & 1u) ? z[k] : fmaxf(run, z[k]);
    mx[k] = run;
  }
#pragma unroll
  for (int k = NCOL - 2; k >= 0; --k)
    if (!((he >> k) & 1u)) mx[k] = mx[k + 1];
  float srun = 0.f;
#pragma unroll
  for (int k = 0; k < NCOL; ++k) {
    const float e = ((hd >> k) & 1u) ? __expf(z[k] - mx[k]) : 0.f;
    srun = ((hs >> k) & 1u) ? e : srun + e;
    se[k] = srun;
  }
#pragma unroll
  for (int k = NCOL - 1; k >= 0; --k) {
    if ((he >> k) & 1u) mx[k] = mx[k] + __logf(se[k]);   // the head's log-sum-exp
    else if (k + 1 < NCOL) mx[k] = mx[k + 1];
  }
  float logp = 0.f;
#pragma unroll
  for (int k = 0; k < NCOL; ++k)
    if ((amask >> k) & 1u) logp += z[k] - mx[k];
  for (int g = 0; g < s.G; ++g) {
    float mu = 0.f;
#pragma unroll
    for (int k = 0; k < NCOL; ++k) mu = (k == off + g) ? z[k] : mu;
    const float ls = __ldg(a.logstd + g);
    const float d = __ldg(a.actc + row * s.G + g) - mu;
    logp += -0.5f * d * d * __expf(-2.f * ls) - ls - 0.91893853320467274f;   // ln(2 pi) / 2
  }
  return logp;
}

// Phase A for one row (thread = row).
template <int NCOL>
__device__ __forceinline__ void eval_row(const FreshAdvArgs& a, const HeadSrc& hs,
                                         const float* w3t, int64_t row) {
  float z[NCOL];
  head_row<NCOL>(hs, w3t, row, z);
  if constexpr (NCOL == 1) {
    a.val[row] = z[0];
  } else {
    float v = 0.f;
#pragma unroll
    for (int c = 0; c < NCOL; ++c) v = (c == a.s.C - 1) ? z[c] : v;
    a.val[row] = v;
    a.ratio[row] = __expf(row_logp<NCOL>(a, row, z) - __ldg(a.logp_old + row));
  }
}

// The rollout inputs of a segment's last window (rewards, dones, bootstrap
// value): they do not depend on phase A, so they are loaded before its barrier.
struct SegPre {
  int64_t e;
  float boot;
  float r[kRun], d[kRun];
};

__device__ __forceinline__ void seg_prefetch(const FreshAdvArgs& a, int64_t e, int lane,
                                             SegPre& p) {
  const int64_t N = a.N;
  p.e = e < 0 ? 0 : (e >= N ? N - 1 : e);
  p.boot = __ldg(a.boot + p.e);
  const int t_lo = a.T - 32 * kRun > 0 ? a.T - 32 * kRun : 0;
  const int start = t_lo + lane * kRun;
#pragma unroll
  for (int q = 0; q < kRun; ++q) {
    p.r[q] = p.d[q] = 0.f;
    if (start + q < a.T) {
      const int64_t i = (int64_t)(start + q) * N + p.e;
      p.r[q] = __ldg(a.rew + i);
      p.d[q] = __ldg(a.done + i);
    }
  }
}

// Many segments (a whole rollout's worth): one thread per segment walks the
// horizon backwards like the GAE kernel, so that a warp reads 32 consecutive
// segments of one time step (coalesced on the [T][ns] arrays, and on the
// [T][N] rollout arrays when the segments are consecutive environments).
constexpr int kSegPerThreadFrom = 16384;
constexpr int kSegU = 16;   // steps whose loads are in flight together

__device__ __forceinline__ void thread_segment(const FreshAdvArgs& a, int j, LaneSums& acc) {
  const int T = a.T, ns = a.ns;
  const int64_t N = a.N;
  int64_t e = __ldg(a.envs + j);
  e = e < 0 ? 0 : (e >= N ? N - 1 : e);
  const bool vtrace = a.ratio != nullptr;
  float A = 0.f;
  float v_next = __ldg(a.boot + e);
  for (int t_hi = T; t_hi > 0; t_hi -= kSegU) {
    float r[kSegU], d[kSegU], v[kSegU], rho[kSegU];
#pragma unroll
    for (int q = 0; q < kSegU; ++q) {
      const int t = t_hi - 1 - q;
      r[q] = d[q] = v[q] = 0.f;
      rho[q] = 1.f;
      if (t >= 0) {
        r[q] = __ldcs(a.rew + (int64_t)t * N + e);
        d[q] = __ldcs(a.done + (int64_t)t * N + e);
        v[q] = a.val[(int64_t)t * ns + j];
        if (vtrace) rho[q] = a.ratio[(int64_t)t * ns + j];
      }
    }
#pragma unroll
    for (int q = 0; q < kSegU; ++q) {
      const int t = t_hi - 1 - q;
      if (t >= 0) {
        const float alive = d[q] != 0.f ? 0.f : 1.f;
        float w = 1.f, c = a.lambda;
        if (vtrace) {
          w = fminf(a.rho_clip, rho[q]);
          c = a.lambda * fminf(a.c_clip, rho[q]);
        }
        A = w * (r[q] + a.gamma * alive * v_next - v[q]) + a.gamma * alive * c * A;
        const int64_t k = (int64_t)t * ns + j;
        a.adv[k] = A;
        a.ret[k] = A + v[q];
        acc.add(A);
        v_next = v[q];
      }
    }
  }
}

// Phase B for segment j: the scan over the horizon, accumulating this lane's
// advantages into its sums.  pre: the segment's prefetched last window.
__device__ __forceinline__ void fresh_segment(const FreshAdvArgs& a, int j, int lane,
                                              const SegPre& pre, LaneSums& acc) {
  const int T = a.T, ns = a.ns;
  const int64_t N = a.N;
  const int64_t e = pre.e;
  const bool vtrace = a.ratio != nullptr;
  float A_in = 0.f;       // advantage at t_hi
  float v_in = pre.boot;  // value at t_hi
  for (int t_hi = T; t_hi > 0; t_hi -= 32 * kRun) {
    const int t_lo = t_hi - 32 * kRun > 0 ? t_hi - 32 * kRun : 0;
    const int start = t_lo + lane * kRun;
    int cnt = t_hi - start;
    cnt = cnt < 0 ? 0 : (cnt > kRun ? kRun : cnt);
    float r[kRun], d[kRun], v[kRun], rho[kRun];
#pragma unroll
    for (int q = 0; q < kRun; ++q) {
      r[q] = pre.r[q];
      d[q] = pre.d[q];
      v[q] = 0.f;
      rho[q] = 1.f;
      if (q < cnt) {
        const int64_t t = start + q;
        const int64_t k = t * ns + j;
        if (t_hi != T) {
          r[q] = __ldg(a.rew + t * N + e);
          d[q] = __ldg(a.done + t * N + e);
        }
        v[q] = a.val[k];          // may have been written by phase A: plain loads
        if (vtrace) rho[q] = a.ratio[k];
      }
    }
    // value after this lane's run: the next lane's first value, or v_in
    const float v_next_lane = __shfl_down_sync(0xffffffffu, v[0], 1);
    const bool last_run = (start + cnt == t_hi) || lane == 31;
    const float v_after = last_run ? v_in : v_next_lane;
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
    const float y_next = __shfl_down_sync(0xffffffffu, beta + alpha * A_in, 1);
    float A = last_run ? A_in : y_next;
#pragma unroll
    for (int q = kRun - 1; q >= 0; --q) {
      if (q < cnt) {
        A = bq[q] + aq[q] * A;
        const int64_t k = (int64_t)(start + q) * ns + j;
        a.adv[k] = A;
        a.ret[k] = A + v[q];
        acc.add(A);
      }
    }
    A_in = __shfl_sync(0xffffffffu, A, 0);
    v_in = __shfl_sync(0xffffffffu, v[0], 0);
  }
}

template <int NCOL>
__global__ void __launch_bounds__(kFreshThreads, 2)
fresh_adv_kernel(FreshAdvArgs a) {
  extern __shared__ float4 smem_dyn[];
  float* w3t = reinterpret_cast<float*>(smem_dyn);
  __shared__ int s_abort;
  __shared__ MomF s_mom[kFreshWarps];
  __shared__ float s_stats[2];
  pdl_wait();
  if (threadIdx.x == 0) s_abort = 0;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t rows = (int64_t)a.T * a.ns;
  unsigned k = 0;
  const int nwarps = gridDim.x * kFreshWarps;
  const int j0 = blockIdx.x * kFreshWarps + warp;
  // the first segment's rollout inputs: its environment index now, the rest
  // after phase A, so that their latency hides behind phase A and the barrier
  const bool warp_path = a.ns < kSegPerThreadFrom;
  const int64_t e0 = warp_path && j0 < a.ns ? (int64_t)__ldg(a.envs + j0) : 0;
  SegPre pre;
  if (a.head) {
    const HeadSrc hs{a.H2, a.h2_bf16, a.W3, a.b3, a.s.H2, a.s.C};
    stage_w3<NCOL>(hs, w3t, kFreshThreads);
    const int64_t stride = (int64_t)gridDim.x * kFreshThreads;
    for (int64_t row = (int64_t)blockIdx.x * kFreshThreads + threadIdx.x; row < rows;
         row += stride)
      eval_row<NCOL>(a, hs, w3t, row);
    if (warp_path && j0 < a.ns) seg_prefetch(a, e0, lane, pre);
    if (!grid_barrier(a.bar, ++k, a.err, a.timeout_ns, &s_abort)) return;
  } else if (warp_path && j0 < a.ns) {
    seg_prefetch(a, e0, lane, pre);
  }
  LaneSums acc{0.f, 0.f, 0.f, 0.f};
  if (a.ns >= kSegPerThreadFrom) {
    for (int j = blockIdx.x * kFreshThreads + threadIdx.x; j < a.ns; j += gridDim.x * kFreshThreads)
      thread_segment(a, j, acc);
  } else {
    for (int j = j0; j < a.ns; j += nwarps) {
      if (j != j0) seg_prefetch(a, __ldg(a.envs + j), lane, pre);
      fresh_segment(a, j, lane, pre, acc);
    }
  }
  const MomF wm = mom_warp(acc.moments());
  if (lane == 0) s_mom[warp] = wm;
  __syncthreads();
  if (threadIdx.x == 0) {
    MomF b = s_mom[0];
    for (int w = 1; w < kFreshWarps; ++w) b = mom_merge(b, s_mom[w]);
    float* part = a.part + 3 * blockIdx.x;
    part[0] = b.n;
    part[1] = b.mean;
    part[2] = b.m2;
  }
  if (!grid_barrier(a.bar, ++k, a.err, a.timeout_ns, &s_abort)) return;
  if (warp == 0) {
    // the same fixed merge order in every block: lane l takes blocks
    // l, l + 32, ... in turn, then the butterfly
    const float* part = a.part;
    MomF m{0.f, 0.f, 0.f};
    for (int b0 = lane; b0 < (int)gridDim.x; b0 += 32 * 8) {
      MomF p[8];   // every load of the batch in flight before the merges
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int b = b0 + 32 * u;
        p[u] = b < (int)gridDim.x ? MomF{part[3 * b], part[3 * b + 1], part[3 * b + 2]}
                                  : MomF{0.f, 0.f, 0.f};
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) m = mom_merge(m, p[u]);
    }
    m = mom_warp(m);
    if (lane == 0) {
      const float sd = m.n > 1.f ? sqrtf(m.m2 / (m.n - 1.f)) : 0.f;
      s_stats[0] = m.mean;
      s_stats[1] = sd;
      if (blockIdx.x == 0 && a.stats) {
        a.stats[0] = m.mean;
        a.stats[1] = sd;
      }
    }
  }
  __syncthreads();
  pdl_trigger();
  if (a.adv_norm) {
    // float4 groups, four groups per thread in flight, then the rows % 4
    // tail (all scalar when a pointer is not 16-byte aligned: a minibatch's
    // rows inside the update start at k * T * ns)
    const float mean = s_stats[0], inv = 1.f / (s_stats[1] + 1e-8f);
    const bool vec = ((reinterpret_cast<uintptr_t>(a.adv) |
                       reinterpret_cast<uintptr_t>(a.adv_norm)) & 15u) == 0;
    const int64_t n4 = vec ? rows / 4 : 0;
    const float4* a4 = reinterpret_cast<const float4*>(a.adv);
    float4* o4 = reinterpret_cast<float4*>(a.adv_norm);
    const int64_t tid = (int64_t)blockIdx.x * kFreshThreads + threadIdx.x;
    const int64_t stride = (int64_t)gridDim.x * kFreshThreads;
    auto nrm = [&](float4 v) {
      return make_float4((v.x - mean) * inv, (v.y - mean) * inv, (v.z - mean) * inv,
                         (v.w - mean) * inv);
    };
    int64_t i = tid;
    for (; i + 3 * stride < n4; i += 4 * stride) {
      float4 v[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) v[u] = __ldcs(a4 + i + u * stride);
#pragma unroll
      for (int u = 0; u < 4; ++u) __stcs(o4 + i + u * stride, nrm(v[u]));
    }
    for (; i < n4; i += stride) __stcs(o4 + i, nrm(__ldcs(a4 + i)));
    for (int64_t k = n4 * 4 + tid; k < rows; k += stride) a.adv_norm[k] = (a.adv[k] - mean) * inv;
  }
  // the last block out resets the barrier counter for the next launch
  if (threadIdx.x == 0) {
    const unsigned total = (k + 1) * gridDim.x;
    if (atomicAdd(a.bar, 1u) == total - 1) atomicExch(a.bar, 0u);
  }
}

// Variants by the number of head columns phase A computes, their shared
// memory at the largest hidden width (512) and resident blocks per SM.
constexpr int kVariants = 3;
constexpr int kVarCols[kVariants] = {1, 16, 32};
int g_blocks_per_sm[kVariants] = {0, 0, 0};

size_t smem_bytes(int ncol, int H2) { return (size_t)w3_floats(ncol, H2) * sizeof(float); }

template <int NCOL>
cudaError_t prepare_one(int v) {
  const size_t smem = smem_bytes(NCOL, 512);
  cudaError_t e = cudaFuncSetAttribute(fresh_adv_kernel<NCOL>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  int n = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, fresh_adv_kernel<NCOL>, kFreshThreads,
                                                    smem);
  if (e != cudaSuccess) return e;
  g_blocks_per_sm[v] = n < 1 ? 1 : n;
  return cudaSuccess;
}

}  // namespace

cudaError_t fresh_prepare() {
  if (g_blocks_per_sm[0] > 0) return cudaSuccess;
  cudaError_t e = prepare_one<1>(0);
  if (e == cudaSuccess) e = prepare_one<16>(1);
  if (e == cudaSuccess) e = prepare_one<32>(2);
  return e;
}

cudaError_t launch_fresh_adv(const FreshAdvArgs& a, int num_sms, cudaStream_t st) {
  if (g_blocks_per_sm[0] <= 0) return cudaErrorInitializationError;
  // GAE needs the value column only; V-trace every head column
  const int v = (!a.head || a.ratio == nullptr) ? 0 : (a.s.C <= 16 ? 1 : 2);
  if (a.head && a.s.H2 > 512) return cudaErrorInvalidValue;
  const int bps = g_blocks_per_sm[v] < 4 ? g_blocks_per_sm[v] : 4;
  int64_t cap = (int64_t)num_sms * bps;
  if (cap > kFreshMaxGrid) cap = kFreshMaxGrid;
  const int64_t rows = (int64_t)a.T * a.ns;
  // enough blocks for one row per thread in phase A (or for the normalisation)
  // and one warp per segment in phase B
  int64_t want = a.ns >= kSegPerThreadFrom ? (a.ns + kFreshThreads - 1) / kFreshThreads
                                           : (a.ns + kFreshWarps - 1) / kFreshWarps;
  const int64_t per_rows = a.head ? (rows + kFreshThreads - 1) / kFreshThreads
                                  : (rows + 8 * kFreshThreads - 1) / (8 * kFreshThreads);
  if (per_rows > want) want = per_rows;
  const int grid = (int)(want > cap ? cap : (want < 1 ? 1 : want));
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kFreshThreads);
  cfg.dynamicSmemBytes = a.head ? smem_bytes(kVarCols[v], a.s.H2) : 0;
  cfg.stream = st;
  // cooperative: all blocks are resident and meet at the grid barriers
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  switch (v) {
    case 0: return cudaLaunchKernelEx(&cfg, fresh_adv_kernel<1>, a);
    case 1: return cudaLaunchKernelEx(&cfg, fresh_adv_kernel<16>, a);
    default: return cudaLaunchKernelEx(&cfg, fresh_adv_kernel<32>, a);
  }
}

}  // namespace ppo
