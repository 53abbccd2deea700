// gae.cu -- reverse-time GAE scan, advantage moments and normalisation.
//
// "Teaching Mario to speedrun", sec. 6 "Better advantages":
//   delta_t = r_t + gamma V(s_{t+1}) - V(s_t),   A_t = delta_t + gamma lambda A_{t+1}
// with sec. 7's terminals (1 where an episode just ended) cutting both the
// bootstrap and the propagation.  One thread owns one environment and walks
// time backwards; a warp therefore reads 32 consecutive environments of one
// time step (128 contiguous bytes per array) -- fully coalesced on the
// time-major [T,N] layout.  Loads for the next chunk of kU time steps are
// issued before the current chunk's dependent arithmetic, so each thread
// keeps 3*kU loads in flight.
#include "common.cuh"

namespace ppo {

namespace {

// Block size: 512 threads when there are at least 32,768 environments
// (measured at T=1024 x N=65,536: 92 % of HBM vs 86 % with 128-thread blocks),
// 128 below that, so that small N still spreads over several SMs.
constexpr int kGaeThreadsBig = 512;
constexpr int kGaeThreadsSmall = 128;
constexpr int kGaeBigN = 32768;
constexpr int kU = 16;

struct Moments {
  double n, mean, m2;
};

// Chan et al. pairwise merge of (count, mean, M2).
__device__ __forceinline__ Moments merge(Moments a, Moments b) {
  if (a.n == 0.0) return b;
  if (b.n == 0.0) return a;
  const double n = a.n + b.n;
  const double d = b.mean - a.mean;
  Moments r;
  r.n = n;
  r.mean = a.mean + d * (b.n / n);
  r.m2 = a.m2 + b.m2 + d * d * (a.n * b.n / n);
  return r;
}

// fp32 variant for the warp level (counts <= 32*T < 2^24 are exact in float)
struct MomentsF {
  float n, mean, m2;
};

__device__ __forceinline__ MomentsF merge_f(MomentsF a, MomentsF b) {
  if (a.n == 0.f) return b;
  if (b.n == 0.f) return a;
  const float n = a.n + b.n;
  const float d = b.mean - a.mean;
  const float fb = b.n / n;
  MomentsF r;
  r.n = n;
  r.mean = a.mean + d * fb;
  r.m2 = a.m2 + b.m2 + d * d * a.n * fb;
  return r;
}

__device__ __forceinline__ Moments shfl_moments(Moments m, int o) {
  Moments r;
  r.n = __shfl_xor_sync(0xffffffffu, m.n, o);
  r.mean = __shfl_xor_sync(0xffffffffu, m.mean, o);
  r.m2 = __shfl_xor_sync(0xffffffffu, m.m2, o);
  return r;
}

__device__ __forceinline__ void load_chunk(const float* __restrict__ rew,
                                           const float* __restrict__ val,
                                           const float* __restrict__ done, int t_hi, int N,
                                           int n, float (&r)[kU], float (&v)[kU],
                                           float (&d)[kU]) {
#pragma unroll
  for (int j = 0; j < kU; ++j) {
    const int t = t_hi - 1 - j;
    if (t >= 0) {
      const int64_t i = (int64_t)t * N + n;
      r[j] = __ldcs(rew + i);
      v[j] = __ldcs(val + i);
      d[j] = __ldcs(done + i);
    }
  }
}

template <int kGaeThreads>
__global__ void __launch_bounds__(kGaeThreads)
gae_kernel(const float* __restrict__ rew, const float* __restrict__ val,
           const float* __restrict__ done, const float* __restrict__ boot, int T, int N,
           float gamma, float gl, float* __restrict__ adv, float* __restrict__ ret,
           double* __restrict__ partials) {
  const int n = blockIdx.x * kGaeThreads + threadIdx.x;
  MomentsF momf{0.f, 0.f, 0.f};
  if (n < N) {
    float next_v = boot[n];
    float next_a = 0.f;
    float shift = 0.f, s1 = 0.f, s2 = 0.f;
    bool have_shift = false;
    float r0[kU], v0[kU], d0[kU], r1[kU], v1[kU], d1[kU];
    load_chunk(rew, val, done, T, N, n, r0, v0, d0);
    for (int t_hi = T; t_hi > 0; t_hi -= 2 * kU) {
      // prefetch the chunk after this one while this one is consumed
      if (t_hi - kU > 0) load_chunk(rew, val, done, t_hi - kU, N, n, r1, v1, d1);
#pragma unroll
      for (int j = 0; j < kU; ++j) {
        const int t = t_hi - 1 - j;
        if (t >= 0) {
          const float alive = d0[j] != 0.f ? 0.f : 1.f;
          const float delta = r0[j] + gamma * alive * next_v - v0[j];
          const float a = delta + gl * alive * next_a;
          const int64_t i = (int64_t)t * N + n;
          __stcs(adv + i, a);
          __stcs(ret + i, a + v0[j]);
          next_v = v0[j];
          next_a = a;
          if (!have_shift) { shift = a; have_shift = true; }
          const float e = a - shift;
          s1 += e;
          s2 += e * e;
        }
      }
      if (t_hi - kU <= 0) break;
      if (t_hi - 2 * kU > 0) load_chunk(rew, val, done, t_hi - 2 * kU, N, n, r0, v0, d0);
#pragma unroll
      for (int j = 0; j < kU; ++j) {
        const int t = t_hi - kU - 1 - j;
        if (t >= 0) {
          const float alive = d1[j] != 0.f ? 0.f : 1.f;
          const float delta = r1[j] + gamma * alive * next_v - v1[j];
          const float a = delta + gl * alive * next_a;
          const int64_t i = (int64_t)t * N + n;
          __stcs(adv + i, a);
          __stcs(ret + i, a + v1[j]);
          next_v = v1[j];
          next_a = a;
          const float e = a - shift;
          s1 += e;
          s2 += e * e;
        }
      }
    }
    const float cnt = (float)T;
    momf.n = cnt;
    momf.mean = shift + s1 / cnt;
    momf.m2 = fmaxf(s2 - s1 * (s1 / cnt), 0.f);
  }
  if (partials == nullptr) return;
  // fixed-order tree: fp32 warp xor-merges, then fp64 over the warps
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    MomentsF other;
    other.n = __shfl_xor_sync(0xffffffffu, momf.n, o);
    other.mean = __shfl_xor_sync(0xffffffffu, momf.mean, o);
    other.m2 = __shfl_xor_sync(0xffffffffu, momf.m2, o);
    momf = merge_f(momf, other);
  }
  Moments mom{(double)momf.n, (double)momf.mean, (double)momf.m2};
  __shared__ Moments wm[kGaeThreads / kWarp];
  const int w = threadIdx.x / kWarp, lane = threadIdx.x % kWarp;
  if (lane == 0) wm[w] = mom;
  __syncthreads();
  if (threadIdx.x == 0) {
    Moments b = wm[0];
    for (int k = 1; k < kGaeThreads / kWarp; ++k) b = merge(b, wm[k]);
    partials[3 * blockIdx.x + 0] = b.n;
    partials[3 * blockIdx.x + 1] = b.mean;
    partials[3 * blockIdx.x + 2] = b.m2;
  }
}

// One block merges the per-block moments in a fixed order and writes
// {mean, unbiased std} as fp32 (kTriple: the merged (count, mean, M2) in fp64
// instead, for a merge with other ranks' shards).
constexpr int kFinThreads = 256;
template <bool kTriple>
__global__ void __launch_bounds__(kFinThreads)
gae_finalize_kernel(const double* __restrict__ partials, int nblocks, float* __restrict__ stats,
                    double* __restrict__ triple) {
  Moments m{0.0, 0.0, 0.0};
  for (int b = threadIdx.x; b < nblocks; b += kFinThreads) {
    Moments p{partials[3 * b], partials[3 * b + 1], partials[3 * b + 2]};
    m = merge(m, p);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = merge(m, shfl_moments(m, o));
  __shared__ Moments wm[kFinThreads / kWarp];
  if (threadIdx.x % kWarp == 0) wm[threadIdx.x / kWarp] = m;
  __syncthreads();
  if (threadIdx.x == 0) {
    Moments b = wm[0];
    for (int k = 1; k < kFinThreads / kWarp; ++k) b = merge(b, wm[k]);
    if constexpr (kTriple) {
      triple[0] = b.n;
      triple[1] = b.mean;
      triple[2] = b.m2;
    } else {
      stats[0] = (float)b.mean;
      stats[1] = (float)(b.n > 1.0 ? sqrt(b.m2 / (b.n - 1.0)) : 0.0);
    }
  }
}

constexpr int kNormThreads = 256;
__global__ void __launch_bounds__(kNormThreads)
normalize_kernel(const float* __restrict__ adv, const float* __restrict__ stats,
                 float* __restrict__ out, int64_t n) {
  const float mean = stats[0];
  const float inv = 1.f / (stats[1] + 1e-8f);
  const int64_t n4 = n / 4;
  const float4* a4 = reinterpret_cast<const float4*>(adv);
  float4* o4 = reinterpret_cast<float4*>(out);
  const int64_t stride = (int64_t)gridDim.x * kNormThreads;
  for (int64_t i = (int64_t)blockIdx.x * kNormThreads + threadIdx.x; i < n4; i += stride) {
    float4 v = __ldcs(a4 + i);
    v.x = (v.x - mean) * inv;
    v.y = (v.y - mean) * inv;
    v.z = (v.z - mean) * inv;
    v.w = (v.w - mean) * inv;
    __stcs(o4 + i, v);
  }
  for (int64_t i = n4 * 4 + (int64_t)blockIdx.x * kNormThreads + threadIdx.x; i < n; i += stride)
    out[i] = (adv[i] - mean) * inv;
}

int g_num_sms = 0;
int num_sms() {
  if (g_num_sms == 0) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&g_num_sms, cudaDevAttrMultiProcessorCount, dev);
    if (g_num_sms <= 0) g_num_sms = 1;
  }
  return g_num_sms;
}

}  // namespace

int gae_num_blocks(int N) {
  const int t = N >= kGaeBigN ? kGaeThreadsBig : kGaeThreadsSmall;
  return (N + t - 1) / t;
}

cudaError_t launch_gae(const float* rew, const float* val, const float* done, const float* boot,
                       int T, int N, float gamma, float lambda, float* adv, float* ret,
                       double* partials, int /*num_partial_blocks*/, cudaStream_t st) {
  if (N >= kGaeBigN)
    gae_kernel<kGaeThreadsBig><<<gae_num_blocks(N), kGaeThreadsBig, 0, st>>>(
        rew, val, done, boot, T, N, gamma, gamma * lambda, adv, ret, partials);
  else
    gae_kernel<kGaeThreadsSmall><<<gae_num_blocks(N), kGaeThreadsSmall, 0, st>>>(
        rew, val, done, boot, T, N, gamma, gamma * lambda, adv, ret, partials);
  return cudaGetLastError();
}

cudaError_t launch_gae_finalize(const double* partials, int nblocks, float* stats,
                                cudaStream_t st) {
  gae_finalize_kernel<false><<<1, kFinThreads, 0, st>>>(partials, nblocks, stats, nullptr);
  return cudaGetLastError();
}

cudaError_t launch_gae_moments(const double* partials, int nblocks, double* triple,
                               cudaStream_t st) {
  gae_finalize_kernel<true><<<1, kFinThreads, 0, st>>>(partials, nblocks, nullptr, triple);
  return cudaGetLastError();
}

cudaError_t launch_normalize(const float* adv, const float* stats, float* out, int64_t n,
                             cudaStream_t st) {
  int64_t blocks = (n / 4 + kNormThreads - 1) / kNormThreads;
  const int64_t cap = (int64_t)num_sms() * 8;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  normalize_kernel<<<(int)blocks, kNormThreads, 0, st>>>(adv, stats, out, n);
  return cudaGetLastError();
}

}  // namespace ppo
