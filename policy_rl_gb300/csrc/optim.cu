// optim.cu -- gradient assembly, gradient-norm clip and fused Adam.
//
// reduce: sums the split-K weight-gradient partials and the per-CTA bias /
// loss partials in a fixed order into the flat fp32 gradient (deterministic).
// sqnorm + adam: "PlayTrain", Table 8 (PPO column): Adam with gradient-norm
// clip.  The squared norm is reduced per block in fp64 and summed in a fixed
// order by every Adam block; Adam then streams p, g, m, v once and
// writes p, m, v and the bf16 weight shadows the tensor-core GEMMs read,
// one coalesced grid-stride pass.
#include "common.cuh"
#include "gemm.h"

namespace ppo {

namespace {

constexpr int kRedThreads = 256;
constexpr int kNormThreads = 256;
constexpr int kNormBlocks = 128;
constexpr int kAdamThreads = 256;

__global__ void __launch_bounds__(kRedThreads) reduce_kernel(ReduceArgs a) {
  const NetShape& s = a.s;
  const int P = (int)s.P;
  const int stride = gridDim.x * kRedThreads;
  double sq = 0.0;
  for (int i = blockIdx.x * kRedThreads + threadIdx.x; i < P; i += stride) {
    float v = 0.f;
    if (i < s.ob1) {
      const int r = i - (int)s.oW1;
      const int j = r / s.D, k = r - j * s.D;
      const float* q = a.pW1 + (int64_t)j * a.ld1 + k;
      const int64_t st = (int64_t)s.H1 * a.ld1;
#pragma unroll 8
      for (int sp = 0; sp < a.s1; ++sp) v += q[sp * st];
    } else if (i < s.oW2) {
      const int j = i - (int)s.ob1;
#pragma unroll 8
      for (int b = 0; b < a.nb1; ++b) v += a.pb1[(int64_t)b * s.H1 + j];
    } else if (i < s.ob2) {
      const int r = i - (int)s.oW2;
      const float* q = a.pW2 + r;
      const int64_t st = (int64_t)s.H2 * s.H1;
#pragma unroll 8
      for (int sp = 0; sp < a.s2; ++sp) v += q[sp * st];
    } else if (i < s.oW3) {
      const int j = i - (int)s.ob2;
#pragma unroll 8
      for (int b = 0; b < a.nb2; ++b) v += a.pb2[(int64_t)b * s.H2 + j];
    } else if (i < s.ob3) {
      const int r = i - (int)s.oW3;
      const int c = r / s.H2, j = r - c * s.H2;
      const float* q = a.pW3t + (int64_t)j * a.ld3 + c;
      const int64_t st = (int64_t)s.H2 * a.ld3;
#pragma unroll 8
      for (int sp = 0; sp < a.s3; ++sp) v += q[sp * st];
    } else if (i < s.ologstd) {
      const int c = i - (int)s.ob3;
#pragma unroll 8
      for (int b = 0; b < a.nb3; ++b) v += a.pb3[(int64_t)b * a.ldb3 + c];
    } else {
      const int gi = i - (int)s.ologstd;
      for (int b = 0; b < a.nl; ++b) v += a.ploss[(int64_t)b * kLossPartials + 6 + gi];
    }
    a.grad[i] = v;
    sq += (double)v * (double)v;
  }
  if (a.sq_part != nullptr) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sq += __shfl_xor_sync(0xffffffffu, sq, o);
    __shared__ double ws[kRedThreads / kWarp];
    if (threadIdx.x % kWarp == 0) ws[threadIdx.x / kWarp] = sq;
    __syncthreads();
    if (threadIdx.x == 0) {
      double t = 0.0;
      for (int w = 0; w < kRedThreads / kWarp; ++w) t += ws[w];
      a.sq_part[blockIdx.x] = t;
    }
  }
  if (blockIdx.x == 0 && a.stats6 != nullptr && threadIdx.x < 6) {
    float v = 0.f;
    for (int b = 0; b < a.nl; ++b) v += a.ploss[(int64_t)b * kLossPartials + threadIdx.x];
    a.stats6[threadIdx.x] = v * a.inv_mb;
  }
}

__global__ void __launch_bounds__(kNormThreads)
sqnorm_kernel(const float* __restrict__ g, int64_t P, double* __restrict__ part) {
  double s = 0.0;
  for (int64_t i = (int64_t)blockIdx.x * kNormThreads + threadIdx.x; i < P;
       i += (int64_t)gridDim.x * kNormThreads) {
    const double x = g[i];
    s += x * x;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  __shared__ double ws[kNormThreads / kWarp];
  if (threadIdx.x % kWarp == 0) ws[threadIdx.x / kWarp] = s;
  __syncthreads();
  if (threadIdx.x == 0) {
    double t = 0.0;
    for (int w = 0; w < kNormThreads / kWarp; ++w) t += ws[w];
    part[blockIdx.x] = t;
  }
}

__device__ __forceinline__ void write_shadow(const NetShape& s, const Shadows& sh, int i,
                                             float p) {
  const __nv_bfloat16 b = __float2bfloat16_rn(p);
  if (i < (int)s.ob1) {
    const int r = i - (int)s.oW1;
    const int j = r / s.D, k = r - j * s.D;
    sh.W1s[j * s.Dp + k] = b;
  } else if (i >= (int)s.oW2 && i < (int)s.ob2) {
    const int r = i - (int)s.oW2;
    const int j = r / s.H1, k = r - j * s.H1;
    sh.W2s[r] = b;
    sh.W2Ts[k * s.H2 + j] = b;
  } else if (i >= (int)s.oW3 && i < (int)s.ob3) {
    const int r = i - (int)s.oW3;
    const int c = r / s.H2, j = r - c * s.H2;
    sh.W3s[r] = b;
    sh.W3Ts[j * sh.ld3t + c] = b;
  }
}

__global__ void __launch_bounds__(kAdamThreads) adam_kernel(AdamArgs a) {
  __shared__ float s_coef, s_norm, s_ibc1, s_ibc2;
  __shared__ long long s_t;
  if (threadIdx.x == 0) {
    double ss = 0.0;
    for (int b = 0; b < a.nsq; ++b) ss += a.sq_part[b];
    const double norm = sqrt(ss);
    double coef = 1.0;
    if (a.max_norm > 0.f) {
      const double c = (double)a.max_norm / (norm + 1e-6);
      coef = c < 1.0 ? c : 1.0;
    }
    const long long t = (long long)(*a.step) + 1;
    s_coef = (float)coef;
    s_norm = (float)norm;
    s_t = t;
    // bias corrections 1 - beta^t, in double, once per block
    s_ibc1 = (float)(1.0 / (1.0 - pow(a.b1, (double)t)));
    s_ibc2 = (float)(1.0 / (1.0 - pow(a.b2, (double)t)));
  }
  __syncthreads();
  const float coef = s_coef, ibc1 = s_ibc1, ibc2 = s_ibc2;
  const float b1 = (float)a.b1, b2 = (float)a.b2, omb1 = a.omb1, omb2 = a.omb2;
  const float lr = a.lr, eps = a.eps;
  const bool shadows = a.sh.W1s != nullptr;
  const int P = (int)a.P;
  const int stride = gridDim.x * kAdamThreads;
  for (int i = blockIdx.x * kAdamThreads + threadIdx.x; i < P; i += stride) {
    const float g = a.g[i] * coef;
    const float m = b1 * a.m[i] + omb1 * g;
    const float v = b2 * a.v[i] + omb2 * g * g;
    const float p = a.p[i] - lr * (m * ibc1) / (sqrtf(v * ibc2) + eps);
    a.m[i] = m;
    a.v[i] = v;
    a.p[i] = p;
    if (shadows) write_shadow(a.s, a.sh, i, p);
  }
  // the last block to finish publishes the new step count (every block has
  // read the old one before its arrival)
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    const unsigned prev = atomicAdd(a.done_ctr, 1u);
    if (prev == gridDim.x - 1) {
      *a.step = (int64_t)s_t;
      if (a.grad_norm_out) *a.grad_norm_out = s_norm;
      *a.done_ctr = 0u;
      __threadfence();
    }
  }
}

__global__ void __launch_bounds__(kAdamThreads)
shadow_kernel(const float* __restrict__ p, NetShape s, Shadows sh) {
  const int64_t stride = (int64_t)gridDim.x * kAdamThreads;
  for (int64_t i = (int64_t)blockIdx.x * kAdamThreads + threadIdx.x; i < s.P; i += stride)
    write_shadow(s, sh, (int)i, p[i]);
}

int blocks_for(int64_t n, int threads, int cap) {
  int64_t b = (n + threads - 1) / threads;
  if (b > cap) b = cap;
  if (b < 1) b = 1;
  return (int)b;
}

}  // namespace

int reduce_blocks(int64_t P) { return blocks_for(P, kRedThreads, 1024); }

cudaError_t launch_reduce(const ReduceArgs& a, cudaStream_t st) {
  reduce_kernel<<<reduce_blocks(a.s.P), kRedThreads, 0, st>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_adam(const AdamArgs& a0, cudaStream_t st, const Trace* tr) {
  AdamArgs a = a0;
  if (a.nsq <= 0) {   // no squared-norm partials supplied: compute them
    sqnorm_kernel<<<kNormBlocks, kNormThreads, 0, st>>>(a.g, a.P, const_cast<double*>(a.sq_part));
    if (tr) tr->mark(ST_SQNORM, st);
    a.nsq = kNormBlocks;
  }
  adam_kernel<<<blocks_for(a.P, kAdamThreads, 152 * 4), kAdamThreads, 0, st>>>(a);
  if (tr) tr->mark(ST_ADAM, st);
  return cudaGetLastError();
}

cudaError_t launch_shadows(const float* p, const NetShape& s, const Shadows& sh, cudaStream_t st) {
  if (sh.W1s == nullptr) return cudaSuccess;
  shadow_kernel<<<blocks_for(s.P, kAdamThreads, 152 * 4), kAdamThreads, 0, st>>>(p, s, sh);
  return cudaGetLastError();
}

}  // namespace ppo
