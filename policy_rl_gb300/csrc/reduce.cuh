// reduce.cuh -- the fixed-order sums that assemble the bias, log-std and loss
// statistic entries of the gradient from per-CTA partial rows (written by the
// GEMM epilogues), shared by the gradient-assembly kernels (optim.cu) and
// the weight-gradient kernel (gemm_tc.cu).
#pragma once

#include "common.cuh"
#include "gemm.h"

namespace ppo {

// Lane l sums rows l, l+32, ... in order (eight loads in flight per lane), then
// a fixed xor-shuffle tree.
__device__ __forceinline__ float warp_rows_sum(const float* base, int rows, int64_t stride) {
  const int lane = threadIdx.x % kWarp;
  float v = 0.f;
  for (int b0 = lane; b0 < rows; b0 += 8 * kWarp) {
    float x[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int b = b0 + u * kWarp;
      x[u] = b < rows ? base[(int64_t)b * stride] : 0.f;
    }
#pragma unroll
    for (int u = 0; u < 8; ++u)
      if (b0 + u * kWarp < rows) v += x[u];
  }
  return warp_sum(v);
}

// Tasks of the vector reduction: one per bias entry (b1, b2, b3), one per
// log-std entry, then the six loss statistics.
__host__ __device__ __forceinline__ int reduce_vector_tasks(const NetShape& s) {
  return s.H1 + s.H2 + s.C + s.G + 6;
}

// Task e of the vector reduction, run by one whole warp: the entry's sum over
// the partial rows is written to the gradient (or, for the statistics, to
// stats6 times 1/mb).  Returns the square of a gradient entry on lane 0, 0
// otherwise.
__device__ __forceinline__ double reduce_vector_task(const ReduceArgs& a, int e) {
  const NetShape& s = a.s;
  const int lane = threadIdx.x % kWarp;
  const int nb = s.H1 + s.H2 + s.C + s.G;
  if (e < nb) {
    float v;
    int i;
    if (e < s.H1) {
      i = (int)s.ob1 + e;
      v = warp_rows_sum(a.pb1 + e, a.nb1, s.H1);
    } else if (e < s.H1 + s.H2) {
      const int j = e - s.H1;
      i = (int)s.ob2 + j;
      v = warp_rows_sum(a.pb2 + j, a.nb2, s.H2);
    } else if (e < s.H1 + s.H2 + s.C) {
      const int c = e - s.H1 - s.H2;
      i = (int)s.ob3 + c;
      v = warp_rows_sum(a.pb3 + c, a.nb3, a.ldb3);
    } else {
      const int g = e - s.H1 - s.H2 - s.C;
      i = (int)s.ologstd + g;
      v = warp_rows_sum(a.ploss + 6 + g, a.nl, kLossPartials);
    }
    if (lane == 0) {
      a.grad[i] = v;
      return (double)(v * v);
    }
  } else if (e < nb + 6) {
    const int q = e - nb;
    const float v = warp_rows_sum(a.ploss + q, a.nl, kLossPartials);
    if (lane == 0 && a.stats6 != nullptr) a.stats6[q] = v * a.inv_mb;
  }
  return 0.0;
}

}  // namespace ppo
