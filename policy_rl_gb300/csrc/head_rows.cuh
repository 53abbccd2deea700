// head_rows.cuh -- per-row head outputs z = W3 h2 + b3 on CUDA cores, one
// thread per row, from the last hidden layer a forward GEMM wrote.
//
// "Teaching Mario to speedrun", sec. 6 "The policy and the value are one
// network": one group of logits per action head, the Gaussian means, then the
// value.  Used where a few head columns of every row are needed outside the
// loss GEMM: the fresh values / ratios of per-minibatch advantages and the
// rollout-side policy step.  The head weights are staged once per block in
// shared memory as fp32 (every lane reads the same unit at the same time, so
// the reads are broadcasts); each thread streams its row of H2 in 16-byte
// chunks, up to 8 chunks in flight.
#pragma once

#include "common.cuh"

namespace ppo {

struct HeadSrc {
  const void* h;    // last hidden layer [rows][H], bf16 (h_bf16) or fp32
  int h_bf16;
  const void* W3;   // bf16 shadow [CP][H] or fp32 [C][H]
  const float* b3;  // [C]
  int H, C;
};

__device__ __forceinline__ float bf_lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf_hi(uint32_t u) { return __uint_as_float(u & 0xffff0000u); }

// Staged layout: unit k's NCOL columns start at w3_off(k); H2 is rounded up
// to whole 8-unit chunks (zero padding).  With several columns, chunk b
// starts 16 b bytes later than packed (lanes reading consecutive chunks of
// one row at once would otherwise share banks).
__host__ __device__ __forceinline__ int w3_rows(int H2) { return (H2 + 7) / 8 * 8; }
template <int NCOL>
__host__ __device__ __forceinline__ int w3_off(int k) {
  return k * NCOL + (NCOL > 1 ? (k >> 3) * 4 : 0);
}
__host__ __device__ __forceinline__ int w3_floats(int ncol, int H2) {
  return w3_rows(H2) * ncol + (ncol > 1 ? w3_rows(H2) / 2 : 0);
}

// Stages the head weights (NCOL == 1: the value column only) with the
// block's nthreads threads, then synchronises the block.  Work item i is 8
// consecutive hidden units of one column (one 16-byte load in bf16 mode);
// the loads of up to 4 items per thread are issued before their stores.
template <int NCOL>
__device__ __forceinline__ void stage_w3(const HeadSrc& hs, float* w3t, int nthreads) {
  const int H = hs.H, C = hs.C, Hp = w3_rows(H);
  const int chunks = Hp / 8, items = NCOL * chunks;
  constexpr int kU = 4;
  for (int i0 = threadIdx.x; i0 < items; i0 += kU * nthreads) {
    float w[kU][8];
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const int i = i0 + u * nthreads;
      const int c = i / chunks, k0 = (i - c * chunks) * 8;
      const int col = NCOL == 1 ? C - 1 : c;
#pragma unroll
      for (int j = 0; j < 8; ++j) w[u][j] = 0.f;
      if (i < items && col < C) {
        const int64_t o = (int64_t)col * H + k0;
        if (hs.h_bf16) {   // H is a multiple of 128 in bf16 mode: whole chunks
          const uint4 q =
              *reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(hs.W3) + o);
          w[u][0] = bf_lo(q.x); w[u][1] = bf_hi(q.x); w[u][2] = bf_lo(q.y); w[u][3] = bf_hi(q.y);
          w[u][4] = bf_lo(q.z); w[u][5] = bf_hi(q.z); w[u][6] = bf_lo(q.w); w[u][7] = bf_hi(q.w);
        } else {
          const float* src = static_cast<const float*>(hs.W3) + o;
#pragma unroll
          for (int j = 0; j < 8; ++j) w[u][j] = k0 + j < H ? src[j] : 0.f;
        }
      }
    }
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const int i = i0 + u * nthreads;
      if (i < items) {
        const int c = i / chunks, k0 = (i - c * chunks) * 8;
#pragma unroll
        for (int j = 0; j < 8; ++j) w3t[w3_off<NCOL>(k0 + j) + c] = w[u][j];
      }
    }
  }
  __syncthreads();
}

// z[c] += h * w3t[unit k][c].
template <int NCOL>
__device__ __forceinline__ void fma_unit(float h, const float* w3t, int k, float (&z)[NCOL]) {
  const float* w = w3t + w3_off<NCOL>(k);
  if constexpr (NCOL == 1) {
    z[0] = fmaf(h, w[0], z[0]);
  } else {
#pragma unroll
    for (int c4 = 0; c4 < NCOL; c4 += 4) {
      const float4 q = *reinterpret_cast<const float4*>(w + c4);
      z[c4 + 0] = fmaf(h, q.x, z[c4 + 0]);
      z[c4 + 1] = fmaf(h, q.y, z[c4 + 1]);
      z[c4 + 2] = fmaf(h, q.z, z[c4 + 2]);
      z[c4 + 3] = fmaf(h, q.w, z[c4 + 3]);
    }
  }
}

// Head outputs of one row: NCOL == 1 gives z[0] = the value (column C - 1);
// otherwise z[c] = column c for c < C and 0 beyond.  Biases included.
// SPLIT > 1: this thread is lane q of the SPLIT consecutive lanes that share
// the row; it sums the row's 8-unit chunks q, q + SPLIT, ... only (bias on
// lane 0), and the caller adds the lanes' partials (split_sum).
template <int NCOL, int SPLIT = 1>
__device__ __forceinline__ void head_row(const HeadSrc& hs, const float* w3t, int64_t row,
                                         float (&z)[NCOL], int q = 0) {
  const int H = hs.H, C = hs.C;
#pragma unroll
  for (int c = 0; c < NCOL; ++c) z[c] = 0.f;
  if (hs.h_bf16) {
    const uint4* hp =
        reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(hs.h) + row * H);
    constexpr int kBatch = 8;   // chunks in flight before any arithmetic
    for (int kb = 8 * q; kb < H; kb += 8 * SPLIT * kBatch) {
      uint4 u[kBatch];
#pragma unroll
      for (int i = 0; i < kBatch; ++i) {
        const int k0 = kb + 8 * SPLIT * i;
        u[i] = k0 < H ? hp[k0 / 8] : make_uint4(0u, 0u, 0u, 0u);
      }
#pragma unroll
      for (int i = 0; i < kBatch; ++i) {
        const int k0 = kb + 8 * SPLIT * i;
        if (k0 < H) {
          const float h[8] = {bf_lo(u[i].x), bf_hi(u[i].x), bf_lo(u[i].y), bf_hi(u[i].y),
                              bf_lo(u[i].z), bf_hi(u[i].z), bf_lo(u[i].w), bf_hi(u[i].w)};
#pragma unroll
          for (int j = 0; j < 8; ++j) fma_unit<NCOL>(h[j], w3t, k0 + j, z);
        }
      }
    }
  } else {
    const float* hp = static_cast<const float*>(hs.h) + row * H;
    for (int k0 = 8 * q; k0 < H; k0 += 8 * SPLIT) {
#pragma unroll
      for (int j = 0; j < 8; ++j)   // staged units below w3_rows(H) are zero past H
        fma_unit<NCOL>(k0 + j < H ? hp[k0 + j] : 0.f, w3t, k0 + j, z);
    }
  }
  if (q != 0) return;
  if constexpr (NCOL == 1) {
    z[0] += __ldg(hs.b3 + C - 1);
  } else {
#pragma unroll
    for (int c = 0; c < NCOL; ++c) z[c] += c < C ? __ldg(hs.b3 + c) : 0.f;
  }
}

// Sums the partials of the SPLIT consecutive lanes of a row (all lanes of the
// warp must call it); every lane of the group ends with the total.
template <int NCOL, int SPLIT>
__device__ __forceinline__ void split_sum(float (&z)[NCOL]) {
#pragma unroll
  for (int c = 0; c < NCOL; ++c)
#pragma unroll
    for (int o = 1; o < SPLIT; o <<= 1) z[c] += __shfl_xor_sync(0xffffffffu, z[c], o);
}

}  // namespace ppo
