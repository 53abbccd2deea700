// tc_tile.cuh -- pieces shared by the tensor-core kernels (the standalone
// GEMM kernels and the persistent minibatch kernel): tile constants, bounded
// mbarrier waits, the shared-memory barrier block, and the per-tile
// epilogues that drain a TMEM accumulator.
#pragma once

#include "common.cuh"
#include "tc_ptx.cuh"

namespace ppo {
namespace tc {

using namespace ptx;

constexpr int BM = 128;
constexpr int BK = 64;          // 64 bf16 = 128 bytes = one swizzle atom row
constexpr int kColsumCap = 512;

// EPI_DACT_K1: EPI_DACT for products with a single k-tile (K <= 64), whose
// pace is set by the activation tiles rather than by the operand ring
enum Epi { EPI_BIAS_ACT = 0, EPI_DACT = 1, EPI_LOSS = 2, EPI_DACT_K1 = 3 };

struct Guard {
  volatile int* abort;
  int* err;
  uint64_t limit_ns;
};

// Bounded wait on an mbarrier phase: gives up after limit_ns (latching
// kDevTimeout and the CTA's abort flag) or when another role aborted.
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, const Guard& g) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer();
  while (true) {
#pragma unroll 1
    for (int i = 0; i < 32; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (*g.abort) return false;
    if (globaltimer() - t0 > g.limit_ns) {
      *g.abort = 1;
      atomicOr(g.err, kDevTimeout);
      return false;
    }
  }
}

// wait used while draining after an abort: never sets the abort flag again
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
  const uint64_t t0 = globaltimer();
  while (!mbar_try_wait(bar, parity))
    if (globaltimer() - t0 > limit_ns) return;
}

__device__ __forceinline__ void store_bf16x32(__nv_bfloat16* dst, const float (&y)[32]) {
  uint4* d = reinterpret_cast<uint4*>(dst);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    uint4 u;
    u.x = pack_bf16x2(y[8 * i + 0], y[8 * i + 1]);
    u.y = pack_bf16x2(y[8 * i + 2], y[8 * i + 3]);
    u.z = pack_bf16x2(y[8 * i + 4], y[8 * i + 5]);
    u.w = pack_bf16x2(y[8 * i + 6], y[8 * i + 7]);
    d[i] = u;
  }
}

// mbarriers of a tensor-core CTA: S smem stages (full/empty), two TMEM
// accumulators (full/empty), a drain barrier and (persistent kernel) an
// epilogue-group barrier.
struct Ctrl {
  uint64_t* bars;
  int S;
  __device__ uint32_t full(int s) const { return smem_u32(&bars[s]); }
  __device__ uint32_t empty(int s) const { return smem_u32(&bars[S + s]); }
  // up to three TMEM accumulators (full / empty each)
  __device__ uint32_t tfull(int a) const { return smem_u32(&bars[2 * S + a]); }
  __device__ uint32_t tempty(int a) const { return smem_u32(&bars[2 * S + 3 + a]); }
  __device__ uint32_t drain() const { return smem_u32(&bars[2 * S + 6]); }
  __device__ uint32_t epi() const { return smem_u32(&bars[2 * S + 7]); }
  __host__ __device__ static constexpr int count(int S) { return 2 * S + 8; }
};

// Element-wise epilogue of one 128 x BN tile for one epilogue warp: TMEM lane
// quarter (the warp's rows), columns [h*PART, (h+1)*PART) of the tile.
//   DACT = false: out = act(acc + bias)                          (forward)
//   DACT = true : out = acc * act'(aux); per-warp column sums into cs_q
// The TMEM load (and the aux operand) of chunk k+1 are in flight while chunk
// k is processed; the two register buffers alternate by chunk parity (the
// loop is fully unrolled, so the index is a compile-time constant) and each
// buffer is read only after its own wait.
template <int BN, int EW, bool DACT>
__device__ __forceinline__ void epi_elem_tile(uint32_t taddr, int row, bool rok, int col_tile,
                                              int h, int act, const float* bias_s,
                                              const __nv_bfloat16* aux, int ldaux,
                                              __nv_bfloat16* out, int ldo, float* cs_q,
                                              int lane) {
  constexpr int PART = BN / (EW / 4);   // columns per epilogue warp
  constexpr int NCH = PART / 32;
  const int cbase = h * PART;
  uint32_t r[2][32];
  uint4 ax[2][4];
  const __nv_bfloat16* auxrow = DACT ? aux + (int64_t)row * ldaux + col_tile + cbase : nullptr;
  tmem_ld32_async(taddr + (uint32_t)cbase, r[0]);
  if constexpr (DACT) {
#pragma unroll
    for (int i = 0; i < 4; ++i)
      ax[0][i] = rok ? __ldg(reinterpret_cast<const uint4*>(auxrow) + i) : make_uint4(0, 0, 0, 0);
  }
#pragma unroll
  for (int k = 0; k < NCH; ++k) {
    const int cur = k & 1, nxt = cur ^ 1;
    const int c0 = cbase + 32 * k;
    tmem_wait_ld(r[cur]);
    if (k + 1 < NCH) {
      tmem_ld32_async(taddr + (uint32_t)(c0 + 32), r[nxt]);
      if constexpr (DACT) {
#pragma unroll
        for (int i = 0; i < 4; ++i)
          ax[nxt][i] = rok ? __ldg(reinterpret_cast<const uint4*>(auxrow + 32 * (k + 1)) + i)
                           : make_uint4(0, 0, 0, 0);
      }
    }
    float v[32];
#pragma unroll
    for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(r[cur][j]);
    const int col0 = col_tile + c0;
    if constexpr (!DACT) {
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        const float x = v[j] + bias_s[col0 + j];
        v[j] = act == 0 ? tanh_fast(x) : (act == 1 ? fmaxf(x, 0.f) : x);
      }
      if (rok) store_bf16x32(out + (int64_t)row * ldo + col0, v);
    } else {
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint32_t w4[4] = {ax[cur][i].x, ax[cur][i].y, ax[cur][i].z, ax[cur][i].w};
#pragma unroll
        for (int hh = 0; hh < 4; ++hh) {
          const float2 hv = unpack_bf16x2(w4[hh]);
          const int j = 8 * i + 2 * hh;
          const float d0 = act == 0 ? 1.f - hv.x * hv.x : (hv.x > 0.f ? 1.f : 0.f);
          const float d1 = act == 0 ? 1.f - hv.y * hv.y : (hv.y > 0.f ? 1.f : 0.f);
          v[j] = rok ? v[j] * d0 : 0.f;
          v[j + 1] = rok ? v[j + 1] * d1 : 0.f;
        }
      }
      if (rok) store_bf16x32(out + (int64_t)row * ldo + col0, v);
      const float colsum = warp_reduce_scatter32(v);
      cs_q[col0 + lane] += colsum;
    }
  }
}

// Walks the NCH 32-column chunks [cbase + 32k, cbase + 32k + 32) of a TMEM
// accumulator (this warp's lane quarter), calling body(regs, c0) per chunk.
// The load of chunk k+1 is in flight while chunk k is processed.  The loop is
// rolled two chunks at a time (two register buffers with compile-time names),
// so the body's code appears twice rather than NCH times: the epilogues run
// once or twice per CTA and kernel at small minibatches, where instruction-
// cache misses on long unrolled code cost more than the loop.
template <int NCH, class Body>
__device__ __forceinline__ void tmem_chunks(uint32_t taddr, int cbase, Body&& body) {
  uint32_t r0[32], r1[32];
  tmem_ld32_async(taddr + (uint32_t)cbase, r0);
  if constexpr (NCH == 1) {
    tmem_wait_ld(r0);
    body(r0, cbase);
  } else {
    static_assert(NCH % 2 == 0, "chunk pairs");
#pragma unroll 1
    for (int k = 0; k < NCH; k += 2) {
      const int c0 = cbase + 32 * k;
      tmem_wait_ld(r0);
      tmem_ld32_async(taddr + (uint32_t)(c0 + 32), r1);
      body(r0, c0);
      tmem_wait_ld(r1);
      if (k + 2 < NCH) tmem_ld32_async(taddr + (uint32_t)(c0 + 64), r0);
      body(r1, c0 + 32);
    }
  }
}

// 32 values -> four 16-byte bf16 chunks of a 128-byte-swizzled row at `row`
// (chunk c of row r at (c ^ (r & 7)) * 16), starting at chunk c16.
__device__ __forceinline__ void put_row_chunks(uint8_t* row, int r, int c16, const float (&v)[32]) {
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    uint4 o;
    o.x = pack_bf16x2(v[8 * i + 0], v[8 * i + 1]);
    o.y = pack_bf16x2(v[8 * i + 2], v[8 * i + 3]);
    o.z = pack_bf16x2(v[8 * i + 4], v[8 * i + 5]);
    o.w = pack_bf16x2(v[8 * i + 6], v[8 * i + 7]);
    *reinterpret_cast<uint4*>(row + (((c16 + i) ^ (r & 7)) << 4)) = o;
  }
}

// 32 values -> one 64-byte bf16 row of a 64-byte-swizzled 32-column tile
// (16-byte chunk c of row r at (c ^ ((r >> 1) & 3)) * 16)
__device__ __forceinline__ void put_row_chunks_sw64(uint8_t* row, int r, const float (&v)[32]) {
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    uint4 o;
    o.x = pack_bf16x2(v[8 * i + 0], v[8 * i + 1]);
    o.y = pack_bf16x2(v[8 * i + 2], v[8 * i + 3]);
    o.z = pack_bf16x2(v[8 * i + 4], v[8 * i + 5]);
    o.w = pack_bf16x2(v[8 * i + 6], v[8 * i + 7]);
    *reinterpret_cast<uint4*>(row + ((i ^ ((r >> 1) & 3)) << 4)) = o;
  }
}

// act(acc + bias) for one 32-column chunk, the bias read as float4 through the
// read-only cache (16-byte aligned); act 0 tanh, 1 ReLU, 2 identity
__device__ __forceinline__ void act_bias_chunk_ldg(const uint32_t (&r)[32], const float* bias,
                                                   int act, float (&v)[32]) {
  const float4* b4 = reinterpret_cast<const float4*>(bias);
#pragma unroll
  for (int j4 = 0; j4 < 8; ++j4) {
    const float4 b = __ldg(b4 + j4);
    const float bb[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float x = __uint_as_float(r[4 * j4 + e]) + bb[e];
      v[4 * j4 + e] = act == 0 ? tanh_fast(x) : (act == 1 ? fmaxf(x, 0.f) : x);
    }
  }
}

// act(acc + bias) for one 32-column chunk (bias read as float4 from shared
// memory); act 0 tanh, 1 ReLU, 2 identity (a plain product)
__device__ __forceinline__ void act_bias_chunk(const uint32_t (&r)[32], const float* bias, int act,
                                               float (&v)[32]) {
  const float4* b4 = reinterpret_cast<const float4*>(bias);   // 16-byte aligned
#pragma unroll
  for (int j4 = 0; j4 < 8; ++j4) {
    const float4 b = b4[j4];
    const float bb[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float x = __uint_as_float(r[4 * j4 + e]) + bb[e];
      v[4 * j4 + e] = act == 0 ? tanh_fast(x) : (act == 1 ? fmaxf(x, 0.f) : x);
    }
  }
}

// Backward-data epilogue with the activation operand already in shared
// memory: `aux` is a 128 x BN bf16 tile loaded by TMA with the 128-byte
// swizzle (BN/64 blocks of 128 rows x 128 bytes, 16-byte chunk c of row r at
// r*128 + ((c ^ (r & 7)) * 16)).  out = acc * act'(aux) is written back in
// place (same thread, same bytes) for a TMA store of the tile; per-warp column
// sums of out go to cs_q (rows >= M count as zero).
// act == 3 instead: out = alpha * aux + beta * acc, no column sums (a
// product added to a multiple of a tile of the same shape).
template <int BN, int EW>
__device__ __forceinline__ void epi_dact_smem_tile(uint32_t taddr, int rl, bool rok, int col_tile,
                                                   int h, int act, uint8_t* aux, float* cs_q,
                                                   int lane, float alpha = 0.f,
                                                   float beta = 0.f) {
  constexpr int PART = BN / (EW / 4);
  tmem_chunks<PART / 32>(taddr, h * PART, [&](const uint32_t (&r)[32], int c0) {
    float v[32];
#pragma unroll
    for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(r[j]);
    uint8_t* blk = aux + (c0 / 64) * 16384 + rl * 128;
    const int c16 = (c0 % 64) / 8;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint4 a4 = *reinterpret_cast<const uint4*>(blk + (((c16 + i) ^ (rl & 7)) << 4));
      const uint32_t w4[4] = {a4.x, a4.y, a4.z, a4.w};
#pragma unroll
      for (int hh = 0; hh < 4; ++hh) {
        const float2 hv = unpack_bf16x2(w4[hh]);
        const int j = 8 * i + 2 * hh;
        if (act == 3) {
          v[j] = rok ? alpha * hv.x + beta * v[j] : 0.f;
          v[j + 1] = rok ? alpha * hv.y + beta * v[j + 1] : 0.f;
        } else {
          const float d0 = act == 0 ? 1.f - hv.x * hv.x : (hv.x > 0.f ? 1.f : 0.f);
          const float d1 = act == 0 ? 1.f - hv.y * hv.y : (hv.y > 0.f ? 1.f : 0.f);
          v[j] = rok ? v[j] * d0 : 0.f;
          v[j + 1] = rok ? v[j + 1] * d1 : 0.f;
        }
      }
    }
    put_row_chunks(blk, rl, c16, v);
    if (act != 3) {
      const float colsum = warp_reduce_scatter32(v);
      cs_q[col_tile + c0 + lane] += colsum;
    }
  });
}

// dP = a * act'(H) for one warp's 32 rows (rl = row in the tile) of one
// 64-column block, from the NEGATED accumulator -a in TMEM columns
// [taddr, taddr + 64) of the warp's lane quarter (the product was run with
// -dz): for tanh, dP = (-a) * (H^2 - 1) in packed fp32 pairs, which rounds
// exactly as a * (1 - H^2) does.  H is in `blk` (128 rows x 128 bytes,
// 128-byte swizzle), overwritten in place by dP (bf16); the block's column
// sums are added to cs[0, 64).  Rows past the last one need no masking:
// their H rows are TMA zero fill and their accumulator rows are zero (a zero
// dz row), so dP is zero there.  mid() runs between the two 32-column chunks.
template <class Mid>
__device__ __forceinline__ void epi_dact_block(uint32_t taddr, int rl, int act, uint8_t* blk,
                                               float* cs, int lane, Mid&& mid) {
  uint8_t* row = blk + rl * 128;
  tmem_chunks<2>(taddr, 0, [&](const uint32_t (&r)[32], int c0) {
    float v[32];
    const int c16 = c0 / 8;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint4 a4 = *reinterpret_cast<const uint4*>(row + (((c16 + i) ^ (rl & 7)) << 4));
      const uint32_t w4[4] = {a4.x, a4.y, a4.z, a4.w};
#pragma unroll
      for (int hh = 0; hh < 4; ++hh) {
        const float2 hv = unpack_bf16x2(w4[hh]);
        const float2 na = make_float2(__uint_as_float(r[8 * i + 2 * hh]),
                                      __uint_as_float(r[8 * i + 2 * hh + 1]));
        float2 dp;
        if (act == 0) {
          dp = fmul2(na, ffma2(hv, hv, make_float2(-1.f, -1.f)));
        } else {
          dp.x = hv.x > 0.f ? -na.x : 0.f;
          dp.y = hv.y > 0.f ? -na.y : 0.f;
        }
        v[8 * i + 2 * hh] = dp.x;
        v[8 * i + 2 * hh + 1] = dp.y;
      }
    }
    put_row_chunks(row, rl, c16, v);
    const float colsum = warp_reduce_scatter32(v);
    cs[c0 + lane] += colsum;
    if (c0 == 0) mid();
  });
}

// The same with the column sums kept in registers: lane j of the warp holds
// column tn * BN + h * PART + 32 k + j of column tile tn in csr[CPW tn + k]
// (NT column tiles at most; the warp's part is PART = 32 CPW columns).
template <int BN, int EW, int NT>
__device__ __forceinline__ void epi_dact_smem_tile_r(uint32_t taddr, int rl, bool rok, int tn,
                                                     int h, int act, uint8_t* aux,
                                                     float (&csr)[NT * (BN / (EW / 4) / 32)],
                                                     int lane, float alpha = 0.f,
                                                     float beta = 0.f) {
  constexpr int PART = BN / (EW / 4);
  tmem_chunks<PART / 32>(taddr, h * PART, [&](const uint32_t (&r)[32], int c0) {
    float v[32];
#pragma unroll
    for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(r[j]);
    uint8_t* blk = aux + (c0 / 64) * 16384 + rl * 128;
    const int c16 = (c0 % 64) / 8;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint4 a4 = *reinterpret_cast<const uint4*>(blk + (((c16 + i) ^ (rl & 7)) << 4));
      const uint32_t w4[4] = {a4.x, a4.y, a4.z, a4.w};
#pragma unroll
      for (int hh = 0; hh < 4; ++hh) {
        const float2 hv = unpack_bf16x2(w4[hh]);
        const int j = 8 * i + 2 * hh;
        if (act == 3) {
          v[j] = rok ? alpha * hv.x + beta * v[j] : 0.f;
          v[j + 1] = rok ? alpha * hv.y + beta * v[j + 1] : 0.f;
        } else {
          const float d0 = act == 0 ? 1.f - hv.x * hv.x : (hv.x > 0.f ? 1.f : 0.f);
          const float d1 = act == 0 ? 1.f - hv.y * hv.y : (hv.y > 0.f ? 1.f : 0.f);
          v[j] = rok ? v[j] * d0 : 0.f;
          v[j + 1] = rok ? v[j + 1] * d1 : 0.f;
        }
      }
    }
    put_row_chunks(blk, rl, c16, v);
    if (act != 3) {
      const float colsum = warp_reduce_scatter32(v);
      constexpr int CPW = PART / 32;
      const int kk = (c0 - h * PART) >> 5;   // chunk of the warp's PART columns
#pragma unroll
      for (int t = 0; t < NT; ++t)
#pragma unroll
        for (int k2 = 0; k2 < CPW; ++k2)
          if (tn == t && kk == k2) csr[CPW * t + k2] += colsum;
    }
  });
}

// Forward epilogue, out = act(acc + bias), for one epilogue warp: its 32 rows
// (lane = row) and columns [h*PART, (h+1)*PART) of the tile go to the warp's
// staging buffer stg as PART/64 blocks of 32 rows x 128 bytes in the 128-byte
// swizzled layout, ready for one TMA store per block.
template <int BN, int EW>
__device__ __forceinline__ void epi_act_stage_tile(uint32_t taddr, int col_tile, int h, int act,
                                                   const float* bias_s, uint8_t* stg, int lane) {
  constexpr int PART = BN / (EW / 4);
  const int cbase = h * PART;
  tmem_chunks<PART / 32>(taddr, cbase, [&](const uint32_t (&r)[32], int c0) {
    float v[32];
    act_bias_chunk(r, bias_s + col_tile + c0, act, v);
    const int lc = c0 - cbase;   // column within the warp's part
    put_row_chunks(stg + (lc / 64) * 4096 + lane * 128, lane, (lc % 64) / 8, v);
  });
}

// Forward epilogue into a 128-row operand tile: out = act(acc + bias) for the
// warp's row rl (thread = row) and columns [h*PART, (h+1)*PART) of an N-column
// accumulator, written as bf16 into 128-row x 64-column blocks (16 KB each,
// 128-byte swizzle) at dst + (column / 64) * 16384 -- the K-major layout of a
// tensor-core A operand, and the layout of 32-row TMA store boxes.
template <int N, int EW>
__device__ __forceinline__ void epi_act_to_blocks(uint32_t taddr, int h, int act,
                                                  const float* bias_s, uint8_t* dst, int rl) {
  constexpr int PART = N / (EW / 4);
  tmem_chunks<PART / 32>(taddr, h * PART, [&](const uint32_t (&r)[32], int c0) {
    float v[32];
    act_bias_chunk(r, bias_s + c0, act, v);
    put_row_chunks(dst + (c0 / 64) * 16384 + rl * 128, rl, (c0 % 64) / 8, v);
  });
}

// Column masks of the head layout (bit k = column k): first / last column of
// each discrete head, all discrete columns, Gaussian means (column g0 + g).
struct HeadMasks {
  uint32_t hs, he, hd, gm;
  int g0, vcol, G;
};

__host__ __device__ constexpr HeadMasks head_masks(const NetShape& s) {
  HeadMasks m{0u, 0u, 0u, 0u, 0, s.C - 1, s.G};
  int off = 0;
  for (int h = 0; h < s.NH; ++h) {
    const int n = s.head_n[h];
    m.hs |= 1u << off;
    m.he |= 1u << (off + n - 1);
    m.hd |= ((1u << n) - 1u) << off;
    off += n;
  }
  m.g0 = off;
  m.gm = s.G > 0 ? ((1u << s.G) - 1u) << off : 0u;
  return m;
}

// Four discrete heads of 9, 2, 2 and 2 actions and the value column (16
// columns, no Gaussian dimensions): with its masks as compile-time constants
// the compiler resolves every per-column test of the loss, and the running
// scans become straight-line per-head code (measured 6x faster than with
// run-time masks).  Every other layout takes the run-time masks.
__host__ __device__ constexpr NetShape shape_9222() {
  NetShape s{};
  s.NH = 4;
  s.head_n[0] = 9;
  s.head_n[1] = 2;
  s.head_n[2] = 2;
  s.head_n[3] = 2;
  s.G = 0;
  s.C = 16;
  s.CP = 16;
  return s;
}
constexpr HeadMasks kMasks9222 = head_masks(shape_9222());
static_assert(kMasks9222.hs == 0x2A01u && kMasks9222.he == 0x5500u && kMasks9222.hd == 0x7FFFu &&
                  kMasks9222.gm == 0u && kMasks9222.g0 == 15 && kMasks9222.vcol == 15 &&
                  kMasks9222.G == 0,
              "head masks of the 9-2-2-2 layout");
__host__ __device__ inline bool is_layout_9222(const NetShape& s) {
  return s.NH == 4 && s.head_n[0] == 9 && s.head_n[1] == 2 && s.head_n[2] == 2 &&
         s.head_n[3] == 2 && s.G == 0 && s.C == 16 && s.CP == 16;
}

// Per-row PPO loss and d(loss)/dz for one row of head outputs z (CP columns),
// the same quantities as row_loss: log-softmax per discrete head, Gaussian
// log-density, entropy, clipped surrogate, value loss, and their gradients
// ("Proximal Policy Optimization Algorithms", sec. 3 and 5).  Heads are
// contiguous column segments, so every per-head reduction is a segmented scan
// over the compile-time-indexed columns and all state stays in registers.
// exp and log are the hardware approximations (__expf/__logf, relative error
// about 1e-6, far inside the bf16 path's tolerance).  amask has one bit per
// head: the column of the taken action.
template <int CP>
__device__ __forceinline__ void row_loss_seg(const HeadMasks& hm, const LossCoef& lc, float inv_mb,
                                             const float (&z)[32], uint32_t amask,
                                             const float* actc, const float* logstd,
                                             float logp_old, float A, float R, float (&dz)[32],
                                             float (&t6)[6], float (&dls)[4]) {
  const float LOG_2PI = 1.8378770664093453f;
  float u[CP], w[CP];
  // head max: running max from each head's first column, broadcast back from its last
  float run = 0.f;
#pragma unroll
  for (int k = 0; k < CP; ++k) {
    run = ((hm.hs >> k) & 1u) ? z[k] : fmaxf(run, z[k]);
    u[k] = run;
  }
#pragma unroll
  for (int k = CP - 2; k >= 0; --k)
    if (!((hm.he >> k) & 1u)) u[k] = u[k + 1];
  // sum of exp(z - max) per head, then log-sum-exp broadcast back
  float srun = 0.f;
#pragma unroll
  for (int k = 0; k < CP; ++k) {
    const float e = ((hm.hd >> k) & 1u) ? __expf(z[k] - u[k]) : 0.f;
    srun = ((hm.hs >> k) & 1u) ? e : srun + e;
    w[k] = srun;
  }
#pragma unroll
  for (int k = CP - 1; k >= 0; --k) {
    if ((hm.he >> k) & 1u) u[k] = u[k] + __logf(w[k]);
    else if (k + 1 < CP) u[k] = u[k + 1];
  }
  // log-probabilities, probabilities, per-head entropy (kept in dz for now)
  float logp = 0.f, ent = 0.f, erun = 0.f;
#pragma unroll
  for (int k = 0; k < CP; ++k) {
    const bool d = (hm.hd >> k) & 1u;
    const float lp = z[k] - u[k];
    const float pk = d ? __expf(lp) : 0.f;
    u[k] = lp;
    w[k] = pk;
    const float hk = d ? -(pk * lp) : 0.f;
    erun = ((hm.hs >> k) & 1u) ? hk : erun + hk;
    dz[k] = erun;
    if ((hm.he >> k) & 1u) ent += erun;
    if ((amask >> k) & 1u) logp += lp;
  }
#pragma unroll
  for (int k = CP - 2; k >= 0; --k)
    if (!((hm.he >> k) & 1u)) dz[k] = dz[k + 1];
  // the value and the Gaussian means, picked out of the row with selects (the
  // Gaussian terms are computed once per dimension, not once per column)
  float value = 0.f, mu[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int k = 0; k < CP; ++k) {
    value = (k == hm.vcol) ? z[k] : value;
#pragma unroll
    for (int g = 0; g < 4; ++g) mu[g] = (k == hm.g0 + g) ? z[k] : mu[g];
  }
  float ag[4], lsg[4], ivg[4];
#pragma unroll
  for (int g = 0; g < 4; ++g) {
    ag[g] = 0.f;
    lsg[g] = 0.f;
    ivg[g] = 0.f;
    if (g < hm.G) {
      ag[g] = actc[g];
      lsg[g] = logstd[g];
      ivg[g] = __expf(-2.f * lsg[g]);
      logp += -0.5f * (ag[g] - mu[g]) * (ag[g] - mu[g]) * ivg[g] - lsg[g] - 0.5f * LOG_2PI;
      ent += 0.5f + 0.5f * LOG_2PI + lsg[g];
    }
  }
  const float log_ratio = logp - logp_old;
  const float ratio = __expf(log_ratio);
  const float lo = 1.f - lc.clip, hi = 1.f + lc.clip;
  const float clipped = fminf(fmaxf(ratio, lo), hi);
  const float s1 = ratio * A, s2 = clipped * A;
  const float pg = -fminf(s1, s2);
  const float vdiff = value - R;
  const float vl = vdiff * vdiff;
  t6[0] = pg + lc.vf * vl - lc.ent * ent;
  t6[1] = pg;
  t6[2] = vl;
  t6[3] = ent;
  t6[4] = fabsf(ratio - 1.f) > lc.clip ? 1.f : 0.f;
  t6[5] = (ratio - 1.f) - log_ratio;
  const float g_logp = (s1 <= s2) ? -A * ratio * inv_mb : 0.f;
  const float g_ent = -lc.ent * inv_mb;
  const float dz_value = lc.vf * 2.f * vdiff * inv_mb;
#pragma unroll
  for (int k = 0; k < CP; ++k) {
    const float dlogp = (((amask >> k) & 1u) ? 1.f : 0.f) - w[k];
    const float dent = -w[k] * (u[k] + dz[k]);
    const float dd = g_logp * dlogp + g_ent * dent;
    dz[k] = ((hm.hd >> k) & 1u) ? dd : 0.f;
    dz[k] = (k == hm.vcol) ? dz_value : dz[k];
  }
#pragma unroll
  for (int g = 0; g < 4; ++g) {
    if (g < hm.G) {
      const float d = ag[g] - mu[g];
      const float dzg = g_logp * d * ivg[g];
      dls[g] = g_logp * (d * d * ivg[g] - 1.f) + g_ent;
#pragma unroll
      for (int k = 0; k < CP; ++k) dz[k] = (k == hm.g0 + g) ? dzg : dz[k];
    }
  }
}

// Per-row loss of one 128 x BN head tile (BN = CP columns), thread = row:
// z = TMEM accumulator + b3, then d(loss)/dz, the loss terms and dlogstd in
// registers (all zero for rows >= M).
// The per-row inputs of the loss that do not depend on the head product:
// loaded before the epilogue waits for the accumulator, so that their latency
// overlaps the wait.
struct RowIn {
  int av[PPO_MAX_HEADS];
  float ac[4];
  float logp_old, adv, ret;
};

__device__ __forceinline__ void load_row_in(RowIn& in, int row, bool rok, const NetShape& s,
                                            const LossRows& rows) {
#pragma unroll
  for (int h = 0; h < PPO_MAX_HEADS; ++h) in.av[h] = rok && h < s.NH ? rows.act[(int64_t)row * s.NH + h] : 0;
#pragma unroll
  for (int g = 0; g < 4; ++g) in.ac[g] = rok && g < s.G ? rows.actc[(int64_t)row * s.G + g] : 0.f;
  in.logp_old = rok ? rows.logp_old[row] : 0.f;
  in.adv = rok ? rows.adv[row] : 0.f;
  in.ret = rok ? rows.ret[row] : 0.f;
}

// loss_row_regs with the row inputs already in registers
template <int BN>
__device__ __forceinline__ void loss_row_in(uint32_t taddr, bool rok, const NetShape& s,
                                            const HeadMasks& hm, const LossCoef& lc, float inv_mb,
                                            const RowIn& in, const float* logstd,
                                            const float* bias_s, float (&dzr)[32], float (&t6)[6],
                                            float (&dls)[4]) {
  float v[32];
  if constexpr (BN == 16) tmem_ld16(taddr, v);
  else tmem_ld32(taddr, v);
  float z[32];
#pragma unroll
  for (int j = 0; j < 32; ++j) {
    z[j] = (j < BN && j < s.C) ? v[j] + bias_s[j] : 0.f;
    dzr[j] = 0.f;
  }
#pragma unroll
  for (int k = 0; k < 6; ++k) t6[k] = 0.f;
#pragma unroll
  for (int k = 0; k < 4; ++k) dls[k] = 0.f;
  if (rok) {
    uint32_t amask = 0u;
    int off = 0;
#pragma unroll
    for (int h = 0; h < PPO_MAX_HEADS; ++h) {
      if (h < s.NH) amask |= 1u << (off + in.av[h]);
      off += h < s.NH ? s.head_n[h] : 0;
    }
    row_loss_seg<BN>(hm, lc, inv_mb, z, amask, in.ac, logstd, in.logp_old, in.adv, in.ret, dzr,
                     t6, dls);
  }
}

template <int BN>
__device__ __forceinline__ void loss_row_regs(uint32_t taddr, int row, bool rok,
                                              const NetShape& s, const HeadMasks& hm,
                                              const LossCoef& lc, float inv_mb,
                                              const LossRows& rows, const float* logstd,
                                              const float* bias_s, float (&dzr)[32],
                                              float (&t6)[6], float (&dls)[4]) {
  float v[32];
  if constexpr (BN == 16) tmem_ld16(taddr, v);
  else tmem_ld32(taddr, v);
  float z[32];
#pragma unroll
  for (int j = 0; j < 32; ++j) {
    z[j] = (j < BN && j < s.C) ? v[j] + bias_s[j] : 0.f;
    dzr[j] = 0.f;
  }
#pragma unroll
  for (int k = 0; k < 6; ++k) t6[k] = 0.f;
#pragma unroll
  for (int k = 0; k < 4; ++k) dls[k] = 0.f;
  if (rok) {
    uint32_t amask = 0u;
    int off = 0;
    const int32_t* a = rows.act + (int64_t)row * s.NH;
    int av[PPO_MAX_HEADS];
#pragma unroll
    for (int h = 0; h < PPO_MAX_HEADS; ++h) av[h] = h < s.NH ? a[h] : 0;   // loads in flight together
#pragma unroll
    for (int h = 0; h < PPO_MAX_HEADS; ++h) {
      if (h < s.NH) amask |= 1u << (off + av[h]);
      off += h < s.NH ? s.head_n[h] : 0;
    }
    row_loss_seg<BN>(hm, lc, inv_mb, z, amask, rows.actc + (int64_t)row * s.G, logstd,
                     rows.logp_old[row], rows.adv[row], rows.ret[row], dzr, t6, dls);
  }
}

// Warp-level reductions of the loss epilogue: column sums of dz into cs_q,
// the six loss terms and dlogstd into lp_q (fixed order).
__device__ __forceinline__ void loss_warp_reduce(float (&dzr)[32], const float (&t6)[6],
                                                 const float (&dls)[4], float* cs_q, float* lp_q,
                                                 int lane) {
  const float colsum = warp_reduce_scatter32(dzr);
  cs_q[lane] += colsum;
#pragma unroll
  for (int k = 0; k < 6; ++k) {
    const float s6 = warp_sum(t6[k]);
    if (lane == 0) lp_q[k] += s6;
  }
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const float s4 = warp_sum(dls[k]);
    if (lane == 0) lp_q[6 + k] += s4;
  }
}

// Loss epilogue of one 128 x BN head tile: dz (bf16) to global row by row,
// per-warp reductions into cs_q / lp_q.
template <int BN>
__device__ __forceinline__ void epi_loss_tile(uint32_t taddr, int row, bool rok, const NetShape& s,
                                              const HeadMasks& hm, const LossCoef& lc,
                                              float inv_mb, const RowIn& in,
                                              const float* logstd, const float* bias_s,
                                              __nv_bfloat16* dz, int lddz, float* cs_q,
                                              float* lp_q, int lane) {
  float dzr[32], t6[6], dls[4];
  loss_row_in<BN>(taddr, rok, s, hm, lc, inv_mb, in, logstd, bias_s, dzr, t6, dls);
  if (rok) {
    uint4* d = reinterpret_cast<uint4*>(dz + (int64_t)row * lddz);
#pragma unroll
    for (int i = 0; i < BN / 8; ++i) {
      uint4 u;
      u.x = pack_bf16x2(dzr[8 * i + 0], dzr[8 * i + 1]);
      u.y = pack_bf16x2(dzr[8 * i + 2], dzr[8 * i + 3]);
      u.z = pack_bf16x2(dzr[8 * i + 4], dzr[8 * i + 5]);
      u.w = pack_bf16x2(dzr[8 * i + 6], dzr[8 * i + 7]);
      d[i] = u;
    }
  }
  loss_warp_reduce(dzr, t6, dls, cs_q, lp_q, lane);
}

// Weight-gradient epilogue: the fp32 accumulator of one 128 x bn unit tile
// goes to its split-K partial (rows < M, columns < N).
__device__ __forceinline__ void epi_wgrad_tile(uint32_t taddr, int row, int bn, int M, int N,
                                               int col_tile, float* part_split) {
#pragma unroll 1
  for (int c0 = 0; c0 < bn; c0 += 32) {
    float v[32];
    tmem_ld32(taddr + (uint32_t)c0, v);
    const int col0 = col_tile + c0;
    if (row < M && col0 < N) {
      float4* dst = reinterpret_cast<float4*>(part_split + (int64_t)row * N + col0);
#pragma unroll
      for (int i = 0; i < 8; ++i)
        dst[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
    }
  }
}

}  // namespace tc
}  // namespace ppo
