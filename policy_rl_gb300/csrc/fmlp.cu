// fmlp.cu -- fused forward, loss and backward-data pass of a small
// actor-critic MLP on tensor cores, one 128-row minibatch tile at a time.
//
// "Teaching Mario to speedrun", sec. 5 "Policy network" (two tanh/ReLU
// layers, then the head logits and the value) and sec. 6 "The whole
// algorithm" (the PPO loss and loss.backward()).  For one tile of rows:
//
//   H1 = act(X W1^T + b1)            tensor cores, X from shared memory
//   H2 = act(H1 W2^T + b2)           A operand = H1, still in shared memory
//   Z  = H2 W3^T + b3 -> dz          per-row loss epilogue
//   dP2 = (dz W3) * act'(H2)         A operand = dz; H2 from shared memory
//   dP1 = (dP2 W2) * act'(H1)        A operand = dP2 (in place of H2)
//
// The per-stage kernels write each activation to HBM and read it back in the
// next launch; here the tile's H1, H2/dP2 and dz stay in shared memory (as
// 128-byte-swizzled K-major operand blocks) and each result is written once,
// by TMA stores, for the weight-gradient kernel.  The weights stream through a
// two-stage TMA ring from L2.  TMEM holds two 256-column accumulators, used in
// turn by the five products.  Shapes: padded obs width <= 64, hidden widths
// 128 or 256, head columns <= 32 (shared memory holds X, H1 and H2 tiles).
//
// Roles: warp 0 issues TMA loads, warp 1 issues MMAs, warps 2..9 run the
// epilogues (TMEM lane quarter q = warp % 4, column half h).  Every wait is
// bounded (abort flag + device error latch), as in the other tensor-core
// kernels of this library.
#include <cuda.h>

#include "common.cuh"
#include "gemm.h"
#include "tc_ptx.cuh"
#include "tc_tile.cuh"

namespace ppo {

namespace {

using namespace ptx;
using namespace tc;

constexpr int kFWarps = 10;
constexpr int kFThreads = kFWarps * kWarp;
constexpr int kEpiThreads = 8 * kWarp;
constexpr int kBlk = 128 * 128;           // 128 rows x 64 bf16 columns
constexpr int kWStage = 256 * 64 * 2;     // one [<= 256 rows][64] bf16 weight box
constexpr int kWS = 2;                    // weight ring stages
constexpr int kHMax = 256;

// shared-memory layout (offsets from the 1024-aligned base)
constexpr int kOffX = 0;                          // X tile (Dp <= 64), then dz
constexpr int kOffHA = kOffX + kBlk;              // H1 / dP1: 4 blocks
constexpr int kOffHB = kOffHA + 4 * kBlk;         // H2 / dP2: 4 blocks
constexpr int kOffRing = kOffHB + 4 * kBlk;
constexpr int kOffCtrl = kOffRing + kWS * kWStage;
constexpr int kCtrlBytes = 512;
constexpr int kOffCs1 = kOffCtrl + kCtrlBytes;    // [4][kHMax]
constexpr int kOffCs2 = kOffCs1 + 4 * kHMax * 4;  // [4][kHMax]
constexpr int kOffCs3 = kOffCs2 + 4 * kHMax * 4;  // [4][32]
constexpr int kOffLp = kOffCs3 + 4 * 32 * 4;      // [4][kLossPartials]
constexpr int kOffBias = kOffLp + 4 * kLossPartials * 4;   // b1[256], b2[256], b3[32]
constexpr int kSmemBytes = 1024 + kOffBias + (2 * kHMax + 32) * 4;

// barrier indices inside the control block
constexpr int kBarFull = 0;                 // [kWS]
constexpr int kBarEmpty = kBarFull + kWS;   // [kWS]
constexpr int kBarX = kBarEmpty + kWS;      // X tile landed
constexpr int kBarTf = kBarX + 1;           // [5] product k finished (tcgen05.commit)
constexpr int kBarRdy = kBarTf + 5;         // [5] epilogue k finished
constexpr int kBarDrain = kBarRdy + 5;
constexpr int kNumBars = kBarDrain + 1;

struct FMaps {
  CUtensorMap x, w1, w2, w3, w3t, w2t;     // loads (w3: 3-D, all blocks in one box)
  CUtensorMap h1, h2, dz, dp2, dp1;        // stores (32-row x 64-column boxes)
};

struct FParams {
  int M, tiles, Dp, CP, act;
  const float *b1, *b2, *b3, *logstd;
  NetShape shape;
  LossCoef lc;
  LossRows rows;
  float inv_mb;
  float *cs1, *cs2, *cs3, *lossp;   // per-CTA partial rows
  int* err;
  uint64_t timeout_ns;
};

// 4 k-steps of 16 over one 64-column block: A block (128 rows) x B stage
__device__ __forceinline__ void mma_block(uint32_t d, uint32_t a_blk, uint32_t b_stage,
                                          uint32_t idesc, bool first, int ksteps) {
  for (int kk = 0; kk < ksteps; ++kk)
    tc_mma_bf16(d, sdesc_sw128(a_blk + kk * 32, 16, 1024), sdesc_sw128(b_stage + kk * 32, 16, 1024),
                idesc, (first && kk == 0) ? 0u : 1u);
}

template <int H1, int H2, int CP>
__global__ void __launch_bounds__(kFThreads, 1)
fmlp_kernel(const __grid_constant__ FMaps maps, const FParams p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gb = smem_raw + (base - raw);
  uint8_t* XA = gb + kOffX;
  uint8_t* HA = gb + kOffHA;
  uint8_t* HB = gb + kOffHB;
  uint64_t* bars = reinterpret_cast<uint64_t*>(gb + kOffCtrl);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(bars + kNumBars);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tslot + 1);
  volatile uint32_t* cnt = reinterpret_cast<volatile uint32_t*>(tslot + 2);  // ring issued, consumed, X issued
  float* cs1 = reinterpret_cast<float*>(gb + kOffCs1);
  float* cs2 = reinterpret_cast<float*>(gb + kOffCs2);
  float* cs3 = reinterpret_cast<float*>(gb + kOffCs3);
  float* lp = reinterpret_cast<float*>(gb + kOffLp);
  float* b1s = reinterpret_cast<float*>(gb + kOffBias);
  float* b2s = b1s + kHMax;
  float* b3s = b2s + kHMax;
  auto bar = [&](int i) { return smem_u32(&bars[i]); };
  const uint32_t ring = base + kOffRing;

  const int warp = threadIdx.x / kWarp, lane = threadIdx.x % kWarp;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kWS; ++s) {
      mbar_init(bar(kBarFull + s), 1);
      mbar_init(bar(kBarEmpty + s), 1);
    }
    mbar_init(bar(kBarX), 1);
    for (int k = 0; k < 5; ++k) {
      mbar_init(bar(kBarTf + k), 1);
      mbar_init(bar(kBarRdy + k), kEpiThreads);
    }
    mbar_init(bar(kBarDrain), 1);
    *abort_flag = 0;
    cnt[0] = 0;
    cnt[1] = 0;
    cnt[2] = 0;
    fence_mbar_init();
  }
  for (int i = threadIdx.x; i < (kOffBias - kOffCs1) / 4; i += kFThreads) cs1[i] = 0.f;
  if (warp == 1) tmem_alloc(smem_u32(tslot), 512);
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&maps.x);
    prefetch_tmap(&maps.w1);
    prefetch_tmap(&maps.w2);
    prefetch_tmap(&maps.w3);
    prefetch_tmap(&maps.w3t);
    prefetch_tmap(&maps.w2t);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tslot;
  const Guard g{abort_flag, p.err, p.timeout_ns};
  pdl_wait();
  pdl_trigger();
  for (int i = threadIdx.x; i < H1; i += kFThreads) b1s[i] = p.b1[i];
  for (int i = threadIdx.x; i < H2; i += kFThreads) b2s[i] = p.b2[i];
  for (int i = threadIdx.x; i < 32; i += kFThreads) b3s[i] = i < p.shape.C ? p.b3[i] : 0.f;
  __syncthreads();   // reached by every thread of the block (before the role split)

  const int nx = p.Dp / 64;   // X blocks (1)
  if (warp == 0) {
    if (lane == 0) {
      uint32_t it = 0, t = 0;
      bool ok = true;
      auto put = [&](const CUtensorMap* m, int x, int rows) -> bool {
        const int s = it % kWS;
        const uint32_t r = it / kWS;
        if (!wait_bar(bar(kBarEmpty + s), (r & 1) ^ 1, g)) return false;
        mbar_arrive_expect_tx(bar(kBarFull + s), (uint32_t)rows * 128u);
        tma_load_2d(ring + (uint32_t)(s * kWStage), m, x, 0, bar(kBarFull + s));
        ++it;
        cnt[0] = it;
        return true;
      };
      for (int tile = blockIdx.x; tile < p.tiles && ok; tile += gridDim.x, ++t) {
        // X shares its block with the previous tile's dz: wait for that tile's dz product
        if (t > 0 && !wait_bar(bar(kBarTf + 3), (t - 1) & 1, g)) break;
        mbar_arrive_expect_tx(bar(kBarX), (uint32_t)(nx * kBlk));
        for (int kb = 0; kb < nx; ++kb)
          tma_load_2d(base + kOffX + kb * kBlk, &maps.x, kb * 64, tile * 128, bar(kBarX));
        cnt[2] = t + 1;
        // the weight boxes, in the order the products consume them
        for (int kb = 0; kb < nx && ok; ++kb) ok = put(&maps.w1, kb * 64, H1);
        for (int kb = 0; kb < H1 / 64 && ok; ++kb) ok = put(&maps.w2, kb * 64, H2);
        if (ok) {   // all of W3 (H2/64 blocks of CP rows) in one 3-D box
          const int sw = it % kWS;
          const uint32_t rw = it / kWS;
          ok = wait_bar(bar(kBarEmpty + sw), (rw & 1) ^ 1, g);
          if (ok) {
            mbar_arrive_expect_tx(bar(kBarFull + sw), (uint32_t)(CP * H2 * 2));
            tma_load_3d(ring + (uint32_t)(sw * kWStage), &maps.w3, 0, 0, 0, bar(kBarFull + sw));
            ++it;
            cnt[0] = it;
          }
        }
        if (ok) ok = put(&maps.w3t, 0, H2);
        for (int kb = 0; kb < H2 / 64 && ok; ++kb) ok = put(&maps.w2t, kb * 64, H1);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      uint32_t it = 0, t = 0;
      const uint32_t R0 = tmem, R1 = tmem + 256;
      auto ring_block = [&](uint32_t d, uint32_t a_blk, uint32_t idesc, bool first,
                            int ksteps) -> bool {
        const int s = it % kWS;
        const uint32_t r = it / kWS;
        if (!wait_bar(bar(kBarFull + s), r & 1, g)) return false;
        tc_fence_after();
        mma_block(d, a_blk, ring + (uint32_t)(s * kWStage), idesc, first, ksteps);
        tc_commit(bar(kBarEmpty + s));
        ++it;
        cnt[1] = it;
        return true;
      };
      bool ok = true;
      for (int tile = blockIdx.x; tile < p.tiles && ok; tile += gridDim.x, ++t) {
        const uint32_t ph = t & 1, pph = (t - 1) & 1;
        // 1: R0 = X W1^T  (R0 free once the previous tile's dP1 epilogue is done)
        if (!wait_bar(bar(kBarX), ph, g)) break;
        if (t > 0 && !wait_bar(bar(kBarRdy + 4), pph, g)) break;
        tc_fence_after();
        for (int kb = 0; kb < nx && ok; ++kb)
          ok = ring_block(R0, base + kOffX + kb * kBlk, idesc_bf16(128, H1, false, false), kb == 0, 4);
        if (!ok) break;
        tc_commit(bar(kBarTf + 0));
        // 2: R1 = H1 W2^T
        if (!wait_bar(bar(kBarRdy + 0), ph, g)) break;
        tc_fence_after();
        for (int kb = 0; kb < H1 / 64 && ok; ++kb)
          ok = ring_block(R1, base + kOffHA + kb * kBlk, idesc_bf16(128, H2, false, false), kb == 0, 4);
        if (!ok) break;
        tc_commit(bar(kBarTf + 1));
        // 3: R0[0, CP) = H2 W3^T  (one ring stage: H2/64 blocks of CP rows)
        if (!wait_bar(bar(kBarRdy + 1), ph, g)) break;
        tc_fence_after();
        {
          const int s3 = it % kWS;
          const uint32_t r3 = it / kWS;
          if (!wait_bar(bar(kBarFull + s3), r3 & 1, g)) break;
          tc_fence_after();
          for (int kb = 0; kb < H2 / 64; ++kb)
            mma_block(R0, base + kOffHB + kb * kBlk, ring + (uint32_t)(s3 * kWStage + kb * CP * 128),
                      idesc_bf16(128, CP, false, false), kb == 0, 4);
          tc_commit(bar(kBarEmpty + s3));
          ++it;
          cnt[1] = it;
        }
        tc_commit(bar(kBarTf + 2));
        // 4: R1 = dz W3  (K = CP: CP/16 k-steps of the dz block)
        if (!wait_bar(bar(kBarRdy + 2), ph, g)) break;
        tc_fence_after();
        ok = ring_block(R1, base + kOffX, idesc_bf16(128, H2, false, false), true, CP / 16);
        if (!ok) break;
        tc_commit(bar(kBarTf + 3));
        // 5: R0 = dP2 W2
        if (!wait_bar(bar(kBarRdy + 3), ph, g)) break;
        tc_fence_after();
        for (int kb = 0; kb < H2 / 64 && ok; ++kb)
          ok = ring_block(R0, base + kOffHB + kb * kBlk, idesc_bf16(128, H1, false, false), kb == 0, 4);
        if (!ok) break;
        tc_commit(bar(kBarTf + 4));
      }
    }
  } else {
    const int q = warp & 3;
    const int h = (warp - 2) / 4;
    const int rl = q * 32 + lane;
    const HeadMasks hm = head_masks(p.shape);
    const uint32_t lanes = (uint32_t)(q * 32) << 16;
    const uint32_t R0 = tmem + lanes, R1 = tmem + 256 + lanes;
    // TMA-store this warp's rows of nblk 64-column blocks of a 128-row tile.
    // The store reads shared memory asynchronously: a later write to the same
    // blocks first waits for it (bulk_wait_read0 below, before E1 and E3 -- E1
    // covers the stores of E4/E5, E3 those of E1/E2).
    auto store_rows = [&](const CUtensorMap* m, const uint8_t* tile_base, int blk0, int nblk,
                          int row0) {
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0 && row0 + q * 32 < p.M) {   // boxes wholly below the last row are skipped
        for (int b = blk0; b < blk0 + nblk; ++b)
          tma_store_2d(m, smem_u32(tile_base + b * kBlk + q * 4096), b * 64, row0 + q * 32);
        bulk_commit();
      }
      __syncwarp();
    };
    auto stores_read = [&]() {
      if (lane == 0) bulk_wait_read0();
      __syncwarp();
    };
    uint32_t t = 0;
    for (int tile = blockIdx.x; tile < p.tiles; tile += gridDim.x, ++t) {
      const uint32_t ph = t & 1;
      const int row0 = tile * 128;
      const int row = row0 + rl;
      const bool rok = row < p.M;
      // E1: H1 = act(R0 + b1) -> HA, stored
      if (!wait_bar(bar(kBarTf + 0), ph, g)) break;
      tc_fence_after();
      stores_read();   // HA (dP1) and HB (dP2) of the previous tile have been read out
      epi_act_to_blocks<H1, 8>(R0, h, p.act, b1s, HA, rl);
      tc_fence_before();
      store_rows(&maps.h1, HA, h * (H1 / 128), H1 / 128, row0);
      mbar_arrive(bar(kBarRdy + 0));
      // E2: H2 = act(R1 + b2) -> HB, stored
      if (!wait_bar(bar(kBarTf + 1), ph, g)) break;
      tc_fence_after();
      epi_act_to_blocks<H2, 8>(R1, h, p.act, b2s, HB, rl);
      tc_fence_before();
      store_rows(&maps.h2, HB, h * (H2 / 128), H2 / 128, row0);
      mbar_arrive(bar(kBarRdy + 1));
      // E3: per-row loss on R0[0, CP) -> dz in the X block (columns >= CP zero), stored
      if (!wait_bar(bar(kBarTf + 2), ph, g)) break;
      tc_fence_after();
      if (h == 0) {
        float dzr[32], t6[6], dls[4];
        loss_row_regs<CP>(R0, row, rok, p.shape, hm, p.lc, p.inv_mb, p.rows, p.logstd, b3s, dzr,
                          t6, dls);
        uint8_t* drow = XA + rl * 128;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          uint4 u = make_uint4(0u, 0u, 0u, 0u);
          if (i < CP / 8) {
            u.x = pack_bf16x2(dzr[8 * i + 0], dzr[8 * i + 1]);
            u.y = pack_bf16x2(dzr[8 * i + 2], dzr[8 * i + 3]);
            u.z = pack_bf16x2(dzr[8 * i + 4], dzr[8 * i + 5]);
            u.w = pack_bf16x2(dzr[8 * i + 6], dzr[8 * i + 7]);
          }
          *reinterpret_cast<uint4*>(drow + ((i ^ (rl & 7)) << 4)) = u;
        }
        loss_warp_reduce(dzr, t6, dls, cs3 + q * 32, lp + q * kLossPartials, lane);
        tc_fence_before();
        store_rows(&maps.dz, XA, 0, 1, row0);
      } else {
        tc_fence_before();
      }
      // the X block (dz) is reloaded after the dz product, and HA / HB are
      // rewritten in place by E4 / E5: all stores so far have been read out
      stores_read();
      mbar_arrive(bar(kBarRdy + 2));
      // E4: dP2 = R1 * act'(H2), in place in HB, stored
      if (!wait_bar(bar(kBarTf + 3), ph, g)) break;
      tc_fence_after();
      epi_dact_smem_tile<H2, 8>(R1, rl, rok, 0, h, p.act, HB, cs2 + q * kHMax, lane);
      tc_fence_before();
      store_rows(&maps.dp2, HB, h * (H2 / 128), H2 / 128, row0);
      mbar_arrive(bar(kBarRdy + 3));
      // E5: dP1 = R0 * act'(H1), in place in HA, stored
      if (!wait_bar(bar(kBarTf + 4), ph, g)) break;
      tc_fence_after();
      epi_dact_smem_tile<H1, 8>(R0, rl, rok, 0, h, p.act, HA, cs1 + q * kHMax, lane);
      tc_fence_before();
      store_rows(&maps.dp1, HA, h * (H1 / 128), H1 / 128, row0);
      mbar_arrive(bar(kBarRdy + 4));
    }
    if (lane == 0) bulk_wait0();   // this warp's stores are complete before the CTA exits
  }

  __syncthreads();
  if (*abort_flag) {
    // drain: loads issued but never consumed, and outstanding MMAs
    if (threadIdx.x == 0) {
      const uint32_t issued = cnt[0], consumed = cnt[1];
      for (uint32_t it = consumed; it < issued; ++it)
        drain_wait(bar(kBarFull + it % kWS), (it / kWS) & 1, p.timeout_ns);
      const uint32_t xi = cnt[2];
      if (xi > 0) drain_wait(bar(kBarX), (xi - 1) & 1, p.timeout_ns);
    }
    if (warp == 1 && lane == 0) {
      tc_commit(bar(kBarDrain));
      drain_wait(bar(kBarDrain), 0, p.timeout_ns);
    }
    __syncthreads();
  }
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
  // per-CTA partial rows of the bias gradients and loss terms (fixed order)
  if (warp >= 2) {
    const int et = threadIdx.x - 2 * kWarp;
    auto quad = [&](const float* b, int ld, int c) {
      return ((b[c] + b[ld + c]) + b[2 * ld + c]) + b[3 * ld + c];
    };
    for (int c = et; c < H1; c += kEpiThreads)
      p.cs1[(int64_t)blockIdx.x * H1 + c] = quad(cs1, kHMax, c);
    for (int c = et; c < H2; c += kEpiThreads)
      p.cs2[(int64_t)blockIdx.x * H2 + c] = quad(cs2, kHMax, c);
    if (et < CP) p.cs3[(int64_t)blockIdx.x * CP + et] = quad(cs3, 32, et);
    if (et < kLossPartials)
      p.lossp[(int64_t)blockIdx.x * kLossPartials + et] = quad(lp, kLossPartials, et);
  }
}

template <int H1, int H2, int CP>
cudaError_t set_attr() {
  return cudaFuncSetAttribute(fmlp_kernel<H1, H2, CP>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              kSmemBytes);
}

template <int H1, int H2, int CP>
cudaError_t launch_t(const FMaps& maps, const FParams& p, int grid, cudaStream_t st) {
  return launch_pdl(fmlp_kernel<H1, H2, CP>, dim3(grid), dim3(kFThreads), (size_t)kSmemBytes, st,
                    maps, p);
}

}  // namespace

bool fmlp_supported(const NetShape& s) {
  return s.Dp == 64 && (s.H1 == 128 || s.H1 == 256) && (s.H2 == 128 || s.H2 == 256) &&
         (s.CP == 16 || s.CP == 32) && s.G <= 4;
}

cudaError_t fmlp_prepare() {
  const cudaError_t errs[] = {set_attr<256, 256, 16>(), set_attr<256, 256, 32>(),
                              set_attr<128, 128, 16>(), set_attr<128, 128, 32>(),
                              set_attr<256, 128, 16>(), set_attr<256, 128, 32>(),
                              set_attr<128, 256, 16>(), set_attr<128, 256, 32>()};
  for (cudaError_t e : errs)
    if (e != cudaSuccess) return e;
  return cudaSuccess;
}

cudaError_t fmlp_launch(const FusedMlp& f, int num_sms, cudaStream_t st, int* grid_out) {
  const NetShape& s = f.s;
  if (!fmlp_supported(s) || f.M < 1) return cudaErrorInvalidValue;
  FMaps m;
  cudaError_t e;
#define FM(dst, ptr, cols, rows, ld, bc, br) \
  if ((e = tc_make_tmap(&m.dst, ptr, cols, rows, ld, bc, br)) != cudaSuccess) return e;
  FM(x, f.X, s.Dp, f.M, s.Dp, 64, 128)
  FM(w1, f.W1s, s.Dp, s.H1, s.Dp, 64, s.H1)
  FM(w2, f.W2s, s.H1, s.H2, s.H1, 64, s.H2)
  if ((e = tc_make_tmap_blocks(&m.w3, f.W3s, s.CP, s.H2, s.H2 / 64, s.CP, s.H2 / 64)) !=
      cudaSuccess)
    return e;
  FM(w3t, f.W3Ts, 64, s.H2, f.ld3t, 64, s.H2)
  FM(w2t, f.W2Ts, s.H2, s.H1, s.H2, 64, s.H1)
  FM(h1, f.H1, s.H1, f.M, s.H1, 64, 32)
  FM(h2, f.H2, s.H2, f.M, s.H2, 64, 32)
  FM(dz, f.dZ, 64, f.M, f.lddz, 64, 32)
  FM(dp2, f.dP2, s.H2, f.M, s.H2, 64, 32)
  FM(dp1, f.dP1, s.H1, f.M, s.H1, 64, 32)
#undef FM
  FParams p{};
  p.M = f.M;
  p.tiles = (f.M + 127) / 128;
  p.Dp = s.Dp;
  p.CP = s.CP;
  p.act = s.act;
  p.b1 = f.b1;
  p.b2 = f.b2;
  p.b3 = f.b3;
  p.logstd = f.logstd;
  p.shape = s;
  p.lc = f.lc;
  p.rows = f.rows;
  p.inv_mb = f.inv_mb;
  p.cs1 = f.cs1;
  p.cs2 = f.cs2;
  p.cs3 = f.cs3;
  p.lossp = f.lossp;
  p.err = f.err;
  p.timeout_ns = f.timeout_ns;
  const int grid = p.tiles < num_sms ? p.tiles : num_sms;
  if (grid_out) *grid_out = grid;
  const int key = (s.H1 == 256 ? 4 : 0) + (s.H2 == 256 ? 2 : 0) + (s.CP == 32 ? 1 : 0);
  switch (key) {
    case 0: return launch_t<128, 128, 16>(m, p, grid, st);
    case 1: return launch_t<128, 128, 32>(m, p, grid, st);
    case 2: return launch_t<128, 256, 16>(m, p, grid, st);
    case 3: return launch_t<128, 256, 32>(m, p, grid, st);
    case 4: return launch_t<256, 128, 16>(m, p, grid, st);
    case 5: return launch_t<256, 128, 32>(m, p, grid, st);
    case 6: return launch_t<256, 256, 16>(m, p, grid, st);
    default: return launch_t<256, 256, 32>(m, p, grid, st);
  }
}

}  // namespace ppo
