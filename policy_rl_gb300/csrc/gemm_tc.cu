// gemm_tc.cu -- tcgen05 / TMA tensor-core GEMMs of the MLP actor-critic.
//
// The only dense contraction on the learner path is the MLP ("Teaching Mario
// to speedrun", sec. 6 "The policy and the value are one network"; its
// backward is sec. 6's loss.backward()).  Two persistent, warp-specialised
// kernels cover all of it:
//
//  * tc_gemm_kernel<BN, EPI>:  D[M,N] = A[M,K] * B[N,K]^T with both operands
//    K-major in global memory (activations [rows][features], weights
//    [out][in]).  Warp 0 issues TMA loads (128B swizzle) into an S-stage
//    shared-memory ring, warp 1 issues tcgen05.mma (128 x BN x 16 per
//    instruction) into a double-buffered TMEM accumulator, warps 2-5 drain
//    TMEM with tcgen05.ld and run the fused epilogue while the next tile's
//    MMAs proceed:
//      EPI_BIAS_ACT  h = act(acc + b)                      (forward layers)
//      EPI_DACT      dpre = acc * act'(h), column sums     (backward data)
//      EPI_LOSS      z = acc + b3 -> per-row PPO loss, dz  (head + loss)
//  * tc_wgrad_kernel: weight gradients dW = dPre^T X with K = minibatch rows.
//    Both operands are read MN-major straight from the row-major activation
//    buffers; K is split across CTAs and every split writes its own fp32
//    partial tile.  In the learner step the launch is cooperative and the
//    kernel assembles the gradient itself: the CTAs of an output tile meet at
//    a per-tile counter and each sums a slice of the tile's rows over the
//    splits in split order (deterministic, no float atomics), then runs a
//    share of the bias / log-std / statistic sums and writes its part of the
//    squared gradient norm.
//
// Every wait on an mbarrier is bounded (globaltimer); on expiry the kernel
// latches kDevTimeout, stops issuing work, drains what it has in flight and
// releases its TMEM before returning.
#include <cudaTypedefs.h>

#include <cmath>

#include "common.cuh"
#include "gemm.h"
#include "reduce.cuh"
#include "tc_ptx.cuh"
#include "tc_tile.cuh"

namespace ppo {

namespace {

using namespace ptx;
using namespace tc;

constexpr int kThreads = 192;

// minibatch rows from which the single-k-tile backward-data kernel is used: it
// trades latency for bandwidth, which short minibatches cannot afford
constexpr int64_t kTallRows = 65536;

// the bias of a forward product launched without one
__device__ __align__(16) float g_zero_bias[kColsumCap];

// Epilogue warps: 16 for the element-wise epilogues of 256-column tiles (four
// per TMEM lane quarter, each taking 64 of the tile's columns; measured faster
// than 8), 8 otherwise (two per lane quarter).  The per-row loss epilogue runs
// two groups of four warps on alternate tiles, one accumulator each (a third
// group would cap the registers at 128 per thread and spill: measured slower).
template <int BN, int EPI>
__host__ __device__ constexpr int epi_warps() { return BN >= 256 && EPI == EPI_BIAS_ACT ? 16 : 8; }
// TMEM accumulators: one per loss group, otherwise a double buffer
template <int BN, int EPI>
__host__ __device__ constexpr int n_acc() { return EPI == EPI_LOSS ? epi_warps<BN, EPI>() / 4 : 2; }
template <int BN, int EPI>
__host__ __device__ constexpr int gemm_threads() { return 2 * kWarp + kWarp * epi_warps<BN, EPI>(); }

template <int EPI>
__host__ __device__ constexpr bool is_dact() { return EPI == EPI_DACT || EPI == EPI_DACT_K1; }

template <int BN, int EPI>
struct Cfg {
  // backward-data kernels keep NAUX TMA-loaded activation tiles (aux), which
  // also stage their output (four when the product has one k-tile, so that
  // the loads run several tiles ahead of the epilogue); forward kernels stage
  // their output per warp
  static constexpr int AUX_SLOT = is_dact<EPI>() ? BM * BN * 2 : 0;
  // 256-column backward data: one activation tile, each epilogue warp
  // reloading its own rows of it for its next tile as soon as its stores have
  // read them (the operand ring takes the rest of the shared memory)
  static constexpr bool WARP_AUX = EPI == EPI_DACT && BN >= 256;
  static constexpr int NAUX = EPI == EPI_DACT_K1 ? 5 : (WARP_AUX ? 1 : 2);
  // per-warp output staging of the forward kernels: one 32-row x 32-column
  // bf16 chunk (2 KB, 64-byte swizzle), stored by TMA before the next chunk
  // is written, so that the ring gets the shared memory: 4 stages of 48 KB
  // at BN = 256
  static constexpr int STG_WARP = EPI == EPI_BIAS_ACT ? 2048 : 0;
  static constexpr int S = EPI == EPI_DACT ? (BN >= 256 ? 3 : 5)
                         : EPI == EPI_DACT_K1 ? 2
                         : EPI == EPI_BIAS_ACT ? (BN >= 256 ? 4 : 6)
                                               : 10;   // loss: H2 rows stream through 10 stages
  static constexpr int A_BYTES = BM * BK * 2;
  static constexpr int B_BYTES = BN * BK * 2;
  static constexpr int STAGE = A_BYTES + B_BYTES;
  static constexpr int ACC_COLS = n_acc<BN, EPI>() * BN;
  static constexpr int TMEM_COLS = ACC_COLS <= 32 ? 32 : (ACC_COLS <= 64 ? 64 : (ACC_COLS <= 128 ? 128 : (ACC_COLS <= 256 ? 256 : 512)));
  // barriers, TMEM slot, flags (<= 244 bytes for S <= 8)
  static constexpr int CTRL = EPI == EPI_LOSS ? 512 : 256;
  // column sums, loss partials (one row per group and lane quarter) and the
  // staged bias of the loss kernel (the forward kernels read their bias
  // through the read-only cache; the backward-data kernels keep their column
  // sums in registers)
  static constexpr size_t EXTRA =
      EPI == EPI_LOSS ? 4 * kColsumCap * 4 + 12 * kLossPartials * 4 + kColsumCap * 4 : 0;
  static constexpr size_t SMEM = 1024 + (size_t)S * STAGE + NAUX * (size_t)AUX_SLOT +
                                 epi_warps<BN, EPI>() * (size_t)STG_WARP + CTRL + EXTRA;
  static_assert(SMEM <= 232448, "shared memory per CTA");
};



// The loss epilogue's tile loop: groups of four warps (lane quarter q =
// warp % 4) take rotating tiles, i.e. the tiles of accumulator grp; column
// sums of group grp sit 64 floats after those of group grp - 1 in each
// quarter's slot.  The row inputs are loaded before the wait for the
// accumulator.  Inlined once with run-time head masks and once with the
// compile-time masks of the common layout.
template <int BN, int NA>
__device__ __forceinline__ void loss_epilogue(const TcParams& p, const HeadMasks hm, const Ctrl& cb,
                                              const Guard& g, uint32_t tmem, int total, float* cs,
                                              float* lp, const float* bias_s, int warp, int lane) {
  const int q = warp & 3;
  const int grp = (warp - 2) / 4;
  uint32_t i = 0;
  for (int tile = blockIdx.x + grp * gridDim.x; tile < total; tile += NA * gridDim.x, ++i) {
    const int tm = tile / p.tiles_n;
    const int row = tm * BM + q * 32 + lane;
    RowIn in;
    load_row_in(in, row, row < p.M, p.shape, p.rows);
    if (!wait_bar(cb.tfull(grp), i & 1, g)) break;
    tc_fence_after();
    const uint32_t taddr = tmem + (uint32_t)(grp * BN) + ((uint32_t)(q * 32) << 16);
    epi_loss_tile<BN>(taddr, row, row < p.M, p.shape, hm, p.lc, p.inv_mb, in, p.logstd, bias_s,
                      p.dz, p.lddz, cs + q * kColsumCap + grp * 64,
                      lp + (grp * 4 + q) * kLossPartials, lane);
    tc_fence_before();
    mbar_arrive(cb.tempty(grp));
  }
}

// ---------------------------------------------------------------------------
template <int BN, int EPI>
__global__ void __launch_bounds__(gemm_threads<BN, EPI>(), 1)
tc_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
               const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmO,
               const TcParams p) {
  using C = Cfg<BN, EPI>;
  constexpr int S = C::S;
  constexpr int EW = epi_warps<BN, EPI>();
  constexpr int NT = gemm_threads<BN, EPI>();
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);
  uint8_t* auxs = gbase + (size_t)S * C::STAGE;          // [2][BM x BN] (DACT only)
  uint8_t* stgs = auxs + C::NAUX * (size_t)C::AUX_SLOT;  // [EW warps][STG_WARP] (BIAS_ACT only)
  uint8_t* ctrl = stgs + EW * (size_t)C::STG_WARP;
  Ctrl cb{reinterpret_cast<uint64_t*>(ctrl), S};
  // aux full[NAUX], empty[NAUX]; with WARP_AUX one barrier per epilogue warp
  constexpr int XB = C::WARP_AUX ? EW : 2 * C::NAUX;
  uint64_t* xbar = reinterpret_cast<uint64_t*>(ctrl) + Ctrl::count(S);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(xbar + XB);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tslot + 1);
  volatile uint32_t* cnt = reinterpret_cast<volatile uint32_t*>(tslot + 2);  // issued, consumed, aux issued
  float* cs = reinterpret_cast<float*>(ctrl + C::CTRL);                      // [4][kColsumCap]
  float* lp = cs + 4 * kColsumCap;                                           // [12][kLossPartials]
  float* bias_s = lp + 12 * kLossPartials;                                   // [kColsumCap]

  const int warp = threadIdx.x / kWarp, lane = threadIdx.x % kWarp;
  auto sA = [&](int s) { return base + (uint32_t)(s * C::STAGE); };
  // backward-data column sums of this epilogue warp (see epi_dact_smem_tile_r)
  constexpr int NTC = kColsumCap / BN;
  constexpr int PART = BN / (EW / 4);   // columns of an epilogue warp
  constexpr int CPW = PART / 32;
  static_assert(EPI == EPI_LOSS || PART % 64 == 0, "whole 64-column blocks per epilogue warp");
  float csr[is_dact<EPI>() ? NTC * CPW : 1];
#pragma unroll
  for (int j = 0; j < (is_dact<EPI>() ? NTC * CPW : 1); ++j) csr[j] = 0.f;
  auto sB = [&](int s) { return base + (uint32_t)(s * C::STAGE + C::A_BYTES); };

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(cb.full(s), 1);
      mbar_init(cb.empty(s), 1);
    }
    for (int a = 0; a < n_acc<BN, EPI>(); ++a) {
      mbar_init(cb.tfull(a), 1);
      mbar_init(cb.tempty(a), (EPI == EPI_LOSS ? 4 : EW) * kWarp);
    }
    mbar_init(cb.drain(), 1);
    if constexpr (C::WARP_AUX) {
      for (int w = 0; w < EW; ++w) mbar_init(smem_u32(&xbar[w]), 1);
    } else {
      for (int a = 0; a < C::NAUX; ++a) {
        mbar_init(smem_u32(&xbar[a]), 1);
        mbar_init(smem_u32(&xbar[C::NAUX + a]), EW * kWarp);
      }
    }
    *abort_flag = 0;
    cnt[0] = 0;
    cnt[1] = 0;
    cnt[2] = 0;
    fence_mbar_init();
  }
  if (EPI == EPI_LOSS)
    for (int i = threadIdx.x; i < 4 * kColsumCap + 12 * kLossPartials; i += NT) cs[i] = 0.f;
  if (warp == 1) tmem_alloc(smem_u32(tslot), C::TMEM_COLS);
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tmA);
    prefetch_tmap(&tmB);
    if (is_dact<EPI>()) prefetch_tmap(&tmX);
    if (EPI != EPI_LOSS) prefetch_tmap(&tmO);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tslot;
  const Guard g{abort_flag, p.err, p.timeout_ns};
  const int total = p.tiles_m * p.tiles_n;
  pdl_wait();      // inputs are written by the previous kernel of the chain
  pdl_trigger();
  if (EPI == EPI_LOSS) {  // the bias, read by every epilogue thread, staged once
    for (int i = threadIdx.x; i < p.N; i += NT) bias_s[i] = p.bias ? p.bias[i] : 0.f;
    __syncthreads();      // reached by every thread of the block (before the role split)
  }

  if (warp == 0) {
    if (lane == 0) {
      uint32_t it = 0;
      bool ok = true;
      uint32_t lt = 0;
      for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x, ++lt) {
        const int tm = tile / p.tiles_n, tn = tile % p.tiles_n;
        // the streamed operands of this CTA's next tile (activation rows, and
        // the act' tile) into L2 one tile ahead, so that the ring's loads wait
        // for L2 rather than DRAM
        if (tile + (int)gridDim.x < total) {
          const int nt = tile + (int)gridDim.x;
          const int tmn = nt / p.tiles_n;
          // A's rows are contiguous in memory: one linear prefetch of them (the
          // k-tile boxes would visit the region in 128-byte column strips)
          const int rows = min(BM, p.M - tmn * BM);
          if (rows > 0)
            bulk_prefetch_l2(p.a_rows + (int64_t)tmn * BM * p.lda,
                             (uint32_t)rows * (uint32_t)p.lda * 2u);
          if constexpr (is_dact<EPI>())   // (the per-warp map's boxes are 32 rows high)
            for (int j = 0; j < BN / 64; ++j)
              for (int r0 = 0; r0 < BM; r0 += C::WARP_AUX ? 32 : BM)
                tma_prefetch_2d(&tmX, (nt % p.tiles_n) * BN + 64 * j, tmn * BM + r0);
        }
        if constexpr (is_dact<EPI>() && !C::WARP_AUX) {
          // this tile's activation operand, one slot of NAUX, ahead of its k-loop
          const int xs = lt % C::NAUX;
          const uint32_t xu = lt / C::NAUX;
          if (!wait_bar(smem_u32(&xbar[C::NAUX + xs]), (xu & 1) ^ 1, g)) { ok = false; break; }
          mbar_arrive_expect_tx(smem_u32(&xbar[xs]), C::AUX_SLOT);
          for (int j = 0; j < BN / 64; ++j)
            tma_load_2d(smem_u32(auxs) + (uint32_t)(xs * C::AUX_SLOT + j * 16384), &tmX,
                        tn * BN + 64 * j, tm * BM, smem_u32(&xbar[xs]));
          cnt[2] = lt + 1;
        }
        for (int kt = 0; kt < p.k_tiles; ++kt) {
          const int s = it % S;
          const uint32_t r = it / S;
          if (!wait_bar(cb.empty(s), (r & 1) ^ 1, g)) { ok = false; break; }
          mbar_arrive_expect_tx(cb.full(s), C::STAGE);
          tma_load_2d(sA(s), &tmA, kt * BK, tm * BM, cb.full(s));
          tma_load_2d(sB(s), &tmB, kt * BK, tn * BN, cb.full(s));
          ++it;
          cnt[0] = it;
        }
      }
      // tail: wait until the MMA warp has released every stage, so that no
      // tcgen05.commit arrival is still pending when the CTA exits
      if (ok)
        for (int j = 0; j < S; ++j, ++it) {
          const int s = it % S;
          const uint32_t r = it / S;
          if (!wait_bar(cb.empty(s), (r & 1) ^ 1, g)) break;
        }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16(BM, BN, false, false);
      uint32_t it = 0, tc = 0;
      bool ok = true;
      for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x) {
        const int acc = (int)(tc % n_acc<BN, EPI>());
        const uint32_t use = tc / n_acc<BN, EPI>();
        if (!wait_bar(cb.tempty(acc), (use & 1) ^ 1, g)) break;
        tc_fence_after();
        const uint32_t d = tmem + (uint32_t)(acc * BN);
        for (int kt = 0; kt < p.k_tiles; ++kt) {
          const int s = it % S;
          const uint32_t r = it / S;
          if (!wait_bar(cb.full(s), r & 1, g)) { ok = false; break; }
          tc_fence_after();
          const int nk = (kt == p.k_tiles - 1) ? p.last_k_steps : BK / 16;
          for (int kk = 0; kk < nk; ++kk) {
            const uint64_t da = sdesc_sw128(sA(s) + kk * 32, 16, 1024);
            const uint64_t db = sdesc_sw128(sB(s) + kk * 32, 16, 1024);
            tc_mma_bf16(d, da, db, idesc, (kt | kk) != 0 ? 1u : 0u);
          }
          tc_commit(cb.empty(s));
          ++it;
          cnt[1] = it;
        }
        if (!ok) break;
        tc_commit(cb.tfull(acc));
        ++tc;
      }
    }
  } else if constexpr (EPI == EPI_LOSS) {
    // groups of four warps (lane quarter q = warp % 4) take rotating tiles,
    // i.e. the tiles of accumulator grp; column sums of group grp sit 64
    // floats after those of group grp - 1 in each quarter's slot.  The row
    // inputs are loaded before the wait for the accumulator.
    if (p.layout9222)
      loss_epilogue<BN, n_acc<BN, EPI>()>(p, kMasks9222, cb, g, tmem, total, cs, lp, bias_s, warp,
                                         lane);
    else
      loss_epilogue<BN, n_acc<BN, EPI>()>(p, head_masks(p.shape), cb, g, tmem, total, cs, lp,
                                         bias_s, warp, lane);
  } else {
    // epilogue warps 2..2+EW: TMEM lane quarter q = warp % 4, column part h
    const int q = warp & 3;
    const int h = (warp - 2) / 4;
    uint32_t tc = 0;
    // WARP_AUX: this warp's rows of the activation tile, [PART/64 blocks of 32
    // rows x 64 columns] at auxs + block * 16384 + q * 4096, loaded by lane 0
    const uint32_t wb = smem_u32(&xbar[C::WARP_AUX ? warp - 2 : 0]);
    uint32_t xi = 0;   // WARP_AUX loads issued by this warp
    auto load_part = [&](int t) {
      const int tm = t / p.tiles_n, tn = t % p.tiles_n;
      mbar_arrive_expect_tx(wb, (uint32_t)(PART / 64) * 4096u);
#pragma unroll
      for (int b = 0; b < PART / 64; ++b) {
        const int cb64 = (h * PART) / 64 + b;
        tma_load_2d(smem_u32(auxs + cb64 * 16384 + q * 4096), &tmX, tn * BN + cb64 * 64,
                    tm * BM + q * 32, wb);
      }
      ++xi;
    };
    if constexpr (C::WARP_AUX)
      if (lane == 0 && (int)blockIdx.x < total) load_part(blockIdx.x);
    for (int tile = blockIdx.x; tile < total; tile += gridDim.x) {
      const int acc = tc & 1;
      const uint32_t use = tc >> 1;
      if (!wait_bar(cb.tfull(acc), use & 1, g)) break;
      tc_fence_after();
      const int tm = tile / p.tiles_n, tn = tile % p.tiles_n;
      const int row = tm * BM + q * 32 + lane;
      const bool rok = row < p.M;
      const uint32_t taddr = tmem + (uint32_t)(acc * BN) + ((uint32_t)(q * 32) << 16);
      if constexpr (C::WARP_AUX) {
        if (!wait_bar(wb, tc & 1, g)) break;
        epi_dact_smem_tile_r<BN, EW, NTC>(taddr, q * 32 + lane, rok, tn, h, p.act, auxs, csr,
                                          lane, p.alpha, p.beta);
        tc_fence_before();
        mbar_arrive(cb.tempty(acc));
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          if (tm * BM + q * 32 < p.M) {   // rows of the box exist
#pragma unroll
            for (int b = 0; b < PART / 64; ++b) {
              const int cb64 = (h * PART) / 64 + b;
              tma_store_2d(&tmO, smem_u32(auxs + cb64 * 16384 + q * 4096), tn * BN + cb64 * 64,
                           tm * BM + q * 32);
            }
            bulk_commit();
          }
          bulk_wait_read0();   // the rows are reloaded for the next tile
          if (tile + (int)gridDim.x < total) load_part(tile + gridDim.x);
        }
        __syncwarp();
      } else if constexpr (is_dact<EPI>()) {
        // tile tc uses aux slot tc % NAUX (same tile order as the producer); the
        // result overwrites the warp's rows of the slot and leaves by TMA
        const int xs = tc % C::NAUX;
        if (!wait_bar(smem_u32(&xbar[xs]), (tc / C::NAUX) & 1, g)) break;
        uint8_t* slot = auxs + xs * C::AUX_SLOT;
        epi_dact_smem_tile_r<BN, EW, NTC>(taddr, q * 32 + lane, rok, tn, h, p.act, slot, csr, lane,
                                          p.alpha, p.beta);
        tc_fence_before();
        mbar_arrive(cb.tempty(acc));
        fence_proxy_async_smem();
        __syncwarp();
        // With two slots the slot is released as soon as its stores have read
        // it; with more, a tile releases the previous tile's slot, so that the
        // warp does not wait for its own stores
        constexpr bool kDefer = C::NAUX >= 3;
        if (lane == 0) {
          if (tm * BM + q * 32 < p.M) {   // rows of the box exist
#pragma unroll
            for (int b = 0; b < PART / 64; ++b) {
              const int cb64 = (h * PART) / 64 + b;
              tma_store_2d(&tmO, smem_u32(slot + cb64 * 16384 + q * 4096), tn * BN + cb64 * 64,
                           tm * BM + q * 32);
            }
            bulk_commit();
            if constexpr (kDefer) bulk_wait_read1();
            else bulk_wait_read0();
          } else {
            bulk_wait_read0();
          }
        }
        __syncwarp();
        if constexpr (kDefer) {
          if (tc > 0) mbar_arrive(smem_u32(&xbar[C::NAUX + (tc - 1) % C::NAUX]));
        } else {
          mbar_arrive(smem_u32(&xbar[C::NAUX + xs]));
        }
      } else {
        // 32-column chunks through the warp's 2 KB staging buffer: each waits
        // until the previous chunk's store has read the buffer
        uint8_t* stg = stgs + (warp - 2) * C::STG_WARP;
        const float* bias = (p.bias ? p.bias : g_zero_bias) + tn * BN;
        const bool rows_exist = tm * BM + q * 32 < p.M;
        tmem_chunks<PART / 32>(taddr, h * PART, [&](const uint32_t (&r)[32], int c0) {
          float v[32];
          act_bias_chunk_ldg(r, bias + c0, p.act, v);
          if (lane == 0) bulk_wait_read0();
          __syncwarp();
          put_row_chunks_sw64(stg + lane * 64, lane, v);
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0 && rows_exist) {
            tma_store_2d(&tmO, smem_u32(stg), tn * BN + c0, tm * BM + q * 32);
            bulk_commit();
          }
        });
        tc_fence_before();
        mbar_arrive(cb.tempty(acc));
      }
      ++tc;
    }
    if constexpr (C::WARP_AUX)   // a load issued for a tile this warp did not reach
      if (lane == 0 && xi > tc) drain_wait(wb, (xi - 1) & 1, p.timeout_ns);
    if (lane == 0) bulk_wait0();   // this warp's stores are complete before the CTA exits
  }

  __syncthreads();
  if (*abort_flag) {
    // drain: TMA loads issued but never consumed, and outstanding MMAs
    if (threadIdx.x == 0) {
      const uint32_t issued = cnt[0], consumed = cnt[1];
      for (uint32_t it = consumed; it < issued; ++it)
        drain_wait(cb.full(it % S), (it / S) & 1, p.timeout_ns);
      const uint32_t xi = cnt[2];   // the last NAUX activation-tile loads
      for (uint32_t l = xi >= (uint32_t)C::NAUX ? xi - C::NAUX : 0; l < xi; ++l)
        drain_wait(smem_u32(&xbar[l % C::NAUX]), (l / C::NAUX) & 1, p.timeout_ns);
    }
    if (warp == 1 && lane == 0) {
      tc_commit(cb.drain());
      drain_wait(cb.drain(), 0, p.timeout_ns);
    }
    __syncthreads();
  }
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
  if constexpr (is_dact<EPI>()) {
    // every stage has been released: the first ones take the per-quarter
    // column sums [4][kColsumCap], summed in quarter order as in the loss
    static_assert((size_t)C::S * C::STAGE >= 4 * kColsumCap * 4, "column-sum scratch");
    float* scr = reinterpret_cast<float*>(gbase);
    if (warp >= 2) {
      const int q = warp & 3, h = (warp - 2) / 4;
#pragma unroll
      for (int t = 0; t < NTC; ++t)
#pragma unroll
        for (int k2 = 0; k2 < CPW; ++k2)
          scr[q * kColsumCap + t * BN + h * PART + k2 * 32 + lane] = csr[CPW * t + k2];
    }
    __syncthreads();
    if (warp >= 2) {
      const int et = threadIdx.x - 2 * kWarp;
      for (int c = et; c < p.epi_n; c += EW * kWarp)
        p.colsum_part[(int64_t)blockIdx.x * p.epi_n + c] =
            ((scr[c] + scr[kColsumCap + c]) + scr[2 * kColsumCap + c]) + scr[3 * kColsumCap + c];
    }
  }
  if constexpr (EPI == EPI_LOSS) {
    if (warp >= 2) {
      const int et = threadIdx.x - 2 * kWarp;
      auto quad = [&](const float* b, int c) {
        return ((b[c] + b[kColsumCap + c]) + b[2 * kColsumCap + c]) + b[3 * kColsumCap + c];
      };
      for (int c = et; c < p.epi_n; c += EW * kWarp)
        p.colsum_part[(int64_t)blockIdx.x * p.epi_n + c] =
            (quad(cs, c) + quad(cs + 64, c)) + quad(cs + 128, c);
      if (et < kLossPartials) {
        float t = 0.f;
        for (int k = 0; k < 12; ++k) t += lp[k * kLossPartials + et];
        p.loss_part[(int64_t)blockIdx.x * kLossPartials + et] = t;
      }
    }
  }
}

// ---------------------------------------------------------------------------
// Weight-gradient kernel: P[M][N] = sum_rows U[row][m] * V[row][n] over a
// K-split of the minibatch rows; both operands MN-major in shared memory.
// Output tiles are WBM = 256 rows x bn <= 256 columns: two 128-row MMAs share
// each B tile, one accumulator pair [rows 0..127 | 128..255] in TMEM, 3
// stages of 64 KB -- per k-tile an SM takes in 64 KB for 256 x 256 x 64
// products (measured against 128-row tiles with a double-buffered
// accumulator: 212 vs 238 us per large-batch minibatch, 116 vs 172 us per
// DDNet-like one, 32 vs 30 us per Mario-like one).  A tile's lower half may
// lie beyond M (M a multiple of 128): its A blocks are zero-filled and its
// MMAs and stores skipped.
constexpr int WBM = 256;
constexpr int WBN = 256;
constexpr int WS = 3;
constexpr int W_STAGE = (WBM + WBN) * BK * 2;   // A: 4 blocks of 64 features x 64 rows, B: up to 4
constexpr int W_STG = 2 * 4096;   // per epilogue warp: two 32 x 32 fp32 store boxes
constexpr size_t W_SMEM = 1024 + (size_t)WS * W_STAGE + 4 * W_STG + 512;
static_assert(W_SMEM + 64 <= 232448, "shared memory per CTA");
constexpr int W_TMEM_COLS = 512;

__device__ __forceinline__ void decode_unit(const WParams& p, int u, int& reg, int& tm, int& tn,
                                            int& kt0, int& kt1, int& split) {
  reg = 0;
  while (reg + 1 < p.nreg && u >= p.r[reg + 1].unit_begin) ++reg;
  const WRegion& R = p.r[reg];
  const int local = u - R.unit_begin;
  const int per = R.tiles_m * R.tiles_n;
  split = local / per;
  const int rem = local % per;
  tm = rem / R.tiles_n;
  tn = rem % R.tiles_n;
  kt0 = split * R.kt_per_split;
  kt1 = min(R.k_tiles, kt0 + R.kt_per_split);
}

// Sum of the n <= kWgMaxSplits split partials q[0], q[st], ... (four
// consecutive columns each) in split order; the loads of 16 splits are issued
// before their adds.  L2 loads: the partials were written by other CTAs of
// this launch.
constexpr int kWgMaxSplits = 64;
__device__ __forceinline__ float4 split_sum4_cg(const float* q, int64_t st, int n) {
  float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int s0 = 0; s0 < n; s0 += 16) {
    float4 x[16];
#pragma unroll
    for (int j = 0; j < 16; ++j)
      x[j] = s0 + j < n ? __ldcg(reinterpret_cast<const float4*>(q + (s0 + j) * st))
                        : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int j = 0; j < 16; ++j)
      if (s0 + j < n) {
        v.x += x[j].x;
        v.y += x[j].y;
        v.z += x[j].z;
        v.w += x[j].w;
      }
  }
  return v;
}

// In-kernel assembly of the weight gradient (cooperative launch: every CTA
// is resident).  Each CTA first arrives on the counter of every output tile
// it stored a split partial of; then, per unit, it waits (bounded) until all
// splits of the tile have arrived and sums its share of the tile's rows --
// split s of S takes rows [256 s / S, 256 (s + 1) / S) below M -- over the splits in
// split order, writing the final gradient entries and the sum of their
// squares (per CTA, fixed order) for the clip norm.  The last CTA of a tile to
// finish clears its counters for the next launch.  On a timeout (or an
// earlier abort of this CTA) it latches the error and writes no gradient.
__device__ __noinline__ void wgrad_fixup(const WParams& p, bool aborted) {
  __shared__ int s_ok;
  __shared__ double s_sq[kThreads / kWarp];
  double sq = 0.0;
  if (!aborted) {
    if (threadIdx.x == 0) {
      __threadfence();
      for (int u = blockIdx.x; u < p.total_units; u += gridDim.x) {
        int reg, tm, tn, kt0, kt1, split;
        decode_unit(p, u, reg, tm, tn, kt0, kt1, split);
        atomicAdd(p.tile_ctr + p.tile_begin[reg] + tm * p.r[reg].tiles_n + tn, 1u);
      }
    }
    // the bias / log-std / statistic sums (their partial rows come from the
    // kernels before this one), while the tiles' other CTAs finish
    constexpr int kFixWarps = kThreads / kWarp;
    for (int e = blockIdx.x * kFixWarps + (int)(threadIdx.x / kWarp); e < p.nvt;
         e += gridDim.x * kFixWarps)
      sq += reduce_vector_task(p.ra, e);
    for (int u = blockIdx.x; u < p.total_units; u += gridDim.x) {
      int reg, tm, tn, kt0, kt1, split;
      decode_unit(p, u, reg, tm, tn, kt0, kt1, split);
      const WRegion& R = p.r[reg];
      const int t = p.tile_begin[reg] + tm * R.tiles_n + tn;
      if (threadIdx.x == 0) {
        int ok = 1;
        if (ld_acquire_gpu(p.tile_ctr + t) < (unsigned)R.splits) {
          const uint64_t t0 = ptx::globaltimer();
          while (ld_acquire_gpu(p.tile_ctr + t) < (unsigned)R.splits) {
            if (ptx::globaltimer() - t0 > p.tile_wait_ns) {
              atomicOr(p.err, kDevTimeout);
              ok = 0;
              break;
            }
          }
        }
        s_ok = ok;
      }
      __syncthreads();
      if (!s_ok) break;
      const WFinal& F = p.f[reg];
      const int r0 = WBM * split / R.splits, r1 = WBM * (split + 1) / R.splits;
      const int q4 = R.bn / 4;   // four columns per work item
      const int n_it = (r1 - r0) * q4;
      const int64_t pst = (int64_t)R.M * R.N;
      for (int e = threadIdx.x; e < n_it; e += kThreads) {
        const int m = tm * WBM + r0 + e / q4, n = tn * R.bn + 4 * (e % q4);
        if (m >= R.M) break;   // (e grows with m)
        const float4 v = split_sum4_cg(R.part + (int64_t)m * R.N + n, pst, R.splits);
        const float vv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int j = 0; j < 4; ++j)
          if (m < F.rows && n + j < F.cols) {
            F.dst[m * F.ldm + (n + j) * F.ldn] = vv[j];
            sq += (double)(vv[j] * vv[j]);
          }
      }
      __syncthreads();
      if (threadIdx.x == 0 &&
          atomicAdd(p.tile_ctr + kWgradMaxTiles + t, 1u) == (unsigned)R.splits - 1) {
        p.tile_ctr[t] = 0u;   // every CTA of the tile has passed its wait
        p.tile_ctr[kWgradMaxTiles + t] = 0u;
      }
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) sq += __shfl_xor_sync(0xffffffffu, sq, o);
  if (threadIdx.x % kWarp == 0) s_sq[threadIdx.x / kWarp] = sq;
  __syncthreads();
  if (threadIdx.x == 0) {
    double tot = 0.0;
    for (int w = 0; w < kThreads / kWarp; ++w) tot += s_sq[w];
    p.sq_part[blockIdx.x] = tot;
  }
}

__global__ void __launch_bounds__(kThreads, 1)
tc_wgrad_kernel(const __grid_constant__ CUtensorMap tmU0, const __grid_constant__ CUtensorMap tmV0,
                const __grid_constant__ CUtensorMap tmU1, const __grid_constant__ CUtensorMap tmV1,
                const __grid_constant__ CUtensorMap tmU2, const __grid_constant__ CUtensorMap tmV2,
                const __grid_constant__ CUtensorMap tmP0, const __grid_constant__ CUtensorMap tmP1,
                const __grid_constant__ CUtensorMap tmP2, const WParams p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);
  uint8_t* wstg = gbase + (size_t)WS * W_STAGE;   // [4 warps][2][32 rows x 128 B]
  uint8_t* ctrl = wstg + 4 * W_STG;
  Ctrl cb{reinterpret_cast<uint64_t*>(ctrl), WS};
  uint32_t* tslot = reinterpret_cast<uint32_t*>(ctrl + 8 * Ctrl::count(WS));
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tslot + 1);
  volatile uint32_t* cnt = reinterpret_cast<volatile uint32_t*>(tslot + 2);
  const int warp = threadIdx.x / kWarp, lane = threadIdx.x % kWarp;
  auto sA = [&](int s) { return base + (uint32_t)(s * W_STAGE); };
  auto sB = [&](int s) { return base + (uint32_t)(s * W_STAGE + WBM * BK * 2); };

  if (threadIdx.x == 0) {
    for (int s = 0; s < WS; ++s) {
      mbar_init(cb.full(s), 1);
      mbar_init(cb.empty(s), 1);
    }
    mbar_init(cb.tfull(0), 1);
    mbar_init(cb.tempty(0), 128);
    mbar_init(cb.drain(), 1);
    *abort_flag = 0;
    cnt[0] = 0;
    cnt[1] = 0;
    fence_mbar_init();
  }
  if (warp == 1) tmem_alloc(smem_u32(tslot), W_TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tslot;
  const Guard g{abort_flag, p.err, p.timeout_ns};
  pdl_wait();
  pdl_trigger();

  if (warp == 0) {
    if (lane == 0) {
      uint32_t it = 0;
      int ws_s = 0;          // stage of `it` (it % WS) and its phase parity ((it / WS) & 1)
      uint32_t ws_ph = 0;
      bool ok = true;
      for (int u = blockIdx.x; u < p.total_units && ok; u += gridDim.x) {
        int reg, tm, tn, kt0, kt1, split;
        decode_unit(p, u, reg, tm, tn, kt0, kt1, split);
        const int bn = p.r[reg].bn;
        const CUtensorMap* tu = reg == 0 ? &tmU0 : (reg == 1 ? &tmU1 : &tmU2);
        const CUtensorMap* tv = reg == 0 ? &tmV0 : (reg == 1 ? &tmV1 : &tmV2);
        const uint32_t bytes = (uint32_t)(WBM + bn) * BK * 2;
        for (int kt = kt0; kt < kt1; ++kt) {
          const int s = ws_s;
          const uint32_t r = ws_ph;
          if (!wait_bar(cb.empty(s), (r & 1) ^ 1, g)) { ok = false; break; }
          mbar_arrive_expect_tx(cb.full(s), bytes);
          // one 3-D box per operand: 64 rows x {4, bn/64} blocks of 64 features
          // (blocks beyond M read as zeros)
          tma_load_3d(sA(s), tu, 0, kt * BK, tm * (WBM / 64), cb.full(s));
          tma_load_3d(sB(s), tv, 0, kt * BK, tn * (bn / 64), cb.full(s));
          ++it;
          cnt[0] = it;
          if (++ws_s == WS) { ws_s = 0; ws_ph ^= 1u; }
        }
      }
      if (ok)
        for (int j = 0; j < WS; ++j, ++it) {
          if (!wait_bar(cb.empty(ws_s), ws_ph ^ 1u, g)) break;
          if (++ws_s == WS) { ws_s = 0; ws_ph ^= 1u; }
        }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      uint32_t it = 0, tc = 0;
      int ws_s = 0;          // as in the producer
      uint32_t ws_ph = 0;
      bool ok = true;
      for (int u = blockIdx.x; u < p.total_units && ok; u += gridDim.x) {
        int reg, tm, tn, kt0, kt1, split;
        decode_unit(p, u, reg, tm, tn, kt0, kt1, split);
        const int bn = p.r[reg].bn;
        const uint32_t idesc = idesc_bf16(BM, bn, true, true);
        const bool lower = tm * WBM + BM < p.r[reg].M;   // the tile's rows 128..255 exist
        // one unit at a time: the accumulators [rows 0..127 | rows 128..255]
        // take 2 bn <= 512 TMEM columns
        const uint32_t d = tmem;
        if (!wait_bar(cb.tempty(0), (tc & 1) ^ 1, g)) break;
        tc_fence_after();
        for (int kt = kt0; kt < kt1; ++kt) {
          const int s = ws_s;
          if (!wait_bar(cb.full(s), ws_ph, g)) { ok = false; break; }
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk) {
            const uint32_t accf = (kt != kt0 || kk != 0) ? 1u : 0u;
            const uint64_t db = sdesc_sw128(sB(s) + kk * 2048, p.mn_lbo, p.mn_sbo);
            tc_mma_bf16(d, sdesc_sw128(sA(s) + kk * 2048, p.mn_lbo, p.mn_sbo), db, idesc, accf);
            if (lower)   // A's features 128..255: two 64-feature blocks further on
              tc_mma_bf16(d + (uint32_t)bn,
                          sdesc_sw128(sA(s) + 2 * (64 * BK * 2) + kk * 2048, p.mn_lbo, p.mn_sbo),
                          db, idesc, accf);
          }
          tc_commit(cb.empty(s));
          ++it;
          cnt[1] = it;
          if (++ws_s == WS) { ws_s = 0; ws_ph ^= 1u; }
        }
        if (!ok) break;
        tc_commit(cb.tfull(0));
        ++tc;
      }
    }
  } else {
    const int q = warp & 3;
    uint32_t tc = 0, sc = 0;
    for (int u = blockIdx.x; u < p.total_units; u += gridDim.x) {
      int reg, tm, tn, kt0, kt1, split;
      decode_unit(p, u, reg, tm, tn, kt0, kt1, split);
      const WRegion& R = p.r[reg];
      if (!wait_bar(cb.tfull(0), tc & 1, g)) break;
      tc_fence_after();
      // fp32 partial tile -> this split's slice of the partial buffer, 32
      // columns at a time through two 32 x 32 staging boxes per warp (128-byte
      // swizzle: float4 c of row r at ((c ^ (r & 7)) * 16)) and TMA stores;
      // half hf = rows 128 hf .. 128 hf + 127 of the tile
      const CUtensorMap* tp = reg == 0 ? &tmP0 : (reg == 1 ? &tmP1 : &tmP2);
      uint8_t* mystg = wstg + (warp - 2) * W_STG;
      for (int hf = 0; hf < WBM / BM; ++hf) {
        if (tm * WBM + hf * BM >= R.M) break;
        const uint32_t taddr = tmem + (uint32_t)(hf * R.bn) + ((uint32_t)(q * 32) << 16);
#pragma unroll 1
        for (int c0 = 0; c0 < R.bn; c0 += 32, ++sc) {
          float v[32];
          tmem_ld32(taddr + (uint32_t)c0, v);
          uint8_t* buf = mystg + (sc & 1) * 4096;
          if (lane == 0) bulk_wait_read1();   // the store that used buf last has read it
          __syncwarp();
#pragma unroll
          for (int i = 0; i < 8; ++i)
            *reinterpret_cast<float4*>(buf + lane * 128 + ((i ^ (lane & 7)) << 4)) =
                make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            tma_store_3d(tp, smem_u32(buf), tn * R.bn + c0, tm * WBM + hf * BM + q * 32, split);
            bulk_commit();
          }
        }
      }
      tc_fence_before();
      mbar_arrive(cb.tempty(0));
      ++tc;
    }
    if (lane == 0) {
      bulk_wait0();   // this warp's stores are complete before the CTA exits
      if (p.fixup) {  // ... and visible to the other CTAs' loads of the tile
        fence_proxy_async_global();
        __threadfence();
      }
    }
  }
  __syncthreads();
  if (*abort_flag) {
    if (threadIdx.x == 0) {
      const uint32_t issued = cnt[0], consumed = cnt[1];
      for (uint32_t it = consumed; it < issued; ++it)
        drain_wait(cb.full(it % WS), (it / WS) & 1, p.timeout_ns);
    }
    if (warp == 1 && lane == 0) {
      tc_commit(cb.drain());
      drain_wait(cb.drain(), 0, p.timeout_ns);
    }
    __syncthreads();
  }
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, W_TMEM_COLS);
  }
  if (p.fixup) wgrad_fixup(p, *abort_flag != 0);
}

// ---------------------------------------------------------------------------
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

cudaError_t get_encode() {
  if (g_encode) return cudaSuccess;
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q;
  cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                                   cudaEnableDefault, &q);
  if (e != cudaSuccess) return e;
  if (q != cudaDriverEntryPointSuccess || fn == nullptr) return cudaErrorNotSupported;
  g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  return cudaSuccess;
}

// bf16 row-major [rows][cols] (row pitch ld elements), box = box_cols x box_rows
cudaError_t make_tmap(CUtensorMap* m, const void* base, int64_t cols, int64_t rows, int64_t ld,
                      int box_cols, int box_rows,
                      CUtensorMapSwizzle swz = CU_TENSOR_MAP_SWIZZLE_128B) {
  // a missing operand is an error here, never a tensor map over address 0
  if (base == nullptr || cols < 1 || rows < 1 || ld < 1) return cudaErrorInvalidValue;
  cudaError_t e = get_encode();
  if (e != cudaSuccess) return e;
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)ld * 2};
  cuuint32_t box[2] = {(cuuint32_t)box_cols, (cuuint32_t)box_rows};
  cuuint32_t es[2] = {1, 1};
  CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims,
                        strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// bf16 row-major [rows][ld] read as 64-feature blocks: x = feature within the
// block, y = row, z = block (of nblk); box = 64 x box_rows x box_blk.  The
// box lands in shared memory as box_blk consecutive [box_rows][64] atoms.
// fp32 split-K partials [splits][rows][cols] as 32-column x 32-row x 1-split boxes
cudaError_t make_tmap_partials(CUtensorMap* m, const float* base, int64_t cols, int64_t rows,
                               int64_t splits) {
  if (base == nullptr || cols < 1 || rows < 1 || splits < 1) return cudaErrorInvalidValue;
  cudaError_t e = get_encode();
  if (e != cudaSuccess) return e;
  cuuint64_t dims[3] = {(cuuint64_t)cols, (cuuint64_t)rows, (cuuint64_t)splits};
  cuuint64_t strides[2] = {(cuuint64_t)cols * 4, (cuuint64_t)(cols * rows * 4)};
  cuuint32_t box[3] = {32, 32, 1};
  cuuint32_t es[3] = {1, 1, 1};
  CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<float*>(base), dims,
                        strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

cudaError_t make_tmap_blocks(CUtensorMap* m, const void* base, int64_t rows, int64_t ld, int nblk,
                             int box_rows, int box_blk) {
  if (base == nullptr || rows < 1 || nblk < 1 || ld < 1) return cudaErrorInvalidValue;
  cudaError_t e = get_encode();
  if (e != cudaSuccess) return e;
  cuuint64_t dims[3] = {64, (cuuint64_t)rows, (cuuint64_t)nblk};
  cuuint64_t strides[2] = {(cuuint64_t)ld * 2, 128};
  cuuint32_t box[3] = {64, (cuuint32_t)box_rows, (cuuint32_t)box_blk};
  cuuint32_t es[3] = {1, 1, 1};
  CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims,
                        strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

template <int BN, int EPI>
cudaError_t launch_tc(const GemmOperands& g, TcParams p, int num_sms, cudaStream_t st,
                      int* grid_out) {
  CUtensorMap ta, tb, tx, to;
  cudaError_t e = make_tmap(&ta, g.A, g.lda, g.M, g.lda, BK, BM);
  if (e != cudaSuccess) return e;
  e = make_tmap(&tb, g.B, g.ldb, g.N, g.ldb, BK, BN);
  if (e != cudaSuccess) return e;
  tx = ta;
  to = ta;
  if (is_dact<EPI>()) {   // activation operand [M][N], 128-row (per-warp: 32-row) x 64-column boxes
    e = make_tmap(&tx, p.aux, g.N, g.M, p.ldaux, 64, Cfg<BN, EPI>::WARP_AUX ? 32 : BM);
    if (e != cudaSuccess) return e;
  }
  if (is_dact<EPI>()) {   // output [M][N] (row pitch ldo), 32-row x 64-column boxes
    e = make_tmap(&to, p.out, g.N, g.M, p.ldo, 64, 32);
    if (e != cudaSuccess) return e;
  }
  if (EPI == EPI_BIAS_ACT) {   // output, 32-row x 32-column boxes, 64-byte swizzle
    e = make_tmap(&to, p.out, g.N, g.M, p.ldo, 32, 32, CU_TENSOR_MAP_SWIZZLE_64B);
    if (e != cudaSuccess) return e;
  }
  p.M = g.M;
  p.N = g.N;
  p.K = g.K;
  p.a_rows = g.A;
  p.lda = g.lda;
  p.tiles_m = (g.M + BM - 1) / BM;
  p.tiles_n = g.N / BN;
  p.k_tiles = (g.K + BK - 1) / BK;
  const int rem = g.K - (p.k_tiles - 1) * BK;
  p.last_k_steps = (rem + 15) / 16;
  const int total = p.tiles_m * p.tiles_n;
  const int grid = total < num_sms ? total : num_sms;
  if (grid_out) *grid_out = grid;
  return launch_pdl(tc_gemm_kernel<BN, EPI>, dim3(grid), dim3(gemm_threads<BN, EPI>()),
                    Cfg<BN, EPI>::SMEM, st, ta, tb, tx, to, p);
}

}  // namespace

template <int BN, int EPI>
cudaError_t set_smem_attr() {
  return cudaFuncSetAttribute(tc_gemm_kernel<BN, EPI>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              (int)Cfg<BN, EPI>::SMEM);
}

// Driver entry point and the shared-memory opt-in of every kernel instance;
// called once per context, outside any stream capture.
cudaError_t tc_prepare() {
  cudaError_t e = get_encode();
  if (e != cudaSuccess) return e;
  const cudaError_t errs[] = {
      set_smem_attr<256, EPI_BIAS_ACT>(), set_smem_attr<128, EPI_BIAS_ACT>(),
      set_smem_attr<128, EPI_DACT>(),     set_smem_attr<128, EPI_DACT_K1>(),
      set_smem_attr<256, EPI_DACT>(),
      set_smem_attr<16, EPI_LOSS>(),      set_smem_attr<32, EPI_LOSS>(),
      cudaFuncSetAttribute(tc_wgrad_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)W_SMEM)};
  for (cudaError_t x : errs)
    if (x != cudaSuccess) return x;
  return cudaSuccess;
}

cudaError_t tc_make_tmap(CUtensorMap* m, const void* base, int64_t cols, int64_t rows, int64_t ld,
                         int box_cols, int box_rows, int swizzle_bytes) {
  if (box_cols * 2 > swizzle_bytes) return cudaErrorInvalidValue;
  const CUtensorMapSwizzle swz = swizzle_bytes == 128  ? CU_TENSOR_MAP_SWIZZLE_128B
                                 : swizzle_bytes == 64 ? CU_TENSOR_MAP_SWIZZLE_64B
                                 : swizzle_bytes == 32 ? CU_TENSOR_MAP_SWIZZLE_32B
                                                       : CU_TENSOR_MAP_SWIZZLE_NONE;
  if (swz == CU_TENSOR_MAP_SWIZZLE_NONE) return cudaErrorInvalidValue;
  return make_tmap(m, base, cols, rows, ld, box_cols, box_rows, swz);
}

cudaError_t tc_make_tmap_blocks(CUtensorMap* m, const void* base, int64_t rows, int64_t ld,
                                int nblk, int box_rows, int box_blk) {
  return make_tmap_blocks(m, base, rows, ld, nblk, box_rows, box_blk);
}

int tc_pick_bn(int N) {
  if (N % 256 == 0) return 256;
  if (N % 128 == 0) return 128;
  if (N % 64 == 0) return 64;
  return 0;
}

cudaError_t tc_gemm_bias_act(const GemmOperands& g, const float* bias, int act,
                             __nv_bfloat16* out, int ldo, int* err, uint64_t timeout_ns,
                             int num_sms, cudaStream_t st) {
  TcParams p{};
  p.bias = bias;
  p.act = act;
  p.out = out;
  p.ldo = ldo;
  p.err = err;
  p.timeout_ns = timeout_ns;
  // output widths are multiples of 128 (64-column TMA-store blocks per warp)
  if (g.N % 256 == 0) return launch_tc<256, EPI_BIAS_ACT>(g, p, num_sms, st, nullptr);
  if (g.N % 128 == 0) return launch_tc<128, EPI_BIAS_ACT>(g, p, num_sms, st, nullptr);
  return cudaErrorInvalidValue;
}

// 256-column backward-data tiles halve the re-reads of the row operand but
// also the number of tiles: used when every SM still gets two (a chain of
// small products, e.g. Newton-Schulz on 256 x 256 matrices, keeps 128 columns)
bool wide_dact(const GemmOperands& g, int num_sms) {
  return g.N % 256 == 0 && (int64_t)((g.M + BM - 1) / BM) * (g.N / 256) >= 2 * num_sms;
}

cudaError_t tc_gemm_dact(const GemmOperands& g, const __nv_bfloat16* aux, int ldaux, int act,
                         __nv_bfloat16* out, int ldo, float* colsum_part, int* err,
                         uint64_t timeout_ns, int num_sms, cudaStream_t st, int* grid_out) {
  if (g.N > kColsumCap) return cudaErrorInvalidValue;
  TcParams p{};
  p.aux = aux;
  p.ldaux = ldaux;
  p.act = act;
  p.out = out;
  p.ldo = ldo;
  p.colsum_part = colsum_part;
  p.epi_n = g.N;
  p.err = err;
  p.timeout_ns = timeout_ns;
  // 128 columns, so that 4 stages and two activation tiles fit (2 stages and
  // four activation tiles for a single k-tile)
  if (g.N % 128 != 0) return cudaErrorInvalidValue;
  // (the single-k-tile configuration pays off on tall minibatches only)
  if (g.K <= BK && g.M >= kTallRows) return launch_tc<128, EPI_DACT_K1>(g, p, num_sms, st, grid_out);
  if (wide_dact(g, num_sms)) return launch_tc<256, EPI_DACT>(g, p, num_sms, st, grid_out);
  return launch_tc<128, EPI_DACT>(g, p, num_sms, st, grid_out);
}

cudaError_t tc_gemm_axpby(const GemmOperands& g, const __nv_bfloat16* aux, int ldaux, float alpha,
                          float beta, __nv_bfloat16* out, int ldo, int* err, uint64_t timeout_ns,
                          int num_sms, cudaStream_t st) {
  if (g.N % 128 != 0) return cudaErrorInvalidValue;
  TcParams p{};
  p.aux = aux;
  p.ldaux = ldaux;
  p.act = 3;
  p.alpha = alpha;
  p.beta = beta;
  p.out = out;
  p.ldo = ldo;
  p.colsum_part = nullptr;
  p.epi_n = 0;   // no column sums
  p.err = err;
  p.timeout_ns = timeout_ns;
  if (g.K <= BK && g.M >= kTallRows) return launch_tc<128, EPI_DACT_K1>(g, p, num_sms, st, nullptr);
  if (wide_dact(g, num_sms)) return launch_tc<256, EPI_DACT>(g, p, num_sms, st, nullptr);
  return launch_tc<128, EPI_DACT>(g, p, num_sms, st, nullptr);
}

cudaError_t tc_gemm_loss(const GemmOperands& g, const NetShape& s, LossCoef lc, LossRows rows,
                         float inv_mb, const float* b3, const float* logstd, __nv_bfloat16* dz,
                         int lddz, float* colsum_part, float* loss_part, int* err,
                         uint64_t timeout_ns, int num_sms, cudaStream_t st, int* grid_out) {
  TcParams p{};
  p.bias = b3;
  p.shape = s;
  p.lc = lc;
  p.rows = rows;
  p.inv_mb = inv_mb;
  p.logstd = logstd;
  p.dz = dz;
  p.lddz = lddz;
  p.colsum_part = colsum_part;
  p.loss_part = loss_part;
  p.layout9222 = is_layout_9222(s) ? 1 : 0;
  p.epi_n = g.N;
  p.err = err;
  p.timeout_ns = timeout_ns;
  if (g.N == 16) return launch_tc<16, EPI_LOSS>(g, p, num_sms, st, grid_out);
  if (g.N == 32) return launch_tc<32, EPI_LOSS>(g, p, num_sms, st, grid_out);
  return cudaErrorInvalidValue;
}

cudaError_t tc_wgrad(const WGradRegion* regs, int nreg, int rows, uint32_t mn_lbo,
                     uint32_t mn_sbo, int* err, uint64_t timeout_ns, int num_sms,
                     cudaStream_t st, unsigned* tile_ctr, double* sq_part, int* grid_out,
                     uint64_t tile_wait_ns, const ReduceArgs* vectors) {
  if (nreg < 1 || nreg > 3) return cudaErrorInvalidValue;
  CUtensorMap tu[3], tv[3], tp[3];
  WParams p{};
  p.nreg = nreg;
  p.err = err;
  p.timeout_ns = timeout_ns;
  p.mn_lbo = mn_lbo;
  p.mn_sbo = mn_sbo;
  p.fixup = tile_ctr != nullptr && sq_part != nullptr;
  p.tile_ctr = tile_ctr;
  p.sq_part = sq_part;
  p.tile_wait_ns = tile_wait_ns ? tile_wait_ns : timeout_ns;
  if (p.fixup && vectors) {
    p.ra = *vectors;
    p.nvt = reduce_vector_tasks(vectors->s);
  }
  int unit = 0, tiles = 0;
  for (int r = 0; r < nreg; ++r) {
    const WGradRegion& G = regs[r];
    if (G.M % BM != 0 || G.N % 64 != 0 || G.M > G.ldu || G.N > G.ldv) return cudaErrorInvalidValue;
    WRegion& R = p.r[r];
    R.bn = tc_wgrad_bn(G.N);
    cudaError_t e = make_tmap_blocks(&tu[r], G.U, rows, G.ldu, G.M / 64, BK, WBM / 64);
    if (e != cudaSuccess) return e;
    e = make_tmap_blocks(&tv[r], G.V, rows, G.ldv, G.N / 64, BK, R.bn / 64);
    if (e != cudaSuccess) return e;
    R.M = G.M;
    R.N = G.N;
    R.tiles_m = (G.M + WBM - 1) / WBM;
    R.tiles_n = G.N / R.bn;
    R.k_tiles = (rows + BK - 1) / BK;
    R.kt_per_split = G.kt_per_split;
    R.splits = (R.k_tiles + R.kt_per_split - 1) / R.kt_per_split;
    e = make_tmap_partials(&tp[r], G.part, G.N, G.M, R.splits);
    if (e != cudaSuccess) return e;
    R.unit_begin = unit;
    R.part = G.part;
    unit += R.tiles_m * R.tiles_n * R.splits;
    if (p.fixup) {
      if (G.fin.dst == nullptr || R.splits > kWgMaxSplits) return cudaErrorInvalidValue;
      p.f[r] = G.fin;
      p.tile_begin[r] = tiles;
    }
    tiles += R.tiles_m * R.tiles_n;
  }
  if (p.fixup && tiles > kWgradMaxTiles) return cudaErrorInvalidValue;
  for (int r = nreg; r < 3; ++r) {
    tu[r] = tu[0];
    tv[r] = tv[0];
    tp[r] = tp[0];
  }
  p.total_units = unit;
  const int grid = unit < num_sms ? unit : num_sms;
  if (grid_out) *grid_out = grid;
  if (!p.fixup)
    return launch_pdl(tc_wgrad_kernel, dim3(grid), dim3(kThreads), W_SMEM, st, tu[0], tv[0],
                      tu[1], tv[1], tu[2], tv[2], tp[0], tp[1], tp[2], p);
  // cooperative: the CTAs of a tile wait for one another (one CTA per SM,
  // grid <= SMs, so the launch is always resident); programmatic
  // serialization lets its prologue overlap the previous kernel's tail (the
  // kernel waits for that kernel's results before its first load)
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = W_SMEM;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, tc_wgrad_kernel, tu[0], tv[0], tu[1], tv[1], tu[2], tv[2],
                            tp[0], tp[1], tp[2], p);
}

int tc_wgrad_bn(int N) { return N % 256 == 0 ? 256 : (N % 128 == 0 ? 128 : 64); }

// At large minibatches the kernel streams its operands (each unit reads
// (128 + bn) features of every row in its k-range) and the tensor pipe is not
// the limit, so units are balanced by the bytes they load: a region of
// bn-column tiles gets q / (128 + bn) k-tiles per unit.  q is the smallest
// budget whose units fit in one wave of num_sms CTAs (a second, partial wave
// would double the kernel's time); every unit covers at least 4 k-tiles and a
// region is split at most max_split times.
void tc_wgrad_plan(const int (*mn)[2], int nreg, int64_t rows, int num_sms, int max_split,
                   int* kt) {
  const int64_t k_tiles = (rows + BK - 1) / BK;
  constexpr int wbm = WBM;
  double total = 0;
  for (int i = 0; i < nreg; ++i) {
    const int bn = tc_wgrad_bn(mn[i][1]);
    total += (double)((mn[i][0] + wbm - 1) / wbm) * (mn[i][1] / bn) * (wbm + bn) * k_tiles;
  }
  for (int64_t q = (int64_t)std::ceil(total / num_sms);; q += (q + 15) / 16) {
    int64_t units = 0;
    for (int i = 0; i < nreg; ++i) {
      const int bn = tc_wgrad_bn(mn[i][1]);
      int64_t kp = q / (wbm + bn);
      if (kp < 4) kp = 4;
      if ((k_tiles + kp - 1) / kp > max_split) kp = (k_tiles + max_split - 1) / max_split;
      if (kp > k_tiles) kp = k_tiles;
      kt[i] = (int)kp;
      units += (int64_t)((mn[i][0] + wbm - 1) / wbm) * (mn[i][1] / bn) * ((k_tiles + kp - 1) / kp);
    }
    if (units <= num_sms || q >= 1024 * k_tiles) return;
  }
}

int tc_wgrad_splits(int rows, int kt_per_split) {
  const int k_tiles = (rows + BK - 1) / BK;
  return (k_tiles + kt_per_split - 1) / kt_per_split;
}

}  // namespace ppo
