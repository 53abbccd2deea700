// hl2.cu -- head + loss + backward-data through the last hidden layer, fused:
// for each 128-row tile of a minibatch
//
//   Z   = H2 W3^T + b3 -> per-row PPO loss -> dz      (N = CP head columns)
//   dP2 = (dz W3) * act'(H2)                            (N = H2, K = CP)
//
// "Teaching Mario to speedrun", sec. 6 (loss_pi, loss_V, entropy and
// loss.backward() through the policy/value head).  Each tile of H2 is loaded
// once by TMA: it is the A operand of the head product and the activation
// operand of act'(H2), and dP2 is written back over it in place and leaves by
// TMA stores.  dz stays in shared memory as the A operand of dz W3 (K = CP)
// and goes to HBM for the weight gradient of W3.  Compared with a head+loss
// kernel followed by a separate backward-data kernel this reads H2 once
// instead of twice and drops the dz round trip and one launch.  Shapes:
// H2 = 256 or 512 with CP = 16 head columns.  Every wait is bounded.
#include <cuda.h>

#include "common.cuh"
#include "gemm.h"
#include "tc_ptx.cuh"
#include "tc_tile.cuh"

namespace ppo {

namespace {

using namespace ptx;
using namespace tc;

constexpr int kHWarps = 10;
constexpr int kHThreads = kHWarps * kWarp;
constexpr int kHEpi = 8 * kWarp;
constexpr int kHGrp = 4 * kWarp;   // one epilogue group
constexpr int kBlk = 128 * 128;   // 128 rows x 64 bf16 columns (16 KB)
constexpr int kCtrlBytes = 512;

struct HMaps {
  CUtensorMap h2, w3;   // loads
  CUtensorMap dz, dp2;  // stores (32-row boxes)
};

struct HParams {
  int M, tiles, act;
  const float *b3, *logstd;
  NetShape shape;
  LossCoef lc;
  LossRows rows;
  float inv_mb;
  float *cs2, *cs3, *lossp;   // per-CTA partial rows
  int* err;
  uint64_t timeout_ns;
  int layout9222;   // the 9-2-2-2 head layout: compile-time masks in the loss
};

// head masks of the loss: the compile-time ones of the common layout, or the
// run-time ones of the shape (two instantiations of the loss loop)
struct FixedMasks {
  __device__ static constexpr HeadMasks get() { return kMasks9222; }
};
struct ShapeMasks {
  HeadMasks m;
  __device__ HeadMasks get() const { return m; }
};

// ---------------------------------------------------------------------------
// H2 = 256 or 512, CP = 16: a tile's dP2 in 128-column quarters (two or
// four), so that the next tile's head product and loss overlap this tile's
// dP2 epilogue.
//
// H2 streams through a ring of kQR 64-column blocks (16 KB each) instead of
// one tile buffer: the next tile's blocks land in slots as the current
// tile's quarters are stored out of theirs, and its head product Z runs
// block by block as they land.  TMEM: three rotating 128-column dP2 quarter
// buffers in columns [0, 384) and Z in [384, 400).  W3 sits in 64-column
// blocks of its 16 rows and is the B operand of both products: K-major for
// Z = H2 W3^T, MN-major for dz W3.  The dz tile (128 x 16) is kept in
// 32-byte swizzled rows, with a negated copy that is the A operand of the
// dP2 product: the epilogue then forms dP2 with two packed fp32-pair
// instructions per pair of columns.
// Roles: warp 0 TMA, warp 1 MMA, warps 2..9 the dP2 epilogue (warps 2..5 the
// first 64 columns of each quarter, warps 6..9 the second; TMEM lane quarter
// q = warp % 4).  Warps 2..5 also run each tile's loss before its quarters.
// A block's slot is handed back once the TMA store of its dP2 has read it:
// each epilogue warp checks that for its previous store half-way through its
// next block, so no warp waits on a store it has just issued.  The loss
// warps keep their loss sums and dz column sums in registers across tiles.
constexpr int kQR = 12;   // ring slots
constexpr int kQCP = 16;
// shared-memory layout for H2 = QH2 (256 or 512) columns
template <int QH2>
struct QL {
  static constexpr int W3 = kQR * kBlk;             // W3: QH2/64 blocks of [16][64]
  static constexpr int DZ = W3 + kQCP * QH2 * 2;    // dz [128][16] (stored out)
  static constexpr int NDZ = DZ + 128 * kQCP * 2;   // -dz, the A operand of the dP2 product
  static constexpr int Ctrl = NDZ + 128 * kQCP * 2;
  static constexpr int Cs2 = Ctrl + kCtrlBytes;     // [4][QH2]
  static constexpr int Cs3 = Cs2 + 4 * QH2 * 4;     // [4][32]
  static constexpr int Lp = Cs3 + 4 * 32 * 4;       // [4][kLossPartials]
  static constexpr int B3 = Lp + 4 * kLossPartials * 4;
  static constexpr int Smem = 1024 + B3 + 32 * 4;
  static_assert(Smem <= 232448, "shared memory of the quarter kernel");
};
constexpr uint32_t kQTZ = 384;   // TMEM column of Z

enum QBar : int {
  Q_FULL = 0, Q_EMPTY = kQR, Q_W3 = 2 * kQR, Q_ZFULL, Q_ZFREE, Q_DZRDY, Q_DZFREE,
  Q_QFULL, Q_QFREE = Q_QFULL + 3, Q_DRAIN = Q_QFREE + 3, Q_COUNT
};
static_assert(Q_COUNT * 8 + 32 <= kCtrlBytes, "barrier block");

template <int QH2, class Masks>
__global__ void __launch_bounds__(kHThreads, 1)
hlq_kernel(const __grid_constant__ HMaps maps, const HParams p, Masks masks) {
  using L = QL<QH2>;
  constexpr int NB = QH2 / 64;    // H2 blocks per tile
  constexpr int NQ = QH2 / 128;   // dP2 quarters per tile
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gb = smem_raw + (base - raw);
  uint8_t* ring = gb;
  uint8_t* DZ = gb + L::DZ;
  uint64_t* bars = reinterpret_cast<uint64_t*>(gb + L::Ctrl);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(bars + Q_COUNT);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tslot + 1);
  volatile uint32_t* cnt = reinterpret_cast<volatile uint32_t*>(tslot + 2);   // H2 blocks issued
  float* cs2 = reinterpret_cast<float*>(gb + L::Cs2);
  float* cs3 = reinterpret_cast<float*>(gb + L::Cs3);
  float* lp = reinterpret_cast<float*>(gb + L::Lp);
  float* b3s = reinterpret_cast<float*>(gb + L::B3);
  auto bar = [&](int i) { return smem_u32(&bars[i]); };

  const int warp = threadIdx.x / kWarp, lane = threadIdx.x % kWarp;
  if (threadIdx.x == 0) {
    for (int b = 0; b < kQR; ++b) {
      mbar_init(bar(Q_FULL + b), 1);
      mbar_init(bar(Q_EMPTY + b), kHGrp);   // the four warps storing the block
    }
    mbar_init(bar(Q_W3), 1);
    mbar_init(bar(Q_ZFULL), 1);
    mbar_init(bar(Q_ZFREE), kHGrp);
    mbar_init(bar(Q_DZRDY), kHGrp);
    mbar_init(bar(Q_DZFREE), 1);
    for (int b = 0; b < 3; ++b) {
      mbar_init(bar(Q_QFULL + b), 1);
      mbar_init(bar(Q_QFREE + b), kHEpi);
    }
    mbar_init(bar(Q_DRAIN), 1);
    *abort_flag = 0;
    cnt[0] = 0;
    fence_mbar_init();
  }
  for (int i = threadIdx.x; i < (L::B3 - L::Cs2) / 4; i += kHThreads) cs2[i] = 0.f;
  if (warp == 1) tmem_alloc(smem_u32(tslot), 512);
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&maps.h2);
    prefetch_tmap(&maps.w3);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tslot;
  const Guard g{abort_flag, p.err, p.timeout_ns};
  pdl_wait();
  pdl_trigger();
  for (int i = threadIdx.x; i < 32; i += kHThreads) b3s[i] = i < p.shape.C ? p.b3[i] : 0.f;
  __syncthreads();   // reached by every thread of the block (before the role split)

  if (warp == 0) {
    if (lane == 0) {
      bool ok = true;
      mbar_arrive_expect_tx(bar(Q_W3), (uint32_t)(kQCP * QH2 * 2));
      tma_load_3d(base + L::W3, &maps.w3, 0, 0, 0, bar(Q_W3));
      uint32_t n = 0, slot = 0, use = 0;   // blocks issued; ring position of the next
      for (int tile = blockIdx.x; tile < p.tiles && ok; tile += gridDim.x) {
        for (int kb = 0; kb < NB; ++kb) {
          if (use > 0 && !wait_bar(bar(Q_EMPTY + slot), (use - 1) & 1, g)) { ok = false; break; }
          mbar_arrive_expect_tx(bar(Q_FULL + slot), (uint32_t)kBlk);
          tma_load_2d(base + slot * kBlk, &maps.h2, kb * 64, tile * 128, bar(Q_FULL + slot));
          cnt[0] = ++n;
          if (++slot == kQR) { slot = 0; ++use; }
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      bool ok = wait_bar(bar(Q_W3), 0, g);
      uint32_t slot = 0, use = 0, qb = 0, qu = 0, t = 0;
      const uint32_t idz = idesc_bf16(128, kQCP, false, false);
      const uint32_t idq = idesc_bf16(128, 128, false, true);   // B = W3, MN-major
      for (int tile = blockIdx.x; tile < p.tiles && ok; tile += gridDim.x, ++t) {
        // Z = H2 W3^T into [kQTZ, kQTZ + 16), block by block as they land,
        // once the loss of the previous tile has read Z
        if (t > 0 && !wait_bar(bar(Q_ZFREE), (t - 1) & 1, g)) break;
        for (int kb = 0; kb < NB && ok; ++kb) {
          if (!wait_bar(bar(Q_FULL + slot), use & 1, g)) { ok = false; break; }
          tc_fence_after();
          for (int kk = 0; kk < 4; ++kk)
            tc_mma_bf16(tmem + kQTZ, sdesc_sw128(base + slot * kBlk + kk * 32, 16, 1024),
                        sdesc_sw128(base + L::W3 + kb * kQCP * 128 + kk * 32, 16, 1024), idz,
                        (kb | kk) ? 1u : 0u);
          if (++slot == kQR) { slot = 0; ++use; }
        }
        if (!ok) break;
        tc_commit(bar(Q_ZFULL));
        // dP2 quarters = dz W3[:, columns of the quarter] (K = 16), each into
        // the next free quarter buffer; B spans two 64-column blocks of W3
        // (leading byte offset: one block) and its 16 rows (stride byte
        // offset: 8 rows of 128 bytes)
        if (!wait_bar(bar(Q_DZRDY), t & 1, g)) break;
        for (int j = 0; j < NQ && ok; ++j) {
          if (qu > 0 && !wait_bar(bar(Q_QFREE + qb), (qu - 1) & 1, g)) { ok = false; break; }
          tc_fence_after();
          tc_mma_bf16(tmem + qb * 128, sdesc_sw32(base + L::NDZ, 256),
                      sdesc_sw128(base + L::W3 + 2 * j * kQCP * 128, kQCP * 128, 1024), idq,
                      0u);
          tc_commit(bar(Q_QFULL + qb));
          if (++qb == 3) { qb = 0; ++qu; }
        }
        if (!ok) break;
        tc_commit(bar(Q_DZFREE));   // the dz tile has been read
      }
    }
  } else {
    const int q = warp & 3;
    const int gi = warp < 6 ? 0 : 1;   // which 64 columns of each quarter
    const bool loss_w = gi == 0;
    const int rl = q * 32 + lane;
    const uint32_t lanes = (uint32_t)(q * 32) << 16;
    const HeadMasks hm = masks.get();
    uint32_t ts = 0, n0 = 0, qb = 0, qu = 0, t = 0;   // ring slot and number of the tile's block 0
    int pend = -1;                            // slot of this warp's last dP2 store
    // the slot of the previous dP2 store goes back once this warp's stores
    // (that one, and the dz tile's for the loss warps) have read shared memory
    auto release = [&]() {
      if (pend >= 0) {
        if (lane == 0) bulk_wait_read0();
        __syncwarp();
        mbar_arrive(bar(Q_EMPTY + pend));
        pend = -1;
      }
    };
    float adz[32], at6[6], adl[4];   // loss warps: sums over their rows of all tiles
#pragma unroll
    for (int k = 0; k < 32; ++k) adz[k] = 0.f;
#pragma unroll
    for (int k = 0; k < 6; ++k) at6[k] = 0.f;
#pragma unroll
    for (int k = 0; k < 4; ++k) adl[k] = 0.f;
    // loss warps: the per-row inputs of the loss, loaded one tile ahead (their
    // latency then overlaps this tile's quarters)
    RowIn in;
    if (loss_w) load_row_in(in, blockIdx.x * 128 + rl, blockIdx.x * 128 + rl < p.M, p.shape, p.rows);
    for (int tile = blockIdx.x; tile < p.tiles; tile += gridDim.x, ++t) {
      const int row0 = tile * 128;
      const int row = row0 + rl;
      const bool rok = row < p.M;
      const bool box_ok = row0 + q * 32 < p.M;   // boxes wholly below the last row are skipped
      if (loss_w) {
        if (!wait_bar(bar(Q_ZFULL), t & 1, g)) break;
        tc_fence_after();
        float dzr[32], t6[6], dls[4];
        loss_row_in<kQCP>(tmem + lanes + kQTZ, rok, p.shape, hm, p.lc, p.inv_mb, in, p.logstd,
                          b3s, dzr, t6, dls);
        tc_fence_before();
        mbar_arrive(bar(Q_ZFREE));
        // the dz tile is free once the previous tile's quarter products have
        // read it (its store was checked by this warp's later stores)
        if (t > 0 && !wait_bar(bar(Q_DZFREE), (t - 1) & 1, g)) break;
        uint8_t* drow = DZ + rl * 32;
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          uint4 u;
          u.x = pack_bf16x2(dzr[8 * i + 0], dzr[8 * i + 1]);
          u.y = pack_bf16x2(dzr[8 * i + 2], dzr[8 * i + 3]);
          u.z = pack_bf16x2(dzr[8 * i + 4], dzr[8 * i + 5]);
          u.w = pack_bf16x2(dzr[8 * i + 6], dzr[8 * i + 7]);
          const int off = (i ^ ((rl >> 2) & 1)) << 4;
          *reinterpret_cast<uint4*>(drow + off) = u;
          constexpr uint32_t kSign = 0x80008000u;   // -dz: both bf16 sign bits flipped
          *reinterpret_cast<uint4*>(drow + (L::NDZ - L::DZ) + off) =
              make_uint4(u.x ^ kSign, u.y ^ kSign, u.z ^ kSign, u.w ^ kSign);
        }
        fence_proxy_async_smem();
        mbar_arrive(bar(Q_DZRDY));
        __syncwarp();
        if (lane == 0) {
          if (box_ok) tma_store_2d(&maps.dz, smem_u32(DZ + q * 1024), 0, row0 + q * 32);
          bulk_commit();
        }
#pragma unroll
        for (int k = 0; k < kQCP; ++k) adz[k] += dzr[k];
#pragma unroll
        for (int k = 0; k < 6; ++k) at6[k] += t6[k];
#pragma unroll
        for (int k = 0; k < 4; ++k) adl[k] += dls[k];
        const int nrow = row + (int)gridDim.x * 128;
        if (tile + (int)gridDim.x < p.tiles) load_row_in(in, nrow, nrow < p.M, p.shape, p.rows);
      }
      bool ok = true;
      for (int j = 0; j < NQ; ++j) {
        const int kb = 2 * j + gi;
        const int slot = ts + kb < kQR ? ts + kb : ts + kb - kQR;
        uint8_t* blk = ring + slot * kBlk;
        // the block's TMA load (complete: the quarter product ran after the
        // head product read it) and the quarter's accumulator
        if (!wait_bar(bar(Q_FULL + slot), ((n0 + kb) / kQR) & 1, g) ||
            !wait_bar(bar(Q_QFULL + qb), qu & 1, g)) { ok = false; break; }
        tc_fence_after();
        epi_dact_block(tmem + lanes + qb * 128 + gi * 64, rl, p.act, blk, cs2 + q * QH2 + kb * 64,
                       lane, release);
        tc_fence_before();
        mbar_arrive(bar(Q_QFREE + qb));
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          if (box_ok) tma_store_2d(&maps.dp2, smem_u32(blk + q * 4096), kb * 64, row0 + q * 32);
          bulk_commit();
        }
        pend = slot;
        if (++qb == 3) { qb = 0; ++qu; }
      }
      if (!ok) break;
      ts = ts + NB < kQR ? ts + NB : ts + NB - kQR;
      n0 += NB;
    }
    if (loss_w) loss_warp_reduce(adz, at6, adl, cs3 + q * 32, lp + q * kLossPartials, lane);
    if (lane == 0) bulk_wait0();
  }

  __syncthreads();
  if (*abort_flag) {
    if (threadIdx.x == 0) {   // loads in flight: the last kQR H2 blocks and W3
      const uint32_t n = cnt[0];
      for (uint32_t l = n >= (uint32_t)kQR ? n - kQR : 0; l < n; ++l)
        drain_wait(bar(Q_FULL + l % kQR), (l / kQR) & 1, p.timeout_ns);
      drain_wait(bar(Q_W3), 0, p.timeout_ns);
    }
    if (warp == 1 && lane == 0) {
      tc_commit(bar(Q_DRAIN));
      drain_wait(bar(Q_DRAIN), 0, p.timeout_ns);
    }
    __syncthreads();
  }
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
  if (warp >= 2) {
    const int et = threadIdx.x - 2 * kWarp;
    auto quad = [&](const float* b, int ld, int c) {
      return ((b[c] + b[ld + c]) + b[2 * ld + c]) + b[3 * ld + c];
    };
    for (int c = et; c < QH2; c += kHEpi)
      p.cs2[(int64_t)blockIdx.x * QH2 + c] = quad(cs2, QH2, c);
    if (et < kQCP) p.cs3[(int64_t)blockIdx.x * kQCP + et] = quad(cs3, 32, et);
    if (et < kLossPartials)
      p.lossp[(int64_t)blockIdx.x * kLossPartials + et] = quad(lp, kLossPartials, et);
  }
}

template <int QH2, class Masks>
cudaError_t launch_q(const HMaps& m, const HParams& p, Masks masks, int grid, cudaStream_t st) {
  return launch_pdl(hlq_kernel<QH2, Masks>, dim3(grid), dim3(kHThreads), (size_t)QL<QH2>::Smem, st,
                    m, p, masks);
}

template <int QH2, class Masks>
cudaError_t set_attr_q() {
  return cudaFuncSetAttribute(hlq_kernel<QH2, Masks>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              QL<QH2>::Smem);
}


}  // namespace

bool hl2_supported(const NetShape& s) {
  return (s.H2 == 256 || s.H2 == 512) && s.CP == kQCP && s.G <= 4;
}

cudaError_t hl2_prepare() {
  const cudaError_t errs[] = {set_attr_q<256, FixedMasks>(), set_attr_q<256, ShapeMasks>(),
                              set_attr_q<512, FixedMasks>(), set_attr_q<512, ShapeMasks>()};
  for (cudaError_t e : errs)
    if (e != cudaSuccess) return e;
  return cudaSuccess;
}

cudaError_t hl2_launch(const HeadLossDact& f, int num_sms, cudaStream_t st, int* grid_out) {
  const NetShape& s = f.s;
  if (!hl2_supported(s) || f.M < 1) return cudaErrorInvalidValue;
  HMaps m;
  cudaError_t e;
  if ((e = tc_make_tmap(&m.h2, f.H2, s.H2, f.M, s.H2, 64, 128)) != cudaSuccess) return e;
  // W3 as H2/64 blocks of its 16 rows: the B operand of both products
  if ((e = tc_make_tmap_blocks(&m.w3, f.W3s, s.CP, s.H2, s.H2 / 64, s.CP, s.H2 / 64)) !=
      cudaSuccess)
    return e;
  if ((e = tc_make_tmap(&m.dz, f.dZ, kQCP, f.M, f.lddz, kQCP, 32, 32)) != cudaSuccess) return e;
  if ((e = tc_make_tmap(&m.dp2, f.dP2, s.H2, f.M, s.H2, 64, 32)) != cudaSuccess) return e;
  HParams p{};
  p.M = f.M;
  p.tiles = (f.M + 127) / 128;
  p.act = s.act;
  p.b3 = f.b3;
  p.logstd = f.logstd;
  p.shape = s;
  p.lc = f.lc;
  p.rows = f.rows;
  p.inv_mb = f.inv_mb;
  p.cs2 = f.cs2;
  p.cs3 = f.cs3;
  p.lossp = f.lossp;
  p.err = f.err;
  p.timeout_ns = f.timeout_ns;
  p.layout9222 = is_layout_9222(s) ? 1 : 0;
  const int grid = p.tiles < num_sms ? p.tiles : num_sms;
  if (grid_out) *grid_out = grid;
  return s.H2 == 512 ? (p.layout9222 ? launch_q<512>(m, p, FixedMasks{}, grid, st)
                                     : launch_q<512>(m, p, ShapeMasks{head_masks(s)}, grid, st))
                     : (p.layout9222 ? launch_q<256>(m, p, FixedMasks{}, grid, st)
                                     : launch_q<256>(m, p, ShapeMasks{head_masks(s)}, grid, st));
}

}  // namespace ppo
