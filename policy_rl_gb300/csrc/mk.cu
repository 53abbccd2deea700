// mk.cu -- one persistent, cooperative kernel for a whole bf16 minibatch step.
//
// "Teaching Mario to speedrun", sec. 6 "The whole algorithm", step 3: for a
// minibatch, loss = ppo_loss(network, minibatch); loss.backward();
// optimizer.step().  The separate-kernel path launches nine kernels per
// minibatch; at the minibatch sizes of the Mario-like workload each of them
// is a few tiles per SM and is dominated by launch and pipeline-fill latency.
// Here one CTA per SM runs every stage as a phase:
//
//   0 gather   1 fwd1   2 fwd2   3 head+loss   4 dact2   5 dact1
//   6 weight gradients   7 gradient assembly   8 clip + Adam (optional)
//
// The roles of the tensor-core kernels persist across phases: warp 0 issues
// TMA loads, warp 1 issues tcgen05 MMAs, warps 2..9 drain TMEM and run the
// epilogues and the CUDA-core phases.  Their smem-ring and TMEM counters run
// on across phases, so every mbarrier parity stays consistent.  Between
// phases a grid barrier (an arrival counter in global memory, acquired with
// ld.acquire.gpu) orders one phase's global writes before the next phase's
// reads; the producer issues a proxy fence after acquiring so that its TMA
// (async-proxy) reads see the epilogues' generic-proxy stores.  Every wait --
// mbarrier or grid barrier -- is bounded (globaltimer); on expiry the kernel
// latches kDevTimeout and unwinds.  The launch is cooperative, so all CTAs
// are co-resident.  Ten warps per CTA put three warps on two of the SM's four
// 16K-register partitions, which caps a thread at 168 registers.
#include "common.cuh"
#include "gemm.h"
#include "tc_ptx.cuh"
#include "tc_tile.cuh"

namespace ppo {

namespace {

using namespace ptx;
using namespace tc;

constexpr int kEW = 8;                       // epilogue warps
constexpr int kMkThreads = 2 * kWarp + kEW * kWarp;
constexpr int kEpiThreads = kEW * kWarp;
constexpr int kS = 4;                        // smem stages
constexpr int kAbytes = BM * BK * 2;         // 16 KB
constexpr int kBbytes = 256 * BK * 2;        // 32 KB (BN <= 256)
constexpr int kStage = kAbytes + kBbytes;
constexpr int kCtrl = 512;
constexpr int kTmemCols = 512;               // two 256-column accumulators
constexpr size_t kMkSmem = 1024 + (size_t)kS * kStage + kCtrl + 4 * kColsumCap * 4 +
                           4 * kLossPartials * 4 + kColsumCap * 4 + 64;

struct MkGemm {
  int M, N, K, BN, tiles_m, tiles_n, k_tiles, last_k_steps;
  int epi;
  const float* bias;
  __nv_bfloat16* out;
  int ldo;
  const __nv_bfloat16* aux;
  int ldaux;
  float* colsum_part;
  int epi_n;
};

struct MkMaps {
  CUtensorMap a[5], b[5], u[3], v[3];
};

struct MkParams {
  NetShape s;
  GatherArgs ga;
  int per_row;
  MkGemm g[5];              // fwd1, fwd2, loss, dact2, dact1
  WParams w;
  ReduceArgs ra;
  int do_adam;
  AdamArgs aa;
  LossCoef lc;
  LossRows rows;
  float inv_mb;
  const float* logstd;
  float* loss_part;
  __nv_bfloat16* dz;
  int lddz;
  unsigned* gbar;           // [0] phase arrivals, [1] exits
  double* sq_part;          // [grid]
  unsigned long long* phase_ns;   // nullable: per-phase time accumulators (profiling)
  int* err;
  uint64_t timeout_ns;
};

__device__ __forceinline__ unsigned ld_acquire(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}

// Bounded wait until `target` arrivals have been counted.
__device__ __forceinline__ bool grid_wait(const unsigned* ctr, unsigned target, const Guard& g) {
  if (ld_acquire(ctr) >= target) return true;
  const uint64_t t0 = globaltimer();
  while (true) {
#pragma unroll 1
    for (int i = 0; i < 16; ++i)
      if (ld_acquire(ctr) >= target) return true;
    if (*g.abort) return false;
    if (globaltimer() - t0 > g.limit_ns) {
      *g.abort = 1;
      atomicOr(g.err, kDevTimeout);
      return false;
    }
  }
}

// ---- CUDA-core phases (run by the 256 epilogue threads of every CTA) --------
__device__ void phase_gather(const MkParams& p, int et) {
  const NetShape& s = p.s;
  const GatherArgs& a = p.ga;
  const int64_t nthreads = (int64_t)gridDim.x * kEpiThreads;
  const int64_t total = a.mb * p.per_row;
  for (int64_t t = (int64_t)blockIdx.x * kEpiThreads + et; t < total; t += nthreads) {
    const int64_t r = t / p.per_row;
    const int c = (int)(t - r * p.per_row);
    int64_t src = __ldg(a.idx + r);
    src = src < 0 ? 0 : (src >= a.B ? a.B - 1 : src);
    if (a.obs_bf16) {
      const uint4* in = reinterpret_cast<const uint4*>(a.obs_bf16 + src * s.Dp);
      reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(a.X) + r * s.Dp)[c] = __ldg(in + c);
    } else {
      const float* in = a.obs_f32 + src * s.D;
      float f[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) f[j] = (8 * c + j < s.D) ? __ldg(in + 8 * c + j) : 0.f;
      uint4 o;
      o.x = pack_bf16x2(f[0], f[1]);
      o.y = pack_bf16x2(f[2], f[3]);
      o.z = pack_bf16x2(f[4], f[5]);
      o.w = pack_bf16x2(f[6], f[7]);
      reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(a.X) + r * s.Dp)[c] = o;
    }
    if (c != 0) continue;
    int32_t act[PPO_MAX_HEADS];
    float actc[4];
    for (int h = 0; h < s.NH; ++h) act[h] = __ldg(a.act + src * s.NH + h);
    for (int g = 0; g < s.G; ++g) actc[g] = __ldg(a.actc + src * s.G + g);
    const float lp = __ldg(a.logp_old + src);
    float A = __ldg(a.adv + src);
    const float R = __ldg(a.ret + src);
    if (a.adv_stats) A = (A - __ldg(a.adv_stats)) / (__ldg(a.adv_stats + 1) + 1e-8f);
    for (int h = 0; h < s.NH; ++h) {
      const int n = s.head_n[h];
      a.act_mb[r * s.NH + h] = act[h] < 0 ? 0 : (act[h] >= n ? n - 1 : act[h]);
    }
    for (int g = 0; g < s.G; ++g) a.actc_mb[r * s.G + g] = actc[g];
    a.logp_mb[r] = lp;
    a.adv_mb[r] = A;
    a.ret_mb[r] = R;
  }
}

__device__ __forceinline__ float rows_sum(const float* base, int rows, int64_t stride, int lane) {
  float v = 0.f;
  for (int b = lane; b < rows; b += kWarp) v += base[(int64_t)b * stride];
  return warp_sum(v);
}

// Gradient assembly: fixed-order sums of the split-K and per-CTA partials;
// returns this thread's sum of squares of what it wrote.
__device__ float phase_reduce(const ReduceArgs& a, int et) {
  const NetShape& s = a.s;
  const int nW1 = s.H1 * s.D, nW2 = s.H2 * s.H1, nW3 = s.C * s.H2;
  const int nW = nW1 + nW2 + nW3;
  float sq = 0.f;
  const int nthreads = gridDim.x * kEpiThreads;
  for (int e = blockIdx.x * kEpiThreads + et; e < nW; e += nthreads) {
    float v = 0.f;
    int i;
    if (e < nW1) {
      i = (int)s.oW1 + e;
      const int j = e / s.D, k = e - j * s.D;
      const float* q = a.pW1 + (int64_t)j * a.ld1 + k;
      const int64_t st = (int64_t)s.H1 * a.ld1;
#pragma unroll 8
      for (int sp = 0; sp < a.s1; ++sp) v += q[sp * st];
    } else if (e < nW1 + nW2) {
      const int r = e - nW1;
      i = (int)s.oW2 + r;
      const int64_t st = (int64_t)s.H2 * s.H1;
#pragma unroll 8
      for (int sp = 0; sp < a.s2; ++sp) v += a.pW2[r + sp * st];
    } else {
      const int r = e - nW1 - nW2;
      i = (int)s.oW3 + r;
      const int c = r / s.H2, j = r - c * s.H2;
      const float* q = a.pW3t + (int64_t)j * a.ld3 + c;
      const int64_t st = (int64_t)s.H2 * a.ld3;
#pragma unroll 8
      for (int sp = 0; sp < a.s3; ++sp) v += q[sp * st];
    }
    a.grad[i] = v;
    sq += v * v;
  }
  // bias / log-std elements and the six statistics: one warp each
  const int lane = et % kWarp;
  const int nb = s.H1 + s.H2 + s.C + s.G;
  const int nwarps = gridDim.x * kEW;
  for (int e = blockIdx.x * kEW + et / kWarp; e < nb + 6; e += nwarps) {
    if (e < nb) {
      float v;
      int i;
      if (e < s.H1) {
        i = (int)s.ob1 + e;
        v = rows_sum(a.pb1 + e, a.nb1, s.H1, lane);
      } else if (e < s.H1 + s.H2) {
        const int j = e - s.H1;
        i = (int)s.ob2 + j;
        v = rows_sum(a.pb2 + j, a.nb2, s.H2, lane);
      } else if (e < s.H1 + s.H2 + s.C) {
        const int c = e - s.H1 - s.H2;
        i = (int)s.ob3 + c;
        v = rows_sum(a.pb3 + c, a.nb3, a.ldb3, lane);
      } else {
        const int g = e - s.H1 - s.H2 - s.C;
        i = (int)s.ologstd + g;
        v = rows_sum(a.ploss + 6 + g, a.nl, kLossPartials, lane);
      }
      if (lane == 0) {
        a.grad[i] = v;
        sq += v * v;
      }
    } else {
      const int q = e - nb;
      const float v = rows_sum(a.ploss + q, a.nl, kLossPartials, lane);
      if (lane == 0 && a.stats6 != nullptr) a.stats6[q] = v * a.inv_mb;
    }
  }
  return sq;
}

__device__ __forceinline__ void write_shadow(const NetShape& s, const Shadows& sh, int i, float p) {
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

// Clip + Adam over the parameters (grid-stride), bias corrections from the
// running beta powers; coef/ibc1/ibc2 computed by the caller.
__device__ void phase_adam(const AdamArgs& a, int et, float coef, float ibc1, float ibc2) {
  const float b1 = (float)a.b1, b2 = (float)a.b2, omb1 = a.omb1, omb2 = a.omb2;
  const float lr = a.lr, eps = a.eps;
  const int P = (int)a.P;
  const int nthreads = gridDim.x * kEpiThreads;
  for (int i = blockIdx.x * kEpiThreads + et; i < P; i += nthreads) {
    const float g = a.g[i] * coef;
    const float m = b1 * a.m[i] + omb1 * g;
    const float v = b2 * a.v[i] + omb2 * g * g;
    const float pnew = a.p[i] - lr * (m * ibc1) / (sqrtf(v * ibc2) + eps);
    a.m[i] = m;
    a.v[i] = v;
    a.p[i] = pnew;
    write_shadow(a.s, a.sh, i, pnew);
  }
}

__device__ __forceinline__ void decode_unit(const WParams& w, int u, int& reg, int& tm, int& tn,
                                            int& kt0, int& kt1, int& split) {
  reg = 0;
  while (reg + 1 < w.nreg && u >= w.r[reg + 1].unit_begin) ++reg;
  const WRegion& R = w.r[reg];
  const int local = u - R.unit_begin;
  const int per = R.tiles_m * R.tiles_n;
  split = local / per;
  const int rem = local % per;
  tm = rem / R.tiles_n;
  tn = rem % R.tiles_n;
  kt0 = split * R.kt_per_split;
  kt1 = min(R.k_tiles, kt0 + R.kt_per_split);
}

// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kMkThreads, 1)
mk_kernel(const __grid_constant__ MkMaps maps, const MkParams p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);
  uint8_t* ctrl = gbase + (size_t)kS * kStage;
  Ctrl cb{reinterpret_cast<uint64_t*>(ctrl), kS};
  uint32_t* tslot = reinterpret_cast<uint32_t*>(ctrl + 8 * Ctrl::count(kS));
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tslot + 1);
  volatile uint32_t* cnt = reinterpret_cast<volatile uint32_t*>(tslot + 2);  // issued, consumed
  float* cs = reinterpret_cast<float*>(ctrl + kCtrl);                        // [4][kColsumCap]
  float* lp = cs + 4 * kColsumCap;                                           // [4][kLossPartials]
  float* bias_s = lp + 4 * kLossPartials;                                    // [kColsumCap]
  float* red = bias_s + kColsumCap;                                          // [kEW] + scalars

  const int warp = threadIdx.x / kWarp, lane = threadIdx.x % kWarp;
  auto sA = [&](int s) { return base + (uint32_t)(s * kStage); };
  auto sB = [&](int s) { return base + (uint32_t)(s * kStage + kAbytes); };

  if (threadIdx.x == 0) {
    for (int s = 0; s < kS; ++s) {
      mbar_init(cb.full(s), 1);
      mbar_init(cb.empty(s), 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(cb.tfull(a), 1);
      mbar_init(cb.tempty(a), kEpiThreads);
    }
    mbar_init(cb.drain(), 1);
    mbar_init(cb.epi(), kEpiThreads);
    *abort_flag = 0;
    cnt[0] = 0;
    cnt[1] = 0;
    fence_mbar_init();
  }
  for (int i = threadIdx.x; i < 4 * kColsumCap + 4 * kLossPartials; i += kMkThreads) cs[i] = 0.f;
  if (warp == 1) tmem_alloc(smem_u32(tslot), kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tslot;
  const Guard g{abort_flag, p.err, p.timeout_ns};
  const unsigned G = gridDim.x;
  unsigned* gbar = p.gbar;

  if (warp == 0) {
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      uint32_t it = 0;
      bool ok = true;
      for (int ph = 1; ph <= 6 && ok; ++ph) {
        if (!grid_wait(gbar, (unsigned)(ph) * G, g)) { ok = false; break; }
        fence_proxy_async_global();
        if (ph <= 5) {
          const MkGemm& m = p.g[ph - 1];
          const CUtensorMap* ta = &maps.a[ph - 1];
          const CUtensorMap* tb = &maps.b[ph - 1];
          const uint32_t bytes = (uint32_t)(kAbytes + m.BN * BK * 2);
          const int total = m.tiles_m * m.tiles_n;
          for (int tile = blockIdx.x; tile < total && ok; tile += G) {
            const int tm = tile / m.tiles_n, tn = tile % m.tiles_n;
            for (int kt = 0; kt < m.k_tiles; ++kt) {
              const int s = it % kS;
              const uint32_t r = it / kS;
              if (!wait_bar(cb.empty(s), (r & 1) ^ 1, g)) { ok = false; break; }
              mbar_arrive_expect_tx(cb.full(s), bytes);
              tma_load_2d(sA(s), ta, kt * BK, tm * BM, cb.full(s));
              tma_load_2d(sB(s), tb, kt * BK, tn * m.BN, cb.full(s));
              ++it;
              cnt[0] = it;
            }
          }
        } else {
          const WParams& w = p.w;
          for (int u = blockIdx.x; u < w.total_units && ok; u += G) {
            int reg, tm, tn, kt0, kt1, split;
            decode_unit(w, u, reg, tm, tn, kt0, kt1, split);
            const int bn = w.r[reg].bn;
            const uint32_t bytes = (uint32_t)(BM + bn) * BK * 2;
            for (int kt = kt0; kt < kt1; ++kt) {
              const int s = it % kS;
              const uint32_t r = it / kS;
              if (!wait_bar(cb.empty(s), (r & 1) ^ 1, g)) { ok = false; break; }
              mbar_arrive_expect_tx(cb.full(s), bytes);
              tma_load_2d(sA(s), &maps.u[reg], tm * BM, kt * BK, cb.full(s));
              tma_load_2d(sA(s) + 8192, &maps.u[reg], tm * BM + 64, kt * BK, cb.full(s));
              for (int j = 0; j < bn / 64; ++j)
                tma_load_2d(sB(s) + 8192 * j, &maps.v[reg], tn * bn + 64 * j, kt * BK, cb.full(s));
              ++it;
              cnt[0] = it;
            }
          }
        }
      }
      if (ok)
        for (int j = 0; j < kS; ++j, ++it) {
          const int s = it % kS;
          const uint32_t r = it / kS;
          if (!wait_bar(cb.empty(s), (r & 1) ^ 1, g)) break;
        }
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      uint32_t it = 0, tc = 0;
      bool ok = true;
      for (int ph = 1; ph <= 6 && ok; ++ph) {
        const bool wg = ph == 6;
        const int total = wg ? p.w.total_units : p.g[ph - 1].tiles_m * p.g[ph - 1].tiles_n;
        for (int t = blockIdx.x; t < total && ok; t += G) {
          int kt0 = 0, kt1, bn, last_steps = BK / 16;
          if (wg) {
            int reg, tm, tn, split;
            decode_unit(p.w, t, reg, tm, tn, kt0, kt1, split);
            bn = p.w.r[reg].bn;
          } else {
            const MkGemm& m = p.g[ph - 1];
            kt1 = m.k_tiles;
            bn = m.BN;
            last_steps = m.last_k_steps;
          }
          const uint32_t idesc = idesc_bf16(BM, bn, wg, wg);
          const int acc = tc & 1;
          const uint32_t use = tc >> 1;
          if (!wait_bar(cb.tempty(acc), (use & 1) ^ 1, g)) { ok = false; break; }
          tc_fence_after();
          const uint32_t d = tmem + (uint32_t)(acc * 256);
          for (int kt = kt0; kt < kt1; ++kt) {
            const int s = it % kS;
            const uint32_t r = it / kS;
            if (!wait_bar(cb.full(s), r & 1, g)) { ok = false; break; }
            tc_fence_after();
            const int nk = (kt == kt1 - 1) ? last_steps : BK / 16;
            for (int kk = 0; kk < nk; ++kk) {
              uint64_t da, db;
              if (wg) {
                da = sdesc_sw128(sA(s) + kk * 2048, 8192, 1024);
                db = sdesc_sw128(sB(s) + kk * 2048, 8192, 1024);
              } else {
                da = sdesc_sw128(sA(s) + kk * 32, 16, 1024);
                db = sdesc_sw128(sB(s) + kk * 32, 16, 1024);
              }
              tc_mma_bf16(d, da, db, idesc, (kt != kt0 || kk != 0) ? 1u : 0u);
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
    }
  } else {
    // ---------------- epilogue warps + CUDA-core phases ----------------
    const int et = threadIdx.x - 2 * kWarp;   // 0..255
    const int q = warp & 3;
    const int h = (warp - 2) / 4;
    uint32_t tc = 0, epi_phase = 0;
    bool ok = true;
    // all epilogue threads: arrive and wait on the epilogue-group barrier
    auto epi_sync = [&]() -> bool {
      mbar_arrive(cb.epi());
      const bool r = wait_bar(cb.epi(), epi_phase & 1, g);
      ++epi_phase;
      return r;
    };
    // phase end: every epilogue thread's writes, then one arrival per CTA
    auto phase_done = [&]() -> bool {
      __threadfence();
      fence_proxy_async_global();
      if (!epi_sync()) return false;
      if (et == 0) {
        __threadfence();      // the group's writes (ordered by epi_sync) before the arrival
        atomicAdd(gbar, 1u);
      }
      return true;
    };
    // profiling: CTA 0 adds the time between consecutive phase starts
    const bool timing = p.phase_ns != nullptr && blockIdx.x == 0 && et == 0;
    uint64_t t_prev = timing ? globaltimer() : 0;
    auto stamp = [&](int ph) {
      if (timing) {
        const uint64_t now = globaltimer();
        p.phase_ns[ph] += now - t_prev;
        t_prev = now;
      }
    };
    auto phase_begin = [&](int ph) -> bool {
      if (et == 0 && !grid_wait(gbar, (unsigned)ph * G, g)) return false;
      stamp(ph - 1);
      return epi_sync();
    };

    // phase 0: gather
    phase_gather(p, et);
    ok = phase_done();
    for (int ph = 1; ph <= 6 && ok; ++ph) {
      if (!(ok = phase_begin(ph))) break;
      const bool wg = ph == 6;
      const MkGemm* m = wg ? nullptr : &p.g[ph - 1];
      if (!wg && m->epi != EPI_DACT) {
        for (int i = et; i < m->N; i += kEpiThreads) bias_s[i] = m->bias[i];
        if (!(ok = epi_sync())) break;
      }
      const int total = wg ? p.w.total_units : m->tiles_m * m->tiles_n;
      for (int t = blockIdx.x; t < total; t += G) {
        const int acc = tc & 1;
        const uint32_t use = tc >> 1;
        if (!(ok = wait_bar(cb.tfull(acc), use & 1, g))) break;
        tc_fence_after();
        const uint32_t taddr = tmem + (uint32_t)(acc * 256) + ((uint32_t)(q * 32) << 16);
        if (wg) {
          int reg, tm, tn, kt0, kt1, split;
          decode_unit(p.w, t, reg, tm, tn, kt0, kt1, split);
          const WRegion& R = p.w.r[reg];
          const int half = R.bn / 2;
          const int row = tm * BM + q * 32 + lane;
          epi_wgrad_tile(taddr + (uint32_t)(h * half), row, half, R.M, R.N,
                         tn * R.bn + h * half, R.part + (int64_t)split * R.M * R.N);
        } else {
          const int tm = t / m->tiles_n, tn = t % m->tiles_n;
          const int row = tm * BM + q * 32 + lane;
          const bool rok = row < m->M;
          float* cs_q = cs + q * kColsumCap;
          if (m->epi == EPI_LOSS) {
            if (h == 0) {
              RowIn in;
              load_row_in(in, row, rok, p.s, p.rows);
              if (m->BN == 16)
                epi_loss_tile<16>(taddr, row, rok, p.s, head_masks(p.s), p.lc, p.inv_mb, in, p.logstd, bias_s,
                                  p.dz, p.lddz, cs_q, lp + q * kLossPartials, lane);
              else
                epi_loss_tile<32>(taddr, row, rok, p.s, head_masks(p.s), p.lc, p.inv_mb, in, p.logstd, bias_s,
                                  p.dz, p.lddz, cs_q, lp + q * kLossPartials, lane);
            }
          } else if (m->epi == EPI_BIAS_ACT) {
            if (m->BN == 256)
              epi_elem_tile<256, kEW, false>(taddr, row, rok, tn * 256, h, p.s.act, bias_s,
                                             nullptr, 0, m->out, m->ldo, cs_q, lane);
            else if (m->BN == 128)
              epi_elem_tile<128, kEW, false>(taddr, row, rok, tn * 128, h, p.s.act, bias_s,
                                             nullptr, 0, m->out, m->ldo, cs_q, lane);
            else
              epi_elem_tile<64, kEW, false>(taddr, row, rok, tn * 64, h, p.s.act, bias_s,
                                            nullptr, 0, m->out, m->ldo, cs_q, lane);
          } else {
            if (m->BN == 256)
              epi_elem_tile<256, kEW, true>(taddr, row, rok, tn * 256, h, p.s.act, bias_s,
                                            m->aux, m->ldaux, m->out, m->ldo, cs_q, lane);
            else if (m->BN == 128)
              epi_elem_tile<128, kEW, true>(taddr, row, rok, tn * 128, h, p.s.act, bias_s,
                                            m->aux, m->ldaux, m->out, m->ldo, cs_q, lane);
            else
              epi_elem_tile<64, kEW, true>(taddr, row, rok, tn * 64, h, p.s.act, bias_s,
                                           m->aux, m->ldaux, m->out, m->ldo, cs_q, lane);
          }
        }
        tc_fence_before();
        mbar_arrive(cb.tempty(acc));
        ++tc;
      }
      if (!ok) break;
      if (!wg && m->epi != EPI_BIAS_ACT) {
        // per-CTA column sums (bias gradients) and loss partials, then clear
        if (!(ok = epi_sync())) break;
        for (int c = et; c < m->epi_n; c += kEpiThreads) {
          m->colsum_part[(int64_t)blockIdx.x * m->epi_n + c] =
              ((cs[c] + cs[kColsumCap + c]) + cs[2 * kColsumCap + c]) + cs[3 * kColsumCap + c];
          cs[c] = cs[kColsumCap + c] = cs[2 * kColsumCap + c] = cs[3 * kColsumCap + c] = 0.f;
        }
        if (m->epi == EPI_LOSS && et < kLossPartials) {
          p.loss_part[(int64_t)blockIdx.x * kLossPartials + et] =
              ((lp[et] + lp[kLossPartials + et]) + lp[2 * kLossPartials + et]) +
              lp[3 * kLossPartials + et];
          lp[et] = lp[kLossPartials + et] = lp[2 * kLossPartials + et] =
              lp[3 * kLossPartials + et] = 0.f;
        }
      }
      ok = phase_done();
    }
    // phase 7: gradient assembly with the per-CTA sum of squares
    if (ok) ok = phase_begin(7);
    if (ok) {
      float sq = phase_reduce(p.ra, et);
      sq = warp_sum(sq);
      if (lane == 0) red[et / kWarp] = sq;
      ok = epi_sync();
      if (ok && et == 0) {
        double t = 0.0;
        for (int w = 0; w < kEW; ++w) t += (double)red[w];
        p.sq_part[blockIdx.x] = t;
      }
      if (ok) ok = phase_done();
    }
    // phase 8: clip + Adam
    if (ok && p.do_adam) {
      ok = phase_begin(8);
      if (ok) {
        if (et < kWarp) {
          double ss = 0.0;
          for (unsigned b = et; b < G; b += kWarp) ss += p.sq_part[b];
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
          if (et == 0) {
            const AdamArgs& a = p.aa;
            const float norm = sqrtf((float)ss);
            red[kEW + 0] = a.max_norm > 0.f ? fminf(1.f, a.max_norm / (norm + 1e-6f)) : 1.f;
            red[kEW + 1] = (float)(1.0 / (1.0 - a.beta_pow[0] * a.b1));
            red[kEW + 2] = (float)(1.0 / (1.0 - a.beta_pow[1] * a.b2));
          }
        }
        ok = epi_sync();
        if (ok) phase_adam(p.aa, et, red[kEW + 0], red[kEW + 1], red[kEW + 2]);
        if (ok) ok = epi_sync();
        if (ok && et == 0) {
          stamp(8);
          // the last CTA out advances the step, the beta powers, and resets
          // the barrier counters for the next launch
          __threadfence();
          const unsigned prev = atomicAdd(gbar + 1, 1u);
          if (prev == G - 1) {
            const AdamArgs& a = p.aa;
            *a.step += 1;
            a.beta_pow[0] *= a.b1;
            a.beta_pow[1] *= a.b2;
            a.beta_pow[2] = 1.0 / (1.0 - a.beta_pow[0] * a.b1);   // next step's corrections
            a.beta_pow[3] = 1.0 / (1.0 - a.beta_pow[1] * a.b2);
            gbar[0] = 0u;
            gbar[1] = 0u;
            __threadfence();
          }
        }
      }
    } else if (ok && et == 0) {
      stamp(7);
      __threadfence();
      const unsigned prev = atomicAdd(gbar + 1, 1u);
      if (prev == G - 1) {
        gbar[0] = 0u;
        gbar[1] = 0u;
        __threadfence();
      }
    }
  }

  __syncthreads();
  if (*abort_flag) {
    if (threadIdx.x == 0) {
      const uint32_t issued = cnt[0], consumed = cnt[1];
      for (uint32_t it = consumed; it < issued; ++it)
        drain_wait(cb.full(it % kS), (it / kS) & 1, p.timeout_ns);
    }
    if (warp == 1 && lane == 0) {
      tc_commit(cb.drain());
      drain_wait(cb.drain(), 0, p.timeout_ns);
    }
    __syncthreads();
  }
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace

cudaError_t mk_prepare() {
  return cudaFuncSetAttribute(mk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              (int)kMkSmem);
}

int mk_grid(int num_sms) { return num_sms; }

cudaError_t mk_launch(const MkLaunch& L, cudaStream_t st) {
  MkMaps maps;
  MkParams p{};
  p.s = L.s;
  p.ga = L.ga;
  p.per_row = L.s.Dp / 8;
  const GemmOperands* ops[5] = {&L.fwd1, &L.fwd2, &L.loss, &L.dact2, &L.dact1};
  const int epis[5] = {EPI_BIAS_ACT, EPI_BIAS_ACT, EPI_LOSS, EPI_DACT, EPI_DACT};
  const float* biases[5] = {L.b1, L.b2, L.b3, nullptr, nullptr};
  __nv_bfloat16* outs[5] = {L.H1, L.H2, nullptr, L.dP2, L.dP1};
  const __nv_bfloat16* auxs[5] = {nullptr, nullptr, nullptr, L.H2, L.H1};
  float* colsums[5] = {nullptr, nullptr, L.cs3, L.cs2, L.cs1};
  for (int i = 0; i < 5; ++i) {
    const GemmOperands& o = *ops[i];
    MkGemm& m = p.g[i];
    m.M = o.M;
    m.N = o.N;
    m.K = o.K;
    m.BN = epis[i] == EPI_LOSS ? o.N : (o.N % 256 == 0 ? 256 : (o.N % 128 == 0 ? 128 : 64));
    m.tiles_m = (o.M + BM - 1) / BM;
    m.tiles_n = o.N / m.BN;
    m.k_tiles = (o.K + BK - 1) / BK;
    m.last_k_steps = (o.K - (m.k_tiles - 1) * BK + 15) / 16;
    m.epi = epis[i];
    m.bias = biases[i];
    m.out = outs[i];
    m.ldo = o.N;
    m.aux = auxs[i];
    m.ldaux = o.N;
    m.colsum_part = colsums[i];
    m.epi_n = o.N;
    cudaError_t e = tc_make_tmap(&maps.a[i], o.A, o.lda, o.M, o.lda, BK, BM);
    if (e != cudaSuccess) return e;
    e = tc_make_tmap(&maps.b[i], o.B, o.ldb, o.N, o.ldb, BK, m.BN);
    if (e != cudaSuccess) return e;
  }
  // weight-gradient regions (MN-major operands)
  p.w = WParams{};
  p.w.nreg = 3;
  p.w.mn_lbo = 8192;
  p.w.mn_sbo = 1024;
  int unit = 0;
  for (int r = 0; r < 3; ++r) {
    const WGradRegion& G = L.wg[r];
    cudaError_t e = tc_make_tmap(&maps.u[r], G.U, G.M, L.rows, G.ldu, 64, BK);
    if (e != cudaSuccess) return e;
    e = tc_make_tmap(&maps.v[r], G.V, G.N, L.rows, G.ldv, 64, BK);
    if (e != cudaSuccess) return e;
    WRegion& R = p.w.r[r];
    R.M = G.M;
    R.N = G.N;
    R.bn = G.N % 128 == 0 ? 128 : 64;
    R.tiles_m = G.M / BM;
    R.tiles_n = G.N / R.bn;
    R.k_tiles = (L.rows + BK - 1) / BK;
    R.kt_per_split = G.kt_per_split;
    R.splits = (R.k_tiles + R.kt_per_split - 1) / R.kt_per_split;
    R.unit_begin = unit;
    R.part = G.part;
    unit += R.tiles_m * R.tiles_n * R.splits;
  }
  p.w.total_units = unit;
  p.ra = L.ra;
  p.do_adam = L.do_adam;
  p.aa = L.aa;
  p.lc = L.lc;
  p.rows = L.rows_in;
  p.inv_mb = L.inv_mb;
  p.logstd = L.logstd;
  p.loss_part = L.loss_part;
  p.dz = L.dz;
  p.lddz = L.lddz;
  p.gbar = L.gbar;
  p.sq_part = L.sq_part;
  p.phase_ns = L.phase_ns;
  p.err = L.err;
  p.timeout_ns = L.timeout_ns;

  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(L.grid);
  cfg.blockDim = dim3(kMkThreads);
  cfg.dynamicSmemBytes = kMkSmem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, mk_kernel, maps, p);
}

int mk_wgrad_bn(int N) { return N % 128 == 0 ? 128 : 64; }

}  // namespace ppo
