// gemm_simt.cu -- fp32 CUDA-core (FFMA) GEMMs of the MLP actor-critic: the
// precision = fp32 mode, where every product and sum stays in fp32 so that
// gradients agree with an fp64 reference to ~1e-6.  Same epilogues as the
// tensor-core path; used for small networks where the tensor cores would
// mostly idle.
#include "common.cuh"
#include "gemm.h"

namespace ppo {

namespace {

constexpr int ST = 64;        // output tile (rows and columns)
constexpr int SK = 16;        // k tile
constexpr int kSimtThreads = 256;

enum { S_BIAS_ACT = 0, S_DACT = 1, S_WGRAD = 2 };

struct SimtEpi {
  const float* bias;
  int act;
  float* out;
  int ldo;
  const float* aux;
  int ldaux;
  float* colsum_part;   // [tiles_m][N]
  float* part;          // [split][M][N]
  int k_per_split;
};

template <int EPI>
__global__ void __launch_bounds__(kSimtThreads) simt_gemm_kernel(SimtOperands g, SimtEpi e) {
  __shared__ float As[SK][ST + 1];
  __shared__ float Bs[SK][ST + 1];
  __shared__ float red[16][ST];
  const int tm = blockIdx.y, tn = blockIdx.x, split = blockIdx.z;
  const int tx = threadIdx.x % 16, ty = threadIdx.x / 16;
  int k0 = 0, k1 = g.K;
  if (EPI == S_WGRAD) {
    k0 = split * e.k_per_split;
    k1 = min(g.K, k0 + e.k_per_split);
  }
  float acc[4][4] = {};
  for (int kb = k0; kb < k1; kb += SK) {
#pragma unroll
    for (int i = 0; i < (SK * ST) / kSimtThreads; ++i) {
      const int idx = threadIdx.x + i * kSimtThreads;
      const int kk = idx / ST, mm = idx % ST;
      const int k = kb + kk;
      const int m = tm * ST + mm, n = tn * ST + mm;
      As[kk][mm] = (k < k1 && m < g.M) ? g.A[m * g.sam + k * g.sak] : 0.f;
      Bs[kk][mm] = (k < k1 && n < g.N) ? g.B[n * g.sbn + k * g.sbk] : 0.f;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < SK; ++kk) {
      float a[4], b[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) a[i] = As[kk][ty * 4 + i];
#pragma unroll
      for (int j = 0; j < 4; ++j) b[j] = Bs[kk][tx * 4 + j];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
    }
    __syncthreads();
  }
  float cs[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int m = tm * ST + ty * 4 + i;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int n = tn * ST + tx * 4 + j;
      if (m >= g.M || n >= g.N) continue;
      float y = acc[i][j];
      if (EPI == S_BIAS_ACT) {
        const float x = y + e.bias[n];
        e.out[(int64_t)m * e.ldo + n] = e.act == 0 ? tanhf(x) : fmaxf(x, 0.f);
      } else if (EPI == S_DACT) {
        const float h = e.aux[(int64_t)m * e.ldaux + n];
        const float d = e.act == 0 ? 1.f - h * h : (h > 0.f ? 1.f : 0.f);
        y *= d;
        e.out[(int64_t)m * e.ldo + n] = y;
        cs[j] += y;
      } else {
        e.part[((int64_t)split * g.M + m) * g.N + n] = y;
      }
    }
  }
  if (EPI == S_DACT) {
#pragma unroll
    for (int j = 0; j < 4; ++j) red[ty][tx * 4 + j] = cs[j];
    __syncthreads();
    if (threadIdx.x < ST) {
      float s = 0.f;
      for (int r = 0; r < 16; ++r) s += red[r][threadIdx.x];
      const int n = tn * ST + threadIdx.x;
      if (n < g.N) e.colsum_part[(int64_t)tm * g.N + n] = s;
    }
  }
}

constexpr int kHeadThreads = 128;

__global__ void __launch_bounds__(kHeadThreads)
simt_head_loss_kernel(NetShape s, LossCoef lc, LossRows rows, float inv_mb,
                      const float* __restrict__ H2, const float* __restrict__ W3,
                      const float* __restrict__ b3, const float* __restrict__ logstd, int mb,
                      float* __restrict__ dz_out, float* __restrict__ colsum_part,
                      float* __restrict__ loss_part) {
  __shared__ float cs[kHeadThreads / kWarp][32];
  __shared__ float lp[kHeadThreads / kWarp][kLossPartials];
  const int row = blockIdx.x * kHeadThreads + threadIdx.x;
  const int warp = threadIdx.x / kWarp, lane = threadIdx.x % kWarp;
  float z[32], dz[32], t6[6] = {0, 0, 0, 0, 0, 0}, dls[4] = {0, 0, 0, 0};
#pragma unroll
  for (int c = 0; c < 32; ++c) {
    z[c] = 0.f;
    dz[c] = 0.f;
  }
  if (row < mb) {
    const float* h = H2 + (int64_t)row * s.H2;
    for (int c = 0; c < s.C; ++c) {
      float acc = 0.f;
      for (int k = 0; k < s.H2; ++k) acc = fmaf(__ldg(W3 + (int64_t)c * s.H2 + k), h[k], acc);
      z[c] = acc + b3[c];
    }
    row_loss(s, lc, inv_mb, z, rows.act + (int64_t)row * s.NH, rows.actc + (int64_t)row * s.G,
             logstd, rows.logp_old[row], rows.adv[row], rows.ret[row], dz, t6, dls);
    for (int c = 0; c < s.CP; ++c) dz_out[(int64_t)row * s.CP + c] = dz[c];
  }
  cs[warp][lane] = warp_reduce_scatter32(dz);
#pragma unroll
  for (int k = 0; k < 6; ++k) {
    const float v = warp_sum(t6[k]);
    if (lane == 0) lp[warp][k] = v;
  }
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const float v = warp_sum(dls[k]);
    if (lane == 0) lp[warp][6 + k] = v;
  }
  if (lane == 0) {
    lp[warp][10] = 0.f;
    lp[warp][11] = 0.f;
  }
  __syncthreads();
  if (threadIdx.x < s.CP) {
    float v = 0.f;
    for (int w = 0; w < kHeadThreads / kWarp; ++w) v += cs[w][threadIdx.x];
    colsum_part[(int64_t)blockIdx.x * s.CP + threadIdx.x] = v;
  }
  if (threadIdx.x < kLossPartials) {
    float v = 0.f;
    for (int w = 0; w < kHeadThreads / kWarp; ++w) v += lp[w][threadIdx.x];
    loss_part[(int64_t)blockIdx.x * kLossPartials + threadIdx.x] = v;
  }
}

}  // namespace

int simt_tiles_m(int M) { return (M + ST - 1) / ST; }
int simt_head_blocks(int mb) { return (mb + kHeadThreads - 1) / kHeadThreads; }

cudaError_t simt_bias_act(const SimtOperands& g, const float* bias, int act, float* out, int ldo,
                          cudaStream_t st) {
  SimtEpi e{};
  e.bias = bias;
  e.act = act;
  e.out = out;
  e.ldo = ldo;
  dim3 grid((g.N + ST - 1) / ST, (g.M + ST - 1) / ST, 1);
  simt_gemm_kernel<S_BIAS_ACT><<<grid, kSimtThreads, 0, st>>>(g, e);
  return cudaGetLastError();
}

cudaError_t simt_dact(const SimtOperands& g, const float* aux, int ldaux, int act, float* out,
                      int ldo, float* colsum_part, cudaStream_t st) {
  SimtEpi e{};
  e.aux = aux;
  e.ldaux = ldaux;
  e.act = act;
  e.out = out;
  e.ldo = ldo;
  e.colsum_part = colsum_part;
  dim3 grid((g.N + ST - 1) / ST, (g.M + ST - 1) / ST, 1);
  simt_gemm_kernel<S_DACT><<<grid, kSimtThreads, 0, st>>>(g, e);
  return cudaGetLastError();
}

cudaError_t simt_wgrad(const SimtOperands& g, int k_per_split, float* part, cudaStream_t st) {
  SimtEpi e{};
  e.part = part;
  e.k_per_split = k_per_split;
  const int splits = (g.K + k_per_split - 1) / k_per_split;
  dim3 grid((g.N + ST - 1) / ST, (g.M + ST - 1) / ST, splits);
  simt_gemm_kernel<S_WGRAD><<<grid, kSimtThreads, 0, st>>>(g, e);
  return cudaGetLastError();
}

cudaError_t simt_head_loss(const NetShape& s, LossCoef lc, LossRows rows, float inv_mb,
                           const float* H2, const float* W3, const float* b3,
                           const float* logstd, int mb, float* dz, float* colsum_part,
                           float* loss_part, cudaStream_t st, int* blocks_out) {
  const int blocks = simt_head_blocks(mb);
  simt_head_loss_kernel<<<blocks, kHeadThreads, 0, st>>>(s, lc, rows, inv_mb, H2, W3, b3, logstd,
                                                         mb, dz, colsum_part, loss_part);
  if (blocks_out) *blocks_out = blocks;
  return cudaGetLastError();
}

}  // namespace ppo
