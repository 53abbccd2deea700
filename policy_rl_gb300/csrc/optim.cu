// optim.cu -- gradient assembly, gradient-norm clip, fused Adam and Muon.
//
// reduce: sums the split-K weight-gradient partials and the per-CTA bias /
// loss partials in a fixed order into the flat fp32 gradient (deterministic).
// sqnorm + adam: "PlayTrain", Table 8 (PPO column): Adam with gradient-norm
// clip.  The squared norm is reduced per block in fp64 and summed in a fixed
// order by every Adam block; Adam then streams p, g, m, v once and
// writes p, m, v and the bf16 weight shadows the tensor-core GEMMs read,
// one coalesced grid-stride pass.
#include <algorithm>
#include <utility>

#include "common.cuh"
#include "gemm.h"
#include "reduce.cuh"
#include "tc_ptx.cuh"

namespace ppo {

namespace {

constexpr int kRedThreads = 256;
constexpr int kNormThreads = 256;
constexpr int kNormBlocks = 152 * 8;
constexpr int kAdamThreads = 256;

// Weight elements: one thread each, summing the split-K partials in split
// order.  Bias / log-std elements and the six loss statistics: one warp each,
// lanes striding over the per-CTA partial rows, then a fixed xor-shuffle tree.
// Every block also writes the sum of squares of the gradient entries it
// produced (fixed order), for the clip norm.
constexpr int kRedWarps = kRedThreads / kWarp;

// Sum of n <= kMaxSplits split-K partials q[0], q[st], ... in split order, with
// every load issued before the first add (one memory latency, not n).
constexpr int kMaxSplits = 64;
__device__ __forceinline__ float split_sum(const float* q, int64_t st, int n) {
  float x[kMaxSplits];
#pragma unroll
  for (int sp = 0; sp < kMaxSplits; ++sp) x[sp] = sp < n ? q[sp * st] : 0.f;
  float v = 0.f;
#pragma unroll
  for (int sp = 0; sp < kMaxSplits; ++sp)
    if (sp < n) v += x[sp];
  return v;
}

// The reduce work of virtual block vb (weight elements for vb < weight_blocks,
// bias / log-std / loss-statistic warps above); writes sq_part[vb].
__device__ __forceinline__ void reduce_block(const ReduceArgs& a, int vb, int weight_blocks) {
  const NetShape& s = a.s;
  const int nW1 = s.H1 * s.D, nW2 = s.H2 * s.H1, nW3 = s.C * s.H2;
  double sq = 0.0;
  if (vb < weight_blocks) {
    const int e = vb * kRedThreads + threadIdx.x;
    float v = 0.f;
    int i = -1;
    if (e < nW1) {
      i = (int)s.oW1 + e;
      const int j = e / s.D, k = e - j * s.D;
      const float* q = a.pW1 + (int64_t)j * a.ld1 + k;
      const int64_t st = (int64_t)s.H1 * a.ld1;
      v = split_sum(q, st, a.s1);
    } else if (e < nW1 + nW2) {
      const int r = e - nW1;
      i = (int)s.oW2 + r;
      const float* q = a.pW2 + r;
      const int64_t st = (int64_t)s.H2 * s.H1;
      v = split_sum(q, st, a.s2);
    } else if (e < nW1 + nW2 + nW3) {
      const int r = e - nW1 - nW2;
      i = (int)s.oW3 + r;
      const int c = r / s.H2, j = r - c * s.H2;
      const float* q = a.pW3t + (int64_t)j * a.ld3 + c;
      const int64_t st = (int64_t)s.H2 * a.ld3;
      v = split_sum(q, st, a.s3);
    }
    if (i >= 0) {
      a.grad[i] = v;
      sq = (double)(v * v);
    }
  } else {
    const int warp = threadIdx.x / kWarp;
    sq = reduce_vector_task(a, (vb - weight_blocks) * kRedWarps + warp);
  }
  if (a.sq_part != nullptr) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sq += __shfl_xor_sync(0xffffffffu, sq, o);
    __shared__ double ws[kRedWarps];
    if (threadIdx.x % kWarp == 0) ws[threadIdx.x / kWarp] = sq;
    __syncthreads();
    if (threadIdx.x == 0) {
      double t = 0.0;
      for (int w = 0; w < kRedWarps; ++w) t += ws[w];
      a.sq_part[vb] = t;
    }
  }
}

__global__ void __launch_bounds__(kRedThreads) reduce_kernel(ReduceArgs a, int weight_blocks) {
  pdl_wait();
  pdl_trigger();
  reduce_block(a, blockIdx.x, weight_blocks);
}

__global__ void __launch_bounds__(kNormThreads)
sqnorm_kernel(const float* __restrict__ g, int64_t P, double* __restrict__ part) {
  pdl_wait();
  pdl_trigger();
  // fp32 within a thread (a few hundred terms at most), fp64 across threads
  float sf = 0.f;
  const int64_t P4 = P / 4;
  const int64_t stride = (int64_t)gridDim.x * kNormThreads;
#pragma unroll 4
  for (int64_t i = (int64_t)blockIdx.x * kNormThreads + threadIdx.x; i < P4; i += stride) {
    const float4 x = __ldcs(reinterpret_cast<const float4*>(g) + i);
    sf = fmaf(x.x, x.x, fmaf(x.y, x.y, fmaf(x.z, x.z, fmaf(x.w, x.w, sf))));
  }
  for (int64_t i = P4 * 4 + (int64_t)blockIdx.x * kNormThreads + threadIdx.x; i < P; i += stride)
    sf = fmaf(g[i], g[i], sf);
  double s = (double)sf;
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

// write_shadow for the four consecutive parameters i0..i0+3 (region starts are
// multiples of 4 in bf16 mode): one row/column division, then increments.
__device__ __forceinline__ void write_shadow4(const NetShape& s, const Shadows& sh, int i0,
                                              float4 p4) {
  const float pv[4] = {p4.x, p4.y, p4.z, p4.w};
  if (i0 < (int)s.ob1) {
    const int r = i0 - (int)s.oW1;
    int j = r / s.D, k = r - j * s.D;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      if (i0 + e < (int)s.ob1) sh.W1s[j * s.Dp + k] = __float2bfloat16_rn(pv[e]);
      if (++k == s.D) { k = 0; ++j; }
    }
  } else if (i0 >= (int)s.oW2 && i0 < (int)s.ob2) {
    const int r = i0 - (int)s.oW2;
    int j = r / s.H1, k = r - j * s.H1;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const __nv_bfloat16 b = __float2bfloat16_rn(pv[e]);
      sh.W2s[r + e] = b;
      sh.W2Ts[k * s.H2 + j] = b;
      if (++k == s.H1) { k = 0; ++j; }
    }
  } else if (i0 >= (int)s.oW3 && i0 < (int)s.ob3) {
    const int r = i0 - (int)s.oW3;
    int c = r / s.H2, j = r - c * s.H2;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const __nv_bfloat16 b = __float2bfloat16_rn(pv[e]);
      sh.W3s[r + e] = b;
      sh.W3Ts[j * sh.ld3t + c] = b;
      if (++j == s.H2) { j = 0; ++c; }
    }
  }
}

// Clip + Adam over the grid-stride share of block `block` of `nblocks`; the
// last block to finish publishes the step count and the beta powers (and
// clears *extra_ctr when given).
__device__ __forceinline__ void adam_body(const AdamArgs& a, int block, int nblocks,
                                          unsigned* extra_ctr) {
  __shared__ float s_coef, s_norm, s_ibc1, s_ibc2;
  __shared__ long long s_t;
  __shared__ double s_ws[kAdamThreads / kWarp];
  {
    // every block sums the norm partials in the same fixed order
    double ss = 0.0;
    for (int b = threadIdx.x; b < a.nsq; b += kAdamThreads) ss += a.sq_part[b];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    if (threadIdx.x % kWarp == 0) s_ws[threadIdx.x / kWarp] = ss;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    double ss = 0.0;
    for (int w = 0; w < kAdamThreads / kWarp; ++w) ss += s_ws[w];
    const float norm = sqrtf((float)ss);
    float coef = 1.f;
    if (a.max_norm > 0.f) coef = fminf(1.f, a.max_norm / (norm + 1e-6f));
    s_coef = coef;
    s_norm = norm;
    s_t = (long long)(*a.step) + 1;
    // bias corrections 1 / (1 - beta^t), computed in double by the block that
    // finished the previous step (no pow(), no division on this path)
    s_ibc1 = (float)a.beta_pow[2];
    s_ibc2 = (float)a.beta_pow[3];
  }
  __syncthreads();
  const float coef = s_coef, ibc1 = s_ibc1, ibc2 = s_ibc2;
  const float b1 = (float)a.b1, b2 = (float)a.b2, omb1 = a.omb1, omb2 = a.omb2;
  const float lr = a.lr, eps = a.eps;
  const bool shadows = a.sh.W1s != nullptr;
  const int P = (int)a.P;
  const int P4 = P / 4;
  const int stride = nblocks * kAdamThreads;
  auto step = [&](float g, float m0, float v0, float p0, float& m, float& v, float& p) {
    g *= coef;
    m = b1 * m0 + omb1 * g;
    v = b2 * v0 + omb2 * g * g;
    p = p0 - lr * (m * ibc1) / (sqrtf(v * ibc2) + eps);
  };
  if (a.vectors_only) {
    // biases and log-std only: b1 [H1], b2 [H2], b3 [C] + log-std [G]
    const int n1 = a.s.H1, n2 = a.s.H2, n3 = a.s.C + a.s.G;
    for (int j = block * kAdamThreads + threadIdx.x; j < n1 + n2 + n3; j += stride) {
      const int i = j < n1 ? (int)a.s.ob1 + j
                           : (j < n1 + n2 ? (int)a.s.ob2 + (j - n1) : (int)a.s.ob3 + (j - n1 - n2));
      float m, v, p;
      step(a.g[i], a.m[i], a.v[i], a.p[i], m, v, p);
      a.m[i] = m;
      a.v[i] = v;
      a.p[i] = p;
    }
  } else {
  const float4* __restrict__ G4 = reinterpret_cast<const float4*>(a.g);
  float4* __restrict__ M4 = reinterpret_cast<float4*>(a.m);
  float4* __restrict__ V4 = reinterpret_cast<float4*>(a.v);
  float4* __restrict__ PP4 = reinterpret_cast<float4*>(a.p);
#pragma unroll 2
  for (int i = block * kAdamThreads + threadIdx.x; i < P4; i += stride) {
    const float4 g4 = __ldcs(G4 + i);
    const float4 m4 = __ldcs(M4 + i);
    const float4 v4 = __ldcs(V4 + i);
    const float4 p4 = __ldcs(PP4 + i);
    float4 mo, vo, po;
    step(g4.x, m4.x, v4.x, p4.x, mo.x, vo.x, po.x);
    step(g4.y, m4.y, v4.y, p4.y, mo.y, vo.y, po.y);
    step(g4.z, m4.z, v4.z, p4.z, mo.z, vo.z, po.z);
    step(g4.w, m4.w, v4.w, p4.w, mo.w, vo.w, po.w);
    __stcs(M4 + i, mo);
    __stcs(V4 + i, vo);
    __stcs(PP4 + i, po);
    if (shadows) write_shadow4(a.s, a.sh, 4 * i, po);
  }
  for (int i = P4 * 4 + block * kAdamThreads + threadIdx.x; i < P; i += stride) {
    float m, v, p;
    step(a.g[i], a.m[i], a.v[i], a.p[i], m, v, p);
    a.m[i] = m;
    a.v[i] = v;
    a.p[i] = p;
    if (shadows) write_shadow(a.s, a.sh, i, p);
  }
  }
  // the last block to finish publishes the new step count (every block has
  // read the old one before its arrival)
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    const unsigned prev = atomicAdd(a.done_ctr, 1u);
    if (prev == (unsigned)nblocks - 1) {
      *a.step = (int64_t)s_t;
      a.beta_pow[0] *= a.b1;
      a.beta_pow[1] *= a.b2;
      a.beta_pow[2] = 1.0 / (1.0 - a.beta_pow[0] * a.b1);   // next step's corrections
      a.beta_pow[3] = 1.0 / (1.0 - a.beta_pow[1] * a.b2);
      if (a.grad_norm_out) *a.grad_norm_out = s_norm;
      *a.done_ctr = 0u;
      if (extra_ctr) *extra_ctr = 0u;
      __threadfence();
    }
  }
}

__global__ void __launch_bounds__(kAdamThreads) adam_kernel(AdamArgs a) {
  pdl_wait();
  pdl_trigger();
  adam_body(a, blockIdx.x, gridDim.x, nullptr);
}

// ---- Muon ("Muon: An optimizer for hidden layers in neural networks") -------
// Newton-Schulz on X (r x k, r <= k): five times A = X X^T, B = b A + c A A,
// X = a X + B X.  Each product is one launch over the tiles of all three
// matrices (fp32 CUDA cores: the matrices are at most 512 x 1408 and the
// products are latency-bound).
constexpr float kNsA = 3.4445f, kNsB = -4.7750f, kNsC = 2.0315f;
constexpr int kNsTile = 32;
constexpr int kNsChunk = 128;   // reduction elements staged per round (all loads in flight)
constexpr int kNsThreads = 256;

// Momentum update of the matrices and the Frobenius partials of u:
//   g' = coef g (clip), mom = beta mom + g', u = g' + beta mom,
// u stored as X0 [r][k] (transposed when the matrix has more rows than columns).
__global__ void __launch_bounds__(kAdamThreads) muon_prep_kernel(MuonArgs mu, AdamArgs a) {
  pdl_wait();
  __shared__ float s_coef;
  __shared__ double s_ws[kAdamThreads / kWarp];
  {
    double ss = 0.0;
    for (int b = threadIdx.x; b < a.nsq; b += kAdamThreads) ss += a.sq_part[b];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    if (threadIdx.x % kWarp == 0) s_ws[threadIdx.x / kWarp] = ss;
  }
  __syncthreads();
  if (threadIdx.x == 0) {   // the same coefficient adam_body computes
    double ss = 0.0;
    for (int w = 0; w < kAdamThreads / kWarp; ++w) ss += s_ws[w];
    const float norm = sqrtf((float)ss);
    s_coef = a.max_norm > 0.f ? fminf(1.f, a.max_norm / (norm + 1e-6f)) : 1.f;
  }
  __syncthreads();
  pdl_trigger();
  const float coef = s_coef;
  __shared__ float s_red[3][kAdamThreads / kWarp];
  for (int mtx = 0; mtx < 3; ++mtx) {
    const MuonMat& m = mu.m[mtx];
    const int n = m.rows * m.cols;
    const bool tr = m.rows > m.cols;
    const int k = tr ? m.rows : m.cols;
    float acc = 0.f;
    for (int i = blockIdx.x * kAdamThreads + threadIdx.x; i < n; i += gridDim.x * kAdamThreads) {
      const float g = m.g[i] * coef;
      const float mo = mu.beta * m.mom[i] + g;
      m.mom[i] = mo;
      const float u = g + mu.beta * mo;
      const int row = i / m.cols, col = i - row * m.cols;
      m.X0[tr ? (int64_t)col * k + row : (int64_t)row * k + col] = u;
      acc = fmaf(u, u, acc);
    }
    acc = warp_sum(acc);
    if (threadIdx.x % kWarp == 0) s_red[mtx][threadIdx.x / kWarp] = acc;
  }
  __syncthreads();
  if (threadIdx.x < 3) {
    float t = 0.f;
    for (int w = 0; w < kAdamThreads / kWarp; ++w) t += s_red[threadIdx.x][w];
    mu.mpart[threadIdx.x * kMuonPrepBlocks + blockIdx.x] = t;
  }
}

// inv[m] = 1 / (||u_m||_F + 1e-7), partials summed in block order.
__global__ void muon_norm_kernel(MuonArgs mu) {
  pdl_wait();
  pdl_trigger();
  if (threadIdx.x < 3) {
    float t = 0.f;
    for (int b = 0; b < kMuonPrepBlocks; ++b) t += mu.mpart[threadIdx.x * kMuonPrepBlocks + b];
    mu.inv[threadIdx.x] = 1.f / (sqrtf(t) + 1e-7f);
  }
}

// One Newton-Schulz product over the tiles of all three matrices:
//   stage 0: A = s^2 X X^T;  stage 1: B = b A + c A A;  stage 2: Xo = a s X + B (s X),
// with s = inv[m] on the first iteration (X = X0 unnormalised) and 1 after.
struct NsStage {
  int stage;
  int first;                 // first iteration: scale X by inv[m]
  const float* src[3];       // X of this iteration per matrix
  float* dst[3];             // Xo (stage 2)
  int tiles[4];              // prefix sums of the tile counts over the matrices
};

__global__ void __launch_bounds__(kNsThreads) ns_stage_kernel(MuonArgs mu, NsStage st) {
  pdl_wait();
  __shared__ float Ps[kNsTile][kNsChunk + 1], Qs[kNsTile][kNsChunk + 1];
  const int b = blockIdx.x;
  const int mtx = b < st.tiles[1] ? 0 : (b < st.tiles[2] ? 1 : 2);
  const MuonMat& m = mu.m[mtx];
  const int r = m.rows < m.cols ? m.rows : m.cols;
  const int kk = m.rows < m.cols ? m.cols : m.rows;
  const float* X = st.src[mtx];
  const float s = st.first ? mu.inv[mtx] : 1.f;
  // output [Mo][No], reduction length K, operands P(i, q) and Q(j, q)
  int No, K;
  const float *P, *Q, *D = nullptr;
  int64_t pi, pq, qj, qq;
  float alpha = 0.f, beta;
  float* out;
  if (st.stage == 0) {          // A[i][j] = sum_q X[i][q] X[j][q]
    No = r; K = kk; P = X; Q = X; pi = kk; pq = 1; qj = kk; qq = 1; beta = s * s; out = m.A;
  } else if (st.stage == 1) {   // B[i][j] = b A[i][j] + c sum_q A[i][q] A[q][j] (A symmetric)
    No = r; K = r; P = m.A; Q = m.A; pi = r; pq = 1; qj = r; qq = 1;
    D = m.A; alpha = kNsB; beta = kNsC; out = m.B;
  } else {                      // Xo[i][j] = a s X[i][j] + s sum_q B[i][q] X[q][j]
    No = kk; K = r; P = m.B; Q = X; pi = r; pq = 1; qj = 1; qq = kk;
    D = X; alpha = kNsA * s; beta = s; out = st.dst[mtx];
  }
  const int tn = (No + kNsTile - 1) / kNsTile;
  const int t = b - st.tiles[mtx];
  const int i0 = (t / tn) * kNsTile, j0 = (t % tn) * kNsTile;
  const int Mo = r;
  // each thread: a 2 x 2 block of the 32 x 32 tile
  const int ty = threadIdx.x / 16, tx = threadIdx.x % 16;
  float acc[2][2] = {{0.f, 0.f}, {0.f, 0.f}};
  constexpr int kPer = kNsTile * kNsChunk / kNsThreads;   // elements per thread per operand
  for (int q0 = 0; q0 < K; q0 += kNsChunk) {
    float pv[kPer], qv[kPer];
#pragma unroll
    for (int u = 0; u < kPer; ++u) {   // every load of the round before any store
      const int e = threadIdx.x + u * kNsThreads;
      const int rr = e / kNsChunk, qc = e % kNsChunk;
      const int q = q0 + qc;
      pv[u] = (i0 + rr < Mo && q < K) ? P[(int64_t)(i0 + rr) * pi + (int64_t)q * pq] : 0.f;
      qv[u] = (j0 + rr < No && q < K) ? Q[(int64_t)(j0 + rr) * qj + (int64_t)q * qq] : 0.f;
    }
#pragma unroll
    for (int u = 0; u < kPer; ++u) {
      const int e = threadIdx.x + u * kNsThreads;
      Ps[e / kNsChunk][e % kNsChunk] = pv[u];
      Qs[e / kNsChunk][e % kNsChunk] = qv[u];
    }
    __syncthreads();
#pragma unroll 8
    for (int qc = 0; qc < kNsChunk; ++qc) {
      const float p0 = Ps[2 * ty][qc], p1 = Ps[2 * ty + 1][qc];
      const float q0v = Qs[2 * tx][qc], q1v = Qs[2 * tx + 1][qc];
      acc[0][0] = fmaf(p0, q0v, acc[0][0]);
      acc[0][1] = fmaf(p0, q1v, acc[0][1]);
      acc[1][0] = fmaf(p1, q0v, acc[1][0]);
      acc[1][1] = fmaf(p1, q1v, acc[1][1]);
    }
    __syncthreads();
  }
  pdl_trigger();
#pragma unroll
  for (int u = 0; u < 2; ++u)
#pragma unroll
    for (int v = 0; v < 2; ++v) {
      const int i = i0 + 2 * ty + u, j = j0 + 2 * tx + v;
      if (i < Mo && j < No) {
        float y = beta * acc[u][v];
        if (D) y = fmaf(alpha, D[(int64_t)i * No + j], y);
        out[(int64_t)i * No + j] = y;
      }
    }
}

// W -= lr sqrt(max(1, rows/cols)) X (transposed back), bf16 shadows refreshed.
// Five iterations ping-pong X0 -> X1 -> X0 -> X1 -> X0 -> X1: the result is X1.
__global__ void __launch_bounds__(kAdamThreads) muon_apply_kernel(MuonArgs mu) {
  pdl_wait();
  pdl_trigger();
  const bool shadows = mu.sh.W1s != nullptr;
  for (int mtx = 0; mtx < 3; ++mtx) {
    const MuonMat& m = mu.m[mtx];
    const int n = m.rows * m.cols;
    const bool tr = m.rows > m.cols;
    const int k = tr ? m.rows : m.cols;
    const float ratio = (float)m.rows / (float)m.cols;
    const float step = mu.lr * sqrtf(ratio > 1.f ? ratio : 1.f);
    const float* X = m.X1;
    for (int i = blockIdx.x * kAdamThreads + threadIdx.x; i < n; i += gridDim.x * kAdamThreads) {
      const int row = i / m.cols, col = i - row * m.cols;
      const float x = X[tr ? (int64_t)col * k + row : (int64_t)row * k + col];
      const float p = m.p[i] - step * x;
      m.p[i] = p;
      if (shadows) write_shadow(mu.s, mu.sh, (int)(m.off + i), p);
    }
  }
}

__device__ __forceinline__ unsigned ld_acquire_u32(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Gradient assembly, then clip + Adam, in one cooperative launch: the grid
// reduces the split-K / per-CTA partials (virtual blocks 0..nvb), meets at a
// grid barrier (bounded: on expiry it latches kDevTimeout and skips Adam), then
// runs Adam with the norm of all nvb partial sums.  Same arithmetic and order
// as reduce_kernel followed by adam_kernel.
__global__ void __launch_bounds__(kRedThreads)
reduce_adam_kernel(ReduceArgs ra, AdamArgs aa, int weight_blocks, int nvb, unsigned* bar,
                   int* err, uint64_t limit_ns) {
  __shared__ int s_abort;
  for (int vb = blockIdx.x; vb < nvb; vb += gridDim.x) {
    reduce_block(ra, vb, weight_blocks);
    __syncthreads();   // the block's shared partials are reused by the next virtual block
  }
  if (threadIdx.x == 0) {
    s_abort = 0;
    __threadfence();
    atomicAdd(bar, 1u);
    if (ld_acquire_u32(bar) < gridDim.x) {
      const uint64_t t0 = ptx::globaltimer();
      while (ld_acquire_u32(bar) < gridDim.x) {
        if (ptx::globaltimer() - t0 > limit_ns) {
          atomicOr(err, kDevTimeout);
          s_abort = 1;
          break;
        }
      }
    }
    __threadfence();
  }
  __syncthreads();
  if (s_abort) return;
  aa.nsq = ra.nsq_pre + nvb;   // the weight-gradient kernel's partials come first
  adam_body(aa, blockIdx.x, gridDim.x, bar);
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

static int reduce_weight_blocks(const NetShape& s) {
  const int64_t nW = (int64_t)s.H1 * s.D + (int64_t)s.H2 * s.H1 + (int64_t)s.C * s.H2;
  return (int)((nW + kRedThreads - 1) / kRedThreads);
}

static int reduce_vector_blocks(const NetShape& s) {
  return (reduce_vector_tasks(s) + kRedWarps - 1) / kRedWarps;
}

int reduce_blocks(const NetShape& s) { return reduce_weight_blocks(s) + reduce_vector_blocks(s); }

// blocks of one reduce launch: the weight blocks only when the weight
// entries are not yet assembled
static int reduce_weight_blocks(const ReduceArgs& a) {
  return a.weights_done ? 0 : reduce_weight_blocks(a.s);
}
int reduce_launch_blocks(const ReduceArgs& a) {
  return reduce_weight_blocks(a) + reduce_vector_blocks(a.s);
}

cudaError_t launch_reduce(const ReduceArgs& a, cudaStream_t st) {
  return launch_pdl(reduce_kernel, dim3(reduce_launch_blocks(a)), dim3(kRedThreads), 0, st, a,
                    reduce_weight_blocks(a));
}

int g_reduce_adam_blocks_per_sm = 0;

cudaError_t reduce_adam_prepare() {
  if (g_reduce_adam_blocks_per_sm > 0) return cudaSuccess;
  int n = 0;
  cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, reduce_adam_kernel, kRedThreads, 0);
  if (e != cudaSuccess) return e;
  g_reduce_adam_blocks_per_sm = n < 1 ? 1 : n;
  return cudaSuccess;
}

cudaError_t launch_reduce_adam(const ReduceArgs& ra, const AdamArgs& aa, unsigned* bar, int* err,
                               uint64_t limit_ns, int num_sms, cudaStream_t st) {
  if (g_reduce_adam_blocks_per_sm <= 0) return cudaErrorInitializationError;
  const int nvb = reduce_launch_blocks(ra);
  // up to 4 resident blocks per SM: one virtual block of reduce work each at
  // the usual sizes (one block per SM measured slower: serial reduce work);
  // at least one block per SM for the Adam pass
  int grid = num_sms * (g_reduce_adam_blocks_per_sm < 4 ? g_reduce_adam_blocks_per_sm : 4);
  if (grid > nvb) grid = nvb > num_sms ? nvb : num_sms;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kRedThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = st;
  // cooperative: all blocks resident, they meet at a barrier.  (Adding
  // programmatic serialization to this launch measured 3 % slower per update.)
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, reduce_adam_kernel, ra, aa, reduce_weight_blocks(ra), nvb, bar,
                            err, limit_ns);
}

cudaError_t launch_adam(const AdamArgs& a0, cudaStream_t st, const Trace* tr) {
  AdamArgs a = a0;
  if (a.nsq <= 0) {   // no squared-norm partials supplied: compute them
    const int nb = blocks_for((a.P + 3) / 4, kNormThreads, kNormBlocks);
    cudaError_t e = launch_pdl(sqnorm_kernel, dim3(nb), dim3(kNormThreads), 0, st, a.g, a.P,
                               const_cast<double*>(a.sq_part));
    if (e != cudaSuccess) return e;
    if (tr) tr->mark(ST_SQNORM, st);
    a.nsq = nb;
  }
  cudaError_t e = launch_pdl(adam_kernel, dim3(blocks_for((a.P + 3) / 4, kAdamThreads, 152 * 8)),
                             dim3(kAdamThreads), 0, st, a);
  if (e != cudaSuccess) return e;
  if (tr) tr->mark(ST_ADAM, st);
  return cudaSuccess;
}

namespace {

// X (bf16) = X0 * inv for the tensor-core iteration, and its transpose; the
// padded rows and columns are never written (zero from allocation).
__global__ void __launch_bounds__(kAdamThreads)
muon_pack_kernel(MuonArgs mu, MuonTcMat t0, MuonTcMat t1, MuonTcMat t2) {
  pdl_wait();
  pdl_trigger();
  const MuonTcMat tm[3] = {t0, t1, t2};
  for (int mtx = 0; mtx < 3; ++mtx) {
    const MuonTcMat& t = tm[mtx];
    const float s = mu.inv[mtx];
    const float* X0 = mu.m[mtx].X0;   // [r][k]
    for (int e = blockIdx.x * kAdamThreads + threadIdx.x; e < t.r * t.k;
         e += gridDim.x * kAdamThreads) {
      const int i = e / t.k, j = e - i * t.k;
      const __nv_bfloat16 v = __float2bfloat16_rn(X0[e] * s);
      t.X[(int64_t)i * t.kp + j] = v;
      t.XT[(int64_t)j * t.rp + i] = v;
    }
  }
}

// XT [kp][rp] = X^T of X [rp][kp] (32 x 32 tiles through shared memory).
__global__ void muon_transpose_kernel(const __nv_bfloat16* __restrict__ X,
                                      __nv_bfloat16* __restrict__ XT, int rp, int kp) {
  __shared__ __nv_bfloat16 tile[32][33];
  const int bx = blockIdx.x * 32, by = blockIdx.y * 32;   // column block of X, row block
  pdl_wait();
  pdl_trigger();
  for (int y = threadIdx.y; y < 32; y += blockDim.y) {
    const int i = by + y, j = bx + threadIdx.x;
    if (i < rp && j < kp) tile[y][threadIdx.x] = X[(int64_t)i * kp + j];
  }
  __syncthreads();
  for (int y = threadIdx.y; y < 32; y += blockDim.y) {
    const int j = bx + y, i = by + threadIdx.x;
    if (i < rp && j < kp) XT[(int64_t)j * rp + i] = tile[threadIdx.x][y];
  }
}

// W -= lr sqrt(max(1, rows/cols)) X with the final bf16 X of the tensor-core
// iteration ([rp][kp], transposed back when tall), bf16 shadows refreshed.
__global__ void __launch_bounds__(kAdamThreads)
muon_apply_tc_kernel(MuonArgs mu, const __nv_bfloat16* X0, const __nv_bfloat16* X1,
                     const __nv_bfloat16* X2, int kp0, int kp1, int kp2) {
  pdl_wait();
  pdl_trigger();
  const bool shadows = mu.sh.W1s != nullptr;
  const __nv_bfloat16* Xs[3] = {X0, X1, X2};
  const int kps[3] = {kp0, kp1, kp2};
  for (int mtx = 0; mtx < 3; ++mtx) {
    const MuonMat& m = mu.m[mtx];
    const int n = m.rows * m.cols;
    const bool tr = m.rows > m.cols;
    const float ratio = (float)m.rows / (float)m.cols;
    const float step = mu.lr * sqrtf(ratio > 1.f ? ratio : 1.f);
    for (int i = blockIdx.x * kAdamThreads + threadIdx.x; i < n; i += gridDim.x * kAdamThreads) {
      const int row = i / m.cols, col = i - row * m.cols;
      const float x = __bfloat162float(
          Xs[mtx][tr ? (int64_t)col * kps[mtx] + row : (int64_t)row * kps[mtx] + col]);
      const float p = m.p[i] - step * x;
      m.p[i] = p;
      if (shadows) write_shadow(mu.s, mu.sh, (int)(m.off + i), p);
    }
  }
}

}  // namespace

// Five Newton-Schulz iterations of the three matrices on the tensor cores,
// each matrix's chain on its own side stream:
//   A = X X^T;  B = b A + c A A (A symmetric: A A = A A^T);  X2 = a X + B X
//   (B X = B (X^T)^T, the transpose held in XT);  XT = X2^T;  swap X, X2.
static cudaError_t muon_tc_iterations(const MuonTc& t, cudaStream_t st, __nv_bfloat16** final) {
  cudaError_t e = cudaEventRecord(t.fork, st);
  if (e != cudaSuccess) return e;
  for (int m = 0; m < 3; ++m) {
    const MuonTcMat& q = t.m[m];
    cudaStream_t s = t.side[m];
    if ((e = cudaStreamWaitEvent(s, t.fork, 0)) != cudaSuccess) return e;
    __nv_bfloat16 *X = q.X, *X2 = q.X2;
    for (int it = 0; it < 5; ++it) {
      const uint64_t to = 2000000000ull;
      e = tc_gemm_bias_act(GemmOperands{X, q.kp, X, q.kp, q.rp, q.rp, q.kp}, nullptr, 2, q.A,
                           q.rp, t.err, to, t.num_sms, s);
      if (e == cudaSuccess)
        e = tc_gemm_axpby(GemmOperands{q.A, q.rp, q.A, q.rp, q.rp, q.rp, q.rp}, q.A, q.rp,
                          kNsB, kNsC, q.B, q.rp, t.err, to, t.num_sms, s);
      if (e == cudaSuccess)
        e = tc_gemm_axpby(GemmOperands{q.B, q.rp, q.XT, q.rp, q.rp, q.kp, q.rp}, X, q.kp, kNsA,
                          1.f, X2, q.kp, t.err, to, t.num_sms, s);
      if (e != cudaSuccess) return e;
      if (it < 4) {   // the last iterate is not transposed: apply reads X
        const dim3 grid((unsigned)(q.kp / 32), (unsigned)(q.rp / 32));
        e = launch_pdl(muon_transpose_kernel, grid, dim3(32, 8), 0, s, X2, q.XT, q.rp, q.kp);
        if (e != cudaSuccess) return e;
      }
      std::swap(X, X2);
    }
    final[m] = X;
    if ((e = cudaEventRecord(t.join[m], s)) != cudaSuccess) return e;
    if ((e = cudaStreamWaitEvent(st, t.join[m], 0)) != cudaSuccess) return e;
  }
  return cudaSuccess;
}

cudaError_t launch_muon(const MuonArgs& mu, const AdamArgs& a0, cudaStream_t st,
                        const Trace* tr, const MuonTc* tc) {
  AdamArgs a = a0;
  if (a.nsq <= 0) {   // no squared-norm partials supplied: compute them
    const int nb = blocks_for((a.P + 3) / 4, kNormThreads, kNormBlocks);
    cudaError_t e = launch_pdl(sqnorm_kernel, dim3(nb), dim3(kNormThreads), 0, st, a.g, a.P,
                               const_cast<double*>(a.sq_part));
    if (e != cudaSuccess) return e;
    if (tr) tr->mark(ST_SQNORM, st);
    a.nsq = nb;
  }
  cudaError_t e = launch_pdl(muon_prep_kernel, dim3(kMuonPrepBlocks), dim3(kAdamThreads), 0, st,
                             mu, a);
  if (e != cudaSuccess) return e;
  if (tr) tr->mark(ST_MUON, st);
  // Adam on the biases and log-std; it also advances the step counter
  a.vectors_only = 1;
  e = launch_pdl(adam_kernel, dim3(4), dim3(kAdamThreads), 0, st, a);
  if (e != cudaSuccess) return e;
  if (tr) tr->mark(ST_ADAM, st);
  e = launch_pdl(muon_norm_kernel, dim3(1), dim3(32), 0, st, mu);
  if (e != cudaSuccess) return e;
  if (tr) tr->mark(ST_MUON, st);
  if (tc) {
    e = launch_pdl(muon_pack_kernel, dim3(152), dim3(kAdamThreads), 0, st, mu, tc->m[0],
                   tc->m[1], tc->m[2]);
    if (e != cudaSuccess) return e;
    if (tr) tr->mark(ST_MUON, st);
    __nv_bfloat16* fin[3];
    if ((e = muon_tc_iterations(*tc, st, fin)) != cudaSuccess) return e;
    if (tr) tr->mark(ST_MUON, st);
    e = launch_pdl(muon_apply_tc_kernel,
                   dim3(blocks_for(mu.m[1].rows * mu.m[1].cols, kAdamThreads, 152)),
                   dim3(kAdamThreads), 0, st, mu, (const __nv_bfloat16*)fin[0],
                   (const __nv_bfloat16*)fin[1], (const __nv_bfloat16*)fin[2], tc->m[0].kp,
                   tc->m[1].kp, tc->m[2].kp);
    if (e != cudaSuccess) return e;
    if (tr) tr->mark(ST_MUON, st);
    return cudaSuccess;
  }
  NsStage sg{};
  int ntile[3][3];   // [stage][matrix]
  for (int m = 0; m < 3; ++m) {
    const int r = std::min(mu.m[m].rows, mu.m[m].cols), k = std::max(mu.m[m].rows, mu.m[m].cols);
    const int tr_ = (r + kNsTile - 1) / kNsTile, tk = (k + kNsTile - 1) / kNsTile;
    ntile[0][m] = tr_ * tr_;
    ntile[1][m] = tr_ * tr_;
    ntile[2][m] = tr_ * tk;
  }
  const float* cur[3] = {mu.m[0].X0, mu.m[1].X0, mu.m[2].X0};
  for (int it = 0; it < 5; ++it) {
    for (int stage = 0; stage < 3; ++stage) {
      sg.stage = stage;
      sg.first = it == 0;
      sg.tiles[0] = 0;
      for (int m = 0; m < 3; ++m) {
        sg.src[m] = cur[m];
        sg.dst[m] = cur[m] == mu.m[m].X0 ? mu.m[m].X1 : mu.m[m].X0;
        sg.tiles[m + 1] = sg.tiles[m] + ntile[stage][m];
      }
      e = launch_pdl(ns_stage_kernel, dim3(sg.tiles[3]), dim3(kNsThreads), 0, st, mu, sg);
      if (e != cudaSuccess) return e;
      if (tr) tr->mark(ST_MUON, st);
    }
    for (int m = 0; m < 3; ++m) cur[m] = sg.dst[m];
  }
  e = launch_pdl(muon_apply_kernel, dim3(blocks_for(mu.m[1].rows * mu.m[1].cols, kAdamThreads, 152)),
                 dim3(kAdamThreads), 0, st, mu);
  if (e != cudaSuccess) return e;
  if (tr) tr->mark(ST_MUON, st);
  return cudaSuccess;
}

cudaError_t launch_shadows(const float* p, const NetShape& s, const Shadows& sh, cudaStream_t st) {
  if (sh.W1s == nullptr) return cudaSuccess;
  shadow_kernel<<<blocks_for(s.P, kAdamThreads, 152 * 4), kAdamThreads, 0, st>>>(p, s, sh);
  return cudaGetLastError();
}

}  // namespace ppo
