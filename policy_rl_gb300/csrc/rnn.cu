// rnn.cu -- loss and gradient of the recurrent (MinGRU) policy on CUDA cores.
//
// "Teaching Mario to speedrun", sec. 8 "The Puffer net, and the trainer":
// bias-free encoder, MinGRU layers (gates from the input only; the state
// carries across horizons and clears when an episode ends), one decoder
// matrix to the heads and the value.  MinGRU (Feng et al. 2024): per layer
//   z = sigmoid(W_z u + b_z),  h~ = W_h u + b_h,  h_t = (1 - z) h_{t-1} + z h~,
// with the state entering step t cleared when the episode ended at t - 1.
// A minibatch is a set of environment segments (rows t*ns + j), the gradient
// backpropagation through time inside each segment.
//
// fp32 throughout (correctness-first version): the products are a generic
// tiled GEMM (split-K with fixed-order partial sums for the weight and bias
// gradients, whose reduction runs over all rows); the recurrence runs one thread per (segment, unit) walking
// time forward (and backward for the gradient); the loss is the MLP path's
// per-row epilogue (tc::row_loss_seg) after a thread-per-row decoder.
#include <utility>

#include "common.cuh"
#include "tc_tile.cuh"

namespace ppo {

namespace {

constexpr int kT = 32;          // GEMM tile
constexpr int kGThreads = 256;

// Writes the constant 1 read by the bias-gradient products.
__global__ void rnn_set_one_kernel(float* one) { *one = 1.f; }

// C[m][n] (+)= sum_k A(m, k) B(n, k) (+ bias[n]) with A(m, k) = A[m sam + k sak],
// B(n, k) = B[n sbn + k sbk]; each output summed over k in order by one thread.
// Split-K (gridDim.z > 1): block z sums k in [z kc, (z + 1) kc) into the
// partial C + z M ldc (no bias, no accumulation); split_reduce_kernel then
// adds the partials in split order.
__global__ void __launch_bounds__(kGThreads)
sgemm_kernel(int M, int N, int K, const float* __restrict__ A, int64_t sam, int64_t sak,
             const float* __restrict__ B, int64_t sbn, int64_t sbk, const float* bias,
             float* C, int64_t ldc, int accumulate, int kc) {
  __shared__ float As[kT][kT + 1], Bs[kT][kT + 1];
  const int m0 = blockIdx.y * kT, n0 = blockIdx.x * kT;
  const int ty = threadIdx.x / 16, tx = threadIdx.x % 16;
  const int kb = blockIdx.z * kc;
  const int ke = kb + kc < K ? kb + kc : K;
  if (gridDim.z > 1) C += (int64_t)blockIdx.z * M * ldc;
  float acc[2][2] = {{0.f, 0.f}, {0.f, 0.f}};
  for (int k0 = kb; k0 < ke; k0 += kT) {
    for (int e = threadIdx.x; e < kT * kT; e += kGThreads) {
      const int r = e / kT, c = e % kT;
      As[r][c] = (m0 + r < M && k0 + c < ke) ? A[(int64_t)(m0 + r) * sam + (int64_t)(k0 + c) * sak]
                                             : 0.f;
      Bs[r][c] = (n0 + r < N && k0 + c < ke) ? B[(int64_t)(n0 + r) * sbn + (int64_t)(k0 + c) * sbk]
                                             : 0.f;
    }
    __syncthreads();
#pragma unroll 8
    for (int c = 0; c < kT; ++c) {
      const float a0 = As[2 * ty][c], a1 = As[2 * ty + 1][c];
      const float b0 = Bs[2 * tx][c], b1 = Bs[2 * tx + 1][c];
      acc[0][0] = fmaf(a0, b0, acc[0][0]);
      acc[0][1] = fmaf(a0, b1, acc[0][1]);
      acc[1][0] = fmaf(a1, b0, acc[1][0]);
      acc[1][1] = fmaf(a1, b1, acc[1][1]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int u = 0; u < 2; ++u)
#pragma unroll
    for (int v = 0; v < 2; ++v) {
      const int m = m0 + 2 * ty + u, n = n0 + 2 * tx + v;
      if (m < M && n < N) {
        float y = acc[u][v];
        if (gridDim.z == 1) {
          y += bias ? bias[n] : 0.f;
          if (accumulate) y += C[(int64_t)m * ldc + n];
        }
        C[(int64_t)m * ldc + n] = y;
      }
    }
}

// C[m][n] = sum over splits of part[s][m][n] (split order).
__global__ void split_reduce_kernel(int M, int N, int splits, const float* __restrict__ part,
                                    float* __restrict__ C, int64_t ldc) {
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= (int64_t)M * N) return;
  const int m = (int)(i / N), n = (int)(i - (int64_t)m * N);
  float y = 0.f;
  for (int sp = 0; sp < splits; ++sp) y += part[((int64_t)sp * M + m) * N + n];
  C[(int64_t)m * ldc + n] = y;
}

cudaError_t sgemm(int M, int N, int K, const float* A, int64_t sam, int64_t sak, const float* B,
                  int64_t sbn, int64_t sbk, const float* bias, float* C, int64_t ldc,
                  int accumulate, cudaStream_t st) {
  if (M <= 0 || N <= 0) return cudaSuccess;
  const dim3 grid((N + kT - 1) / kT, (M + kT - 1) / kT);
  sgemm_kernel<<<grid, kGThreads, 0, st>>>(M, N, K, A, sam, sak, B, sbn, sbk, bias, C, ldc,
                                            accumulate, K);
  return cudaGetLastError();
}

// Weight-gradient form: a long reduction (K = rows) over few output tiles,
// split into kSplitK ranges written to `part` ([kSplitK][M][N]) and summed in
// split order into C.
constexpr int kSplitK = 32;
cudaError_t sgemm_splitk(int M, int N, int K, const float* A, int64_t sam, int64_t sak,
                         const float* B, int64_t sbn, int64_t sbk, float* C, int64_t ldc,
                         float* part, cudaStream_t st) {
  if (M <= 0 || N <= 0) return cudaSuccess;
  int kc = (K + kSplitK - 1) / kSplitK;
  kc = (kc + kT - 1) / kT * kT;
  const int splits = (K + kc - 1) / kc;
  const dim3 grid((N + kT - 1) / kT, (M + kT - 1) / kT, splits);
  sgemm_kernel<<<grid, kGThreads, 0, st>>>(M, N, K, A, sam, sak, B, sbn, sbk, nullptr, part, N,
                                            0, kc);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const int64_t n = (int64_t)M * N;
  split_reduce_kernel<<<(unsigned)((n + 255) / 256), 256, 0, st>>>(M, N, splits, part, C, ldc);
  return cudaGetLastError();
}

struct RnnDims {
  int T, ns, D, H, L, C;
  int64_t N, rows;
};

__device__ __forceinline__ int64_t seg_env(const int32_t* envs, int j, int64_t N) {
  int64_t e = __ldg(envs + j);
  return e < 0 ? 0 : (e >= N ? N - 1 : e);
}

// X[r][k] = obs[(t N + env_j) D + k], r = t ns + j.
__global__ void rnn_gather_kernel(RnnDims d, const float* __restrict__ obs,
                                  const int32_t* __restrict__ envs, float* __restrict__ X) {
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= d.rows * d.D) return;
  const int64_t r = i / d.D;
  const int k = (int)(i - r * d.D);
  const int t = (int)(r / d.ns), j = (int)(r - (int64_t)t * d.ns);
  X[i] = obs[((int64_t)t * d.N + seg_env(envs, j, d.N)) * d.D + k];
}

// Forward recurrence of layer l, one thread per (segment j, unit i): Zg holds
// the gate pre-activations on entry and the gates on exit, HT the candidates;
// HP receives the masked previous state, Hout the new state.
__global__ void rnn_fwd_scan_kernel(RnnDims d, int l, const float* __restrict__ done,
                                    const int32_t* __restrict__ envs,
                                    const float* __restrict__ h0, float* Zg,
                                    const float* __restrict__ HT, float* __restrict__ HP,
                                    float* __restrict__ Hout) {
  const int64_t q = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (q >= (int64_t)d.ns * d.H) return;
  const int j = (int)(q / d.H), i = (int)(q - (int64_t)j * d.H);
  const int64_t e = seg_env(envs, j, d.N);
  float h = h0[(e * d.L + l) * d.H + i];
  for (int t = 0; t < d.T; ++t) {
    const int64_t o = ((int64_t)t * d.ns + j) * d.H + i;
    const float mask = (t > 0 && done[(int64_t)(t - 1) * d.N + e] != 0.f) ? 0.f : 1.f;
    const float z = 1.f / (1.f + expf(-Zg[o]));
    const float hp = mask * h;
    h = (1.f - z) * hp + z * HT[o];
    Zg[o] = z;
    HP[o] = hp;
    Hout[o] = h;
  }
}

// Backward recurrence of layer l, reverse time: dIn holds dL/dh from above;
// dPZ / dPH receive the gradients of the gate / candidate pre-activations.
__global__ void rnn_bwd_scan_kernel(RnnDims d, const float* __restrict__ done,
                                    const int32_t* __restrict__ envs,
                                    const float* __restrict__ Zg, const float* __restrict__ HT,
                                    const float* __restrict__ HP, const float* __restrict__ dIn,
                                    float* __restrict__ dPZ, float* __restrict__ dPH) {
  const int64_t q = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (q >= (int64_t)d.ns * d.H) return;
  const int j = (int)(q / d.H), i = (int)(q - (int64_t)j * d.H);
  const int64_t e = seg_env(envs, j, d.N);
  float dnext = 0.f;   // dL/dh_t through h_{t+1}
  for (int t = d.T - 1; t >= 0; --t) {
    const int64_t o = ((int64_t)t * d.ns + j) * d.H + i;
    const float mask = (t > 0 && done[(int64_t)(t - 1) * d.N + e] != 0.f) ? 0.f : 1.f;
    const float dh = dIn[o] + dnext;
    const float z = Zg[o];
    dPZ[o] = dh * (HT[o] - HP[o]) * z * (1.f - z);
    dPH[o] = dh * z;
    dnext = dh * (1.f - z) * mask;
  }
}

constexpr int kLossThreads = 128;

// Decoder z = W_dec h (thread per row, W_dec staged as [H][32]), then the
// per-row PPO loss epilogue of the MLP path: dz [rows][32] and per-block
// partials {6 loss terms, dlogstd[4]}.
__global__ void __launch_bounds__(kLossThreads)
rnn_loss_kernel(RnnDims d, NetShape s, LossCoef lc, const float* __restrict__ Wdec,
                const float* __restrict__ logstd, const float* __restrict__ Htop,
                const int32_t* __restrict__ act, const float* __restrict__ actc,
                const float* __restrict__ logp_old, const float* __restrict__ adv,
                const float* __restrict__ ret, const float* adv_stats,
                const int32_t* __restrict__ envs, float* __restrict__ dz,
                float* __restrict__ part) {
  extern __shared__ float wsm[];   // [H][32]
  for (int e = threadIdx.x; e < d.H * 32; e += kLossThreads) {
    const int k = e / 32, c = e % 32;
    wsm[e] = c < d.C ? Wdec[(int64_t)c * d.H + k] : 0.f;
  }
  __syncthreads();
  const int64_t r = (int64_t)blockIdx.x * kLossThreads + threadIdx.x;
  float t6[6] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f}, dls[4] = {0.f, 0.f, 0.f, 0.f};
  if (r < d.rows) {
    float z[32];
#pragma unroll
    for (int c = 0; c < 32; ++c) z[c] = 0.f;
    const float* h = Htop + r * d.H;
    for (int k = 0; k < d.H; ++k) {
      const float hk = h[k];
#pragma unroll
      for (int c = 0; c < 32; ++c) z[c] = fmaf(wsm[k * 32 + c], hk, z[c]);
    }
    const int t = (int)(r / d.ns), j = (int)(r - (int64_t)t * d.ns);
    const int64_t src = (int64_t)t * d.N + seg_env(envs, j, d.N);
    uint32_t amask = 0u;
    int off = 0;
    for (int hh = 0; hh < s.NH; ++hh) {
      int a = __ldg(act + src * s.NH + hh);
      a = a < 0 ? 0 : (a >= s.head_n[hh] ? s.head_n[hh] - 1 : a);
      amask |= 1u << (off + a);
      off += s.head_n[hh];
    }
    float A = __ldg(adv + src);
    if (adv_stats) A = (A - __ldg(adv_stats)) / (__ldg(adv_stats + 1) + 1e-8f);
    const tc::HeadMasks hm = tc::head_masks(s);
    float dzr[32];
    tc::row_loss_seg<32>(hm, lc, 1.f / (float)d.rows, z, amask, actc + src * s.G, logstd,
                         __ldg(logp_old + src), A, __ldg(ret + src), dzr, t6, dls);
    for (int c = 0; c < d.C; ++c) dz[r * 32 + c] = dzr[c];
  }
  // fixed-order block reduction of the 10 partials
  __shared__ float red[kLossThreads / 32][10];
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  float v[10] = {t6[0], t6[1], t6[2], t6[3], t6[4], t6[5], dls[0], dls[1], dls[2], dls[3]};
#pragma unroll
  for (int q = 0; q < 10; ++q) {
    const float x = warp_sum(v[q]);
    if (lane == 0) red[w][q] = x;
  }
  __syncthreads();
  if (threadIdx.x < 10) {
    float x = 0.f;
    for (int ww = 0; ww < kLossThreads / 32; ++ww) x += red[ww][threadIdx.x];
    part[(int64_t)blockIdx.x * 10 + threadIdx.x] = x;
  }
}

// stats6 = mean of the six loss terms; the log-std gradient (blocks in order).
__global__ void rnn_finalize_kernel(int nblocks, int64_t rows, int G,
                                    const float* __restrict__ part, float* stats6,
                                    float* glogstd) {
  const int q = threadIdx.x;
  if (q >= 10) return;
  float x = 0.f;
  for (int b = 0; b < nblocks; ++b) x += part[(int64_t)b * 10 + q];
  if (q < 6) {
    if (stats6) stats6[q] = x / (float)rows;
  } else if (q - 6 < G) {
    glogstd[q - 6] = x;
  }
}

}  // namespace

size_t rnn_workspace_floats(int D, int H, int L, int64_t rows) {
  // X, per layer (U, Zg, HT, HP), top state, dz, dIn, dPZ, dPH, dU, loss
  // partials, split-K partials of the largest weight gradient, the constant 1
  const size_t wmax = (size_t)H * (D > H ? (D > 32 ? D : 32) : (H > 32 ? H : 32));
  return (size_t)rows * D + (size_t)L * 4 * rows * H + (size_t)rows * H + (size_t)rows * 32 +
         4 * (size_t)rows * H + 10 * ((size_t)(rows + kLossThreads - 1) / kLossThreads) + 64 +
         (size_t)kSplitK * wmax + 4;
}

cudaError_t launch_rnn_loss_grad(const RnnLaunch& a, cudaStream_t st) {
  const int D = a.D, H = a.H, L = a.L, C = a.s.C;
  const int64_t rows = (int64_t)a.T * a.ns;
  RnnDims d{a.T, a.ns, D, H, L, C, a.N, rows};
  float* w = a.work;
  float* X = w;            w += rows * D;
  float* U = w;            w += (size_t)L * rows * H;   // layer inputs (U[0] = encoder out)
  float* Zg = w;           w += (size_t)L * rows * H;
  float* HT = w;           w += (size_t)L * rows * H;
  float* HPv = w;          w += (size_t)L * rows * H;
  float* Htop = w;         w += rows * H;
  float* dz = w;           w += rows * 32;
  float* dIn = w;          w += rows * H;
  float* dPZ = w;          w += rows * H;
  float* dPH = w;          w += rows * H;
  float* dU = w;           w += rows * H;
  float* part = w;         w += 10 * ((rows + kLossThreads - 1) / kLossThreads) + 64;
  const size_t wmax = (size_t)H * (D > H ? (D > 32 ? D : 32) : (H > 32 ? H : 32));
  float* kpart = w;        w += (size_t)kSplitK * wmax;
  float* one = w;          // the constant 1 (column sums as a product with ones)
  const float* P = a.params;
  const int64_t oLayer0 = (int64_t)H * D, per = 2 * (int64_t)H * H + 2 * H;
  const float* Wenc = P;
  const float* Wdec = P + oLayer0 + L * per;
  const float* logstd = Wdec + (int64_t)C * H;
  float* G = a.grad;
  const int thr = 256;
  cudaError_t e;
#define RNN_TRY(x) do { if ((e = (x)) != cudaSuccess) return e; } while (0)
  // the constant 1 the bias-gradient products read, written on the stream
  // (no host memory involved, so the call can be captured)
  rnn_set_one_kernel<<<1, 1, 0, st>>>(one);
  RNN_TRY(cudaGetLastError());
  rnn_gather_kernel<<<(unsigned)((rows * D + thr - 1) / thr), thr, 0, st>>>(d, a.obs, a.envs, X);
  RNN_TRY(cudaGetLastError());
  // encoder: U0 = X W_enc^T
  RNN_TRY(sgemm((int)rows, H, D, X, D, 1, Wenc, D, 1, nullptr, U, H, 0, st));
  const unsigned sgrid = (unsigned)(((int64_t)a.ns * H + thr - 1) / thr);
  for (int l = 0; l < L; ++l) {
    const float* Wz = P + oLayer0 + l * per;
    const float *bz = Wz + (int64_t)H * H, *Wh = bz + H, *bh = Wh + (int64_t)H * H;
    float* Ul = U + (size_t)l * rows * H;
    float* Zl = Zg + (size_t)l * rows * H;
    float* Tl = HT + (size_t)l * rows * H;
    float* HPl = HPv + (size_t)l * rows * H;
    float* Out = l + 1 < L ? U + (size_t)(l + 1) * rows * H : Htop;
    RNN_TRY(sgemm((int)rows, H, H, Ul, H, 1, Wz, H, 1, bz, Zl, H, 0, st));
    RNN_TRY(sgemm((int)rows, H, H, Ul, H, 1, Wh, H, 1, bh, Tl, H, 0, st));
    rnn_fwd_scan_kernel<<<sgrid, thr, 0, st>>>(d, l, a.done, a.envs, a.h0, Zl, Tl, HPl, Out);
    RNN_TRY(cudaGetLastError());
  }
  // decoder + loss
  const int lblocks = (int)((rows + kLossThreads - 1) / kLossThreads);
  rnn_loss_kernel<<<lblocks, kLossThreads, (size_t)H * 32 * sizeof(float), st>>>(
      d, a.s, a.lc, Wdec, logstd, Htop, a.act, a.actc, a.logp_old, a.adv, a.ret, a.adv_stats,
      a.envs, dz, part);
  RNN_TRY(cudaGetLastError());
  float* gWdec = G + oLayer0 + L * per;
  // gW_dec[c][k] = sum_r dz[r][c] Htop[r][k];  dIn = dz W_dec
  RNN_TRY(sgemm_splitk(C, H, (int)rows, dz, 1, 32, Htop, 1, H, gWdec, H, kpart, st));
  RNN_TRY(sgemm((int)rows, H, C, dz, 32, 1, Wdec, 1, H, nullptr, dIn, H, 0, st));
  for (int l = L - 1; l >= 0; --l) {
    const float* Wz = P + oLayer0 + l * per;
    const float* Wh = Wz + (int64_t)H * H + H;
    float* gWz = G + oLayer0 + l * per;
    float *gbz = gWz + (int64_t)H * H, *gWh = gbz + H, *gbh = gWh + (int64_t)H * H;
    const float* Ul = U + (size_t)l * rows * H;
    rnn_bwd_scan_kernel<<<sgrid, thr, 0, st>>>(d, a.done, a.envs, Zg + (size_t)l * rows * H,
                                               HT + (size_t)l * rows * H,
                                               HPv + (size_t)l * rows * H, dIn, dPZ, dPH);
    RNN_TRY(cudaGetLastError());
    // weight and bias gradients
    RNN_TRY(sgemm_splitk(H, H, (int)rows, dPZ, 1, H, Ul, 1, H, gWz, H, kpart, st));
    RNN_TRY(sgemm_splitk(H, H, (int)rows, dPH, 1, H, Ul, 1, H, gWh, H, kpart, st));
    // bias gradients: column sums, i.e. the product with a column of ones
    RNN_TRY(sgemm_splitk(H, 1, (int)rows, dPZ, 1, H, one, 0, 0, gbz, 1, kpart, st));
    RNN_TRY(sgemm_splitk(H, 1, (int)rows, dPH, 1, H, one, 0, 0, gbh, 1, kpart, st));
    // input gradient: dU = dPZ W_z + dPH W_h -> the layer below
    RNN_TRY(sgemm((int)rows, H, H, dPZ, H, 1, Wz, 1, H, nullptr, dU, H, 0, st));
    RNN_TRY(sgemm((int)rows, H, H, dPH, H, 1, Wh, 1, H, nullptr, dU, H, 1, st));
    std::swap(dIn, dU);
  }
  // encoder gradient: gW_enc[i][k] = sum_r dU0[r][i] X[r][k]
  RNN_TRY(sgemm_splitk(H, D, (int)rows, dIn, 1, H, X, 1, D, G, D, kpart, st));
  rnn_finalize_kernel<<<1, 32, 0, st>>>(lblocks, rows, a.s.G, part, a.stats6,
                                        G + (logstd - P));
  RNN_TRY(cudaGetLastError());
#undef RNN_TRY
  return cudaSuccess;
}

}  // namespace ppo
