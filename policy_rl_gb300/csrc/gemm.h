// gemm.h -- internal interface of the MLP GEMM kernels (tensor-core bf16 and
// CUDA-core fp32) used by the learner-step orchestration in api.cu.
#pragma once

#include "common.cuh"

namespace ppo {

// ---- bf16 tensor-core path --------------------------------------------------
// D[M][N] = A[M][K] * B[N][K]^T; A and B row-major bf16 with row pitches
// lda/ldb (elements, multiples of 8); N a multiple of 64 (or 16/32 for the
// loss head); K <= lda, K <= ldb, columns of A/B between K and the next
// multiple of 64 must be zero or lie beyond lda/ldb.
struct GemmOperands {
  const __nv_bfloat16* A;
  int lda;
  const __nv_bfloat16* B;
  int ldb;
  int M, N, K;
};

struct TcParams {
  int M, N, K;
  int tiles_m, tiles_n, k_tiles, last_k_steps;
  int epi_n;
  const float* bias;
  __nv_bfloat16* out;
  int ldo;
  const __nv_bfloat16* aux;
  int ldaux;
  int act;
  float* colsum_part;
  NetShape shape;
  LossCoef lc;
  LossRows rows;
  float inv_mb;
  const float* logstd;
  float* loss_part;
  __nv_bfloat16* dz;
  int lddz;
  int* err;
  uint64_t timeout_ns;
  float alpha, beta;   // act 3 of the aux-tile epilogue: out = alpha aux + beta acc
  int layout9222;      // loss epilogue: the 9-2-2-2 head layout (compile-time masks)
  const __nv_bfloat16* a_rows;   // A [M][lda] (the producer's L2 prefetch of whole rows)
  int lda;
};

// Gradient assembly from the split-K and per-CTA partials (optim.cu, and the
// weight-gradient kernel's vector tasks).
struct ReduceArgs {
  NetShape s;
  const float* pW1; int s1; int ld1;    // [s1][H1][ld1]
  const float* pW2; int s2;             // [s2][H2][H1]
  const float* pW3t; int s3; int ld3;   // [s3][H2][ld3]  (dW3 transposed)
  const float* pb1; int nb1;            // [nb1][H1]
  const float* pb2; int nb2;            // [nb2][H2]
  const float* pb3; int nb3; int ldb3;  // [nb3][ldb3]
  const float* ploss; int nl;           // [nl][kLossPartials]
  float inv_mb;
  float* grad;                          // [P]
  double* sq_part;                      // nullable: per-block sum of squares of grad
  float* stats6;                        // nullable
  int weights_done;                     // the weight entries of grad are already assembled
                                        // (by the weight-gradient kernel): biases, log-std
                                        // and statistics only
  int nsq_pre;                          // squared-norm partials of the same gradient stored
                                        // just before sq_part (by that kernel)
};

struct WRegion {
  int M, N, bn, tiles_m, tiles_n, splits, kt_per_split, k_tiles, unit_begin;
  float* part;  // [splits][M][N]
};

// Where the assembled gradient of a weight-gradient region goes: element
// (m, n) of the region's product, m < rows and n < cols, is written to
// dst[m * ldm + n * ldn].
struct WFinal {
  float* dst;
  int rows, cols;
  int64_t ldm, ldn;
};

struct WParams {
  WRegion r[3];
  int nreg, total_units;
  uint32_t mn_lbo, mn_sbo;
  int* err;
  uint64_t timeout_ns;
  // in-kernel assembly (fixup != 0): the CTAs of one output tile meet at a
  // per-tile counter and each sums a slice of the tile over the splits
  int fixup;
  WFinal f[3];
  int tile_begin[3];   // first tile index of each region
  unsigned* tile_ctr;  // [2][tiles] arrival / completion counters, zero between launches
  double* sq_part;     // [gridDim.x] per-CTA sums of squares of the entries it wrote
  uint64_t tile_wait_ns;   // limit of the wait for a tile's other CTAs (no copies in flight)
  // the bias / log-std / statistic entries (nvt > 0): ra's vector tasks, one
  // warp each, summed into the same per-CTA squared-norm partials
  ReduceArgs ra;
  int nvt;
};

// One weight-gradient product P[M][N] = sum_r U[r][0..M) (x) V[r][0..N),
// U, V bf16 row-major [rows][ldu/ldv]; M a multiple of 128, N of 64.
struct WGradRegion {
  const __nv_bfloat16* U;
  int ldu, M;
  const __nv_bfloat16* V;
  int ldv, N;
  int kt_per_split;   // 64-row k-tiles per split
  float* part;        // [splits][M][N] fp32
  WFinal fin;         // in-kernel assembly target (fin.dst == nullptr: partials only)
};

// Largest tile count of a tc_wgrad call with in-kernel assembly (size of the
// counter array: 2 * kWgradMaxTiles unsigned), and the most K-splits of a
// product in one call.
constexpr int kWgradMaxTiles = 256;
constexpr int kMaxWgSplit = 64;

// Loss and BPTT gradient of the recurrent policy on the tensor cores
// (rnn_tc.cu): hidden 128 or 256; the workspace holds an error word at its
// start (nonzero after a bounded device wait gave up), *err_out points to it.
struct RnnLaunch;
bool rnn_tc_supported(int D, int H);
size_t rnn_tc_workspace_bytes(int D, int H, int L, int64_t T, int64_t ns, int num_sms);
cudaError_t launch_rnn_loss_grad_tc(const RnnLaunch& a, int num_sms, cudaStream_t st,
                                    int** err_out);

cudaError_t tc_prepare();
int tc_pick_bn(int N);
int tc_wgrad_splits(int rows, int kt_per_split);
int tc_wgrad_bn(int N);   // column width of the weight-gradient tiles of an N-column product
// K-split plan of up to three products mn[i] = {M, N} over `rows` rows: kt[i]
// 64-row k-tiles per unit, all units in one wave of num_sms CTAs when possible.
void tc_wgrad_plan(const int (*mn)[2], int nreg, int64_t rows, int num_sms, int max_split,
                   int* kt);

cudaError_t tc_gemm_bias_act(const GemmOperands& g, const float* bias, int act,
                             __nv_bfloat16* out, int ldo, int* err, uint64_t timeout_ns,
                             int num_sms, cudaStream_t st);
cudaError_t tc_gemm_dact(const GemmOperands& g, const __nv_bfloat16* aux, int ldaux, int act,
                         __nv_bfloat16* out, int ldo, float* colsum_part, int* err,
                         uint64_t timeout_ns, int num_sms, cudaStream_t st, int* grid_out);
// out = alpha * aux + beta * (A B^T), bf16, aux and out [M][N] (N a multiple
// of 128): the aux-tile kernel with its act' replaced by the sum.
cudaError_t tc_gemm_axpby(const GemmOperands& g, const __nv_bfloat16* aux, int ldaux, float alpha,
                          float beta, __nv_bfloat16* out, int ldo, int* err, uint64_t timeout_ns,
                          int num_sms, cudaStream_t st);
cudaError_t tc_gemm_loss(const GemmOperands& g, const NetShape& s, LossCoef lc, LossRows rows,
                         float inv_mb, const float* b3, const float* logstd, __nv_bfloat16* dz,
                         int lddz, float* colsum_part, float* loss_part, int* err,
                         uint64_t timeout_ns, int num_sms, cudaStream_t st, int* grid_out);
// Weight gradients of up to three regions.  With tile_ctr and sq_part given
// (and every region's fin.dst set), the kernel is launched cooperatively and
// also sums the split partials into the final gradient (fixed split order)
// and writes per-CTA squared-norm partials sq_part[0 .. *grid_out).
// timeout_ns bounds the TMA/MMA pipeline waits, tile_wait_ns (0: timeout_ns)
// the wait of a CTA for the other CTAs of its tile.  With `vectors` (and the
// assembly on), the kernel also runs that gradient's bias / log-std /
// statistic sums, so that sq_part covers the whole gradient.
cudaError_t tc_wgrad(const WGradRegion* regs, int nreg, int rows, uint32_t mn_lbo,
                     uint32_t mn_sbo, int* err, uint64_t timeout_ns, int num_sms,
                     cudaStream_t st, unsigned* tile_ctr = nullptr, double* sq_part = nullptr,
                     int* grid_out = nullptr, uint64_t tile_wait_ns = 0,
                     const ReduceArgs* vectors = nullptr);

// ---- fp32 CUDA-core path ----------------------------------------------------
// Generic-stride GEMM: C(m,n) = sum_k A(m,k) B(n,k) with
// A(m,k) = A[m*sam + k*sak], B(n,k) = B[n*sbn + k*sbk].
struct SimtOperands {
  const float* A;
  int64_t sam, sak;
  const float* B;
  int64_t sbn, sbk;
  int M, N, K;
};
int simt_tiles_m(int M);
cudaError_t simt_bias_act(const SimtOperands& g, const float* bias, int act, float* out, int ldo,
                          cudaStream_t st);
cudaError_t simt_dact(const SimtOperands& g, const float* aux, int ldaux, int act, float* out,
                      int ldo, float* colsum_part, cudaStream_t st);
// split-K partial products: part[split][M][N], split covers k_per_split rows
cudaError_t simt_wgrad(const SimtOperands& g, int k_per_split, float* part, cudaStream_t st);
// head + loss: z = H2 W3^T + b3 per row, per-row loss, dz (fp32 [mb][CP]),
// per-block column sums of dz and loss partials; returns the block count.
cudaError_t simt_head_loss(const NetShape& s, LossCoef lc, LossRows rows, float inv_mb,
                           const float* H2, const float* W3, const float* b3,
                           const float* logstd, int mb, float* dz, float* colsum_part,
                           float* loss_part, cudaStream_t st, int* blocks_out);
int simt_head_blocks(int mb);

// ---- reduction and optimizer --------------------------------------------------
int reduce_blocks(const NetShape& s);            // every entry: weights, biases, statistics
int reduce_launch_blocks(const ReduceArgs& a);    // blocks of one launch (and its sq partials)
cudaError_t launch_reduce(const ReduceArgs& a, cudaStream_t st);

struct Shadows {
  __nv_bfloat16 *W1s, *W2s, *W2Ts, *W3s, *W3Ts;  // nullptr in fp32 mode
  int ld3t;                                       // row pitch of W3Ts
};
struct AdamArgs {
  float* p;
  const float* g;
  float* m;
  float* v;
  int64_t P;
  const double* sq_part;   // per-block sums of squares of g (written by the caller's
  int nsq;                 // reduce when nsq > 0; computed by launch_adam when nsq == 0)
  float max_norm, lr, eps;
  double b1, b2;      // for the bias corrections 1 - beta^t
  float omb1, omb2;   // 1 - beta1, 1 - beta2 (rounded once from double)
  int64_t* step;
  double* beta_pow;        // {beta1^step, beta2^step, 1/(1-beta1^(step+1)), 1/(1-beta2^(step+1))},
                           // advanced by the last block
  unsigned* done_ctr;
  float* grad_norm_out;
  NetShape s;
  Shadows sh;
  int vectors_only;        // 1: update only the biases and log-std (the weight
                           // matrices take Muon's update instead)
};
cudaError_t launch_adam(const AdamArgs& a, cudaStream_t st, const Trace* tr = nullptr);

// ---- Muon (optim.cu) ---------------------------------------------------------
// One weight matrix p [rows][cols] of the flat parameter vector, its gradient
// and momentum, and the Newton-Schulz workspaces (r = min(rows, cols),
// k = max): X0, X1 [r][k] (ping-pong), A, B [r][r].
struct MuonMat {
  float* p;
  const float* g;
  float* mom;
  int rows, cols;
  int64_t off;         // flat index of p[0][0]
  float *X0, *X1, *A, *B;
};
constexpr int kMuonPrepBlocks = 64;
struct MuonArgs {
  MuonMat m[3];        // W1, W2, W3
  float beta, lr;      // momentum and Muon learning rate
  float* mpart;        // [3][kMuonPrepBlocks] per-block sums of squares of u
  float* inv;          // [3] 1 / (||u||_F + 1e-7)
  NetShape s;
  Shadows sh;
};
// Clip (coefficient from a's squared-norm partials, computed by launch_muon
// when a.nsq == 0), Muon on the three weight matrices, Adam (a) on the
// biases and log-std, bf16 shadows refreshed.  With tc, the Newton-Schulz
// products run on the tensor cores with bf16 X, A, B (see MuonTc).
struct MuonTc;
cudaError_t launch_muon(const MuonArgs& mu, const AdamArgs& a, cudaStream_t st,
                        const Trace* tr = nullptr, const MuonTc* tc = nullptr);

// Tensor-core Newton-Schulz of one matrix: r x k (r <= k) zero-padded to
// rp x kp (multiples of 128); bf16 X, X2 [rp][kp] (ping-pong), XT [kp][rp]
// (X transposed), A, B [rp][rp].  The padding stays zero.
struct MuonTcMat {
  int r, k, rp, kp;
  __nv_bfloat16 *X, *X2, *XT, *A, *B;
};
// The three matrices' iterations run concurrently on side streams (forked
// from and joined back to the caller's stream with the events).
struct MuonTc {
  MuonTcMat m[3];
  cudaStream_t side[3];
  cudaEvent_t fork, join[3];
  int* err;
  int num_sms;
};
// Gradient assembly + clip + Adam in one cooperative launch (optim.cu); *bar
// is a zeroed grid-barrier counter (cleared again by the kernel).
cudaError_t reduce_adam_prepare();
cudaError_t launch_reduce_adam(const ReduceArgs& ra, const AdamArgs& aa, unsigned* bar, int* err,
                               uint64_t limit_ns, int num_sms, cudaStream_t st);

// ---- persistent minibatch kernel (mk.cu) ------------------------------------
// Everything the fused bf16 minibatch step needs: the five K-major GEMMs, the
// three weight-gradient regions, gradient assembly and (optionally) Adam.
struct MkLaunch {
  NetShape s;
  GatherArgs ga;
  GemmOperands fwd1, fwd2, loss, dact2, dact1;
  const float *b1, *b2, *b3, *logstd;
  __nv_bfloat16 *H1, *H2, *dP2, *dP1, *dz;
  int lddz;
  float *cs1, *cs2, *cs3, *loss_part;   // per-CTA partial rows [grid][...]
  WGradRegion wg[3];
  int rows;                             // minibatch rows
  ReduceArgs ra;
  int do_adam;
  AdamArgs aa;
  LossCoef lc;
  LossRows rows_in;
  float inv_mb;
  unsigned* gbar;                       // [2] grid-barrier counters (zero between launches)
  double* sq_part;                      // [grid]
  unsigned long long* phase_ns;         // nullable: per-phase time sums (profiling)
  int* err;
  uint64_t timeout_ns;
  int grid;
};
constexpr int kMkPhases = 9;   // gather, fwd1, fwd2, loss, dact2, dact1, wgrad, reduce, adam
cudaError_t mk_prepare();
int mk_grid(int num_sms);
int mk_wgrad_bn(int N);
cudaError_t mk_launch(const MkLaunch& L, cudaStream_t st);
// bf16 row-major [rows][ld]: box = box_cols x box_rows, swizzled in rows of
// swizzle_bytes (128, 64 or 32; the box's row must fit in it)
cudaError_t tc_make_tmap(CUtensorMap* m, const void* base, int64_t cols, int64_t rows, int64_t ld,
                         int box_cols, int box_rows, int swizzle_bytes = 128);
// [rows][ld] bf16 viewed as 64-column blocks: box = 64 x box_rows x box_blk,
// landing as box_blk consecutive [box_rows][64] swizzled blocks
cudaError_t tc_make_tmap_blocks(CUtensorMap* m, const void* base, int64_t rows, int64_t ld,
                                int nblk, int box_rows, int box_blk);
cudaError_t launch_shadows(const float* p, const NetShape& s, const Shadows& sh, cudaStream_t st);

// Fused forward + loss + backward-data pass of one minibatch (fmlp.cu): all
// activations bf16 row-major [M][width]; dZ with row pitch lddz (64).
struct FusedMlp {
  NetShape s;
  int M;
  const __nv_bfloat16 *X, *W1s, *W2s, *W3s, *W3Ts, *W2Ts;
  int ld3t;
  const float *b1, *b2, *b3, *logstd;
  __nv_bfloat16 *H1, *H2, *dZ, *dP2, *dP1;
  int lddz;
  LossCoef lc;
  LossRows rows;
  float inv_mb;
  float *cs1, *cs2, *cs3, *lossp;   // per-CTA partial rows (grid of them)
  int* err;
  uint64_t timeout_ns;
};
// Head + loss + backward-data through the last hidden layer (hl2.cu):
// dz [M][lddz] and dP2 [M][H2] from H2 [M][H2], all bf16.
struct HeadLossDact {
  NetShape s;
  int M;
  const __nv_bfloat16 *H2, *W3s;
  const float *b3, *logstd;
  __nv_bfloat16 *dZ, *dP2;
  int lddz;
  LossCoef lc;
  LossRows rows;
  float inv_mb;
  float *cs2, *cs3, *lossp;   // per-CTA partial rows (grid of them)
  int* err;
  uint64_t timeout_ns;
};
// shapes of the fused kernel: H2 = 256 or 512 with 16 head columns
bool hl2_supported(const NetShape& s);
cudaError_t hl2_prepare();
cudaError_t hl2_launch(const HeadLossDact& f, int num_sms, cudaStream_t st, int* grid_out);

bool fmlp_supported(const NetShape& s);
cudaError_t fmlp_prepare();
cudaError_t fmlp_launch(const FusedMlp& f, int num_sms, cudaStream_t st, int* grid_out);

}  // namespace ppo
