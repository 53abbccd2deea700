/*
 * ppo.h -- C ABI of the GB300 (sm_103a) PPO learner step.
 *
 * The library computes, on one GPU, the learner half of PPO over a rollout
 * buffer of T steps x N environments ("Teaching Mario to speedrun",
 * sec. 6 "The whole algorithm", steps 2 "judge" and 3 "learn"):
 *   GAE -> advantage normalisation -> for each epoch, a shuffled set of
 *   minibatches -> MLP actor-critic forward, clipped surrogate + value +
 *   entropy loss, backward -> gradient-norm clip -> Adam.
 * and, from sec. 8 (PufferLib 5.0) and the rollout side of sec. 6-7:
 *   advantages per minibatch of environment segments from fresh values
 *   (GAE or V-trace: ppo_segment_advantage, ppo_minibatch_loss_grad_fresh,
 *   ppo_config.adv_mode), the Muon optimizer (ppo_muon_step,
 *   ppo_config.optimizer), the rollout-side policy step with sampling
 *   (ppo_policy_act), and the loss and gradient of the recurrent MinGRU
 *   policy (ppo_rnn_loss_grad).
 *
 * Conventions shared by every entry point
 *  - Pointers named d_* are DEVICE pointers on the current CUDA device;
 *    pointers named h_* are HOST pointers.  The caller owns every buffer it
 *    passes; the library never frees or retains a caller pointer beyond the
 *    call, except that ppo_update may cache a CUDA graph that refers to the
 *    pointers of its last call (re-captured whenever any argument changes).
 *  - Rollout arrays are time-major: element (t, n) of a [T, N] array is at
 *    t*N + n (environment index fastest).  Flat batch row b = t*N + n.
 *  - Every device pointer must be 16-byte aligned (PPO_ERR_ALIGN otherwise).
 *  - All work is enqueued asynchronously on `stream`; no call synchronises
 *    the device except ppo_create, ppo_destroy, ppo_sync_status and
 *    ppo_update_host.  Argument errors are detected on the host before any
 *    launch and nothing is enqueued.  Errors found on the device (a bounded
 *    wait that timed out) are latched in the context and returned by the next
 *    ppo_sync_status.
 *  - Results are deterministic: the same inputs give bit-identical outputs
 *    (fixed-order reductions, no floating-point atomics).
 *  - There is no CPU fallback: without a usable sm_103a device every call that
 *    launches work returns PPO_ERR_CUDA or PPO_ERR_UNSUPPORTED.
 */
#ifndef PPO_H
#define PPO_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    PPO_OK = 0,
    PPO_ERR_INVALID = 1,      /* bad size, null pointer, inconsistent shapes */
    PPO_ERR_ALIGN = 2,        /* a device pointer is not 16-byte aligned      */
    PPO_ERR_CUDA = 3,         /* a CUDA runtime/driver call failed            */
    PPO_ERR_UNSUPPORTED = 4,  /* shape outside what the kernels implement    */
    PPO_ERR_TIMEOUT = 5,      /* a bounded device-side wait gave up           */
    PPO_ERR_NOMEM = 6         /* device allocation failed                     */
} ppo_status;

#define PPO_MAX_HEADS 8

/* Network and loss configuration (fixed for the life of a context).
 * The MLP is h1 = act(W1 x + b1), h2 = act(W2 h1 + b2), z = W3 h2 + b3
 * ("Teaching Mario to speedrun", sec. 6 "The policy and the value are one
 * network").  The C = sum(head_n) + n_gauss + 1 output columns are, in order:
 * the logits of each discrete head, the means of the diagonal-Gaussian
 * dimensions ("boesch.dev DDNet RL", "What the agent sees and does"), the
 * value.  Flat parameter layout (fp32):
 *   W1[h1][obs_dim], b1[h1], W2[h2][h1], b2[h2], W3[C][h2], b3[C],
 *   logstd[n_gauss]   (state-independent learned log-std per Gaussian dim). */
typedef struct {
    int32_t obs_dim;             /* D                                        */
    int32_t h1, h2;              /* hidden widths                            */
    int32_t act;                 /* 0 = tanh, 1 = ReLU                       */
    int32_t n_heads;             /* discrete heads, 0..PPO_MAX_HEADS          */
    int32_t head_n[PPO_MAX_HEADS];
    int32_t n_gauss;             /* Gaussian action dims, 0..4               */
    int32_t precision;           /* 0 = fp32 (CUDA-core FFMA GEMMs),
                                    1 = bf16 tensor-core GEMMs (tcgen05), fp32
                                        accumulate, fp32 master weights       */
    float clip;                  /* epsilon of clip(ratio, 1-eps, 1+eps)     */
    float vf_coef, ent_coef;     /* loss = pg + vf_coef*V - ent_coef*H       */
    float max_grad_norm;         /* <= 0 disables the clip                   */
    double beta1, beta2;         /* Adam moment decays (double: 1 - beta is
                                    formed without fp32 cancellation)        */
    double adam_eps;
    int64_t max_batch;           /* largest T*N given to ppo_update          */
    int64_t max_minibatch;       /* largest minibatch row count              */
    int32_t max_epochs;          /* largest epoch count given to ppo_update  */
    int32_t persistent_minibatch; /* bf16 mode: 0 (default) launches one kernel
                                    per stage of a minibatch step; 1 runs the
                                    whole step (gather .. Adam) as one
                                    persistent cooperative kernel whose stages
                                    are separated by grid barriers.  Same
                                    results up to fp32 summation order.      */
    int32_t fused_mlp;           /* bf16 mode, persistent_minibatch == 0: 0
                                    (default) launches one kernel per GEMM
                                    stage; 1 runs forward, loss and
                                    backward-data of a minibatch as one fused
                                    kernel when the network fits its shared
                                    memory tiles (padded obs width 64, hidden
                                    widths 128 or 256, <= 32 head columns,
                                    <= 4 Gaussian dims), else per stage.  Same
                                    results up to fp32 summation order.      */
    int32_t fused_loss;          /* bf16 mode: head + loss and
                                    dP2 = (dz W3) * act'(H2) as one kernel
                                    that reads each tile of H2 once, or as two
                                    kernels.  -1: two kernels; 0 (default) or
                                    1: one kernel where it applies (H2 = 256
                                    or 512 with at most 16 head columns), two
                                    elsewhere.  Same results up to fp32
                                    summation order.                         */
    int32_t adv_mode;            /* advantages of ppo_update:
                                    0 (default) GAE once per update over the
                                      whole rollout, normalised over all T*N;
                                    1 per minibatch from fresh values ("Teaching
                                      Mario to speedrun", sec. 8): minibatches
                                      are whole environment segments (epoch e
                                      shuffles the N environments with the rule
                                      of ppo_minibatch_perm, minibatch k takes
                                      N/minibatches of them), and before each
                                      loss the advantages are recomputed by GAE
                                      from the current network's values and
                                      normalised over the minibatch;
                                    2 as 1 with V-trace (see
                                      ppo_segment_advantage) using the current
                                      network's importance ratios.
                                    Modes 1 and 2 run the per-stage kernels
                                    (persistent_minibatch and fused_mlp are
                                    ignored) and need N % minibatches == 0.   */
    float vtrace_rho_clip;       /* V-trace rho_bar (adv_mode 2; IMPALA: 1)    */
    float vtrace_c_clip;         /* V-trace c_bar   (adv_mode 2; IMPALA: 1)    */
    int32_t optimizer;           /* optimizer step of ppo_update:
                                    0 (default) Adam on every parameter;
                                    1 Muon ("Teaching Mario to speedrun",
                                      sec. 8; see ppo_muon_step) on W1, W2,
                                      W3 and Adam on the biases and log-std.
                                    Muon needs persistent_minibatch == 0
                                    (ignored otherwise).                      */
    float muon_lr;               /* Muon learning rate (write-up: 0.02)        */
    float muon_beta;             /* Muon momentum (write-up: 0.95)             */
} ppo_config;

typedef struct ppo_ctx ppo_ctx;

/* Human-readable name of a status code (static string). */
const char *ppo_status_string(ppo_status s);

/* Creates a context on the current device: parameters (initialised from
 * h_init_params, a HOST array of ppo_param_count() floats, or zero if NULL),
 * gradient, Adam moments (zero), step counter (zero), the bf16 weight shadows
 * and every workspace sized from max_batch / max_minibatch / max_epochs.
 * Synchronous.  C <= 32; bf16 mode requires h1 and h2 to be multiples of 128
 * and at most 512 (PPO_ERR_UNSUPPORTED otherwise); requires an sm_103 device. */
ppo_status ppo_create(const ppo_config *cfg, const float *h_init_params, ppo_ctx **out);
ppo_status ppo_destroy(ppo_ctx *ctx);

/* Number of fp32 parameters for cfg (layout above).  No device needed. */
ppo_status ppo_param_count(const ppo_config *cfg, int64_t *n);

/* Device pointers owned by the context (valid until ppo_destroy): params,
 * gradient (written by ppo_minibatch_loss_grad), Adam first and second
 * moments.  Any may be NULL.  Writing d_params directly requires a following
 * ppo_params_changed so that the bf16 shadows are refreshed. */
ppo_status ppo_buffers(ppo_ctx *ctx, float **d_params, float **d_grad, float **d_adam_m,
                       float **d_adam_v);
ppo_status ppo_params_changed(ppo_ctx *ctx, cudaStream_t stream);
/* Adam step counter (number of ppo_adam_step calls so far); synchronous. */
ppo_status ppo_get_step(ppo_ctx *ctx, int64_t *step);

/* ---- GAE ------------------------------------------------------------------
 * "Teaching Mario to speedrun", sec. 6 "Better advantages":
 *   delta_t = r_t + gamma V(s_{t+1}) - V(s_t),  A_t = sum_l (gamma lambda)^l delta_{t+l}
 * computed per environment as a reverse-time scan.  d_done[t,n] != 0 means
 * the episode ended during step t (sec. 7: terminals are 1 where an episode
 * just ended): r[t,n] is its last reward and neither V(s_{t+1}) nor A_{t+1}
 * crosses it.  d_boot[n] = V(s_T) bootstraps the last step.
 * Inputs  d_rew, d_val, d_done: fp32 [T,N];  d_boot: fp32 [N].
 * Outputs d_adv: fp32 [T,N] advantages; d_ret: fp32 [T,N] lambda-returns
 *         A + V;  d_adv_norm (nullable): (A - mean)/(std + 1e-8);
 *         d_stats (nullable): fp32 [2] = {mean, unbiased std} of A over all
 *         T*N entries.
 * d_work: device scratch of ppo_gae_workspace_bytes(T, N) bytes (may be NULL
 * when both d_adv_norm and d_stats are NULL).  Outputs may not alias inputs.
 * T, N >= 1; T*N < 2^31; T <= 2^19 (the per-warp moment counts, at most
 * 32*T, stay exact in fp32; PPO_ERR_UNSUPPORTED above). */
ppo_status ppo_gae_workspace_bytes(int64_t T, int64_t N, size_t *bytes);
ppo_status ppo_gae(const float *d_rew, const float *d_val, const float *d_done,
                   const float *d_boot, int64_t T, int64_t N, float gamma, float lambda,
                   float *d_adv, float *d_ret, float *d_adv_norm, float *d_stats,
                   void *d_work, size_t work_bytes, cudaStream_t stream);

/* ppo_gae without the workspace argument, for callers that cannot allocate
 * device memory (a stream being captured into a CUDA graph where cudaMalloc is
 * not allowed, latency-critical loops that must not enter the allocator,
 * hosts whose device memory is all owned by their own pool).  The pages have
 * no counterpart; the results are those of ppo_gae with the same arguments.
 * The moment partials live in a fixed array in the library's device memory
 * (about 193 KB, held on every GPU that loads the library until exit), so
 * N must be at most 1,048,576 (PPO_ERR_UNSUPPORTED otherwise).  The first
 * call on a device looks that array's address up (cudaGetSymbolAddress with
 * the device current): make it before any stream capture.  The look-up is
 * repeated when another CUDA context has become current on the device (after
 * cudaDeviceReset, say); the first call after such a change must also come
 * before any stream capture.  All calls share
 * the array: calls that may overlap on the GPU (unordered streams, several
 * host threads) race and must be serialised by the caller.  Never calls
 * cudaMalloc or cudaFree. */
ppo_status ppo_gae_noalloc(const float *d_rew, const float *d_val, const float *d_done,
                           const float *d_boot, int64_t T, int64_t N, float gamma, float lambda,
                           float *d_adv, float *d_ret, float *d_adv_norm, float *d_stats,
                           cudaStream_t stream);

/* ---- Advantages of environment segments (per-minibatch recompute) ----------
 * "Teaching Mario to speedrun", sec. 8 "The Puffer net, and the trainer":
 * advantages computed per minibatch from fresh values, by GAE or V-trace.
 * V-trace is defined by Espeholt et al. 2018 ("IMPALA", sec. 4.1, eq. 1 with
 * lambda-weighted traces): with rho_t = min(rho_clip, ratio_t) and
 * c_t = lambda min(c_clip, ratio_t),
 *   A_t = rho_t delta_t + gamma c_t (1 - d_t) A_{t+1},  A_T = 0,
 *   delta_t = r_t + gamma (1 - d_t) V_{t+1} - V_t,      V_T = boot,
 * ret_t = A_t + V_t (the V-trace target v_t).  d_ratio == NULL is GAE
 * (rho = 1, c = lambda; the clips are ignored).  Terminals as in ppo_gae.
 * Segment j is environment d_envs[j] (int32 [ns], each in [0, N); clamped
 * on the device) over the whole horizon; the segment arrays are [T][ns]
 * (element t*ns + j):
 *   d_val    fp32 [T][ns]  values V(s_t) of the segments' steps
 *   d_ratio  fp32 [T][ns]  importance ratios pi/mu, or NULL
 *   d_rew, d_done fp32 [T][N]; d_boot fp32 [N]  (the whole rollout)
 * Outputs d_adv, d_ret fp32 [T][ns]; d_adv_norm (nullable, may equal d_adv)
 * = (A - mean)/(std + 1e-8); d_stats (nullable) fp32 [2] = {mean, unbiased
 * std} of A over the T*ns entries.  d_work: ppo_segment_advantage_workspace_bytes()
 * bytes of device scratch; its int32 at byte offset 4 is set nonzero if a
 * bounded device wait of the call gave up (outputs then unspecified).
 * T, ns >= 1; T*ns < 2^31.  Deterministic. */
ppo_status ppo_segment_advantage_workspace_bytes(size_t *bytes);
ppo_status ppo_segment_advantage(const float *d_rew, const float *d_done, const float *d_boot,
                                 int64_t T, int64_t N, const int32_t *d_envs, int64_t ns,
                                 const float *d_val, const float *d_ratio, float gamma,
                                 float lambda, float rho_clip, float c_clip, float *d_adv,
                                 float *d_ret, float *d_adv_norm, float *d_stats, void *d_work,
                                 size_t work_bytes, cudaStream_t stream);

/* ---- Minibatch permutation -------------------------------------------------
 * "Teaching Mario to speedrun", sec. 6: "for minibatch in shuffle(batch)".
 * Key i = mulberry32 draw number epoch*B + i of the stream seeded with `seed`
 * ("PlayTrain", Appendix F.2 "seeded RNG"); d_perm (int32 [B]) receives
 * 0..B-1 sorted by (key, index).  Minibatch m of an epoch is
 * d_perm[m*mb .. (m+1)*mb).  Bit-exact.  1 <= B < 2^31.
 * d_work: ppo_perm_workspace_bytes(B) bytes of device scratch. */
ppo_status ppo_perm_workspace_bytes(int64_t B, size_t *bytes);
ppo_status ppo_minibatch_perm(uint32_t seed, int64_t epoch, int64_t B, int32_t *d_perm,
                              void *d_work, size_t work_bytes, cudaStream_t stream);

/* ---- Loss and gradient of one minibatch --------------------------------------
 * "Teaching Mario to speedrun", sec. 6 "Don't move too far at once":
 *   ratio = exp(logp - logp_old),  loss_pi = -min(ratio A, clip(ratio, 1-eps, 1+eps) A),
 *   loss_V = (V - R)^2,  loss = mean(loss_pi) + vf_coef mean(loss_V) - ent_coef mean(H)
 * with logp and H summed over the discrete heads (log-softmax) and the
 * Gaussian dimensions.  Rows d_idx[0..mb) (int32, each in [0, B)) are
 * gathered from the full-batch arrays
 *   d_obs      fp32 [B][obs_dim]
 *   d_act_disc int32 [B][n_heads]   (each in [0, head_n[h]))
 *   d_act_cont fp32 [B][n_gauss]    (may be NULL if n_gauss == 0)
 *   d_logp_old fp32 [B], d_adv fp32 [B], d_ret fp32 [B].
 * If d_adv_stats (fp32 [2] = {mean, std}, device) is non-NULL the advantage
 * used is (adv - mean)/(std + 1e-8).  The gradient dloss/dparams (fp32, flat
 * layout) OVERWRITES the context's gradient buffer.  d_stats6 (nullable,
 * fp32 [6]) receives the minibatch means {loss, pg_loss, v_loss, entropy,
 * clipfrac, approx_kl}, with approx_kl = mean((r - 1) - log r).
 * 1 <= mb <= max_minibatch.  An index outside [0, B) or an action outside
 * [0, head_n) is clamped into range on the device (it never faults). */
ppo_status ppo_minibatch_loss_grad(ppo_ctx *ctx, const float *d_obs, const int32_t *d_act_disc,
                                   const float *d_act_cont, const float *d_logp_old,
                                   const float *d_adv, const float *d_ret, const int32_t *d_idx,
                                   int64_t B, int64_t mb, const float *d_adv_stats,
                                   float *d_stats6, cudaStream_t stream);

/* Loss and gradient of a minibatch of environment segments with advantages
 * from fresh values ("Teaching Mario to speedrun", sec. 8): the rows are
 * (t, d_envs[j]) for t < T, j < ns (batch row t*N + d_envs[j]), in the order
 * t*ns + j.  After the forward pass, the value of every row (adv_mode 1: GAE)
 * and, for V-trace (adv_mode 2), the ratio exp(logp - logp_old) of its action
 * feed ppo_segment_advantage's recursion (clips from the config); the
 * advantages are normalised over the minibatch and the loss uses ret = A + V
 * as the value target.  d_rew, d_done [T][N], d_boot [N]; other inputs as in
 * ppo_minibatch_loss_grad (B = T*N).  The gradient overwrites the context's
 * gradient buffer; d_stats6 as there.  d_adv_out / d_ret_out (nullable, fp32
 * [T*ns]) receive the normalised advantages and the value targets.
 * 1 <= T*ns <= max_minibatch; adv_mode 1 or 2. */
ppo_status ppo_minibatch_loss_grad_fresh(ppo_ctx *ctx, const float *d_obs,
                                         const int32_t *d_act_disc, const float *d_act_cont,
                                         const float *d_logp_old, const float *d_rew,
                                         const float *d_done, const float *d_boot, int64_t T,
                                         int64_t N, const int32_t *d_envs, int64_t ns,
                                         int32_t adv_mode, float gamma, float lambda,
                                         float *d_stats6, float *d_adv_out, float *d_ret_out,
                                         cudaStream_t stream);

/* ---- Rollout-side policy step -------------------------------------------------
 * "Teaching Mario to speedrun", sec. 6 "The whole algorithm", step 1, and
 * sec. 7 (the trainer's side of a horizon): for the N agents of one
 * environment step, logits and value from the context's current policy, an
 * action sampled from the logits, and the log-probability of that action
 * (the learner's logp_old).  The forward pass is the learner's (bf16 tensor
 * cores in bf16 mode).  Sampling (the pages leave it open; the plainest
 * reading): per discrete head, the first category whose cumulative softmax
 * probability exceeds a uniform u; per Gaussian dimension
 * mu + exp(logstd) sqrt(-2 ln(1 - u1)) cos(2 pi u2).  The uniforms are
 * u = (x >> 8) / 2^24 for x = draw number draw0 + i*K + k of the mulberry32
 * stream seeded with `seed` ("PlayTrain", Appendix F.2), agent i, slot k
 * (head h: slot h; Gaussian dim g: slots n_heads + 2g and n_heads + 2g + 1),
 * K = n_heads + 2 n_gauss; a horizon advances draw0 by N*K per step.
 * Inputs  d_obs fp32 [N][obs_dim].
 * Outputs d_act_disc int32 [N][n_heads]; d_act_cont fp32 [N][n_gauss] (may
 *         be NULL if n_gauss == 0); d_logp fp32 [N] (nullable) the
 *         log-probability of the stored action; d_value fp32 [N] (nullable).
 * 1 <= N <= max_minibatch (the minibatch workspace holds the activations, so
 * calls on one context are ordered by its stream); h2 <= 512
 * (PPO_ERR_UNSUPPORTED otherwise).  Deterministic: a function of the
 * parameters, the observations, seed and draw0. */
ppo_status ppo_policy_act(ppo_ctx *ctx, const float *d_obs, int64_t N, uint32_t seed,
                          uint64_t draw0, int32_t *d_act_disc, float *d_act_cont, float *d_logp,
                          float *d_value, cudaStream_t stream);

/* ---- Optimizer step ---------------------------------------------------------
 * "PlayTrain", Table 8 (PPO column): Adam with gradient-norm clip.
 * Scales the context gradient by min(1, max_grad_norm/(||g||_2 + 1e-6)) when
 * max_grad_norm > 0, then one bias-corrected Adam step with learning rate
 * lr; increments the step counter and refreshes the bf16 weight shadows.
 * d_grad_norm (nullable, fp32 [1]) receives ||g||_2 before clipping. */
ppo_status ppo_adam_step(ppo_ctx *ctx, float lr, float *d_grad_norm, cudaStream_t stream);

/* Muon step ("Teaching Mario to speedrun", sec. 8 and "puff-rs": the 5.0
 * optimizer orthogonalises each weight matrix's update with five
 * Newton-Schulz iterations).  Definition from Muon's published write-up:
 * after the gradient-norm clip (as in ppo_adam_step), for each weight matrix
 * W (rows x cols) with momentum buffer mom (context-owned, zero at creation):
 *   mom = muon_beta mom + g;  u = g + muon_beta mom  (Nesterov);
 *   X = u / (||u||_F + 1e-7) as an r x k matrix, r = min(rows, cols);
 *   five times: A = X X^T, B = b A + c A A, X = a X + B X,
 *     (a, b, c) = (3.4445, -4.7750, 2.0315);
 *   W -= muon_lr sqrt(max(1, rows / cols)) X.
 * The biases and log-std take the Adam step of ppo_adam_step with rate lr.
 * The Newton-Schulz products run in fp32 (the write-up uses bf16).  Requires
 * a context created with optimizer == 1 (PPO_ERR_INVALID otherwise);
 * increments the step counter; d_grad_norm as in ppo_adam_step. */
ppo_status ppo_muon_step(ppo_ctx *ctx, float lr, float *d_grad_norm, cudaStream_t stream);

/* ---- Recurrent (MinGRU) policy ------------------------------------------------
 * "Teaching Mario to speedrun", sec. 8 "The Puffer net, and the trainer":
 * bias-free encoder (obs_dim -> hidden), `layers` MinGRU layers, one decoder
 * matrix to every head's logits, the Gaussian means and the value.  MinGRU
 * (Feng et al. 2024, "Were RNNs All We Needed?"), layer input u, state h:
 *   z = sigmoid(W_z u + b_z),  h~ = W_h u + b_h,  h_t = (1 - z) h_{t-1} + z h~;
 * the state entering step t is cleared when the episode ended at step t - 1
 * (d_done[t-1][n] != 0).  Parameter layout (fp32): W_enc[hidden][obs_dim];
 * per layer W_z[hidden][hidden], b_z[hidden], W_h[hidden][hidden],
 * b_h[hidden]; W_dec[C][hidden]; logstd[n_gauss]. */
typedef struct {
    int32_t obs_dim, hidden, layers;  /* hidden 1..256, layers 1..8             */
    int32_t n_heads;
    int32_t head_n[PPO_MAX_HEADS];
    int32_t n_gauss;                  /* 0..4; C = sum(head_n) + n_gauss + 1 <= 32 */
    float clip, vf_coef, ent_coef;
    int32_t precision;                /* 0 = fp32 CUDA-core products,
                                         1 = bf16 tensor-core (tcgen05) products,
                                             fp32 accumulate; hidden 128 or 256 */
    /* the update (ppo_rnn_update): gradient-norm clip and Adam */
    float max_grad_norm;
    double beta1, beta2, adam_eps;
} ppo_rnn_config;

ppo_status ppo_rnn_param_count(const ppo_rnn_config *cfg, int64_t *n);
ppo_status ppo_rnn_workspace_bytes(const ppo_rnn_config *cfg, int64_t T, int64_t ns,
                                   size_t *bytes);
/* Loss (sec. 6, as ppo_minibatch_loss_grad) and gradient of a minibatch of
 * environment segments d_envs[0..ns) (rows t*N + d_envs[j], t < T), with
 * backpropagation through time inside each segment; d_h0 (fp32 [N][layers]
 * [hidden]) is the state carried into the horizon, a constant of the loss.
 * d_obs [T*N][obs_dim], d_act_disc [T*N][n_heads], d_act_cont [T*N][n_gauss],
 * d_logp_old, d_adv, d_ret [T*N], d_adv_stats nullable ({mean, std}: the
 * advantage used is (adv - mean)/(std + 1e-8)), d_done [T][N].  d_grad
 * (param_count floats) is overwritten; d_stats6 as in
 * ppo_minibatch_loss_grad.  precision 0: fp32 CUDA-core kernels; precision
 * 1: the products (encoder, gate and candidate pre-activations, input
 * gradients, weight gradients) on the tensor cores with bf16 operands -- the
 * weights, the observations, each layer's input, the stored pre-activations,
 * dL/dz, the pre-activation and input gradients -- and fp32 accumulation;
 * the recurrence, the loss and the bias gradients in fp32.  In precision 1
 * the first int32 of d_work is set nonzero if a bounded device wait of the
 * call gave up (the outputs are then unspecified).  Deterministic. */
ppo_status ppo_rnn_loss_grad(const ppo_rnn_config *cfg, const float *d_params, int64_t T,
                             int64_t N, const int32_t *d_envs, int64_t ns, const float *d_obs,
                             const int32_t *d_act_disc, const float *d_act_cont,
                             const float *d_logp_old, const float *d_adv, const float *d_ret,
                             const float *d_adv_stats, const float *d_done, const float *d_h0,
                             float *d_grad, float *d_stats6, void *d_work, size_t work_bytes,
                             cudaStream_t stream);

/* Update of the recurrent policy ("Teaching Mario to speedrun", sec. 6 "The
 * whole algorithm" with sec. 8's policy and its carried state).  The context
 * owns the parameters (fp32, layout above), the gradient, Adam's m and v and
 * the workspaces for rollouts of up to max_T steps x max_N environments and
 * max_epochs epochs.  ppo_rnn_update: GAE (gamma, lambda, terminals as in
 * ppo_gae) over d_val/d_rew/d_done [T][N] and d_boot [N]; the statistics of
 * all T*N advantages; per epoch e the mulberry32 permutation of the N
 * environments (the rule of ppo_minibatch_perm, B = N); per minibatch k the
 * segments perm_e[k*ns .. (k+1)*ns), ns = N / minibatches, with the loss and
 * gradient of ppo_rnn_loss_grad (normalised advantages, d_h0 [N][layers]
 * [hidden] the state carried into the horizon), the gradient-norm clip
 * (max_grad_norm) and Adam (lr, beta1, beta2, adam_eps of the config).
 * d_obs [T*N][obs_dim], d_act_disc [T*N][n_heads], d_act_cont [T*N][n_gauss]
 * (NULL if n_gauss == 0), d_logp_old [T*N]; d_stats (nullable) fp32
 * [epochs*minibatches][6].  minibatches must divide N.  Asynchronous on
 * `stream`; ppo_rnn_sync_status synchronises it and returns PPO_ERR_TIMEOUT
 * once if a bounded device wait gave up since the last call. */
typedef struct ppo_rnn_ctx ppo_rnn_ctx;
ppo_status ppo_rnn_create(const ppo_rnn_config *cfg, const float *h_init_params, int64_t max_T,
                          int64_t max_N, int32_t max_epochs, ppo_rnn_ctx **out);
ppo_status ppo_rnn_destroy(ppo_rnn_ctx *ctx);
ppo_status ppo_rnn_buffers(ppo_rnn_ctx *ctx, float **d_params, float **d_grad, float **d_m,
                           float **d_v);
ppo_status ppo_rnn_update(ppo_rnn_ctx *ctx, const float *d_obs, const int32_t *d_act_disc,
                          const float *d_act_cont, const float *d_logp_old, const float *d_val,
                          const float *d_rew, const float *d_done, const float *d_boot,
                          const float *d_h0, int64_t T, int64_t N, int32_t epochs,
                          int32_t minibatches, float gamma, float lambda, float lr, uint32_t seed,
                          float *d_stats, cudaStream_t stream);
ppo_status ppo_rnn_sync_status(ppo_rnn_ctx *ctx, cudaStream_t stream);

/* ---- Whole update -------------------------------------------------------------
 * "Teaching Mario to speedrun", sec. 6 "The whole algorithm", steps 2-3:
 * GAE (gamma, lambda) over the [T,N] rollout, advantage statistics over all
 * T*N entries, then for e in [0, epochs): permutation of epoch e (seed), and
 * for m in [0, minibatches): loss+gradient of minibatch m, clip, Adam(lr).
 * With adv_mode 1/2 (ppo_config) the minibatches are environment segments
 * whose advantages are recomputed from fresh values before each loss (GAE
 * or V-trace; d_val is then unused); with optimizer 1 the step is Muon on
 * the weight matrices and Adam(lr) on the biases and log-std.
 * d_obs..d_boot as above (d_val, d_rew, d_done [T,N]; d_boot [N]).
 * d_stats (nullable): fp32 [epochs*minibatches][6] minibatch stats.
 * T*N must be divisible by minibatches; T*N <= max_batch; epochs <=
 * max_epochs; T*N/minibatches <= max_minibatch.  Launched as one CUDA graph
 * (captured on `stream` on the first call with a given argument set; the
 * stream must not be the legacy default stream). */
ppo_status ppo_update(ppo_ctx *ctx, const float *d_obs, const int32_t *d_act_disc,
                      const float *d_act_cont, const float *d_logp_old, const float *d_val,
                      const float *d_rew, const float *d_done, const float *d_boot,
                      int64_t T, int64_t N, int32_t epochs, int32_t minibatches,
                      float gamma, float lambda, float lr, uint32_t seed, float *d_stats,
                      cudaStream_t stream);

/* Same update, from HOST arrays (ideally pinned): copies the rollout into
 * context-owned device buffers, runs ppo_update, copies the stats back into
 * h_stats (nullable, fp32 [epochs*minibatches][6]) and returns when all of
 * it is done.  h_act_cont may be NULL if n_gauss == 0.  Waits first for any
 * ppo_update_host_async still in flight. */
ppo_status ppo_update_host(ppo_ctx *ctx, const float *h_obs, const int32_t *h_act_disc,
                           const float *h_act_cont, const float *h_logp_old, const float *h_val,
                           const float *h_rew, const float *h_done, const float *h_boot,
                           int64_t T, int64_t N, int32_t epochs, int32_t minibatches,
                           float gamma, float lambda, float lr, uint32_t seed, float *h_stats,
                           cudaStream_t stream);

/* Pipelined form of ppo_update_host: enqueues the copies, the update and the
 * stats copy-back and returns without waiting for them, so that the copies
 * of one call run on the copy engines while the previous call's update
 * computes.  The context stages rollouts in two device slots, used in turn.
 * Before enqueueing, a call waits on the host until the call two before it
 * (the last user of its slot) has completed: on return from call k, the
 * update of call k-2 is done, its h_stats written and its host arrays no
 * longer read.  The arrays of calls k-1 and k must stay unchanged, and their
 * h_stats unread, until a later call returns or ppo_host_wait does.
 * The copies overlap compute only from page-locked host memory (pageable
 * arrays still give correct results, without the overlap).  Successive
 * calls belong on one stream; a call on another stream first waits for the
 * calls in flight.  Arguments and errors as ppo_update_host; on an error
 * nothing of the call is enqueued except possibly its copies. */
ppo_status ppo_update_host_async(ppo_ctx *ctx, const float *h_obs, const int32_t *h_act_disc,
                                 const float *h_act_cont, const float *h_logp_old,
                                 const float *h_val, const float *h_rew, const float *h_done,
                                 const float *h_boot, int64_t T, int64_t N, int32_t epochs,
                                 int32_t minibatches, float gamma, float lambda, float lr,
                                 uint32_t seed, float *h_stats, cudaStream_t stream);

/* Waits until every ppo_update_host_async of the context has completed
 * (updates done, stats on the host, host arrays free). */
ppo_status ppo_host_wait(ppo_ctx *ctx);

/* ---- Profiling -----------------------------------------------------------------
 * The library's kernels, by stage; one stage entry is one kernel launch.
 * Entries PPO_NUM_KERNEL_STAGES .. PPO_NUM_STAGES-1 ("phase:*") are the
 * phases inside the persistent minibatch kernel (time between the phase
 * starts seen by its first CTA, summed over minibatches); they are not
 * separate launches. */
#define PPO_NUM_KERNEL_STAGES 25
#define PPO_NUM_STAGES 34
/* Name of a stage (static string; "unknown" outside [0, PPO_NUM_STAGES)). */
const char *ppo_stage_name(int32_t stage);

/* Runs one whole update exactly as ppo_update would (same arguments, same
 * effect on parameters, Adam state and step counter), from a CUDA graph in
 * which a CUDA event is recorded after every kernel, then returns per stage
 * the summed device time in milliseconds (h_stage_ms[PPO_NUM_STAGES], HOST)
 * and the number of launches (h_stage_launches[PPO_NUM_STAGES], HOST).  A
 * launch's time is the interval since the previous kernel's event, so it
 * includes its own launch gap.  Phase entries hold times within the
 * persistent kernel's launches.  Synchronous; `stream` must not be the legacy
 * default stream. */
ppo_status ppo_update_profile(ppo_ctx *ctx, const float *d_obs, const int32_t *d_act_disc,
                              const float *d_act_cont, const float *d_logp_old,
                              const float *d_val, const float *d_rew, const float *d_done,
                              const float *d_boot, int64_t T, int64_t N, int32_t epochs,
                              int32_t minibatches, float gamma, float lambda, float lr,
                              uint32_t seed, float *d_stats, float *h_stage_ms,
                              int32_t *h_stage_launches, cudaStream_t stream);

/* Synchronises `stream` and returns any error latched on the device since
 * the last call (PPO_ERR_TIMEOUT if a bounded wait gave up), clearing it. */
ppo_status ppo_sync_status(ppo_ctx *ctx, cudaStream_t stream);

/* ---- Data-parallel learner ---------------------------------------------------
 * "PlayTrain", App. C.3 (the learner trained data-parallel over GPUs with DDP,
 * Table 8 "2 DDP + 2 inference GPUs"), applied to the update of sec. 6 of
 * "Teaching Mario to speedrun".  With world > 1, each of `world` processes
 * (one GPU each) calls ppo_update on its own shard of environments -- the
 * [T, N_r] rollout of its N_r envs, the same T, epochs, minibatches and
 * seed on every rank, the same N_r on every rank -- and the update becomes:
 *   GAE on the shard; the shard's advantage moments (count, mean, M2) in
 *   fp64, all-gathered, merged in a fixed order into the global mean and
 *   std (every rank the same values); per epoch the shard's own
 *   permutation by the single-GPU rule (seed, epoch, B_r = T*N_r); minibatch
 *   m is the union of the ranks' m-th slices, so the loss of rank r's rows
 *   is scaled by 1/(world * B_r/minibatches); after gradient assembly the
 *   flat gradient (and the minibatch statistics) are sum-all-reduced, and
 *   every rank takes the same clip + optimizer step.
 * The library issues its collectives through `fn`, called on the host while
 * the update is enqueued, in the same order on every rank:
 *   op PPO_COLL_ALLREDUCE_SUM_F32: d_buf fp32 [count], summed in place over
 *     the ranks;
 *   op PPO_COLL_ALLGATHER_F64: d_buf fp64 [world][count], this rank's count
 *     values at d_buf + rank*count on entry, every rank's on return;
 * each enqueued on `stream` (device pointers, stream order); fn returns 0 on
 * success (anything else: the update returns PPO_ERR_CUDA).  The Python
 * binding supplies one over torch.distributed.  With world > 1 ppo_update is
 * enqueued directly rather than from a cached CUDA graph; the fresh-advantage
 * modes (adv_mode 1, 2), the persistent minibatch kernel and
 * ppo_update_profile return PPO_ERR_UNSUPPORTED.  world == 1 (the default)
 * restores the single-GPU update; fn may then be NULL. */
typedef enum {
    PPO_COLL_ALLREDUCE_SUM_F32 = 0,
    PPO_COLL_ALLGATHER_F64 = 1
} ppo_collective_op;
typedef int (*ppo_collective_fn)(void *user, int32_t op, void *d_buf, int64_t count,
                                 cudaStream_t stream);
ppo_status ppo_set_collective(ppo_ctx *ctx, int32_t world, int32_t rank, ppo_collective_fn fn,
                              void *user);

/* ---- Inspection and failure handling ----------------------------------------
 * Step trace of the whole update ("Teaching Mario to speedrun", sec. 6 "The
 * whole algorithm": one backward pass and one optimizer step per minibatch).
 * With a trace set, ppo_update records for minibatch step j (j = e *
 * minibatches + m, the first max_steps steps of each update) into
 * d_trace + j*4*P (P = ppo_param_count) four fp32 vectors of P values:
 *   [0] the parameters before the step, [1] Adam's m and [2] Adam's v before
 *   the step, [3] the assembled gradient of the step's minibatch (before the
 *   gradient-norm clip).
 * The copies are device-to-device on the update's stream, inside its graph;
 * the kernels and their results are unchanged.  d_trace (DEVICE, 16-byte
 * aligned, max_steps*4*P floats, owned by the caller, kept until the trace is
 * cleared or the context destroyed); d_trace NULL with max_steps 0 clears it.
 * The next ppo_update re-captures its graph. */
ppo_status ppo_set_step_trace(ppo_ctx *ctx, float *d_trace, int64_t max_steps);

/* Limit, in nanoseconds of the GPU's global timer, of the bounded waits of
 * the cooperative kernels for one another's blocks: the grid barrier of
 * gradient assembly + Adam inside ppo_update, those of the fresh-advantage
 * kernel, and the weight-gradient kernel's wait for the other blocks of its
 * output tile (taken after its own copies have completed and its tensor
 * memory is freed).  A wait that runs past it latches PPO_ERR_TIMEOUT
 * (returned by the next ppo_sync_status); the kernel then skips the rest of
 * its work and returns, with no asynchronous copy or tensor memory held.  The results of an update that timed out are
 * undefined; the next update starts from cleared barrier counters.  0
 * restores the default (2 s).  The tensor-core kernels' pipeline waits keep
 * their own 2 s limit.  The next ppo_update re-captures its graph. */
ppo_status ppo_set_wait_limit(ppo_ctx *ctx, uint64_t limit_ns);

#ifdef __cplusplus
}
#endif
#endif /* PPO_H */
