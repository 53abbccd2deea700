/*
 * ppo_oracle.h -- plain CPU reference of the PPO learner step.
 *
 * TEST INFRASTRUCTURE ONLY.  This is the slow, obviously-correct restatement
 * of what the learner step computes, written from the pages' text in fp64.
 * It exists so that tests, the package smoke check and the bench's CPU
 * baseline leg can compare against it.  The CUDA library never includes,
 * links or calls anything here, and this code includes nothing of the CUDA
 * library: the two share no code.
 *
 * Sources (page title, section):
 *   "Teaching Mario to speedrun" (bigmah.com rl_blog) sec. 4  -- discounted return
 *   same page, sec. 5  -- gradient of a log-softmax: (a == action) - probs[a]
 *   same page, sec. 6 "Better advantages" -- delta_t and the GAE sum
 *   same page, sec. 6 "Don't move too far at once" -- clipped ratio, value and
 *                     entropy terms and their weights
 *   same page, sec. 6 "The whole algorithm" -- epochs x shuffled minibatches,
 *                     backward, optimizer step
 *   same page, sec. 7 -- terminals are 1 where an episode just ended
 *   "PlayTrain" (arXiv 2609.09059) Table 8 -- Adam, grad-norm clip 0.5, PPO
 *                     hyper-parameters
 *   "PlayTrain" Appendix F.2 listing "seeded RNG" -- mulberry32 definition
 *   "boesch.dev DDNet RL" sec. "What the agent sees and does" -- hybrid
 *                     discrete + continuous action space (diagonal Gaussian)
 */
#ifndef PPO_ORACLE_H
#define PPO_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* One draw of mulberry32; *state is the generator's 32-bit counter. */
uint32_t orc_mulberry32_next(uint32_t *state);

/* GAE over a [T,N] rollout (time-major, env fastest).  done[t,n] != 0 means
 * the episode ended during step t: rew[t,n] is its last reward, nothing is
 * bootstrapped across it.  boot[n] is V(s_T).  Outputs adv, ret [T,N]. */
void orc_gae(int64_t T, int64_t N, const float *rew, const float *val,
             const float *done, const float *boot, double gamma, double lambda,
             double *adv, double *ret);

/* Advantages of whole environment segments from given values: V-trace
 * (Espeholt et al. 2018, sec. 4.1) with rho = min(rho_clip, ratio) and
 * c = lambda min(c_clip, ratio); ratio == NULL gives GAE (rho = 1, c = lambda).
 * Segment j is environment envs[j]; val, ratio, adv, ret are [T][ns]
 * (element t*ns + j); rew, done [T][N]; boot [N].  adv = v - V, ret = v. */
void orc_segment_advantage(int64_t T, int64_t N, const float *rew, const float *done,
                           const float *boot, int64_t ns, const int32_t *envs,
                           const double *val, const double *ratio, double gamma,
                           double lambda, double rho_clip, double c_clip, double *adv,
                           double *ret);

/* Mean and unbiased (n-1) standard deviation, two passes. */
void orc_moments(int64_t n, const double *x, double *mean, double *std_unbiased);

/* out[i] = (x[i] - mean) / (std + 1e-8) */
/* (count, mean, M2) of x[0..n) (two-pass), and the pairwise merge of two
 * such triples (Chan, Golub and LeVeque); out may alias a or b. */
void orc_moments3(int64_t n, const double *x, double out[3]);
void orc_moments_merge(const double a[3], const double b[3], double out[3]);
void orc_normalize(int64_t n, const double *x, double mean, double std_, double *out);

/* Minibatch permutation of epoch `epoch`: key i = mulberry32 draw number
 * epoch*B + i of the stream seeded with `seed`; perm lists 0..B-1 sorted by
 * (key, index). */
void orc_perm(uint32_t seed, int64_t epoch, int64_t B, int32_t *perm);

/* MLP actor-critic.  Output columns: head logits in head order, then the
 * Gaussian means, then the value.  act: 0 = tanh, 1 = ReLU. */
typedef struct {
    int32_t obs_dim, h1, h2, act;
    int32_t n_heads;
    int32_t head_n[8];
    int32_t n_gauss;
} orc_net;

/* Number of output columns C = sum(head_n) + n_gauss + 1. */
int64_t orc_out_cols(const orc_net *net);
/* Flat parameter count.  Layout: W1[h1][D], b1[h1], W2[h2][h1], b2[h2],
 * W3[C][h2], b3[C], logstd[n_gauss]. */
int64_t orc_num_params(const orc_net *net);

/* x rounded to fp32, then to bfloat16, both to nearest even (the rounding of
 * the bf16-operand mode below). */
double orc_round_bf16(double x);

/* Forward pass of one observation; z has C entries. */
void orc_forward(const orc_net *net, const double *params, const float *x, double *z);

/* Per-row log-probability of the given action and policy entropy at params
 * (rows 0..n of obs [n][D], act_disc [n][n_heads], act_cont [n][n_gauss]). */
void orc_policy_logp(const orc_net *net, const double *params, int64_t n, const float *obs,
                     const int32_t *act_disc, const float *act_cont, double *logp, double *ent);

typedef struct {
    double clip, vf_coef, ent_coef;
    /* 0: every product in fp64.  1: bf16-operand mode -- the operands of
     * every GEMM (observation, weights W1..W3, stored activations, the
     * backpropagated signals dz, dpre2, dpre1) are rounded to bfloat16 where
     * a bf16 tensor-core implementation stores them; sums stay in fp64 and
     * bias gradients use the unrounded signals. */
    int bf16_operands;
} orc_loss_cfg;

/* Loss and gradient of one minibatch.
 * rows idx[0..mb) select from the full-batch arrays obs [B][D],
 * act_disc [B][n_heads], act_cont [B][n_gauss], logp_old [B], adv [B], ret [B].
 * If normalize != 0 the advantage used is (adv - adv_mean)/(adv_std + 1e-8).
 * grad (length num_params) is OVERWRITTEN with dL/dparams.
 * stats6 = {loss, pg_loss, v_loss, entropy, clipfrac, approx_kl} (means).
 * scale6 = mean |per-row term| of the same six quantities (may be NULL);
 *          used by tests to form absolute tolerances for near-zero means.
 * Returns the loss. */
/* Number of threads the OpenMP row loops use (1 when built without OpenMP). */
int orc_threads(void);
/* Sets the thread count of those loops (no effect without OpenMP). */
void orc_set_threads(int n);

double orc_loss_grad(const orc_net *net, const orc_loss_cfg *cfg, const double *params,
                     int64_t mb, const int32_t *idx,
                     const float *obs, const int32_t *act_disc, const float *act_cont,
                     const float *logp_old, const double *adv, const double *ret,
                     int normalize, double adv_mean, double adv_std,
                     double *grad, double *stats6, double *scale6);

/* Fresh values (value column at params) and ratios exp(logp - logp_old) of
 * rows idx[0..n).  bf16: operand rounding as in orc_loss_cfg.  ratio nullable. */
void orc_fresh_values(const orc_net *net, int bf16, const double *params, int64_t n,
                      const int32_t *idx, const float *obs, const int32_t *act_disc,
                      const float *act_cont, const float *logp_old, double *val, double *ratio);

/* Loss and gradient of the minibatch of environment segments envs[0..ns)
 * (rows t*N + envs[j], in the order t*ns + j) with advantages from fresh
 * values: GAE (vtrace 0) or V-trace (vtrace 1), normalised over the
 * minibatch.  adv_norm_out / ret_out nullable [T*ns].  Returns the loss. */
double orc_loss_grad_fresh(const orc_net *net, const orc_loss_cfg *cfg, const double *params,
                           int64_t T, int64_t N, int64_t ns, const int32_t *envs,
                           const float *obs, const int32_t *act_disc, const float *act_cont,
                           const float *logp_old, const float *rew, const float *done,
                           const float *boot, int vtrace, double gamma, double lambda,
                           double rho_clip, double c_clip, double *grad, double *stats6,
                           double *scale6, double *adv_norm_out, double *ret_out);

/* Rollout-side policy step (sample actions for n agents at params): see
 * ppo_oracle.c.  act [n][n_heads] int32, actc [n][n_gauss], logp [n] (of the
 * sampled action, Gaussian part at the fp32-rounded action), value [n].
 * bf16: operand rounding as in orc_loss_cfg. */
double orc_uniform24(uint32_t x);
uint32_t orc_mulberry32_at(uint32_t seed, uint64_t draw);
int orc_sample_categorical(const double *z, int n, double u);
double orc_box_muller(double u1, double u2);
void orc_policy_act(const orc_net *net, int bf16, const double *params, int64_t n,
                    const float *obs, uint32_t seed, uint64_t draw0, int32_t *act,
                    double *actc, double *logp, double *value);

/* Recurrent policy (see ppo_oracle.c): bias-free encoder, `layers` MinGRU
 * layers of width `hidden`, bias-free decoder to the head columns. */
typedef struct {
    int32_t obs_dim, hidden, layers;
    int32_t n_heads;
    int32_t head_n[8];
    int32_t n_gauss;
} orc_rnn;
int64_t orc_rnn_out_cols(const orc_rnn *r);
int64_t orc_rnn_num_params(const orc_rnn *r);
void orc_rnn_forward(const orc_rnn *r, const double *params, int64_t T, int64_t N, int64_t n,
                     const float *obs, const float *done, const double *h0, double *zout,
                     double *su, double *sz, double *sht, double *shp, double *sh);
double orc_rnn_loss_grad(const orc_rnn *r, const orc_loss_cfg *cfg, const double *params,
                         int64_t T, int64_t N, int64_t ns, const int32_t *envs,
                         const float *obs, const int32_t *act_disc, const float *act_cont,
                         const float *logp_old, const double *adv, const double *ret,
                         int normalize, double adv_mean, double adv_std, const float *done,
                         const double *h0, double *grad, double *stats6, double *scale6);

/* L2 norm of g; if max_norm > 0, g *= min(1, max_norm/(norm + 1e-6)).
 * Returns the norm before clipping. */
double orc_clip_grad_norm(int64_t P, double *g, double max_norm);

/* One Adam step (bias-corrected); `step` is the 1-based step number. */
void orc_adam(int64_t P, double *p, const double *g, double *m, double *v, int64_t step,
              double lr, double beta1, double beta2, double eps);

/* Muon ("Muon: An optimizer for hidden layers in neural networks"): the
 * quintic Newton-Schulz orthogonalisation of a rows x cols matrix (steps
 * iterations), and one Muon step of the MLP (matrices W1..W3 by Muon with
 * Nesterov momentum mom, biases and log-std by Adam).  See ppo_oracle.c. */
void orc_newton_schulz5(int64_t rows, int64_t cols, const double *G, int steps, double *out);
/* The same with X, A, B stored as bf16 (each product rounded once computed). */
void orc_newton_schulz5_bf16(int64_t rows, int64_t cols, const double *G, int steps,
                             double *out);
void orc_muon(const orc_net *net, double *params, const double *g, double *mom,
              double *adam_m, double *adam_v, int64_t step, double muon_lr, double muon_beta,
              double lr, double beta1, double beta2, double eps);
/* orc_muon with the bf16 Newton-Schulz iteration (orc_newton_schulz5_bf16). */
void orc_muon_bf16(const orc_net *net, double *params, const double *g, double *mom,
                   double *adam_m, double *adam_v, int64_t step, double muon_lr,
                   double muon_beta, double lr, double beta1, double beta2, double eps);

typedef struct {
    double gamma, lambda, clip, vf_coef, ent_coef;
    double lr, beta1, beta2, adam_eps, max_grad_norm;
    uint32_t seed;
    int bf16_operands;   /* as in orc_loss_cfg */
    int adv_mode;        /* 0: GAE once per update over the whole rollout;
                            1: per minibatch of env segments, GAE from fresh values;
                            2: the same with V-trace */
    double rho_clip, c_clip;   /* V-trace truncation levels (adv_mode 2) */
    int optimizer;             /* 0 Adam; 1 Muon for the weight matrices (orc_muon) */
    double muon_lr, muon_beta;
} orc_hyper;

/* One whole PPO update: GAE, global advantage statistics, then for each epoch
 * a fresh permutation and M minibatch steps (loss+grad, norm clip, Adam).
 * adv_mode 1/2: each epoch permutes the N environments instead, minibatch k
 * is the segments of envs perm[k*N/M .. (k+1)*N/M) with orc_loss_grad_fresh,
 * and adv_out/ret_out are not written.
 * params, m, v are updated in place; *step is incremented per minibatch.
 * stats (E*M*6) receives the per-minibatch stats6.  adv_out/ret_out [T*N]
 * may be NULL. */
void orc_update(const orc_net *net, const orc_hyper *hp, int64_t T, int64_t N,
                int64_t epochs, int64_t minibatches,
                const float *obs, const int32_t *act_disc, const float *act_cont,
                const float *logp_old, const float *val, const float *rew,
                const float *done, const float *boot,
                double *params, double *m, double *v, double *mom, int64_t *step,
                double *stats, double *adv_out, double *ret_out);

/* One update of the recurrent policy: GAE, global advantage statistics, per
 * epoch an environment permutation and minibatches of whole segments with
 * orc_rnn_loss_grad, clip and Adam (see ppo_oracle.c).  h0 [N][layers][hidden].
 * Returns -1 unless minibatches >= 1 divides N. */
int orc_rnn_update(const orc_rnn *r, const orc_hyper *hp, int64_t T, int64_t N, int64_t epochs,
                   int64_t minibatches, const float *obs, const int32_t *act_disc,
                   const float *act_cont, const float *logp_old, const float *val,
                   const float *rew, const float *done, const float *boot, const double *h0,
                   double *params, double *m, double *v, int64_t *step, double *stats);

/* The update data-parallel over `world` ranks, emulated in one process: rank
 * r holds envs [r N/world, (r+1) N/world) of the [T][N] rollout; shard GAE,
 * statistics from the merged shard moments, per-rank permutations of the
 * shard's rows, minibatch k = the union of the ranks' k-th slices, gradient
 * = mean over the ranks (see ppo_oracle.c).  Returns -1 unless world divides
 * N and minibatches divides T*N/world. */
int orc_update_sharded(const orc_net *net, const orc_hyper *hp, int64_t world, int64_t T,
                       int64_t N, int64_t epochs, int64_t minibatches, const float *obs,
                       const int32_t *act_disc, const float *act_cont, const float *logp_old,
                       const float *val, const float *rew, const float *done, const float *boot,
                       double *params, double *m, double *v, double *mom, int64_t *step,
                       double *stats);

#ifdef __cplusplus
}
#endif
#endif
