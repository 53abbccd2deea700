/*
 * ppo_oracle.c -- plain CPU reference of the PPO learner step (fp64).
 *
 * TEST INFRASTRUCTURE ONLY: used by tests/, the package smoke check and the
 * bench's CPU-baseline leg.  Shares no code with the CUDA library.
 * Every function follows the passage cited above it, in the pages' order;
 * sums run in the plain order of their definition, in double precision.
 */
#include "ppo_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ------------------------------------------------------------------------ */
/* "PlayTrain", Appendix F.2 listing "seeded RNG" (mulberry32).
 * The state is a counter advanced by 0x6D2B79F5 per draw; the output is a
 * xor-shift / multiply mix of it.  The listing's Math.imul and >>> are 32-bit
 * wrapping multiply and logical shift, i.e. uint32_t arithmetic here. */
uint32_t orc_mulberry32_next(uint32_t *state)
{
    uint32_t t = *state + 0x6D2B79F5u;
    *state = t;
    uint32_t n = (t ^ (t >> 15)) * (t | 1u);
    n ^= n + (n ^ (n >> 7)) * (n | 61u);
    return n ^ (n >> 14);
}

/* ------------------------------------------------------------------------ */
/* "Teaching Mario to speedrun", sec. 6 "Better advantages":
 *   delta_t = r_t + gamma V(s_{t+1}) - V(s_t)
 *   A_t     = delta_t + (gamma lambda) delta_{t+1} + (gamma lambda)^2 delta_{t+2} + ...
 * written as the backward recursion A_t = delta_t + gamma lambda A_{t+1}.
 * Sec. 7: terminals are 1 where an episode just ended, so a done at step t
 * stops both the bootstrap V(s_{t+1}) and the propagation of A_{t+1}.
 * The return used by the value loss is the lambda-return A_t + V(s_t). */
void orc_gae(int64_t T, int64_t N, const float *rew, const float *val,
             const float *done, const float *boot, double gamma, double lambda,
             double *adv, double *ret)
{
    for (int64_t n = 0; n < N; ++n) {
        double next_value = (double)boot[n];
        double next_adv = 0.0;
        for (int64_t t = T - 1; t >= 0; --t) {
            int64_t i = t * N + n;
            double alive = (done[i] != 0.0f) ? 0.0 : 1.0;
            double v = (double)val[i];
            double delta = (double)rew[i] + gamma * alive * next_value - v;
            double a = delta + gamma * lambda * alive * next_adv;
            adv[i] = a;
            ret[i] = a + v;
            next_value = v;
            next_adv = a;
        }
    }
}

/* ------------------------------------------------------------------------ */
/* "Teaching Mario to speedrun", sec. 8 "The Puffer net, and the trainer":
 * PufferLib 5.0 computes the advantages of each minibatch from fresh values,
 * by GAE or by V-trace.  The pages give V-trace no formula; it is taken from
 * its published definition (Espeholt et al. 2018, "IMPALA", sec. 4.1, eq. 1
 * and Remarks 1-2): with truncated importance weights
 * rho_t = min(rho_bar, pi/mu) and lambda-weighted traces
 * c_t = lambda min(c_bar, pi/mu), the value target is
 *   v_s = V(x_s) + sum_{t >= s} gamma^{t-s} (c_s ... c_{t-1}) rho_t delta_t,
 *   delta_t = r_t + gamma V(x_{t+1}) - V(x_t),
 * computed here by its backward recursion
 *   v_s - V(x_s) = rho_s delta_s + gamma c_s (v_{s+1} - V(x_{s+1})).
 * Terminals cut the bootstrap and the trace exactly as in orc_gae.  The
 * advantage is v_s - V(x_s) and the value target v_s, so that, as for GAE,
 * ret = adv + V.  ratio == NULL is on-policy GAE: rho = 1, c = lambda.
 * Segment j is environment envs[j] over the whole horizon; val, ratio, adv
 * and ret are [T][ns] (element t*ns + j); rew, done [T][N]; boot [N]. */
void orc_segment_advantage(int64_t T, int64_t N, const float *rew, const float *done,
                           const float *boot, int64_t ns, const int32_t *envs,
                           const double *val, const double *ratio, double gamma,
                           double lambda, double rho_clip, double c_clip, double *adv,
                           double *ret)
{
    for (int64_t j = 0; j < ns; ++j) {
        const int64_t n = envs[j];
        double next_value = (double)boot[n];
        double next_corr = 0.0;   /* v_{t+1} - V(x_{t+1}) */
        for (int64_t t = T - 1; t >= 0; --t) {
            const int64_t i = t * N + n, k = t * ns + j;
            const double alive = (done[i] != 0.0f) ? 0.0 : 1.0;
            double rho = 1.0, c = lambda;
            if (ratio) {
                rho = ratio[k] < rho_clip ? ratio[k] : rho_clip;
                c = lambda * (ratio[k] < c_clip ? ratio[k] : c_clip);
            }
            const double v = val[k];
            const double delta = (double)rew[i] + gamma * alive * next_value - v;
            const double corr = rho * delta + gamma * alive * c * next_corr;
            adv[k] = corr;
            ret[k] = v + corr;
            next_value = v;
            next_corr = corr;
        }
    }
}

/* Global advantage statistics: mean and the unbiased standard deviation. */
void orc_moments(int64_t n, const double *x, double *mean, double *std_unbiased)
{
    double s = 0.0;
    for (int64_t i = 0; i < n; ++i) s += x[i];
    double mu = (n > 0) ? s / (double)n : 0.0;
    double ss = 0.0;
    for (int64_t i = 0; i < n; ++i) ss += (x[i] - mu) * (x[i] - mu);
    *mean = mu;
    *std_unbiased = (n > 1) ? sqrt(ss / (double)(n - 1)) : 0.0;
}

/* (count, mean, M2) of x[0..n), M2 the sum of squared deviations from the
 * mean, by the two-pass definition. */
void orc_moments3(int64_t n, const double *x, double out[3])
{
    double s = 0.0;
    for (int64_t i = 0; i < n; ++i) s += x[i];
    const double mu = (n > 0) ? s / (double)n : 0.0;
    double ss = 0.0;
    for (int64_t i = 0; i < n; ++i) ss += (x[i] - mu) * (x[i] - mu);
    out[0] = (double)n;
    out[1] = mu;
    out[2] = ss;
}

/* The (count, mean, M2) of the union of two sets from theirs (Chan, Golub
 * and LeVeque's pairwise combination): with d = mean_b - mean_a,
 *   n = n_a + n_b,  mean = mean_a + d n_b / n,  M2 = M2_a + M2_b + d^2 n_a n_b / n.
 * out may alias a or b. */
void orc_moments_merge(const double a[3], const double b[3], double out[3])
{
    if (a[0] == 0.0) { out[0] = b[0]; out[1] = b[1]; out[2] = b[2]; return; }
    if (b[0] == 0.0) { out[0] = a[0]; out[1] = a[1]; out[2] = a[2]; return; }
    const double n = a[0] + b[0], d = b[1] - a[1];
    const double mean = a[1] + d * (b[0] / n);
    const double m2 = a[2] + b[2] + d * d * (a[0] * b[0] / n);
    out[0] = n;
    out[1] = mean;
    out[2] = m2;
}

void orc_normalize(int64_t n, const double *x, double mean, double std_, double *out)
{
    for (int64_t i = 0; i < n; ++i) out[i] = (x[i] - mean) / (std_ + 1e-8);
}

/* ------------------------------------------------------------------------ */
/* "Teaching Mario to speedrun", sec. 6: "for minibatch in shuffle(batch)".
 * The shuffle of epoch e sorts the indices by mulberry32 keys, key i being
 * draw number e*B + i of the stream seeded with `seed`; equal keys keep index
 * order.  Skipping e*B draws is adding e*B*0x6D2B79F5 to the counter. */
typedef struct { uint32_t key; int32_t idx; } orc_kv;

static int orc_kv_cmp(const void *a, const void *b)
{
    const orc_kv *x = (const orc_kv *)a, *y = (const orc_kv *)b;
    if (x->key != y->key) return x->key < y->key ? -1 : 1;
    return (x->idx > y->idx) - (x->idx < y->idx);
}

void orc_perm(uint32_t seed, int64_t epoch, int64_t B, int32_t *perm)
{
    orc_kv *kv = (orc_kv *)malloc((size_t)B * sizeof(orc_kv));
    uint32_t state = seed + (uint32_t)((uint64_t)epoch * (uint64_t)B) * 0x6D2B79F5u;
    for (int64_t i = 0; i < B; ++i) {
        kv[i].key = orc_mulberry32_next(&state);
        kv[i].idx = (int32_t)i;
    }
    qsort(kv, (size_t)B, sizeof(orc_kv), orc_kv_cmp);
    for (int64_t i = 0; i < B; ++i) perm[i] = kv[i].idx;
    free(kv);
}

/* ------------------------------------------------------------------------ */
/* "Teaching Mario to speedrun", sec. 6 "The policy and the value are one
 * network": observation in, one group of logits per action head plus one
 * value out.  The MLP is h1 = act(W1 x + b1), h2 = act(W2 h1 + b2),
 * z = W3 h2 + b3.  Hybrid action spaces ("boesch.dev DDNet RL", "What the
 * agent sees and does") add diagonal-Gaussian means before the value. */
int64_t orc_out_cols(const orc_net *net)
{
    int64_t c = 0;
    for (int h = 0; h < net->n_heads; ++h) c += net->head_n[h];
    return c + net->n_gauss + 1;
}

int64_t orc_num_params(const orc_net *net)
{
    int64_t D = net->obs_dim, H1 = net->h1, H2 = net->h2, C = orc_out_cols(net);
    return H1 * D + H1 + H2 * H1 + H2 + C * H2 + C + net->n_gauss;
}

typedef struct {
    const double *W1, *b1, *W2, *b2, *W3, *b3, *logstd;
} orc_views;

static orc_views orc_split(const orc_net *net, const double *p)
{
    int64_t D = net->obs_dim, H1 = net->h1, H2 = net->h2, C = orc_out_cols(net);
    orc_views v;
    v.W1 = p;
    v.b1 = v.W1 + H1 * D;
    v.W2 = v.b1 + H1;
    v.b2 = v.W2 + H2 * H1;
    v.W3 = v.b2 + H2;
    v.b3 = v.W3 + C * H2;
    v.logstd = v.b3 + C;
    return v;
}

static double orc_act(int act, double pre)
{
    return act == 0 ? tanh(pre) : (pre > 0.0 ? pre : 0.0);
}

/* derivative of the activation, from its input and output:
 * tanh' = 1 - tanh^2, ReLU' = 1[pre > 0] (0 at pre == 0). */
static double orc_act_grad(int act, double pre, double post)
{
    return act == 0 ? 1.0 - post * post : (pre > 0.0 ? 1.0 : 0.0);
}

/* bf16-operand mode: the value a bf16 tensor-core GEMM reads for operand x --
 * x rounded to fp32, then to bfloat16 (8-bit significand), both to nearest
 * even.  Identity when the mode is off. */
static double orc_bf16(double x)
{
    float f = (float)x;
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    if ((u & 0x7F800000u) != 0x7F800000u) u += 0x7FFFu + ((u >> 16) & 1u);
    u &= 0xFFFF0000u;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

static double orc_rnd(int bf16, double x) { return bf16 ? orc_bf16(x) : x; }

double orc_round_bf16(double x) { return orc_bf16(x); }

/* bf16-operand mode: the GEMMs read bf16-rounded weights; biases and
 * log-std stay in full precision.  Returns a rounded copy of params (caller
 * frees), or NULL when the mode is off. */
static double *orc_gemm_weights(const orc_net *net, const double *params, int bf16)
{
    if (!bf16) return NULL;
    const int64_t D = net->obs_dim, H1 = net->h1, H2 = net->h2, C = orc_out_cols(net);
    const int64_t P = orc_num_params(net);
    double *wr = (double *)malloc(sizeof(double) * (size_t)P);
    memcpy(wr, params, sizeof(double) * (size_t)P);
    orc_views v0 = orc_split(net, params);
    const int64_t nW1 = H1 * D, nW2 = H2 * H1, nW3 = C * H2;
    for (int64_t i = 0; i < nW1; ++i) wr[(v0.W1 - params) + i] = orc_bf16(v0.W1[i]);
    for (int64_t i = 0; i < nW2; ++i) wr[(v0.W2 - params) + i] = orc_bf16(v0.W2[i]);
    for (int64_t i = 0; i < nW3; ++i) wr[(v0.W3 - params) + i] = orc_bf16(v0.W3[i]);
    return wr;
}

/* Forward pass of one row.  In bf16-operand mode the observation and the
 * stored activations are rounded to bf16 (the weights are rounded by the
 * caller); the accumulation stays in double. */
static void orc_forward_full(const orc_net *net, const orc_views *w, const float *x,
                             double *pre1, double *h1, double *pre2, double *h2, double *z,
                             int bf16)
{
    int64_t D = net->obs_dim, H1 = net->h1, H2 = net->h2, C = orc_out_cols(net);
    for (int64_t j = 0; j < H1; ++j) {
        double s = w->b1[j];
        for (int64_t k = 0; k < D; ++k) s += w->W1[j * D + k] * orc_rnd(bf16, (double)x[k]);
        pre1[j] = s;
        h1[j] = orc_rnd(bf16, orc_act(net->act, s));
    }
    for (int64_t j = 0; j < H2; ++j) {
        double s = w->b2[j];
        for (int64_t k = 0; k < H1; ++k) s += w->W2[j * H1 + k] * h1[k];
        pre2[j] = s;
        h2[j] = orc_rnd(bf16, orc_act(net->act, s));
    }
    for (int64_t c = 0; c < C; ++c) {
        double s = w->b3[c];
        for (int64_t k = 0; k < H2; ++k) s += w->W3[c * H2 + k] * h2[k];
        z[c] = s;
    }
}

void orc_forward(const orc_net *net, const double *params, const float *x, double *z)
{
    orc_views w = orc_split(net, params);
    double *buf = (double *)malloc(sizeof(double) * 2 * (size_t)(net->h1 + net->h2));
    orc_forward_full(net, &w, x, buf, buf + net->h1, buf + 2 * net->h1,
                     buf + 2 * net->h1 + net->h2, z, 0);
    free(buf);
}

/* Log-probability of one row's action and the policy entropy, from the
 * row's output columns z: log-softmax per discrete head (probabilities
 * multiply over heads, so log-probabilities and entropies add), then the
 * diagonal-Gaussian dimensions.  logprob[] receives each head logit's
 * log-softmax, head_ent[] each head's entropy. */
static void orc_row_policy(const orc_net *net, const double *logstd, const double *z,
                           const int32_t *act, const float *actc, double *logprob,
                           double *head_ent, double *logp_out, double *ent_out)
{
    const double LOG_2PI = log(2.0 * acos(-1.0));
    double logp = 0.0, ent = 0.0;
    int64_t off = 0;
    for (int64_t h = 0; h < net->n_heads; ++h) {
        int64_t n = net->head_n[h];
        double zmax = z[off];
        for (int64_t k = 1; k < n; ++k) if (z[off + k] > zmax) zmax = z[off + k];
        double se = 0.0;
        for (int64_t k = 0; k < n; ++k) se += exp(z[off + k] - zmax);
        double lse = zmax + log(se);
        double eh = 0.0;
        for (int64_t k = 0; k < n; ++k) {
            logprob[off + k] = z[off + k] - lse;
            eh -= exp(logprob[off + k]) * logprob[off + k];
        }
        head_ent[h] = eh;
        ent += eh;
        logp += logprob[off + act[h]];
        off += n;
    }
    for (int64_t g = 0; g < net->n_gauss; ++g) {
        double mu = z[off + g], s = logstd[g];
        double a = (double)actc[g];
        double var = exp(2.0 * s);
        logp += -(a - mu) * (a - mu) / (2.0 * var) - s - 0.5 * LOG_2PI;
        ent += 0.5 + 0.5 * LOG_2PI + s;
    }
    *logp_out = logp;
    *ent_out = ent;
}

void orc_policy_logp(const orc_net *net, const double *params, int64_t n, const float *obs,
                     const int32_t *act_disc, const float *act_cont, double *logp, double *ent)
{
    const int64_t C = orc_out_cols(net);
    orc_views w = orc_split(net, params);
    /* rows are independent: with OpenMP each thread takes a share of them */
#ifdef _OPENMP
#pragma omp parallel
#endif
    {
        double *z = (double *)malloc(sizeof(double) * (size_t)C);
        double *logprob = (double *)malloc(sizeof(double) * (size_t)C);
        double head_ent[8];
#ifdef _OPENMP
#pragma omp for schedule(static)
#endif
        for (int64_t r = 0; r < n; ++r) {
            orc_forward(net, params, obs + r * net->obs_dim, z);
            orc_row_policy(net, w.logstd, z, act_disc + r * net->n_heads,
                           act_cont + r * net->n_gauss, logprob, head_ent, &logp[r], &ent[r]);
        }
        free(z);
        free(logprob);
    }
}

/* Per-row loss terms and dL/dz of one row of head outputs z (the body of
 * orc_loss_grad's row loop, also used by the recurrent policy):
 *   ratio = exp(logp - logp_old), pg = -min(ratio A, clip(ratio) A),
 *   vl = (V - R)^2, total = pg + c_v vl - c_e H, clipfrac, approx_kl;
 * dz gets dL/dz (with the 1/mb of the mean), glogstd accumulates the row's
 * log-std gradient, terms = {total, pg, vl, H, clipfrac, kl}. */
static void orc_ppo_row(const orc_net *net, const orc_loss_cfg *cfg, const double *logstd,
                        const double *z, const int32_t *act, const float *actc,
                        double logp_old, double A, double R, double inv_mb, double *logprob,
                        double *dz, double *glogstd, double terms[6])
{
    const int64_t NH = net->n_heads, G = net->n_gauss, C = orc_out_cols(net);
    /* log-probability and entropy of the taken action */
    double logp, ent, head_ent[8];
    orc_row_policy(net, logstd, z, act, actc, logprob, head_ent, &logp, &ent);
    const double value = z[C - 1];

    const double log_ratio = logp - logp_old;
    const double ratio = exp(log_ratio);
    const double lo = 1.0 - cfg->clip, hi = 1.0 + cfg->clip;
    const double clipped = ratio < lo ? lo : (ratio > hi ? hi : ratio);
    const double s1 = ratio * A, s2 = clipped * A;
    const double pg = -(s1 < s2 ? s1 : s2);
    const double vl = (value - R) * (value - R);
    terms[0] = pg + cfg->vf_coef * vl - cfg->ent_coef * ent;
    terms[1] = pg;
    terms[2] = vl;
    terms[3] = ent;
    terms[4] = fabs(ratio - 1.0) > cfg->clip ? 1.0 : 0.0;
    terms[5] = (ratio - 1.0) - log_ratio;

    /* dL/dlogp: the unclipped term is active when s1 <= s2 */
    const double g_logp = (s1 <= s2) ? -A * ratio * inv_mb : 0.0;
    const double g_ent = -cfg->ent_coef * inv_mb;

    int64_t off = 0;
    for (int64_t h = 0; h < NH; ++h) {
        int64_t n = net->head_n[h];
        int64_t a = act[h];
        for (int64_t k = 0; k < n; ++k) {
            double p = exp(logprob[off + k]);
            double dlogp_dz = (k == a ? 1.0 : 0.0) - p;
            double dent_dz = -p * (logprob[off + k] + head_ent[h]);
            dz[off + k] = g_logp * dlogp_dz + g_ent * dent_dz;
        }
        off += n;
    }
    for (int64_t g = 0; g < G; ++g) {
        double mu = z[off + g], s = logstd[g];
        double a = (double)actc[g];
        double var = exp(2.0 * s);
        dz[off + g] = g_logp * (a - mu) / var;
        glogstd[g] += g_logp * ((a - mu) * (a - mu) / var - 1.0) + g_ent * 1.0;
    }
    dz[C - 1] = cfg->vf_coef * 2.0 * (value - R) * inv_mb;
}

/* Forward, loss terms and backward of one row; accumulates the row's
 * gradient into grad (layout of the flat parameter vector) and returns its
 * loss terms in terms[6].  buf holds 6 H + 3 C doubles of scratch. */
static void orc_row_grad(const orc_net *net, const orc_loss_cfg *cfg, const orc_views *w,
                         const float *x, const int32_t *act, const float *actc,
                         double logp_old, double A, double R, double inv_mb, double *buf,
                         double *grad, double terms[6])
{
    const int64_t D = net->obs_dim, H1 = net->h1, H2 = net->h2, C = orc_out_cols(net);
    const int bf16 = cfg->bf16_operands;
    double *gW1 = grad, *gb1 = gW1 + H1 * D, *gW2 = gb1 + H1, *gb2 = gW2 + H2 * H1;
    double *gW3 = gb2 + H2, *gb3 = gW3 + C * H2, *glogstd = gb3 + C;
    double *pre1 = buf, *h1 = pre1 + H1, *dh1 = h1 + H1;
    double *pre2 = dh1 + H1, *h2 = pre2 + H2, *dh2 = h2 + H2;
    double *z = dh2 + H2, *logprob = z + C, *dz = logprob + C;

    orc_forward_full(net, w, x, pre1, h1, pre2, h2, z, bf16);
    orc_ppo_row(net, cfg, w->logstd, z, act, actc, logp_old, A, R, inv_mb, logprob, dz, glogstd,
                terms);

    /* backward through z = W3 h2 + b3 (bias gradients take the unrounded
     * signal; GEMM operands are rounded in bf16-operand mode) */
    for (int64_t j = 0; j < H2; ++j) dh2[j] = 0.0;
    for (int64_t c = 0; c < C; ++c) {
        gb3[c] += dz[c];
        const double dzc = orc_rnd(bf16, dz[c]);
        for (int64_t j = 0; j < H2; ++j) {
            gW3[c * H2 + j] += dzc * h2[j];
            dh2[j] += dzc * w->W3[c * H2 + j];
        }
    }
    /* through h2 = act(W2 h1 + b2) */
    for (int64_t k = 0; k < H1; ++k) dh1[k] = 0.0;
    for (int64_t j = 0; j < H2; ++j) {
        double dpre = dh2[j] * orc_act_grad(net->act, pre2[j], h2[j]);
        gb2[j] += dpre;
        dpre = orc_rnd(bf16, dpre);
        for (int64_t k = 0; k < H1; ++k) {
            gW2[j * H1 + k] += dpre * h1[k];
            dh1[k] += dpre * w->W2[j * H1 + k];
        }
    }
    /* through h1 = act(W1 x + b1) */
    for (int64_t j = 0; j < H1; ++j) {
        double dpre = dh1[j] * orc_act_grad(net->act, pre1[j], h1[j]);
        gb1[j] += dpre;
        dpre = orc_rnd(bf16, dpre);
        for (int64_t k = 0; k < D; ++k) gW1[j * D + k] += dpre * orc_rnd(bf16, (double)x[k]);
    }
}

int orc_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void orc_set_threads(int n)
{
#ifdef _OPENMP
    if (n >= 1) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

/* ------------------------------------------------------------------------ */
/* "Teaching Mario to speedrun", sec. 6 "Don't move too far at once":
 *   ratio  = new_prob(action) / old_prob(action)
 *   loss_pi = -min(ratio A, clip(ratio, 1 - eps, 1 + eps) A)
 *   loss_V  = (value - return)^2
 *   loss    = loss_pi + c_v loss_V - c_e entropy
 * averaged over the minibatch.  A multi-discrete action's probability is the
 * product of its heads' softmax probabilities (sec. 6: each head sampled
 * separately), so log-probabilities and entropies add over heads.  A Gaussian
 * dimension g with mean mu_g and learned log-std s_g adds
 *   log N(a; mu, e^s) = -(a-mu)^2 / (2 e^{2s}) - s - ln(2 pi)/2
 * and entropy 1/2 + ln(2 pi)/2 + s.
 * Gradient of the log-probability w.r.t. head logits: 1[k == a] - p_k
 * (sec. 5, "the gradient of log probs[action]").  The clipped branch, where
 * min() picks the clipped term, has zero gradient w.r.t. the ratio.
 *
 * The gradient is a sum over rows.  With OpenMP the rows are cut into one
 * contiguous range per thread, each thread sums its range into its own
 * gradient, and the per-thread sums are added in thread order (deterministic
 * for a given thread count). */
double orc_loss_grad(const orc_net *net, const orc_loss_cfg *cfg, const double *params,
                     int64_t mb, const int32_t *idx,
                     const float *obs, const int32_t *act_disc, const float *act_cont,
                     const float *logp_old, const double *adv, const double *ret,
                     int normalize, double adv_mean, double adv_std,
                     double *grad, double *stats6, double *scale6)
{
    const int64_t D = net->obs_dim, H1 = net->h1, H2 = net->h2, C = orc_out_cols(net);
    const int64_t NH = net->n_heads, G = net->n_gauss;
    const int64_t P = orc_num_params(net);
    double *wr = orc_gemm_weights(net, params, cfg->bf16_operands);
    const orc_views w = orc_split(net, cfg->bf16_operands ? wr : params);
    const double inv_mb = 1.0 / (double)mb;

    int nt = orc_threads();
    if (nt > mb) nt = (int)(mb > 0 ? mb : 1);
    double *acc = (double *)calloc((size_t)nt * (size_t)P, sizeof(double));
    double *tsum = (double *)calloc((size_t)nt * 12, sizeof(double));

#ifdef _OPENMP
#pragma omp parallel num_threads(nt)
#endif
    {
#ifdef _OPENMP
        const int t = omp_get_thread_num();
#else
        const int t = 0;
#endif
        const int64_t r0 = mb * t / nt, r1 = mb * (t + 1) / nt;
        double *buf = (double *)malloc(sizeof(double) * (size_t)(3 * H1 + 3 * H2 + 3 * C));
        double *g = acc + (size_t)t * (size_t)P;
        double *sum = tsum + 12 * t, *asum = sum + 6;
        for (int64_t r = r0; r < r1; ++r) {
            const int64_t row = idx[r];
            double A = adv[row];
            if (normalize) A = (A - adv_mean) / (adv_std + 1e-8);
            double terms[6];
            orc_row_grad(net, cfg, &w, obs + row * D, act_disc + row * NH, act_cont + row * G,
                         (double)logp_old[row], A, ret[row], inv_mb, buf, g, terms);
            for (int q = 0; q < 6; ++q) { sum[q] += terms[q]; asum[q] += fabs(terms[q]); }
        }
        free(buf);
    }

    memset(grad, 0, sizeof(double) * (size_t)P);
    double sum[6] = {0, 0, 0, 0, 0, 0}, asum[6] = {0, 0, 0, 0, 0, 0};
    for (int t = 0; t < nt; ++t) {
        const double *g = acc + (size_t)t * (size_t)P;
        for (int64_t i = 0; i < P; ++i) grad[i] += g[i];
        for (int q = 0; q < 6; ++q) { sum[q] += tsum[12 * t + q]; asum[q] += tsum[12 * t + 6 + q]; }
    }
    for (int q = 0; q < 6; ++q) {
        if (stats6) stats6[q] = sum[q] * inv_mb;
        if (scale6) scale6[q] = asum[q] * inv_mb;
    }
    free(acc);
    free(tsum);
    free(wr);
    return sum[0] * inv_mb;
}

/* ------------------------------------------------------------------------ */
/* "Teaching Mario to speedrun", sec. 8 "The Puffer net, and the trainer":
 * fresh values for the advantages of a minibatch.  For rows idx[0..n): the
 * value column of the forward pass at params, and the importance ratio
 * pi/mu = exp(logp - logp_old) of the taken action (sec. 6 "Don't move too
 * far at once").  bf16: the operand rounding of orc_loss_cfg.  ratio may be
 * NULL. */
void orc_fresh_values(const orc_net *net, int bf16, const double *params, int64_t n,
                      const int32_t *idx, const float *obs, const int32_t *act_disc,
                      const float *act_cont, const float *logp_old, double *val, double *ratio)
{
    const int64_t H1 = net->h1, H2 = net->h2, C = orc_out_cols(net);
    double *wr = orc_gemm_weights(net, params, bf16);
    orc_views w = orc_split(net, bf16 ? wr : params);
    /* rows are independent: with OpenMP each thread takes a share of them */
#ifdef _OPENMP
#pragma omp parallel
#endif
    {
        double *buf = (double *)malloc(sizeof(double) * (size_t)(2 * H1 + 2 * H2 + 2 * C));
        double *pre1 = buf, *h1 = pre1 + H1, *pre2 = h1 + H1, *h2 = pre2 + H2, *z = h2 + H2;
        double *logprob = z + C;
        double head_ent[8];
#ifdef _OPENMP
#pragma omp for schedule(static)
#endif
        for (int64_t r = 0; r < n; ++r) {
            const int64_t row = idx[r];
            orc_forward_full(net, &w, obs + row * net->obs_dim, pre1, h1, pre2, h2, z, bf16);
            val[r] = z[C - 1];
            if (ratio) {
                double logp, ent;
                orc_row_policy(net, w.logstd, z, act_disc + row * net->n_heads,
                               act_cont + row * net->n_gauss, logprob, head_ent, &logp, &ent);
                ratio[r] = exp(logp - (double)logp_old[row]);
            }
        }
        free(buf);
    }
    free(wr);
}

/* One minibatch made of whole environment segments, with advantages computed
 * from fresh values ("Teaching Mario to speedrun", sec. 8: per minibatch,
 * GAE or V-trace).  The rows are (t, envs[j]) for t < T, j < ns, in the order
 * t*ns + j, i.e. flat batch rows t*N + envs[j].  Steps: fresh values (and,
 * for V-trace, ratios) at params; orc_segment_advantage; the minibatch's own
 * mean and unbiased std; orc_loss_grad with the normalised advantages and the
 * targets ret.  vtrace: 0 GAE, 1 V-trace.  adv_norm_out / ret_out (nullable,
 * [T*ns]) receive the normalised advantages and the value targets. */
double orc_loss_grad_fresh(const orc_net *net, const orc_loss_cfg *cfg, const double *params,
                           int64_t T, int64_t N, int64_t ns, const int32_t *envs,
                           const float *obs, const int32_t *act_disc, const float *act_cont,
                           const float *logp_old, const float *rew, const float *done,
                           const float *boot, int vtrace, double gamma, double lambda,
                           double rho_clip, double c_clip, double *grad, double *stats6,
                           double *scale6, double *adv_norm_out, double *ret_out)
{
    const int64_t mb = T * ns, B = T * N;
    int32_t *idx = (int32_t *)malloc(sizeof(int32_t) * (size_t)mb);
    double *val = (double *)malloc(sizeof(double) * (size_t)mb);
    double *ratio = vtrace ? (double *)malloc(sizeof(double) * (size_t)mb) : NULL;
    double *adv = (double *)malloc(sizeof(double) * (size_t)mb);
    double *ret = (double *)malloc(sizeof(double) * (size_t)mb);
    double *adv_full = (double *)calloc((size_t)B, sizeof(double));
    double *ret_full = (double *)calloc((size_t)B, sizeof(double));
    for (int64_t t = 0; t < T; ++t)
        for (int64_t j = 0; j < ns; ++j) idx[t * ns + j] = (int32_t)(t * N + envs[j]);
    orc_fresh_values(net, cfg->bf16_operands, params, mb, idx, obs, act_disc, act_cont,
                     logp_old, val, ratio);
    orc_segment_advantage(T, N, rew, done, boot, ns, envs, val, ratio, gamma, lambda, rho_clip,
                          c_clip, adv, ret);
    double mean, sd;
    orc_moments(mb, adv, &mean, &sd);
    for (int64_t r = 0; r < mb; ++r) {
        adv_full[idx[r]] = adv[r];
        ret_full[idx[r]] = ret[r];
        if (adv_norm_out) adv_norm_out[r] = (adv[r] - mean) / (sd + 1e-8);
        if (ret_out) ret_out[r] = ret[r];
    }
    const double loss = orc_loss_grad(net, cfg, params, mb, idx, obs, act_disc, act_cont,
                                      logp_old, adv_full, ret_full, 1, mean, sd, grad, stats6,
                                      scale6);
    free(idx); free(val); free(ratio); free(adv); free(ret); free(adv_full); free(ret_full);
    return loss;
}

/* ------------------------------------------------------------------------ */
/* Rollout side: "Teaching Mario to speedrun", sec. 6 "The whole algorithm",
 * step 1, and sec. 7 (the trainer's side of a horizon): for every agent,
 * logits and value from the policy, an action sampled from the logits, and
 * its probability kept as old_prob.  The pages do not define sample(); the
 * plainest reading is used: per discrete head, inverse-CDF sampling of the
 * softmax with one uniform u (the first category whose cumulative
 * probability exceeds u); per Gaussian dimension, mu + e^s n with n from the
 * Box-Muller transform of two uniforms.  Uniforms come from mulberry32
 * ("PlayTrain", Appendix F.2) used as a counter: for agent i, slot k (head h
 * is slot h, Gaussian dim g uses slots NH + 2g and NH + 2g + 1, K = NH + 2G
 * slots per agent) the draw number is draw0 + i K + k of the stream seeded
 * with `seed`, and u = (draw >> 8) / 2^24, a 24-bit uniform in [0, 1). */
double orc_uniform24(uint32_t x) { return (double)(x >> 8) / 16777216.0; }

uint32_t orc_mulberry32_at(uint32_t seed, uint64_t draw)
{
    uint32_t state = seed + (uint32_t)draw * 0x6D2B79F5u;   /* skip `draw` draws */
    return orc_mulberry32_next(&state);
}

/* Inverse CDF of softmax(z[0..n)): the smallest k with u < sum_{i<=k} p_i,
 * compared as u * sum_i e^{z_i - max} < sum_{i<=k} e^{z_i - max}; n - 1 if
 * rounding leaves no such k. */
int orc_sample_categorical(const double *z, int n, double u)
{
    double zmax = z[0];
    for (int k = 1; k < n; ++k) if (z[k] > zmax) zmax = z[k];
    double total = 0.0;
    for (int k = 0; k < n; ++k) total += exp(z[k] - zmax);
    double cum = 0.0;
    for (int k = 0; k < n; ++k) {
        cum += exp(z[k] - zmax);
        if (u * total < cum) return k;
    }
    return n - 1;
}

/* Box-Muller: n = sqrt(-2 ln(1 - u1)) cos(2 pi u2) (1 - u1 lies in (0, 1]). */
double orc_box_muller(double u1, double u2)
{
    return sqrt(-2.0 * log(1.0 - u1)) * cos(2.0 * acos(-1.0) * u2);
}

void orc_policy_act(const orc_net *net, int bf16, const double *params, int64_t n,
                    const float *obs, uint32_t seed, uint64_t draw0, int32_t *act,
                    double *actc, double *logp, double *value)
{
    const int64_t H1 = net->h1, H2 = net->h2, C = orc_out_cols(net);
    const int64_t NH = net->n_heads, G = net->n_gauss, K = NH + 2 * G;
    double *wr = orc_gemm_weights(net, params, bf16);
    orc_views w = orc_split(net, bf16 ? wr : params);
    double *buf = (double *)malloc(sizeof(double) * (size_t)(2 * H1 + 2 * H2 + 2 * C));
    double *pre1 = buf, *h1 = pre1 + H1, *pre2 = h1 + H1, *h2 = pre2 + H2, *z = h2 + H2;
    double *logprob = z + C;
    double head_ent[8];
    float actc_f[4];
    for (int64_t i = 0; i < n; ++i) {
        orc_forward_full(net, &w, obs + i * net->obs_dim, pre1, h1, pre2, h2, z, bf16);
        const uint64_t d0 = draw0 + (uint64_t)i * (uint64_t)K;
        int64_t off = 0;
        for (int64_t h = 0; h < NH; ++h) {
            const double u = orc_uniform24(orc_mulberry32_at(seed, d0 + (uint64_t)h));
            act[i * NH + h] = orc_sample_categorical(z + off, net->head_n[h], u);
            off += net->head_n[h];
        }
        for (int64_t g = 0; g < G; ++g) {
            const double u1 = orc_uniform24(orc_mulberry32_at(seed, d0 + (uint64_t)(NH + 2 * g)));
            const double u2 = orc_uniform24(orc_mulberry32_at(seed, d0 + (uint64_t)(NH + 2 * g + 1)));
            const double a = z[off + g] + exp(w.logstd[g]) * orc_box_muller(u1, u2);
            actc[i * G + g] = a;
            actc_f[g] = (float)a;
        }
        /* the kept log-probability: of the action as stored (fp32) */
        double ent;
        orc_row_policy(net, w.logstd, z, act + i * NH, actc_f, logprob, head_ent, &logp[i], &ent);
        value[i] = z[C - 1];
    }
    free(buf);
    free(wr);
}

/* ------------------------------------------------------------------------ */
/* "Teaching Mario to speedrun", sec. 8 "The Puffer net, and the trainer":
 * PufferLib 5.0's policy is a bias-free linear encoder (observation -> H),
 * four MinGRU layers, and one matrix from the hidden state to every head's
 * logits plus the value.  The MinGRU's gates depend only on its input; its
 * state carries across horizons and clears when an episode ends.  The pages
 * give no equations; the MinGRU is the minimal GRU of Feng et al. 2024 ("Were
 * RNNs All We Needed?"), layer input u, state h:
 *   z_t = sigmoid(W_z u_t + b_z),  h~_t = W_h u_t + b_h,
 *   h_t = (1 - z_t) h_{t-1} + z_t h~_t,
 * layer l + 1 reading layer l's h (no residual, no normalisation: the pages
 * name none).  A terminal at step t - 1 (the episode ended there) clears the
 * state entering step t; h0 is the state carried into the segment.
 * Parameter layout: W_enc[H][D]; per layer W_z[H][H], b_z[H], W_h[H][H],
 * b_h[H]; W_dec[C][H]; logstd[G]. */
int64_t orc_rnn_out_cols(const orc_rnn *r)
{
    int64_t c = 0;
    for (int h = 0; h < r->n_heads; ++h) c += r->head_n[h];
    return c + r->n_gauss + 1;
}

int64_t orc_rnn_num_params(const orc_rnn *r)
{
    const int64_t D = r->obs_dim, H = r->hidden, L = r->layers, C = orc_rnn_out_cols(r);
    return H * D + L * (2 * H * H + 2 * H) + C * H + r->n_gauss;
}

/* the head layout of the recurrent policy as an orc_net (for orc_ppo_row) */
static orc_net orc_rnn_heads(const orc_rnn *r)
{
    orc_net n;
    memset(&n, 0, sizeof n);
    n.obs_dim = r->obs_dim;
    n.h1 = r->hidden;
    n.h2 = r->hidden;
    n.n_heads = r->n_heads;
    for (int h = 0; h < 8; ++h) n.head_n[h] = r->head_n[h];
    n.n_gauss = r->n_gauss;
    return n;
}

static double orc_sigmoid(double x) { return 1.0 / (1.0 + exp(-x)); }

/* bf16-operand mode of the recurrent policy (the reading of the MLP's mode
 * applied to its products): the GEMMs read bf16-rounded weights (W_enc,
 * W_z, W_h, W_dec) and bf16 operands -- the observation, every layer input
 * u (the encoder's output and each layer's new state as the next layer's or
 * the decoder's input), and in the backward pass dL/dz, the pre-activation
 * gradients dpz, dph and the input gradients du -- and the products that are
 * stored between kernels are rounded when stored: u, the pre-activations
 * pz, ph (bias added first), du.  The recurrence itself (z, the state h,
 * dL/dh) and the bias gradients stay unrounded.  Identity when off. */
static double *orc_rnn_gemm_weights(const orc_rnn *r, const double *params, int bf16)
{
    if (!bf16) return NULL;
    const int64_t D = r->obs_dim, H = r->hidden, L = r->layers, C = orc_rnn_out_cols(r);
    const int64_t P = orc_rnn_num_params(r), per = 2 * H * H + 2 * H;
    double *wr = (double *)malloc(sizeof(double) * (size_t)P);
    memcpy(wr, params, sizeof(double) * (size_t)P);
    for (int64_t i = 0; i < H * D; ++i) wr[i] = orc_bf16(params[i]);
    for (int64_t l = 0; l < L; ++l) {
        const int64_t oz = H * D + l * per, oh = oz + H * H + H;
        for (int64_t i = 0; i < H * H; ++i) {
            wr[oz + i] = orc_bf16(params[oz + i]);
            wr[oh + i] = orc_bf16(params[oh + i]);
        }
    }
    const int64_t od = H * D + L * per;
    for (int64_t i = 0; i < C * H; ++i) wr[od + i] = orc_bf16(params[od + i]);
    return wr;
}

/* Forward of one segment (env n, steps 0..T-1).  obs rows t*N + n, done
 * [T][N], h0 [L][H].  zout [T][C]; when non-NULL, per step and layer
 * [T][L][H]: the layer input u, the gate z, the candidate h~, the masked
 * previous state hp and the new state h.  bf16: the operand rounding above
 * (params must then hold the rounded weights, see orc_rnn_gemm_weights). */
static void orc_rnn_forward_mode(const orc_rnn *r, const double *params, int64_t T, int64_t N,
                                 int64_t n, const float *obs, const float *done, const double *h0,
                                 int bf16, double *zout, double *su, double *sz, double *sht,
                                 double *shp, double *sh)
{
    const int64_t D = r->obs_dim, H = r->hidden, L = r->layers, C = orc_rnn_out_cols(r);
    const double *Wenc = params;
    const double *Wdec = params + H * D + L * (2 * H * H + 2 * H);
    double *state = (double *)malloc(sizeof(double) * (size_t)(L * H));
    double *u = (double *)malloc(sizeof(double) * (size_t)H);
    double *hn = (double *)malloc(sizeof(double) * (size_t)H);
    memcpy(state, h0, sizeof(double) * (size_t)(L * H));
    for (int64_t t = 0; t < T; ++t) {
        const float *x = obs + (t * N + n) * D;
        const double mask = (t > 0 && done[(t - 1) * N + n] != 0.0f) ? 0.0 : 1.0;
        for (int64_t i = 0; i < H; ++i) {
            double e = 0.0;
            for (int64_t k = 0; k < D; ++k) e += Wenc[i * D + k] * orc_rnd(bf16, (double)x[k]);
            u[i] = orc_rnd(bf16, e);
        }
        for (int64_t l = 0; l < L; ++l) {
            const double *Wz = params + H * D + l * (2 * H * H + 2 * H);
            const double *bz = Wz + H * H, *Wh = bz + H, *bh = Wh + H * H;
            for (int64_t i = 0; i < H; ++i) {
                double pz = bz[i], ph = bh[i];
                for (int64_t k = 0; k < H; ++k) {
                    pz += Wz[i * H + k] * u[k];
                    ph += Wh[i * H + k] * u[k];
                }
                pz = orc_rnd(bf16, pz);
                ph = orc_rnd(bf16, ph);
                const double z = orc_sigmoid(pz);
                const double hp = mask * state[l * H + i];
                hn[i] = (1.0 - z) * hp + z * ph;
                const int64_t o = (t * L + l) * H + i;
                if (su) { su[o] = u[i]; sz[o] = z; sht[o] = ph; shp[o] = hp; sh[o] = hn[i]; }
            }
            memcpy(state + l * H, hn, sizeof(double) * (size_t)H);
            for (int64_t i = 0; i < H; ++i) u[i] = orc_rnd(bf16, hn[i]);
        }
        for (int64_t c = 0; c < C; ++c) {
            double acc = 0.0;
            for (int64_t k = 0; k < H; ++k) acc += Wdec[c * H + k] * u[k];
            zout[t * C + c] = acc;
        }
    }
    free(state); free(u); free(hn);
}

void orc_rnn_forward(const orc_rnn *r, const double *params, int64_t T, int64_t N, int64_t n,
                     const float *obs, const float *done, const double *h0, double *zout,
                     double *su, double *sz, double *sht, double *shp, double *sh)
{
    orc_rnn_forward_mode(r, params, T, N, n, obs, done, h0, 0, zout, su, sz, sht, shp, sh);
}

/* Loss and gradient of a minibatch of environment segments envs[0..ns)
 * (rows t*N + envs[j], t < T), with backpropagation through time inside each
 * segment (h0, carried in from the previous horizon, is a constant).  The
 * per-row loss is orc_loss_grad's (orc_ppo_row), with advantages optionally
 * normalised by (adv_mean, adv_std); adv, ret [T*N]; h0 [N][L][H].
 * grad overwritten; stats6 / scale6 as in orc_loss_grad. */
/* One segment's contribution (env n) to the recurrent policy's loss and
 * gradient: forward, per-row loss, backpropagation through time.  Adds into
 * grad (layout of the parameters) and the loss-term sums; buf holds the
 * segment's scratch (see orc_rnn_loss_grad). */
static void orc_rnn_segment_grad(const orc_rnn *r, const orc_loss_cfg *cfg, const double *params,
                                 const double *pw, int64_t T, int64_t N, int64_t n,
                                 const float *obs, const int32_t *act_disc,
                                 const float *act_cont, const float *logp_old, const double *adv,
                                 const double *ret, int normalize, double adv_mean,
                                 double adv_std, const float *done, const double *h0,
                                 double inv_mb, double *buf, double *grad, double sum[6],
                                 double asum[6])
{
    const int64_t D = r->obs_dim, H = r->hidden, L = r->layers, C = orc_rnn_out_cols(r);
    const int64_t NH = r->n_heads, G = r->n_gauss;
    const orc_net heads = orc_rnn_heads(r);
    const int bf16 = cfg->bf16_operands;
    const double *Wdec = pw + H * D + L * (2 * H * H + 2 * H);
    const double *logstd = params + (Wdec - pw) + C * H;
    double *gWenc = grad;
    double *gWdec = grad + (Wdec - pw), *glogstd = grad + (logstd - params);
    const int64_t TLH = T * L * H;
    double *su = buf, *sz = su + TLH, *sht = sz + TLH, *shp = sht + TLH, *sh = shp + TLH;
    double *zout = sh + TLH, *logprob = zout + T * C, *dz = logprob + C, *dnext = dz + C;
    double *din = dnext + L * H, *du = din + H;
    orc_rnn_forward_mode(r, pw, T, N, n, obs, done, h0 + n * L * H, bf16, zout, su, sz, sht,
                         shp, sh);
    memset(dnext, 0, sizeof(double) * (size_t)(L * H));
    for (int64_t t = T - 1; t >= 0; --t) {
        const int64_t row = t * N + n;
        double A = adv[row];
        if (normalize) A = (A - adv_mean) / (adv_std + 1e-8);
        double terms[6];
        orc_ppo_row(&heads, cfg, logstd, zout + t * C, act_disc + row * NH,
                    act_cont + row * G, (double)logp_old[row], A, ret[row], inv_mb,
                    logprob, dz, glogstd, terms);
        for (int q = 0; q < 6; ++q) { sum[q] += terms[q]; asum[q] += fabs(terms[q]); }
        /* decoder: z = W_dec u^L_t (u^L the top state, as an operand) */
        const double *htop = sh + (t * L + (L - 1)) * H;
        for (int64_t k = 0; k < H; ++k) din[k] = 0.0;
        for (int64_t c = 0; c < C; ++c) {
            const double dzc = orc_rnd(bf16, dz[c]);
            for (int64_t k = 0; k < H; ++k) {
                gWdec[c * H + k] += dzc * orc_rnd(bf16, htop[k]);
                din[k] += dzc * Wdec[c * H + k];
            }
        }
        for (int64_t k = 0; k < H; ++k) din[k] = orc_rnd(bf16, din[k]);
        /* layers, top to bottom: h = (1 - z) hp + z h~ */
        const double mask = (t > 0 && done[(t - 1) * N + n] != 0.0f) ? 0.0 : 1.0;
        for (int64_t l = L - 1; l >= 0; --l) {
            const double *Wz = pw + H * D + l * (2 * H * H + 2 * H);
            const double *Wh = Wz + H * H + H;
            double *gWz = grad + (Wz - pw), *gbz = gWz + H * H;
            double *gWh = gbz + H, *gbh = gWh + H * H;
            const int64_t o = (t * L + l) * H;
            for (int64_t k = 0; k < H; ++k) du[k] = 0.0;
            for (int64_t i = 0; i < H; ++i) {
                const double dh = din[i] + dnext[l * H + i];
                const double z = sz[o + i];
                const double dpz = dh * (sht[o + i] - shp[o + i]) * z * (1.0 - z);
                const double dht = dh * z;
                dnext[l * H + i] = dh * (1.0 - z) * mask;   /* into h_{t-1} */
                gbz[i] += dpz;
                gbh[i] += dht;
                const double dpzr = orc_rnd(bf16, dpz), dhtr = orc_rnd(bf16, dht);
                for (int64_t k = 0; k < H; ++k) {
                    gWz[i * H + k] += dpzr * su[o + k];
                    gWh[i * H + k] += dhtr * su[o + k];
                    du[k] += Wz[i * H + k] * dpzr + Wh[i * H + k] * dhtr;
                }
            }
            for (int64_t k = 0; k < H; ++k) din[k] = orc_rnd(bf16, du[k]);
        }
        /* encoder: u^0 = W_enc x */
        const float *x = obs + row * D;
        for (int64_t i = 0; i < H; ++i)
            for (int64_t k = 0; k < D; ++k)
                gWenc[i * D + k] += din[i] * orc_rnd(bf16, (double)x[k]);
    }
}

double orc_rnn_loss_grad(const orc_rnn *r, const orc_loss_cfg *cfg, const double *params,
                         int64_t T, int64_t N, int64_t ns, const int32_t *envs,
                         const float *obs, const int32_t *act_disc, const float *act_cont,
                         const float *logp_old, const double *adv, const double *ret,
                         int normalize, double adv_mean, double adv_std, const float *done,
                         const double *h0, double *grad, double *stats6, double *scale6)
{
    const int64_t H = r->hidden, L = r->layers, C = orc_rnn_out_cols(r);
    const int64_t P = orc_rnn_num_params(r);
    double *wr = orc_rnn_gemm_weights(r, params, cfg->bf16_operands);
    const double *pw = cfg->bf16_operands ? wr : params;   /* the weights the products read */
    const double inv_mb = 1.0 / (double)(T * ns);
    const int64_t nbuf = 5 * T * L * H + T * C + 2 * C + L * H + 2 * H;
    /* segments are independent: with OpenMP each thread takes a contiguous
     * range of them into its own gradient, summed in thread order */
    int nt = orc_threads();
    if (nt > ns) nt = (int)(ns > 0 ? ns : 1);
    double *acc = (double *)calloc((size_t)nt * (size_t)P, sizeof(double));
    double *tsum = (double *)calloc((size_t)nt * 12, sizeof(double));
#ifdef _OPENMP
#pragma omp parallel num_threads(nt)
#endif
    {
#ifdef _OPENMP
        const int th = omp_get_thread_num();
#else
        const int th = 0;
#endif
        double *buf = (double *)malloc(sizeof(double) * (size_t)nbuf);
        for (int64_t j = ns * th / nt; j < ns * (th + 1) / nt; ++j) {
            const int64_t n = envs[j];
            orc_rnn_segment_grad(r, cfg, params, pw, T, N, n, obs, act_disc, act_cont, logp_old,
                                 adv, ret, normalize, adv_mean, adv_std, done, h0, inv_mb, buf,
                                 acc + (size_t)th * (size_t)P, tsum + 12 * th, tsum + 12 * th + 6);
        }
        free(buf);
    }
    memset(grad, 0, sizeof(double) * (size_t)P);
    double sum[6] = {0, 0, 0, 0, 0, 0}, asum[6] = {0, 0, 0, 0, 0, 0};
    for (int th = 0; th < nt; ++th) {
        for (int64_t i = 0; i < P; ++i) grad[i] += acc[(size_t)th * (size_t)P + i];
        for (int q = 0; q < 6; ++q) { sum[q] += tsum[12 * th + q]; asum[q] += tsum[12 * th + 6 + q]; }
    }
    for (int q = 0; q < 6; ++q) {
        if (stats6) stats6[q] = sum[q] * inv_mb;
        if (scale6) scale6[q] = asum[q] * inv_mb;
    }
    free(acc);
    free(tsum);
    free(wr);
    return sum[0] * inv_mb;
}

/* ------------------------------------------------------------------------ */
/* "PlayTrain", Table 8 (PPO column): gradient-norm clip 0.5.  The global L2
 * norm over all parameters; if above max_norm, scale by max_norm/(norm+1e-6). */
double orc_clip_grad_norm(int64_t P, double *g, double max_norm)
{
    double ss = 0.0;
    for (int64_t i = 0; i < P; ++i) ss += g[i] * g[i];
    double norm = sqrt(ss);
    if (max_norm > 0.0) {
        double coef = max_norm / (norm + 1e-6);
        if (coef < 1.0)
            for (int64_t i = 0; i < P; ++i) g[i] *= coef;
    }
    return norm;
}

/* "PlayTrain", Table 8 (PPO column): optimizer Adam (Kingma & Ba), with the
 * usual bias correction:
 *   m = b1 m + (1-b1) g;  v = b2 v + (1-b2) g^2
 *   p -= lr * (m / (1 - b1^t)) / (sqrt(v / (1 - b2^t)) + eps)            */
void orc_adam(int64_t P, double *p, const double *g, double *m, double *v, int64_t step,
              double lr, double beta1, double beta2, double eps)
{
    double bc1 = 1.0 - pow(beta1, (double)step);
    double bc2 = 1.0 - pow(beta2, (double)step);
    for (int64_t i = 0; i < P; ++i) {
        m[i] = beta1 * m[i] + (1.0 - beta1) * g[i];
        v[i] = beta2 * v[i] + (1.0 - beta2) * g[i] * g[i];
        double mhat = m[i] / bc1;
        double vhat = v[i] / bc2;
        p[i] -= lr * mhat / (sqrt(vhat) + eps);
    }
}

/* ------------------------------------------------------------------------ */
/* "Teaching Mario to speedrun", sec. 8 "The Puffer net, and the trainer" and
 * "puff-rs": the 5.0 optimizer is Muon, which orthogonalises each weight
 * matrix's update, with five Newton-Schulz iterations.  The pages give no
 * formula; the definition is Muon's published write-up (K. Jordan et al.,
 * 2024, "Muon: An optimizer for hidden layers in neural networks"):
 *   X = G / (||G||_F + 1e-7), as an r x k matrix with r <= k (transposed if
 *   G has more rows than columns); five times
 *     A = X X^T,  B = b A + c A A,  X = a X + B X,
 *   with (a, b, c) = (3.4445, -4.7750, 2.0315); transposed back.
 * The write-up runs the iteration in bf16; here it is fp64. */
/* bf16 mode (the write-up's precision): X, A and B are stored as bf16 --
 * the normalised input, each product A = X X^T, B = b A + c A A and
 * X = a X + B X rounded once computed (sums in fp64 of the rounded values).
 * Identity when off. */
static void orc_newton_schulz5_mode(int64_t rows, int64_t cols, const double *G, int steps,
                                    int bf16, double *out)
{
    const double ca = 3.4445, cb = -4.7750, cc = 2.0315;
    const int tr = rows > cols;
    const int64_t r = tr ? cols : rows, k = tr ? rows : cols;
    double *X = (double *)malloc(sizeof(double) * (size_t)(r * k));
    double *Xn = (double *)malloc(sizeof(double) * (size_t)(r * k));
    double *A = (double *)malloc(sizeof(double) * (size_t)(r * r));
    double *B = (double *)malloc(sizeof(double) * (size_t)(r * r));
    double ss = 0.0;
    for (int64_t i = 0; i < rows * cols; ++i) ss += G[i] * G[i];
    const double inv = 1.0 / (sqrt(ss) + 1e-7);
    for (int64_t i = 0; i < r; ++i)
        for (int64_t j = 0; j < k; ++j)
            X[i * k + j] = orc_rnd(bf16, (tr ? G[j * cols + i] : G[i * cols + j]) * inv);
    for (int s = 0; s < steps; ++s) {
        for (int64_t i = 0; i < r; ++i)
            for (int64_t j = 0; j < r; ++j) {
                double t = 0.0;
                for (int64_t q = 0; q < k; ++q) t += X[i * k + q] * X[j * k + q];
                A[i * r + j] = orc_rnd(bf16, t);
            }
        for (int64_t i = 0; i < r; ++i)
            for (int64_t j = 0; j < r; ++j) {
                double t = 0.0;
                for (int64_t q = 0; q < r; ++q) t += A[i * r + q] * A[q * r + j];
                B[i * r + j] = orc_rnd(bf16, cb * A[i * r + j] + cc * t);
            }
        for (int64_t i = 0; i < r; ++i)
            for (int64_t j = 0; j < k; ++j) {
                double t = 0.0;
                for (int64_t q = 0; q < r; ++q) t += B[i * r + q] * X[q * k + j];
                Xn[i * k + j] = orc_rnd(bf16, ca * X[i * k + j] + t);
            }
        memcpy(X, Xn, sizeof(double) * (size_t)(r * k));
    }
    for (int64_t i = 0; i < r; ++i)
        for (int64_t j = 0; j < k; ++j) {
            if (tr) out[j * cols + i] = X[i * k + j];
            else out[i * cols + j] = X[i * k + j];
        }
    free(X); free(Xn); free(A); free(B);
}

void orc_newton_schulz5(int64_t rows, int64_t cols, const double *G, int steps, double *out)
{
    orc_newton_schulz5_mode(rows, cols, G, steps, 0, out);
}

void orc_newton_schulz5_bf16(int64_t rows, int64_t cols, const double *G, int steps, double *out)
{
    orc_newton_schulz5_mode(rows, cols, G, steps, 1, out);
}

/* One Muon step of the MLP's parameters (write-up's update with Nesterov
 * momentum): for each weight matrix W1, W2, W3 (rows x cols)
 *   mom = beta mom + g;  u = g + beta mom;
 *   W -= muon_lr sqrt(max(1, rows / cols)) NS5(u),
 * and, as the write-up prescribes for parameters that are not matrices, Adam
 * for the biases and the log-std (orc_adam's update, this `step`).  mom
 * covers the whole parameter vector (only the matrix entries are used);
 * adam_m, adam_v likewise (only the vector entries). */
static void orc_muon_mode(const orc_net *net, double *params, const double *g, double *mom,
                          double *adam_m, double *adam_v, int64_t step, double muon_lr,
                          double muon_beta, double lr, double beta1, double beta2, double eps,
                          int bf16)
{
    const int64_t D = net->obs_dim, H1 = net->h1, H2 = net->h2, C = orc_out_cols(net);
    const int64_t P = orc_num_params(net);
    orc_views v = orc_split(net, params);
    const int64_t offs[3] = {v.W1 - params, v.W2 - params, v.W3 - params};
    const int64_t rows[3] = {H1, H2, C}, cols[3] = {D, H1, H2};
    char *is_mat = (char *)calloc((size_t)P, 1);
    for (int mtx = 0; mtx < 3; ++mtx) {
        const int64_t o = offs[mtx], n = rows[mtx] * cols[mtx];
        double *u = (double *)malloc(sizeof(double) * (size_t)n);
        double *x = (double *)malloc(sizeof(double) * (size_t)n);
        for (int64_t i = 0; i < n; ++i) {
            mom[o + i] = muon_beta * mom[o + i] + g[o + i];
            u[i] = g[o + i] + muon_beta * mom[o + i];
            is_mat[o + i] = 1;
        }
        orc_newton_schulz5_mode(rows[mtx], cols[mtx], u, 5, bf16, x);
        const double ratio = (double)rows[mtx] / (double)cols[mtx];
        const double scale = sqrt(ratio > 1.0 ? ratio : 1.0);
        for (int64_t i = 0; i < n; ++i) params[o + i] -= muon_lr * scale * x[i];
        free(u); free(x);
    }
    const double bc1 = 1.0 - pow(beta1, (double)step);
    const double bc2 = 1.0 - pow(beta2, (double)step);
    for (int64_t i = 0; i < P; ++i) {
        if (is_mat[i]) continue;
        adam_m[i] = beta1 * adam_m[i] + (1.0 - beta1) * g[i];
        adam_v[i] = beta2 * adam_v[i] + (1.0 - beta2) * g[i] * g[i];
        params[i] -= lr * (adam_m[i] / bc1) / (sqrt(adam_v[i] / bc2) + eps);
    }
    free(is_mat);
}

void orc_muon(const orc_net *net, double *params, const double *g, double *mom,
              double *adam_m, double *adam_v, int64_t step, double muon_lr, double muon_beta,
              double lr, double beta1, double beta2, double eps)
{
    orc_muon_mode(net, params, g, mom, adam_m, adam_v, step, muon_lr, muon_beta, lr, beta1,
                  beta2, eps, 0);
}

void orc_muon_bf16(const orc_net *net, double *params, const double *g, double *mom,
                   double *adam_m, double *adam_v, int64_t step, double muon_lr,
                   double muon_beta, double lr, double beta1, double beta2, double eps)
{
    orc_muon_mode(net, params, g, mom, adam_m, adam_v, step, muon_lr, muon_beta, lr, beta1,
                  beta2, eps, 1);
}

/* One update of the recurrent policy ("Teaching Mario to speedrun", sec. 6
 * "The whole algorithm" with sec. 8's policy): GAE over the stored values,
 * advantage statistics over all T*N entries, then per epoch the mulberry32
 * permutation of the N environments (orc_perm) and per minibatch the segments
 * envs perm[k*ns .. (k+1)*ns) (ns = N / minibatches): orc_rnn_loss_grad
 * (normalised advantages, carried state h0), gradient-norm clip, Adam.
 * params, m, v updated in place; *step incremented per minibatch; stats
 * (epochs*minibatches*6) nullable.  Returns -1 (and changes nothing) unless
 * minibatches >= 1 divides N. */
int orc_rnn_update(const orc_rnn *r, const orc_hyper *hp, int64_t T, int64_t N, int64_t epochs,
                   int64_t minibatches, const float *obs, const int32_t *act_disc,
                   const float *act_cont, const float *logp_old, const float *val,
                   const float *rew, const float *done, const float *boot, const double *h0,
                   double *params, double *m, double *v, int64_t *step, double *stats)
{
    /* every minibatch takes N / minibatches whole segments: no remainder */
    if (minibatches < 1 || N % minibatches != 0) return -1;
    const int64_t B = T * N, ns = N / minibatches, P = orc_rnn_num_params(r);
    double *adv = (double *)malloc(sizeof(double) * (size_t)B);
    double *ret = (double *)malloc(sizeof(double) * (size_t)B);
    int32_t *perm = (int32_t *)malloc(sizeof(int32_t) * (size_t)N);
    double *grad = (double *)malloc(sizeof(double) * (size_t)P);
    orc_gae(T, N, rew, val, done, boot, hp->gamma, hp->lambda, adv, ret);
    double mean, sd;
    orc_moments(B, adv, &mean, &sd);
    const orc_loss_cfg lc = {hp->clip, hp->vf_coef, hp->ent_coef, hp->bf16_operands};
    for (int64_t e = 0; e < epochs; ++e) {
        orc_perm(hp->seed, e, N, perm);
        for (int64_t k = 0; k < minibatches; ++k) {
            double tmp[6];
            double *st = stats ? stats + (e * minibatches + k) * 6 : tmp;
            orc_rnn_loss_grad(r, &lc, params, T, N, ns, perm + k * ns, obs, act_disc, act_cont,
                              logp_old, adv, ret, 1, mean, sd, done, h0, grad, st, NULL);
            orc_clip_grad_norm(P, grad, hp->max_grad_norm);
            *step += 1;
            orc_adam(P, params, grad, m, v, *step, hp->lr, hp->beta1, hp->beta2, hp->adam_eps);
        }
    }
    free(adv); free(ret); free(perm); free(grad);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* "Teaching Mario to speedrun", sec. 6 "The whole algorithm": judge with GAE,
 * then learn for a few epochs over shuffled minibatches, one backward pass
 * and one optimizer step per minibatch.  The advantages are normalised with
 * the statistics of the whole batch. */
/* The optimizer step of orc_update: Adam (optimizer 0) or Muon (1). */
static void orc_optimize(const orc_net *net, const orc_hyper *hp, int64_t P, double *params,
                         const double *grad, double *m, double *v, double *mom, int64_t step)
{
    if (hp->optimizer == 1)
        orc_muon_mode(net, params, grad, mom, m, v, step, hp->muon_lr, hp->muon_beta, hp->lr,
                      hp->beta1, hp->beta2, hp->adam_eps, hp->bf16_operands);
    else
        orc_adam(P, params, grad, m, v, step, hp->lr, hp->beta1, hp->beta2, hp->adam_eps);
}

void orc_update(const orc_net *net, const orc_hyper *hp, int64_t T, int64_t N,
                int64_t epochs, int64_t minibatches,
                const float *obs, const int32_t *act_disc, const float *act_cont,
                const float *logp_old, const float *val, const float *rew,
                const float *done, const float *boot,
                double *params, double *m, double *v, double *mom, int64_t *step,
                double *stats, double *adv_out, double *ret_out)
{
    const int64_t B = T * N, mb = B / minibatches, P = orc_num_params(net);
    double *adv = (double *)malloc(sizeof(double) * (size_t)B);
    double *ret = (double *)malloc(sizeof(double) * (size_t)B);
    int32_t *perm = (int32_t *)malloc(sizeof(int32_t) * (size_t)B);
    double *grad = (double *)malloc(sizeof(double) * (size_t)P);

    orc_loss_cfg lc = {hp->clip, hp->vf_coef, hp->ent_coef, hp->bf16_operands};
    if (hp->adv_mode != 0) {
        /* sec. 8: minibatches of whole environment segments, advantages
         * recomputed per minibatch from fresh values (GAE or V-trace); epoch
         * e shuffles the N environments with the rule of orc_perm */
        const int64_t ns = N / minibatches;
        for (int64_t e = 0; e < epochs; ++e) {
            orc_perm(hp->seed, e, N, perm);
            for (int64_t k = 0; k < minibatches; ++k) {
                double *st = stats ? stats + (e * minibatches + k) * 6 : NULL;
                double tmp[6];
                orc_loss_grad_fresh(net, &lc, params, T, N, ns, perm + k * ns, obs, act_disc,
                                    act_cont, logp_old, rew, done, boot, hp->adv_mode == 2,
                                    hp->gamma, hp->lambda, hp->rho_clip, hp->c_clip, grad,
                                    st ? st : tmp, NULL, NULL, NULL);
                orc_clip_grad_norm(P, grad, hp->max_grad_norm);
                *step += 1;
                orc_optimize(net, hp, P, params, grad, m, v, mom, *step);
            }
        }
        free(adv); free(ret); free(perm); free(grad);
        return;
    }

    orc_gae(T, N, rew, val, done, boot, hp->gamma, hp->lambda, adv, ret);
    double mean, sd;
    orc_moments(B, adv, &mean, &sd);

    for (int64_t e = 0; e < epochs; ++e) {
        orc_perm(hp->seed, e, B, perm);
        for (int64_t k = 0; k < minibatches; ++k) {
            double *st = stats ? stats + (e * minibatches + k) * 6 : NULL;
            double tmp[6];
            orc_loss_grad(net, &lc, params, mb, perm + k * mb, obs, act_disc, act_cont,
                          logp_old, adv, ret, 1, mean, sd, grad, st ? st : tmp, NULL);
            orc_clip_grad_norm(P, grad, hp->max_grad_norm);
            *step += 1;
            orc_optimize(net, hp, P, params, grad, m, v, mom, *step);
        }
    }
    if (adv_out) memcpy(adv_out, adv, sizeof(double) * (size_t)B);
    if (ret_out) memcpy(ret_out, ret, sizeof(double) * (size_t)B);
    free(adv); free(ret); free(perm); free(grad);
}

/* ------------------------------------------------------------------------ */
/* The update of "Teaching Mario to speedrun", sec. 6, data-parallel over
 * `world` learners ("PlayTrain", App. C.3: the learner trained with DDP on
 * several GPUs), emulated in one process.  The rollout [T][N] is split by
 * environment: rank r holds envs [r Nr, (r + 1) Nr), Nr = N / world.  Each
 * rank runs GAE on its shard; the advantage statistics are those of all T*N
 * advantages, from the shards' (count, mean, M2) merged in rank order; per
 * epoch every rank permutes its own Br = T*Nr rows with orc_perm(seed, e, Br)
 * and minibatch k is the union of the ranks' k-th slices of Br/minibatches
 * rows.  The minibatch loss is the mean over that union, so its gradient is
 * the mean over the ranks of each rank's own minibatch gradient (equal
 * slice sizes); then clip and the optimizer, as in orc_update.  Returns -1
 * (changing nothing) unless world divides N and minibatches divides Br. */
int orc_update_sharded(const orc_net *net, const orc_hyper *hp, int64_t world, int64_t T,
                       int64_t N, int64_t epochs, int64_t minibatches, const float *obs,
                       const int32_t *act_disc, const float *act_cont, const float *logp_old,
                       const float *val, const float *rew, const float *done, const float *boot,
                       double *params, double *m, double *v, double *mom, int64_t *step,
                       double *stats)
{
    if (world < 1 || N % world != 0 || minibatches < 1) return -1;
    const int64_t Nr = N / world, Br = T * Nr;
    if (Br % minibatches != 0) return -1;
    const int64_t mbr = Br / minibatches, P = orc_num_params(net);
    double *adv = (double *)malloc(sizeof(double) * (size_t)(T * N));
    double *ret = (double *)malloc(sizeof(double) * (size_t)(T * N));
    float *sr = (float *)malloc(sizeof(float) * (size_t)Br);
    float *sv = (float *)malloc(sizeof(float) * (size_t)Br);
    float *sd = (float *)malloc(sizeof(float) * (size_t)Br);
    double *sa = (double *)malloc(sizeof(double) * (size_t)Br);
    double *sret = (double *)malloc(sizeof(double) * (size_t)Br);
    int32_t *perm = (int32_t *)malloc(sizeof(int32_t) * (size_t)Br);
    int32_t *idx = (int32_t *)malloc(sizeof(int32_t) * (size_t)mbr);
    double *g = (double *)malloc(sizeof(double) * (size_t)P);
    double *gsum = (double *)malloc(sizeof(double) * (size_t)P);

    /* judge: GAE per shard, statistics of the union */
    double tot[3] = {0.0, 0.0, 0.0};
    for (int64_t r = 0; r < world; ++r) {
        for (int64_t t = 0; t < T; ++t)
            for (int64_t j = 0; j < Nr; ++j) {
                const int64_t gi = t * N + r * Nr + j;
                sr[t * Nr + j] = rew[gi];
                sv[t * Nr + j] = val[gi];
                sd[t * Nr + j] = done[gi];
            }
        orc_gae(T, Nr, sr, sv, sd, boot + r * Nr, hp->gamma, hp->lambda, sa, sret);
        for (int64_t t = 0; t < T; ++t)
            for (int64_t j = 0; j < Nr; ++j) {
                adv[t * N + r * Nr + j] = sa[t * Nr + j];
                ret[t * N + r * Nr + j] = sret[t * Nr + j];
            }
        double mr[3];
        orc_moments3(Br, sa, mr);
        orc_moments_merge(tot, mr, tot);
    }
    const double mean = tot[1];
    const double sdv = tot[0] > 1.0 ? sqrt(tot[2] / (tot[0] - 1.0)) : 0.0;

    /* learn */
    const orc_loss_cfg lc = {hp->clip, hp->vf_coef, hp->ent_coef, hp->bf16_operands};
    for (int64_t e = 0; e < epochs; ++e) {
        orc_perm(hp->seed, e, Br, perm);   /* every rank: the same rule over its Br rows */
        for (int64_t k = 0; k < minibatches; ++k) {
            double st[6] = {0, 0, 0, 0, 0, 0};
            memset(gsum, 0, sizeof(double) * (size_t)P);
            for (int64_t r = 0; r < world; ++r) {
                for (int64_t i = 0; i < mbr; ++i) {
                    const int64_t b = perm[k * mbr + i];   /* local row t * Nr + j */
                    idx[i] = (int32_t)((b / Nr) * N + r * Nr + b % Nr);
                }
                double st_r[6];
                orc_loss_grad(net, &lc, params, mbr, idx, obs, act_disc, act_cont, logp_old,
                              adv, ret, 1, mean, sdv, g, st_r, NULL);
                for (int64_t i = 0; i < P; ++i) gsum[i] += g[i];
                for (int q = 0; q < 6; ++q) st[q] += st_r[q];
            }
            for (int64_t i = 0; i < P; ++i) gsum[i] /= (double)world;
            if (stats)
                for (int q = 0; q < 6; ++q)
                    stats[(e * minibatches + k) * 6 + q] = st[q] / (double)world;
            orc_clip_grad_norm(P, gsum, hp->max_grad_norm);
            *step += 1;
            orc_optimize(net, hp, P, params, gsum, m, v, mom, *step);
        }
    }
    free(adv); free(ret); free(sr); free(sv); free(sd); free(sa); free(sret);
    free(perm); free(idx); free(g); free(gsum);
    return 0;
}
