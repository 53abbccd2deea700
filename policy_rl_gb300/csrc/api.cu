// api.cu -- the C ABI of include/ppo.h: context lifetime, argument checks,
// and the orchestration of one learner update ("Teaching Mario to speedrun",
// sec. 6 "The whole algorithm", steps 2 "judge" and 3 "learn") as a sequence
// of kernel launches on the caller's stream, captured once into a CUDA graph.
#include <algorithm>
#include <cmath>
#include <cstdio>
#include <cstring>
#include <new>
#include <vector>

#include "common.cuh"
#include "gemm.h"

using namespace ppo;

namespace {

constexpr uint64_t kTimeoutNs = 2000000000ull;  // bounded device waits: 2 s
constexpr int kMaxSplit = 64;

bool al16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

#define PPO_CUDA(x)                              \
  do {                                           \
    cudaError_t e_ = (x);                        \
    if (e_ != cudaSuccess) return PPO_ERR_CUDA;  \
  } while (0)

int64_t round_up(int64_t x, int64_t m) { return (x + m - 1) / m * m; }

struct UpdateKey {
  const void* p[9];
  int64_t T, N;
  int32_t epochs, minibatches;
  float gamma, lambda, lr;
  uint32_t seed;
  const void* stats;
  cudaStream_t stream;
  bool operator==(const UpdateKey& o) const { return std::memcmp(this, &o, sizeof(*this)) == 0; }
};

// one cached update: part 1 (GAE, moments, permutations) and part 2 (the
// rest) as two executable graphs, so that a host update can make part 2 wait
// for its observation copy
struct GraphEntry {
  UpdateKey key{};
  cudaGraphExec_t pre = nullptr, main = nullptr;
  uint64_t used = 0;
  bool valid = false;
  void reset() {
    // an executable graph still in flight is released when it completes
    if (pre) cudaGraphExecDestroy(pre);
    if (main) cudaGraphExecDestroy(main);
    pre = main = nullptr;
    valid = false;
  }
};
constexpr int kGraphCache = 4;

// device copy of one host rollout and the events that order its use:
// gae_in (values, rewards, dones, bootstrap) copied, rest (observations,
// actions, old log-probs) copied, freed (the update that read it and its
// stats copy-back done)
struct HostSlot {
  float *obs = nullptr, *actc = nullptr, *logp = nullptr, *val = nullptr, *rew = nullptr,
        *done = nullptr, *boot = nullptr;
  int32_t* act = nullptr;
  cudaEvent_t gae_in = nullptr, rest = nullptr, freed = nullptr;
  bool used = false;   // freed has been recorded at least once
  void destroy_events() {
    for (cudaEvent_t e : {gae_in, rest, freed})
      if (e) cudaEventDestroy(e);
    gae_in = rest = freed = nullptr;
  }
};

}  // namespace

struct ppo_ctx {
  ppo_config cfg;
  NetShape s;
  int bf16 = 0;
  int use_mk = 0;        // bf16: one persistent kernel per minibatch
  int num_sms = 1;
  unsigned* gbar = nullptr;
  unsigned long long* phase_ns = nullptr;   // persistent-kernel phase times (profiling)
  bool profiling = false;
  std::vector<void*> allocs;

  float *params = nullptr, *grad = nullptr, *m = nullptr, *v = nullptr;
  int64_t* step = nullptr;
  double* beta_pow = nullptr;
  unsigned* done_ctr = nullptr;
  int* err = nullptr;
  double* sq = nullptr;
  unsigned* wctr = nullptr;   // weight-gradient tile counters [2][kWgradMaxTiles]
  Shadows sh{};

  // minibatch workspace
  int64_t mbmax = 0;
  bool use_fmlp = false;   // fused forward + loss + backward-data kernel
  bool use_hl2 = false;    // head + loss + layer-2 backward-data kernel
  unsigned* rbar = nullptr; // grid-barrier counter of the reduce + Adam kernel
  // per-minibatch advantages from fresh values (adv_mode 1, 2)
  float *vfresh = nullptr, *rfresh = nullptr;   // [mbmax] fresh values / ratios
  float* fpart = nullptr;                       // [kFreshMaxGrid][3] moment partials
  // Muon (optimizer 1): momentum [P] and the Newton-Schulz workspaces
  float* mom = nullptr;
  float *ns_ws[3][4] = {};                      // per matrix: X0, X1 [r][k], A, B [r][r]
  float *mpart = nullptr, *minv = nullptr;
  MuonTc mtc{};                                 // bf16 contexts: tensor-core Newton-Schulz
  bool has_mtc = false;
  unsigned* fbar = nullptr;                     // grid-barrier counter of that kernel
  void* X = nullptr;
  // one epoch of minibatch rows gathered in permutation order (ppo_update)
  void* X_ep = nullptr;
  int32_t* act_ep = nullptr;
  float *actc_ep = nullptr, *logp_ep = nullptr, *adv_ep = nullptr, *ret_ep = nullptr;
  int32_t* act_mb = nullptr;
  float *actc_mb = nullptr, *logp_mb = nullptr, *adv_mb = nullptr, *ret_mb = nullptr;
  void *H1 = nullptr, *H2 = nullptr, *dZ = nullptr, *dP2 = nullptr, *dP1 = nullptr;
  int lddz = 0;
  float *pW1 = nullptr, *pW2 = nullptr, *pW3 = nullptr;
  float *cs1 = nullptr, *cs2 = nullptr, *cs3 = nullptr, *lossp = nullptr;

  // update workspace
  int64_t bmax = 0;
  int emax = 0;
  __nv_bfloat16* obs_packed = nullptr;
  float *adv = nullptr, *ret = nullptr, *advstats = nullptr;
  double* gae_part = nullptr;
  int32_t* perm = nullptr;
  void* perm_work = nullptr;

  // step trace (ppo_set_step_trace): per minibatch step, params, m, v before
  // the step and the assembled gradient after it, [trace_cap][4][P] fp32
  float* trace = nullptr;
  int64_t trace_cap = 0;
  // limit of the cooperative kernels' grid-barrier waits (ppo_set_wait_limit)
  uint64_t wait_ns = kTimeoutNs;
  // data-parallel learner (ppo_set_collective): this rank of `world`, the
  // caller's collective, the gathered shard moments [world][3]
  int world = 1, rank = 0;
  ppo_collective_fn coll = nullptr;
  void* coll_user = nullptr;
  double* mom_all = nullptr;
  int mom_cap = 0;

  // host-update staging (allocated on first ppo_update_host[_async]): two
  // slots, so that the copies of one call run while the previous call's
  // update still reads the other slot
  HostSlot hs[2];
  float* st_stats = nullptr;
  int64_t st_stats_cap = 0;
  int hs_next = 0;                  // slot of the next host update
  cudaStream_t hs_stream = nullptr; // the stream of the host updates in flight
  int hs_inflight = 0;              // host updates enqueued and not yet waited for

  // kernel-boundary trace hook (profiling) and its events
  Trace tr;
  std::vector<cudaEvent_t> prof_events;
  std::vector<int> prof_stages;

  // graph cache of ppo_update, least recently used entry replaced: one
  // entry per argument set (the two host staging slots are two)
  GraphEntry gc[kGraphCache];
  uint64_t gclock = 0;
  cudaStream_t cst = nullptr;             // host updates: the rollout copies

  void invalidate_graphs() {
    for (GraphEntry& g : gc) g.reset();
  }

  ppo_status alloc(void** p, size_t bytes) {
    void* q = nullptr;
    if (bytes == 0) bytes = 16;
    if (cudaMalloc(&q, bytes) != cudaSuccess) {
      cudaGetLastError();
      return PPO_ERR_NOMEM;
    }
    // zeroed on the legacy stream, which the library's non-blocking streams
    // do not wait for: finish it before any of them writes the buffer
    if (cudaMemset(q, 0, bytes) != cudaSuccess ||
        cudaStreamSynchronize(cudaStreamLegacy) != cudaSuccess) {
      cudaFree(q);
      return PPO_ERR_CUDA;
    }
    allocs.push_back(q);
    *p = q;
    return PPO_OK;
  }
  template <class T>
  ppo_status alloc_n(T** p, int64_t n) {
    return alloc(reinterpret_cast<void**>(p), (size_t)n * sizeof(T));
  }
  ~ppo_ctx() {
    if (has_mtc) {
      for (int i = 0; i < 3; ++i) {
        if (mtc.side[i]) cudaStreamDestroy(mtc.side[i]);
        if (mtc.join[i]) cudaEventDestroy(mtc.join[i]);
      }
      if (mtc.fork) cudaEventDestroy(mtc.fork);
    }
    invalidate_graphs();
    for (HostSlot& h : hs) h.destroy_events();
    if (cst) cudaStreamDestroy(cst);
    for (cudaEvent_t e : prof_events) cudaEventDestroy(e);
    for (void* p : allocs) cudaFree(p);
  }
};

#define TRY(x)                           \
  do {                                   \
    ppo_status s_ = (x);                 \
    if (s_ != PPO_OK) return s_;         \
  } while (0)

namespace {

ppo_status shape_from(const ppo_config* c, NetShape* s) {
  if (!c) return PPO_ERR_INVALID;
  if (c->obs_dim < 1 || c->h1 < 1 || c->h2 < 1) return PPO_ERR_INVALID;
  if (c->act != 0 && c->act != 1) return PPO_ERR_INVALID;
  if (c->n_heads < 0 || c->n_heads > PPO_MAX_HEADS) return PPO_ERR_INVALID;
  if (c->n_gauss < 0 || c->n_gauss > 4) return PPO_ERR_INVALID;
  if (c->precision != 0 && c->precision != 1) return PPO_ERR_INVALID;
  if (c->adv_mode < 0 || c->adv_mode > 2) return PPO_ERR_INVALID;
  if (c->optimizer != 0 && c->optimizer != 1) return PPO_ERR_INVALID;
  std::memset(s, 0, sizeof(*s));
  s->D = c->obs_dim;
  s->H1 = c->h1;
  s->H2 = c->h2;
  s->act = c->act;
  s->NH = c->n_heads;
  int C = 0;
  for (int h = 0; h < c->n_heads; ++h) {
    if (c->head_n[h] < 1) return PPO_ERR_INVALID;
    s->head_n[h] = c->head_n[h];
    C += c->head_n[h];
  }
  s->G = c->n_gauss;
  C += c->n_gauss + 1;
  if (C > 32) return PPO_ERR_UNSUPPORTED;
  s->C = C;
  s->CP = C <= 16 ? 16 : 32;
  s->Dp = c->precision == 1 ? (int)round_up(c->obs_dim, 64) : c->obs_dim;
  const int64_t D = s->D, H1 = s->H1, H2 = s->H2;
  s->oW1 = 0;
  s->ob1 = s->oW1 + H1 * D;
  s->oW2 = s->ob1 + H1;
  s->ob2 = s->oW2 + H2 * H1;
  s->oW3 = s->ob2 + H2;
  s->ob3 = s->oW3 + (int64_t)C * H2;
  s->ologstd = s->ob3 + C;
  s->P = s->ologstd + s->G;
  return PPO_OK;
}

// K-split length (64-row k-tiles) of the persistent kernel's weight-gradient
// units (at most 128 columns), chosen so that the units of all three products
// have roughly equal cost and number about the SM count, with at least 8
// k-tiles per unit.  In 128-column units: 64-column regions take twice as many.
int wgrad_kt_per_split(const NetShape& s, int64_t mb, int num_sms) {
  const int64_t kt = (mb + 63) / 64;
  auto tiles = [](int M, int N) { return (double)(M / 128) * (N / 128.0); };
  const double cost = (tiles(s.H2, s.H1) + tiles(s.H1, s.Dp) + tiles(s.H2, 64)) * (double)kt;
  int per = (int)std::ceil(cost / (double)num_sms);
  if (per < 8) per = 8;
  if ((kt + per - 1) / per > kMaxSplit) per = (int)((kt + kMaxSplit - 1) / kMaxSplit);
  return per;
}

// Split plan of the weight-gradient kernel for the MLP's three products:
// W2 (H2 x H1), W1 (H1 x Dp), W3 (H2 x 64); see tc_wgrad_plan.
struct WgradPlan {
  int kt[3];   // k-tiles per unit: W2 (H2 x H1), W1 (H1 x Dp), W3 (H2 x 64)
};

WgradPlan wgrad_plan(const NetShape& s, int64_t mb, int num_sms) {
  const int regs[3][2] = {{s.H2, s.H1}, {s.H1, s.Dp}, {s.H2, 64}};
  WgradPlan P{};
  tc_wgrad_plan(regs, 3, mb, num_sms, kMaxSplit, P.kt);
  return P;
}

ppo_status check_minibatch_args(ppo_ctx* c, const float* obs, const int32_t* act,
                                const float* actc, const float* logp, const float* adv,
                                const float* ret, const int32_t* idx, int64_t B, int64_t mb) {
  if (!c || !obs || !logp || !adv || !ret || !idx) return PPO_ERR_INVALID;
  if (c->s.NH > 0 && !act) return PPO_ERR_INVALID;
  if (c->s.G > 0 && !actc) return PPO_ERR_INVALID;
  if (mb < 1 || mb > c->mbmax || B < 1 || B >= (1ll << 31)) return PPO_ERR_INVALID;
  const void* ps[] = {obs, act, actc, logp, adv, ret, idx};
  for (const void* p : ps)
    if (p && !al16(p)) return PPO_ERR_ALIGN;
  return PPO_OK;
}

// Rows of one minibatch in minibatch order: X (bf16 [mb][Dp] or fp32 [mb][D]),
// actions, logp_old, normalised advantages, returns.
struct MbRows {
  void* X;
  int32_t* act;
  float *actc, *logp, *adv, *ret;
};

// Gathers rows idx[0..n) of the rollout into r (advantages normalised).
cudaError_t enqueue_gather(ppo_ctx* c, const float* obs, const __nv_bfloat16* obs_packed,
                           const int32_t* act, const float* actc, const float* logp_old,
                           const float* adv, const float* ret, const int32_t* idx, int64_t B,
                           int64_t n, const float* adv_stats, const MbRows& r, cudaStream_t st) {
  GatherArgs ga{};
  ga.obs_f32 = obs;
  ga.obs_bf16 = obs_packed;
  ga.act = act;
  ga.actc = actc;
  ga.logp_old = logp_old;
  ga.adv = adv;
  ga.ret = ret;
  ga.adv_stats = adv_stats;
  ga.idx = idx;
  ga.mb = n;
  ga.B = B;
  ga.X = r.X;
  ga.x_bf16 = c->bf16;
  ga.act_mb = r.act;
  ga.actc_mb = r.actc;
  ga.logp_mb = r.logp;
  ga.adv_mb = r.adv;
  ga.ret_mb = r.ret;
  return launch_gather(c->s, ga, st);
}

// Gathers the rows of minibatches of environment segments: n rows, minibatch m
// being envs[m*ns .. (m+1)*ns) over the horizon T, rows ordered t*ns + j.
// Advantages and returns are left to the fresh-advantage kernel.
cudaError_t enqueue_gather_seg(ppo_ctx* c, const float* obs, const __nv_bfloat16* obs_packed,
                               const int32_t* act, const float* actc, const float* logp_old,
                               const int32_t* envs, int T, int ns, int64_t N, int64_t n,
                               const MbRows& r, cudaStream_t st) {
  GatherArgs ga{};
  ga.obs_f32 = obs;
  ga.obs_bf16 = obs_packed;
  ga.act = act;
  ga.actc = actc;
  ga.logp_old = logp_old;
  ga.mb = n;
  ga.B = (int64_t)T * N;
  ga.seg_envs = envs;
  ga.seg_T = T;
  ga.seg_ns = ns;
  ga.seg_N = N;
  ga.X = r.X;
  ga.x_bf16 = c->bf16;
  ga.act_mb = r.act;
  ga.actc_mb = r.actc;
  ga.logp_mb = r.logp;
  return launch_gather(c->s, ga, st);
}

// Advantages of one minibatch from fresh values: the rollout's rewards, dones
// and bootstrap values, the minibatch's environments, and the scan's settings.
struct FreshSpec {
  const float *rew, *done, *boot;
  const int32_t* envs;   // [ns]
  int T, ns;
  int64_t N;
  float gamma, lambda;
  int vtrace;
};

// One minibatch: gather (unless its rows are given, already gathered),
// forward, [advantages from fresh values], loss, backward, gradient assembly.
ppo_status enqueue_minibatch(ppo_ctx* c, const float* obs, const __nv_bfloat16* obs_packed,
                             const int32_t* act, const float* actc, const float* logp_old,
                             const float* adv, const float* ret, const int32_t* idx, int64_t B,
                             int64_t mb, const float* adv_stats, float* stats6, cudaStream_t st,
                             int* nsq_out = nullptr, const MbRows* pre = nullptr,
                             const AdamArgs* adam = nullptr, const FreshSpec* fr = nullptr,
                             int64_t mb_global = 0) {
  const NetShape& s = c->s;
  MbRows mr{c->X, c->act_mb, c->actc_mb, c->logp_mb, c->adv_mb, c->ret_mb};
  if (pre) {
    mr = *pre;
  } else {
    PPO_CUDA(enqueue_gather(c, obs, obs_packed, act, actc, logp_old, adv, ret, idx, B, mb,
                            adv_stats, mr, st));
    c->tr.mark(ST_GATHER, st);
  }

  LossRows rows{mr.act, mr.actc, mr.logp, mr.adv, mr.ret};
  LossCoef lc{c->cfg.clip, c->cfg.vf_coef, c->cfg.ent_coef};
  // the loss is a mean over the minibatch: over all ranks' rows when the
  // minibatch is the union of the ranks' slices (data-parallel update)
  const float inv_mb = 1.0f / (float)(mb_global > 0 ? mb_global : mb);
  const float* P = c->params;
  const int M = (int)mb;
  // advantages from the values (and ratios) of the forward pass just run;
  // they overwrite the minibatch rows' advantages (normalised) and returns
  auto fresh_adv = [&](const void* H2) -> cudaError_t {
    FreshAdvArgs f{};
    f.head = 1;
    f.s = s;
    f.H2 = H2;
    f.h2_bf16 = c->bf16;
    f.W3 = c->bf16 ? static_cast<const void*>(c->sh.W3s) : static_cast<const void*>(P + s.oW3);
    f.b3 = P + s.ob3;
    f.logstd = P + s.ologstd;
    f.act = mr.act;
    f.actc = mr.actc;
    f.logp_old = mr.logp;
    f.rew = fr->rew;
    f.done = fr->done;
    f.boot = fr->boot;
    f.envs = fr->envs;
    f.T = fr->T;
    f.ns = fr->ns;
    f.N = fr->N;
    f.val = c->vfresh;
    f.ratio = fr->vtrace ? c->rfresh : nullptr;
    f.gamma = fr->gamma;
    f.lambda = fr->lambda;
    f.rho_clip = c->cfg.vtrace_rho_clip;
    f.c_clip = c->cfg.vtrace_c_clip;
    f.adv = mr.adv;
    f.ret = mr.ret;
    f.adv_norm = mr.adv;
    f.part = c->fpart;
    f.bar = c->fbar;
    f.err = c->err;
    f.timeout_ns = c->wait_ns;
    cudaError_t e = launch_fresh_adv(f, c->num_sms, st);
    if (e == cudaSuccess) c->tr.mark(ST_FRESH_ADV, st);
    return e;
  };

  ReduceArgs ra{};
  ra.s = s;
  ra.inv_mb = inv_mb;
  ra.grad = c->grad;
  ra.stats6 = stats6;
  ra.sq_part = nsq_out ? c->sq : nullptr;   // fused squared-norm partials for Adam
  ra.weights_done = 0;
  ra.nsq_pre = 0;

  if (c->bf16) {
    auto* X = static_cast<__nv_bfloat16*>(mr.X);
    auto* H1 = static_cast<__nv_bfloat16*>(c->H1);
    auto* H2 = static_cast<__nv_bfloat16*>(c->H2);
    auto* dZ = static_cast<__nv_bfloat16*>(c->dZ);
    auto* dP2 = static_cast<__nv_bfloat16*>(c->dP2);
    auto* dP1 = static_cast<__nv_bfloat16*>(c->dP1);
    const int ns = c->num_sms;
    int n3 = 0, n2 = 0, n1 = 0;
    if (c->use_fmlp && !fr) {
      // forward, loss and backward-data in one kernel (activations stay on chip)
      FusedMlp f{};
      f.s = s;
      f.M = M;
      f.X = X;
      f.W1s = c->sh.W1s;
      f.W2s = c->sh.W2s;
      f.W3s = c->sh.W3s;
      f.W3Ts = c->sh.W3Ts;
      f.W2Ts = c->sh.W2Ts;
      f.ld3t = c->sh.ld3t;
      f.b1 = P + s.ob1;
      f.b2 = P + s.ob2;
      f.b3 = P + s.ob3;
      f.logstd = P + s.ologstd;
      f.H1 = H1;
      f.H2 = H2;
      f.dZ = dZ;
      f.dP2 = dP2;
      f.dP1 = dP1;
      f.lddz = c->lddz;
      f.lc = lc;
      f.rows = rows;
      f.inv_mb = inv_mb;
      f.cs1 = c->cs1;
      f.cs2 = c->cs2;
      f.cs3 = c->cs3;
      f.lossp = c->lossp;
      f.err = c->err;
      f.timeout_ns = kTimeoutNs;
      PPO_CUDA(fmlp_launch(f, ns, st, &n1));
      n2 = n3 = n1;
      c->tr.mark(ST_FUSED_MLP, st);
    } else {
    // forward: H1 = act(X W1^T + b1), H2 = act(H1 W2^T + b2)
    GemmOperands g1{X, s.Dp, c->sh.W1s, s.Dp, M, s.H1, s.Dp};
    PPO_CUDA(tc_gemm_bias_act(g1, P + s.ob1, s.act, H1, s.H1, c->err, kTimeoutNs, ns, st));
    c->tr.mark(ST_FWD1, st);
    GemmOperands g2{H1, s.H1, c->sh.W2s, s.H1, M, s.H2, s.H1};
    PPO_CUDA(tc_gemm_bias_act(g2, P + s.ob2, s.act, H2, s.H2, c->err, kTimeoutNs, ns, st));
    c->tr.mark(ST_FWD2, st);
    if (fr) PPO_CUDA(fresh_adv(H2));
    if (c->use_hl2) {
      // head + loss + dP2 = (dz W3) * act'(H2) in one kernel (H2 read once)
      HeadLossDact f{};
      f.s = s;
      f.M = M;
      f.H2 = H2;
      f.W3s = c->sh.W3s;
      f.b3 = P + s.ob3;
      f.logstd = P + s.ologstd;
      f.dZ = dZ;
      f.dP2 = dP2;
      f.lddz = c->lddz;
      f.lc = lc;
      f.rows = rows;
      f.inv_mb = inv_mb;
      f.cs2 = c->cs2;
      f.cs3 = c->cs3;
      f.lossp = c->lossp;
      f.err = c->err;
      f.timeout_ns = kTimeoutNs;
      PPO_CUDA(hl2_launch(f, ns, st, &n3));
      n2 = n3;
      c->tr.mark(ST_LOSS_DACT2, st);
    } else {
      // head + loss: z = H2 W3^T + b3 -> dz
      GemmOperands g3{H2, s.H2, c->sh.W3s, s.H2, M, s.CP, s.H2};
      PPO_CUDA(tc_gemm_loss(g3, s, lc, rows, inv_mb, P + s.ob3, P + s.ologstd, dZ, c->lddz,
                            c->cs3, c->lossp, c->err, kTimeoutNs, ns, st, &n3));
      c->tr.mark(ST_LOSS, st);
      // backward data: dP2 = (dz W3) * act'(H2)
      GemmOperands g4{dZ, c->lddz, c->sh.W3Ts, c->sh.ld3t, M, s.H2, s.CP};
      PPO_CUDA(tc_gemm_dact(g4, H2, s.H2, s.act, dP2, s.H2, c->cs2, c->err, kTimeoutNs, ns, st,
                            &n2));
      c->tr.mark(ST_DACT2, st);
    }
    // backward data: dP1 = (dP2 W2) * act'(H1)
    GemmOperands g5{dP2, s.H2, c->sh.W2Ts, s.H2, M, s.H1, s.H2};
    PPO_CUDA(tc_gemm_dact(g5, H1, s.H1, s.act, dP1, s.H1, c->cs1, c->err, kTimeoutNs, ns, st, &n1));
    c->tr.mark(ST_DACT1, st);
    }
    // weight gradients, split over the minibatch rows; the kernel also sums
    // the split partials into the flat gradient (dW3 from its transpose) and
    // writes the squared-norm partials of those entries to sq[0 .. wg_grid)
    const WgradPlan wp = wgrad_plan(s, mb, ns);
    float* G = c->grad;
    WGradRegion regs[3] = {
        {dP2, s.H2, s.H2, H1, s.H1, s.H1, wp.kt[0], c->pW2, {G + s.oW2, s.H2, s.H1, s.H1, 1}},
        {dP1, s.H1, s.H1, X, s.Dp, s.Dp, wp.kt[1], c->pW1, {G + s.oW1, s.H1, s.D, s.D, 1}},
        {H2, s.H2, s.H2, dZ, c->lddz, 64, wp.kt[2], c->pW3, {G + s.oW3, s.H2, s.C, 1, s.H2}}};
    // ... and the bias / log-std / statistic entries from the epilogues'
    // per-CTA partial rows, so that its squared-norm partials cover the
    // whole gradient and the optimizer follows directly
    ra.pb1 = c->cs1; ra.nb1 = n1;
    ra.pb2 = c->cs2; ra.nb2 = n2;
    ra.pb3 = c->cs3; ra.nb3 = n3; ra.ldb3 = s.CP;
    ra.ploss = c->lossp; ra.nl = n3;
    if (!pre)   // standalone call: the tile counters start at zero (also after a timeout)
      PPO_CUDA(cudaMemsetAsync(c->wctr, 0, 2 * kWgradMaxTiles * sizeof(unsigned), st));
    int wg_grid = 0;
    PPO_CUDA(tc_wgrad(regs, 3, M, 8192, 1024, c->err, kTimeoutNs, ns, st, c->wctr, c->sq,
                      &wg_grid, c->wait_ns, &ra));
    c->tr.mark(ST_WGRAD, st);
    if (adam) {   // clip + Adam (its norm from the weight-gradient kernel's partials)
      AdamArgs aa = *adam;
      aa.sq_part = c->sq;
      aa.nsq = wg_grid;
      PPO_CUDA(launch_adam(aa, st, &c->tr));
    }
    if (nsq_out) *nsq_out = wg_grid;
    return PPO_OK;
  } else {
    auto* X = static_cast<float*>(mr.X);
    auto* H1 = static_cast<float*>(c->H1);
    auto* H2 = static_cast<float*>(c->H2);
    auto* dZ = static_cast<float*>(c->dZ);
    auto* dP2 = static_cast<float*>(c->dP2);
    auto* dP1 = static_cast<float*>(c->dP1);
    SimtOperands g1{X, s.D, 1, P + s.oW1, s.D, 1, M, s.H1, s.D};
    PPO_CUDA(simt_bias_act(g1, P + s.ob1, s.act, H1, s.H1, st));
    c->tr.mark(ST_FWD1, st);
    SimtOperands g2{H1, s.H1, 1, P + s.oW2, s.H1, 1, M, s.H2, s.H1};
    PPO_CUDA(simt_bias_act(g2, P + s.ob2, s.act, H2, s.H2, st));
    c->tr.mark(ST_FWD2, st);
    if (fr) PPO_CUDA(fresh_adv(H2));
    int n3 = 0;
    PPO_CUDA(simt_head_loss(s, lc, rows, inv_mb, H2, P + s.oW3, P + s.ob3, P + s.ologstd, M, dZ,
                            c->cs3, c->lossp, st, &n3));
    c->tr.mark(ST_LOSS, st);
    // dP2(m, n) = sum_c dz(m, c) W3[c][n] * act'(H2)
    SimtOperands g4{dZ, s.CP, 1, P + s.oW3, 1, s.H2, M, s.H2, s.C};
    PPO_CUDA(simt_dact(g4, H2, s.H2, s.act, dP2, s.H2, c->cs2, st));
    c->tr.mark(ST_DACT2, st);
    SimtOperands g5{dP2, s.H2, 1, P + s.oW2, 1, s.H1, M, s.H1, s.H2};
    PPO_CUDA(simt_dact(g5, H1, s.H1, s.act, dP1, s.H1, c->cs1, st));
    c->tr.mark(ST_DACT1, st);
    // split-K weight gradients (transposed dW3 like the tensor-core path)
    auto kps = [&](int Mo, int No) {
      const int tiles = ((Mo + 63) / 64) * ((No + 63) / 64);
      int splits = (2 * c->num_sms + tiles - 1) / tiles;
      if (splits > kMaxSplit) splits = kMaxSplit;
      if (splits < 1) splits = 1;
      int k = (int)((mb + splits - 1) / splits);
      k = (int)round_up(k, 16);
      return k;
    };
    const int k2 = kps(s.H2, s.H1), k1 = kps(s.H1, s.D), k3 = kps(s.H2, s.CP);
    SimtOperands w2{dP2, 1, s.H2, H1, 1, s.H1, s.H2, s.H1, M};
    PPO_CUDA(simt_wgrad(w2, k2, c->pW2, st));
    c->tr.mark(ST_WGRAD, st);
    SimtOperands w1{dP1, 1, s.H1, X, 1, s.D, s.H1, s.D, M};
    PPO_CUDA(simt_wgrad(w1, k1, c->pW1, st));
    c->tr.mark(ST_WGRAD, st);
    SimtOperands w3{H2, 1, s.H2, dZ, 1, s.CP, s.H2, s.CP, M};
    PPO_CUDA(simt_wgrad(w3, k3, c->pW3, st));
    c->tr.mark(ST_WGRAD, st);
    ra.pW1 = c->pW1; ra.s1 = (int)((mb + k1 - 1) / k1); ra.ld1 = s.D;
    ra.pW2 = c->pW2; ra.s2 = (int)((mb + k2 - 1) / k2);
    ra.pW3t = c->pW3; ra.s3 = (int)((mb + k3 - 1) / k3); ra.ld3 = s.CP;
    ra.pb1 = c->cs1; ra.nb1 = simt_tiles_m(M);
    ra.pb2 = c->cs2; ra.nb2 = simt_tiles_m(M);
    ra.pb3 = c->cs3; ra.nb3 = n3; ra.ldb3 = s.CP;
    ra.ploss = c->lossp; ra.nl = n3;
  }
  if (adam) {   // gradient assembly, clip and Adam in one cooperative launch
    ra.sq_part = c->sq + ra.nsq_pre;
    PPO_CUDA(launch_reduce_adam(ra, *adam, c->rbar, c->err, c->wait_ns, c->num_sms, st));
    c->tr.mark(ST_REDUCE_ADAM, st);
    return PPO_OK;
  }
  PPO_CUDA(launch_reduce(ra, st));
  c->tr.mark(ST_REDUCE, st);
  if (nsq_out) *nsq_out = ra.nsq_pre + reduce_launch_blocks(ra);
  return PPO_OK;
}

AdamArgs make_adam_args(ppo_ctx* c, float lr, float* grad_norm_out, int nsq) {
  AdamArgs a{};
  a.p = c->params;
  a.g = c->grad;
  a.m = c->m;
  a.v = c->v;
  a.P = c->s.P;
  a.sq_part = c->sq;
  a.nsq = nsq;
  a.max_norm = c->cfg.max_grad_norm;
  a.lr = lr;
  a.b1 = c->cfg.beta1;
  a.b2 = c->cfg.beta2;
  a.eps = c->cfg.adam_eps;
  a.omb1 = (float)(1.0 - c->cfg.beta1);   // 1 - beta in double: no cancellation in fp32
  a.omb2 = (float)(1.0 - c->cfg.beta2);
  a.step = c->step;
  a.beta_pow = c->beta_pow;
  a.done_ctr = c->done_ctr;
  a.grad_norm_out = grad_norm_out;
  a.s = c->s;
  a.sh = c->sh;
  return a;
}

MuonArgs make_muon_args(ppo_ctx* c) {
  const NetShape& s = c->s;
  MuonArgs mu{};
  const int64_t offs[3] = {s.oW1, s.oW2, s.oW3};
  const int rows[3] = {s.H1, s.H2, s.C}, cols[3] = {s.D, s.H1, s.H2};
  for (int m = 0; m < 3; ++m) {
    MuonMat& w = mu.m[m];
    w.p = c->params + offs[m];
    w.g = c->grad + offs[m];
    w.mom = c->mom + offs[m];
    w.rows = rows[m];
    w.cols = cols[m];
    w.off = offs[m];
    w.X0 = c->ns_ws[m][0];
    w.X1 = c->ns_ws[m][1];
    w.A = c->ns_ws[m][2];
    w.B = c->ns_ws[m][3];
  }
  mu.beta = c->cfg.muon_beta;
  mu.lr = c->cfg.muon_lr;
  mu.mpart = c->mpart;
  mu.inv = c->minv;
  mu.s = s;
  mu.sh = c->sh;
  return mu;
}

ppo_status enqueue_muon(ppo_ctx* c, float lr, float* grad_norm_out, cudaStream_t st, int nsq) {
  if (!c->mom) return PPO_ERR_INVALID;   // context created with optimizer 0
  const AdamArgs a = make_adam_args(c, lr, grad_norm_out, nsq);
  PPO_CUDA(launch_muon(make_muon_args(c), a, st, &c->tr, c->has_mtc ? &c->mtc : nullptr));
  return PPO_OK;
}

ppo_status enqueue_adam(ppo_ctx* c, float lr, float* grad_norm_out, cudaStream_t st,
                        int nsq = 0) {
  const AdamArgs a = make_adam_args(c, lr, grad_norm_out, nsq);
  PPO_CUDA(launch_adam(a, st, &c->tr));
  return PPO_OK;
}

// One bf16 minibatch (gather .. gradient assembly, and Adam when do_adam) as
// one persistent cooperative kernel.
ppo_status enqueue_minibatch_mk(ppo_ctx* c, const float* obs, const __nv_bfloat16* obs_packed,
                                const int32_t* act, const float* actc, const float* logp_old,
                                const float* adv, const float* ret, const int32_t* idx, int64_t B,
                                int64_t mb, const float* adv_stats, float* stats6, int do_adam,
                                float lr, cudaStream_t st) {
  const NetShape& s = c->s;
  const float* P = c->params;
  const int M = (int)mb;
  const int grid = mk_grid(c->num_sms);
  auto* X = static_cast<__nv_bfloat16*>(c->X);
  auto* H1 = static_cast<__nv_bfloat16*>(c->H1);
  auto* H2 = static_cast<__nv_bfloat16*>(c->H2);
  auto* dZ = static_cast<__nv_bfloat16*>(c->dZ);
  auto* dP2 = static_cast<__nv_bfloat16*>(c->dP2);
  auto* dP1 = static_cast<__nv_bfloat16*>(c->dP1);
  MkLaunch L{};
  L.s = s;
  L.ga.obs_f32 = obs;
  L.ga.obs_bf16 = obs_packed;
  L.ga.act = act;
  L.ga.actc = actc;
  L.ga.logp_old = logp_old;
  L.ga.adv = adv;
  L.ga.ret = ret;
  L.ga.adv_stats = adv_stats;
  L.ga.idx = idx;
  L.ga.mb = mb;
  L.ga.B = B;
  L.ga.X = X;
  L.ga.x_bf16 = 1;
  L.ga.act_mb = c->act_mb;
  L.ga.actc_mb = c->actc_mb;
  L.ga.logp_mb = c->logp_mb;
  L.ga.adv_mb = c->adv_mb;
  L.ga.ret_mb = c->ret_mb;
  L.fwd1 = GemmOperands{X, s.Dp, c->sh.W1s, s.Dp, M, s.H1, s.Dp};
  L.fwd2 = GemmOperands{H1, s.H1, c->sh.W2s, s.H1, M, s.H2, s.H1};
  L.loss = GemmOperands{H2, s.H2, c->sh.W3s, s.H2, M, s.CP, s.H2};
  L.dact2 = GemmOperands{dZ, c->lddz, c->sh.W3Ts, c->sh.ld3t, M, s.H2, s.CP};
  L.dact1 = GemmOperands{dP2, s.H2, c->sh.W2Ts, s.H2, M, s.H1, s.H2};
  L.b1 = P + s.ob1;
  L.b2 = P + s.ob2;
  L.b3 = P + s.ob3;
  L.logstd = P + s.ologstd;
  L.H1 = H1;
  L.H2 = H2;
  L.dP2 = dP2;
  L.dP1 = dP1;
  L.dz = dZ;
  L.lddz = c->lddz;
  L.cs1 = c->cs1;
  L.cs2 = c->cs2;
  L.cs3 = c->cs3;
  L.loss_part = c->lossp;
  const int per = wgrad_kt_per_split(s, mb, grid);
  L.wg[0] = {dP2, s.H2, s.H2, H1, s.H1, s.H1, per, c->pW2};
  L.wg[1] = {dP1, s.H1, s.H1, X, s.Dp, s.Dp, s.Dp % 128 == 0 ? per : 2 * per, c->pW1};
  L.wg[2] = {H2, s.H2, s.H2, dZ, c->lddz, 64, 2 * per, c->pW3};
  for (auto& r : L.wg)
    if (tc_wgrad_splits(M, r.kt_per_split) > kMaxSplit)
      r.kt_per_split = (int)(((mb + 63) / 64 + kMaxSplit - 1) / kMaxSplit);
  L.rows = M;
  ReduceArgs& ra = L.ra;
  ra.s = s;
  ra.inv_mb = 1.0f / (float)mb;
  ra.grad = c->grad;
  ra.stats6 = stats6;
  ra.pW1 = c->pW1; ra.s1 = tc_wgrad_splits(M, L.wg[1].kt_per_split); ra.ld1 = s.Dp;
  ra.pW2 = c->pW2; ra.s2 = tc_wgrad_splits(M, L.wg[0].kt_per_split);
  ra.pW3t = c->pW3; ra.s3 = tc_wgrad_splits(M, L.wg[2].kt_per_split); ra.ld3 = 64;
  ra.pb1 = c->cs1; ra.nb1 = grid;
  ra.pb2 = c->cs2; ra.nb2 = grid;
  ra.pb3 = c->cs3; ra.nb3 = grid; ra.ldb3 = s.CP;
  ra.ploss = c->lossp; ra.nl = grid;
  L.do_adam = do_adam;
  AdamArgs& a = L.aa;
  a.p = c->params;
  a.g = c->grad;
  a.m = c->m;
  a.v = c->v;
  a.P = s.P;
  a.max_norm = c->cfg.max_grad_norm;
  a.lr = lr;
  a.b1 = c->cfg.beta1;
  a.b2 = c->cfg.beta2;
  a.eps = (float)c->cfg.adam_eps;
  a.omb1 = (float)(1.0 - c->cfg.beta1);
  a.omb2 = (float)(1.0 - c->cfg.beta2);
  a.step = c->step;
  a.beta_pow = c->beta_pow;
  a.s = s;
  a.sh = c->sh;
  L.lc = LossCoef{c->cfg.clip, c->cfg.vf_coef, c->cfg.ent_coef};
  L.rows_in = LossRows{c->act_mb, c->actc_mb, c->logp_mb, c->adv_mb, c->ret_mb};
  L.inv_mb = 1.0f / (float)mb;
  L.gbar = c->gbar;
  L.sq_part = c->sq;
  L.phase_ns = c->profiling ? c->phase_ns : nullptr;
  L.err = c->err;
  L.timeout_ns = kTimeoutNs;
  L.grid = grid;
  PPO_CUDA(mk_launch(L, st));
  c->tr.mark(ST_MINIBATCH, st);
  return PPO_OK;
}

ppo_status collective(ppo_ctx* c, int32_t op, void* buf, int64_t count, cudaStream_t st) {
  return c->coll(c->coll_user, op, buf, count, st) == 0 ? PPO_OK : PPO_ERR_CUDA;
}

// Step trace of minibatch step j: params, m, v before the step (after == 0),
// the assembled (unclipped) gradient after it (after == 1).
cudaError_t trace_step(ppo_ctx* c, int64_t j, int after, cudaStream_t st) {
  if (!c->trace || j >= c->trace_cap) return cudaSuccess;
  const int64_t P = c->s.P;
  float* slot = c->trace + j * 4 * P;
  const size_t bytes = sizeof(float) * (size_t)P;
  if (after) return cudaMemcpyAsync(slot + 3 * P, c->grad, bytes, cudaMemcpyDeviceToDevice, st);
  const float* src[3] = {c->params, c->m, c->v};
  for (int i = 0; i < 3; ++i) {
    cudaError_t e = cudaMemcpyAsync(slot + i * P, src[i], bytes, cudaMemcpyDeviceToDevice, st);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

ppo_status enqueue_update(ppo_ctx* c, const float* obs, const int32_t* act, const float* actc,
                          const float* logp_old, const float* val, const float* rew,
                          const float* done, const float* boot, int64_t T, int64_t N,
                          int32_t epochs, int32_t minibatches, float gamma, float lambda,
                          float lr, uint32_t seed, float* stats, cudaStream_t st,
                          int parts = 3) {
  const int64_t B = T * N, mb = B / minibatches;
  const __nv_bfloat16* packed = c->bf16 ? c->obs_packed : nullptr;
  if (c->cfg.adv_mode != 0) {
    // advantages per minibatch of environment segments, from fresh values
    // ("Teaching Mario to speedrun", sec. 8); epoch e shuffles the N
    // environments with the mulberry32 rule, minibatch k takes N/M of them
    const int ns = (int)(N / minibatches);
    if (parts & 1) {
      // barrier and Adam completion counters start at zero (also after a
      // launch that gave up on a bounded wait)
      PPO_CUDA(cudaMemsetAsync(c->rbar, 0, sizeof(unsigned), st));
      PPO_CUDA(cudaMemsetAsync(c->fbar, 0, sizeof(unsigned), st));
      PPO_CUDA(cudaMemsetAsync(c->done_ctr, 0, sizeof(unsigned), st));
      PPO_CUDA(cudaMemsetAsync(c->wctr, 0, 2 * kWgradMaxTiles * sizeof(unsigned), st));
      PPO_CUDA(launch_perm(seed, 0, epochs, N, c->perm, c->perm_work, st, &c->tr));
    }
    if (!(parts & 2)) return PPO_OK;
    if (c->bf16) {
      PPO_CUDA(launch_pack_obs(obs, B, c->s.D, c->s.Dp, c->obs_packed, st));
      c->tr.mark(ST_PACK, st);
    }
    const MbRows ep{c->X_ep, c->act_ep, c->actc_ep, c->logp_ep, c->adv_ep, c->ret_ep};
    const int64_t xrow = c->bf16 ? (int64_t)c->s.Dp * 2 : (int64_t)c->s.D * 4;
    const int NH = c->s.NH > 0 ? c->s.NH : 1, G = c->s.G > 0 ? c->s.G : 1;
    for (int e = 0; e < epochs; ++e) {
      const int32_t* perm_e = c->perm + (int64_t)e * N;
      PPO_CUDA(enqueue_gather_seg(c, obs, packed, act, actc, logp_old, perm_e, (int)T, ns, N, B,
                                  ep, st));
      c->tr.mark(ST_GATHER, st);
      for (int k = 0; k < minibatches; ++k) {
        float* st6 = stats ? stats + ((int64_t)e * minibatches + k) * 6 : nullptr;
        const int64_t r0 = (int64_t)k * mb;
        const MbRows mr{static_cast<uint8_t*>(ep.X) + r0 * xrow, ep.act + r0 * NH,
                        ep.actc + r0 * G, ep.logp + r0, ep.adv + r0, ep.ret + r0};
        const AdamArgs aa = make_adam_args(c, lr, nullptr, 0);
        const FreshSpec fs{rew, done, boot, perm_e + (int64_t)k * ns, (int)T, ns, N, gamma,
                           lambda, c->cfg.adv_mode == 2};
        const int64_t j = (int64_t)e * minibatches + k;
        PPO_CUDA(trace_step(c, j, 0, st));
        if (c->cfg.optimizer == 1) {
          int nsq = 0;
          TRY(enqueue_minibatch(c, obs, packed, act, actc, logp_old, nullptr, nullptr, nullptr,
                                B, mb, nullptr, st6, st, &nsq, &mr, nullptr, &fs));
          PPO_CUDA(trace_step(c, j, 1, st));
          TRY(enqueue_muon(c, lr, nullptr, st, nsq));
        } else {
          TRY(enqueue_minibatch(c, obs, packed, act, actc, logp_old, nullptr, nullptr, nullptr,
                                B, mb, nullptr, st6, st, nullptr, &mr, &aa, &fs));
          PPO_CUDA(trace_step(c, j, 1, st));
        }
      }
    }
    return PPO_OK;
  }
  if (parts & 1) {
    // part 1 reads only rewards, values, dones and bootstrap values
    if (c->use_mk)   // grid-barrier counters start at zero (also after an aborted launch)
      PPO_CUDA(cudaMemsetAsync(c->gbar, 0, 2 * sizeof(unsigned), st));
    else
      PPO_CUDA(cudaMemsetAsync(c->rbar, 0, sizeof(unsigned), st));
    PPO_CUDA(cudaMemsetAsync(c->done_ctr, 0, sizeof(unsigned), st));
    PPO_CUDA(cudaMemsetAsync(c->wctr, 0, 2 * kWgradMaxTiles * sizeof(unsigned), st));
    PPO_CUDA(launch_gae(rew, val, done, boot, (int)T, (int)N, gamma, lambda, c->adv, c->ret,
                        c->gae_part, gae_num_blocks((int)N), st));
    c->tr.mark(ST_GAE, st);
    if (c->world > 1) {
      // this shard's (count, mean, M2), every rank's gathered, merged in a
      // fixed order: the same global statistics on every rank
      PPO_CUDA(launch_gae_moments(c->gae_part, gae_num_blocks((int)N), c->mom_all + 3 * c->rank,
                                  st));
      TRY(collective(c, PPO_COLL_ALLGATHER_F64, c->mom_all, 3, st));
      PPO_CUDA(launch_gae_finalize(c->mom_all, c->world, c->advstats, st));
    } else {
      PPO_CUDA(launch_gae_finalize(c->gae_part, gae_num_blocks((int)N), c->advstats, st));
    }
    c->tr.mark(ST_GAE_FINALIZE, st);
    PPO_CUDA(launch_perm(seed, 0, epochs, B, c->perm, c->perm_work, st, &c->tr));
  }
  if (!(parts & 2)) return PPO_OK;
  if (c->bf16) {
    PPO_CUDA(launch_pack_obs(obs, B, c->s.D, c->s.Dp, c->obs_packed, st));
    c->tr.mark(ST_PACK, st);
  }
  const MbRows ep{c->X_ep, c->act_ep, c->actc_ep, c->logp_ep, c->adv_ep, c->ret_ep};
  const int64_t xrow = c->bf16 ? (int64_t)c->s.Dp * 2 : (int64_t)c->s.D * 4;
  const int NH = c->s.NH > 0 ? c->s.NH : 1, G = c->s.G > 0 ? c->s.G : 1;
  for (int e = 0; e < epochs; ++e) {
    const int32_t* perm_e = c->perm + (int64_t)e * B;
    if (!c->use_mk) {
      // the epoch's rows in permutation order: one gather for all its minibatches
      PPO_CUDA(enqueue_gather(c, obs, packed, act, actc, logp_old, c->adv, c->ret, perm_e, B, B,
                              c->advstats, ep, st));
      c->tr.mark(ST_GATHER, st);
    }
    for (int k = 0; k < minibatches; ++k) {
      const int32_t* idx = perm_e + (int64_t)k * mb;
      float* st6 = stats ? stats + ((int64_t)e * minibatches + k) * 6 : nullptr;
      const int64_t j = (int64_t)e * minibatches + k;
      PPO_CUDA(trace_step(c, j, 0, st));
      if (c->use_mk) {
        TRY(enqueue_minibatch_mk(c, obs, packed, act, actc, logp_old, c->adv, c->ret, idx, B, mb,
                                 c->advstats, st6, 1, lr, st));
        PPO_CUDA(trace_step(c, j, 1, st));
      } else if (c->world > 1) {
        // data-parallel step: this rank's slice of minibatch k, scaled for the
        // union of the ranks' slices; the gradient (and the statistics) summed
        // over the ranks before the optimizer, which recomputes the norm
        const int64_t r0 = (int64_t)k * mb;
        const MbRows mr{static_cast<uint8_t*>(ep.X) + r0 * xrow, ep.act + r0 * NH,
                        ep.actc + r0 * G, ep.logp + r0, ep.adv + r0, ep.ret + r0};
        TRY(enqueue_minibatch(c, obs, packed, act, actc, logp_old, c->adv, c->ret, idx, B, mb,
                              c->advstats, st6, st, nullptr, &mr, nullptr, nullptr,
                              mb * c->world));
        TRY(collective(c, PPO_COLL_ALLREDUCE_SUM_F32, c->grad, c->s.P, st));
        if (st6) TRY(collective(c, PPO_COLL_ALLREDUCE_SUM_F32, st6, 6, st));
        PPO_CUDA(trace_step(c, j, 1, st));
        if (c->cfg.optimizer == 1)
          TRY(enqueue_muon(c, lr, nullptr, st, 0));
        else
          TRY(enqueue_adam(c, lr, nullptr, st, 0));
      } else {
        const int64_t r0 = (int64_t)k * mb;
        const MbRows mr{static_cast<uint8_t*>(ep.X) + r0 * xrow, ep.act + r0 * NH,
                        ep.actc + r0 * G, ep.logp + r0, ep.adv + r0, ep.ret + r0};
        const AdamArgs aa = make_adam_args(c, lr, nullptr, 0);
        if (c->cfg.optimizer == 1) {
          int nsq = 0;
          TRY(enqueue_minibatch(c, obs, packed, act, actc, logp_old, c->adv, c->ret, idx, B, mb,
                                c->advstats, st6, st, &nsq, &mr));
          PPO_CUDA(trace_step(c, j, 1, st));
          TRY(enqueue_muon(c, lr, nullptr, st, nsq));
        } else {
          TRY(enqueue_minibatch(c, obs, packed, act, actc, logp_old, c->adv, c->ret, idx, B, mb,
                                c->advstats, st6, st, nullptr, &mr, &aa));
          PPO_CUDA(trace_step(c, j, 1, st));
        }
      }
    }
  }
  return PPO_OK;
}

}  // namespace

// =============================================================================
extern "C" {

const char* ppo_status_string(ppo_status s) {
  switch (s) {
    case PPO_OK: return "ok";
    case PPO_ERR_INVALID: return "invalid argument";
    case PPO_ERR_ALIGN: return "device pointer not 16-byte aligned";
    case PPO_ERR_CUDA: return "CUDA error";
    case PPO_ERR_UNSUPPORTED: return "unsupported shape or device";
    case PPO_ERR_TIMEOUT: return "device-side wait timed out";
    case PPO_ERR_NOMEM: return "device allocation failed";
  }
  return "unknown status";
}

ppo_status ppo_param_count(const ppo_config* cfg, int64_t* n) {
  if (!n) return PPO_ERR_INVALID;
  NetShape s;
  TRY(shape_from(cfg, &s));
  *n = s.P;
  return PPO_OK;
}

ppo_status ppo_create(const ppo_config* cfg, const float* h_init_params, ppo_ctx** out) {
  if (!out) return PPO_ERR_INVALID;
  *out = nullptr;
  NetShape s;
  TRY(shape_from(cfg, &s));
  if (cfg->max_batch < 1 || cfg->max_batch >= (1ll << 31) || cfg->max_minibatch < 1 ||
      cfg->max_minibatch > cfg->max_batch || cfg->max_epochs < 1)
    return PPO_ERR_INVALID;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return PPO_ERR_CUDA;
  int major = 0, minor = 0;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
    return PPO_ERR_CUDA;
  if (major != 10 || minor != 3) return PPO_ERR_UNSUPPORTED;  // built for sm_103a only
  if (cfg->precision == 1 && (s.H1 % 64 != 0 || s.H2 % 64 != 0 || s.H1 > 512 || s.H2 > 512))
    return PPO_ERR_UNSUPPORTED;
  if (cfg->precision == 1 && (s.H2 % 128 != 0 || s.H1 % 128 != 0))
    return PPO_ERR_UNSUPPORTED;  // the weight-gradient tiles are 128 rows of features

  ppo_ctx* c = new (std::nothrow) ppo_ctx();
  if (!c) return PPO_ERR_NOMEM;
  c->cfg = *cfg;
  c->s = s;
  c->bf16 = cfg->precision == 1;
  // the persistent and fused-MLP kernels have no step between the forward
  // pass and the loss, where per-minibatch advantages are computed
  c->use_mk = c->bf16 && cfg->persistent_minibatch != 0 && cfg->adv_mode == 0 &&
              cfg->optimizer == 0;   // the persistent kernel runs Adam itself
  c->use_fmlp = c->bf16 && !c->use_mk && cfg->fused_mlp != 0 && cfg->adv_mode == 0 &&
                fmlp_supported(s);
  c->use_hl2 = c->bf16 && !c->use_mk && cfg->fused_loss >= 0 && hl2_supported(s);
  cudaDeviceGetAttribute(&c->num_sms, cudaDevAttrMultiProcessorCount, dev);
  if (c->num_sms < 1) c->num_sms = 1;
  c->mbmax = cfg->max_minibatch;
  c->bmax = cfg->max_batch;
  c->emax = cfg->max_epochs;

  auto fail = [&](ppo_status st) {
    delete c;
    return st;
  };
  ppo_status r;
#define A(ptr, n)                                   \
  if ((r = c->alloc_n(&(ptr), (n))) != PPO_OK) return fail(r);

  const int64_t P = s.P;
  A(c->params, P);
  A(c->grad, P);
  A(c->m, P);
  A(c->v, P);
  A(c->step, 1);
  A(c->beta_pow, 4);
  A(c->gbar, 2);
  A(c->phase_ns, kMkPhases);
  A(c->done_ctr, 1);
  A(c->err, 1);
  // squared-norm partials: the weight-gradient kernel's (<= SMs), then the reduce's
  A(c->sq, std::max(4096, reduce_blocks(s)) + c->num_sms);
  A(c->wctr, 2 * kWgradMaxTiles);
  A(c->rbar, 1);
  A(c->fbar, 1);
  A(c->fpart, 3 * (int64_t)kFreshMaxGrid);
  A(c->vfresh, cfg->max_minibatch);
  A(c->rfresh, cfg->max_minibatch);
  if (cfg->optimizer == 1) {
    A(c->mom, P);
    A(c->mpart, 3 * kMuonPrepBlocks);
    A(c->minv, 4);
    const int64_t rows[3] = {s.H1, s.H2, s.C}, cols[3] = {s.D, s.H1, s.H2};
    for (int m = 0; m < 3; ++m) {
      const int64_t nr = std::min(rows[m], cols[m]), nk = std::max(rows[m], cols[m]);
      A(c->ns_ws[m][0], nr * nk);
      A(c->ns_ws[m][1], nr * nk);
      A(c->ns_ws[m][2], nr * nr);
      A(c->ns_ws[m][3], nr * nr);
      if (c->bf16) {   // tensor-core iteration: bf16 X, X2, XT, A, B padded to 128
        MuonTcMat& q = c->mtc.m[m];
        q.r = (int)nr;
        q.k = (int)nk;
        q.rp = (int)round_up(nr, 128);
        q.kp = (int)round_up(nk, 128);
        A(q.X, (int64_t)q.rp * q.kp);
        A(q.X2, (int64_t)q.rp * q.kp);
        A(q.XT, (int64_t)q.kp * q.rp);
        A(q.A, (int64_t)q.rp * q.rp);
        A(q.B, (int64_t)q.rp * q.rp);
      }
    }
    if (c->bf16) {
      c->has_mtc = true;
      for (int i = 0; i < 3; ++i) {
        if (cudaStreamCreateWithFlags(&c->mtc.side[i], cudaStreamNonBlocking) != cudaSuccess ||
            cudaEventCreateWithFlags(&c->mtc.join[i], cudaEventDisableTiming) != cudaSuccess)
          return fail(PPO_ERR_CUDA);
      }
      if (cudaEventCreateWithFlags(&c->mtc.fork, cudaEventDisableTiming) != cudaSuccess)
        return fail(PPO_ERR_CUDA);
      c->mtc.err = c->err;
      c->mtc.num_sms = c->num_sms;
    }
  }
  if (c->bf16) {
    c->sh.ld3t = 64;
    A(c->sh.W1s, (int64_t)s.H1 * s.Dp);
    A(c->sh.W2s, (int64_t)s.H2 * s.H1);
    A(c->sh.W2Ts, (int64_t)s.H1 * s.H2);
    A(c->sh.W3s, (int64_t)s.CP * s.H2);
    A(c->sh.W3Ts, (int64_t)s.H2 * 64);
  }
  const int64_t mbm = c->mbmax;
  const int esz = c->bf16 ? 2 : 4;
  c->lddz = c->bf16 ? 64 : s.CP;
  {
    void* t;
    if ((r = c->alloc(&t, (size_t)mbm * (c->bf16 ? s.Dp : s.D) * esz)) != PPO_OK) return fail(r);
    c->X = t;
    if ((r = c->alloc(&t, (size_t)mbm * s.H1 * esz)) != PPO_OK) return fail(r);
    c->H1 = t;
    if ((r = c->alloc(&t, (size_t)mbm * s.H2 * esz)) != PPO_OK) return fail(r);
    c->H2 = t;
    if ((r = c->alloc(&t, (size_t)mbm * c->lddz * esz)) != PPO_OK) return fail(r);
    c->dZ = t;
    if ((r = c->alloc(&t, (size_t)mbm * s.H2 * esz)) != PPO_OK) return fail(r);
    c->dP2 = t;
    if ((r = c->alloc(&t, (size_t)mbm * s.H1 * esz)) != PPO_OK) return fail(r);
    c->dP1 = t;
  }
  {
    void* t;
    if ((r = c->alloc(&t, (size_t)c->bmax * (c->bf16 ? s.Dp : s.D) * esz)) != PPO_OK)
      return fail(r);
    c->X_ep = t;
  }
  A(c->act_ep, c->bmax * (s.NH > 0 ? s.NH : 1));
  A(c->actc_ep, c->bmax * (s.G > 0 ? s.G : 1));
  A(c->logp_ep, c->bmax);
  A(c->adv_ep, c->bmax);
  A(c->ret_ep, c->bmax);
  A(c->act_mb, mbm * (s.NH > 0 ? s.NH : 1));
  A(c->actc_mb, mbm * (s.G > 0 ? s.G : 1));
  A(c->logp_mb, mbm);
  A(c->adv_mb, mbm);
  A(c->ret_mb, mbm);
  const int ldW1 = c->bf16 ? s.Dp : s.D;
  // split-K partials: a split covers at least 16 rows (fp32) / 4 k-tiles (bf16)
  const int64_t max_split = std::min<int64_t>(kMaxSplit, c->bf16 ? (mbm + 255) / 256 + 1
                                                                   : (mbm + 15) / 16 + 1);
  A(c->pW1, max_split * s.H1 * ldW1);
  A(c->pW2, max_split * s.H2 * s.H1);
  A(c->pW3, max_split * s.H2 * (c->bf16 ? 64 : s.CP));
  const int64_t part_rows = std::max<int64_t>(c->num_sms, (mbm + 63) / 64) + 1;
  A(c->cs1, part_rows * s.H1);
  A(c->cs2, part_rows * s.H2);
  A(c->cs3, part_rows * 32);
  A(c->lossp, part_rows * kLossPartials);
  // update workspace
  const int64_t B = c->bmax;
  if (c->bf16) A(c->obs_packed, B * s.Dp);
  A(c->adv, B);
  A(c->ret, B);
  A(c->advstats, 4);
  A(c->gae_part, 3 * (int64_t)gae_num_blocks((int)B));
  A(c->perm, B * c->emax);
  {
    void* t;
    if ((r = c->alloc(&t, perm_workspace_bytes(B, c->emax))) != PPO_OK) return fail(r);
    c->perm_work = t;
  }
#undef A
  if (c->bf16 && tc_prepare() != cudaSuccess) return fail(PPO_ERR_CUDA);
  if (c->use_fmlp && fmlp_prepare() != cudaSuccess) return fail(PPO_ERR_CUDA);
  if (c->use_hl2 && hl2_prepare() != cudaSuccess) return fail(PPO_ERR_CUDA);
  if (reduce_adam_prepare() != cudaSuccess) return fail(PPO_ERR_CUDA);
  if (fresh_prepare() != cudaSuccess) return fail(PPO_ERR_CUDA);
  if (policy_act_prepare() != cudaSuccess) return fail(PPO_ERR_CUDA);
  if (c->use_mk && mk_prepare() != cudaSuccess) return fail(PPO_ERR_CUDA);
  if (h_init_params) {
    if (cudaMemcpy(c->params, h_init_params, sizeof(float) * P, cudaMemcpyHostToDevice) !=
        cudaSuccess)
      return fail(PPO_ERR_CUDA);
  }
  {
    // beta^0 and the first step's bias corrections 1 / (1 - beta^1)
    const double one[4] = {1.0, 1.0, 1.0 / (1.0 - cfg->beta1), 1.0 / (1.0 - cfg->beta2)};
    if (cudaMemcpy(c->beta_pow, one, sizeof one, cudaMemcpyHostToDevice) != cudaSuccess)
      return fail(PPO_ERR_CUDA);
  }
  if (launch_shadows(c->params, s, c->sh, 0) != cudaSuccess) return fail(PPO_ERR_CUDA);
  if (cudaDeviceSynchronize() != cudaSuccess) return fail(PPO_ERR_CUDA);
  *out = c;
  return PPO_OK;
}

ppo_status ppo_destroy(ppo_ctx* ctx) {
  if (!ctx) return PPO_ERR_INVALID;
  cudaDeviceSynchronize();
  delete ctx;
  return PPO_OK;
}

ppo_status ppo_buffers(ppo_ctx* c, float** d_params, float** d_grad, float** d_m, float** d_v) {
  if (!c) return PPO_ERR_INVALID;
  if (d_params) *d_params = c->params;
  if (d_grad) *d_grad = c->grad;
  if (d_m) *d_m = c->m;
  if (d_v) *d_v = c->v;
  return PPO_OK;
}

ppo_status ppo_params_changed(ppo_ctx* c, cudaStream_t st) {
  if (!c) return PPO_ERR_INVALID;
  PPO_CUDA(launch_shadows(c->params, c->s, c->sh, st));
  return PPO_OK;
}

ppo_status ppo_get_step(ppo_ctx* c, int64_t* step) {
  if (!c || !step) return PPO_ERR_INVALID;
  PPO_CUDA(cudaDeviceSynchronize());
  PPO_CUDA(cudaMemcpy(step, c->step, sizeof(int64_t), cudaMemcpyDeviceToHost));
  return PPO_OK;
}

ppo_status ppo_gae_workspace_bytes(int64_t T, int64_t N, size_t* bytes) {
  if (!bytes || T < 1 || N < 1 || T * N >= (1ll << 31)) return PPO_ERR_INVALID;
  if (T > kGaeMaxT) return PPO_ERR_UNSUPPORTED;
  *bytes = (size_t)round_up(24 * (int64_t)gae_num_blocks((int)N), 256) + 256;
  return PPO_OK;
}

ppo_status ppo_gae(const float* rew, const float* val, const float* done, const float* boot,
                   int64_t T, int64_t N, float gamma, float lambda, float* adv, float* ret,
                   float* adv_norm, float* stats, void* work, size_t work_bytes,
                   cudaStream_t st) {
  if (!rew || !val || !done || !boot || !adv || !ret) return PPO_ERR_INVALID;
  if (T < 1 || N < 1 || T * N >= (1ll << 31)) return PPO_ERR_INVALID;
  if (T > kGaeMaxT) return PPO_ERR_UNSUPPORTED;
  const void* ps[] = {rew, val, done, boot, adv, ret, adv_norm, stats, work};
  for (const void* p : ps)
    if (p && !al16(p)) return PPO_ERR_ALIGN;
  const bool need_stats = adv_norm || stats;
  size_t need = 0;
  TRY(ppo_gae_workspace_bytes(T, N, &need));
  if (need_stats && (!work || work_bytes < need)) return PPO_ERR_INVALID;
  const int nb = gae_num_blocks((int)N);
  double* part = need_stats ? static_cast<double*>(work) : nullptr;
  PPO_CUDA(launch_gae(rew, val, done, boot, (int)T, (int)N, gamma, lambda, adv, ret, part, nb, st));
  if (need_stats) {
    float* sbuf = stats ? stats
                        : reinterpret_cast<float*>(static_cast<char*>(work) + round_up(24 * nb, 256));
    PPO_CUDA(launch_gae_finalize(part, nb, sbuf, st));
    if (adv_norm) PPO_CUDA(launch_normalize(adv, sbuf, adv_norm, T * N, st));
  }
  return PPO_OK;
}

ppo_status ppo_perm_workspace_bytes(int64_t B, size_t* bytes) {
  if (!bytes || B < 1 || B >= (1ll << 31)) return PPO_ERR_INVALID;
  *bytes = perm_workspace_bytes(B, 1);
  return PPO_OK;
}

ppo_status ppo_minibatch_perm(uint32_t seed, int64_t epoch, int64_t B, int32_t* perm, void* work,
                              size_t work_bytes, cudaStream_t st) {
  if (!perm || !work || B < 1 || B >= (1ll << 31) || epoch < 0) return PPO_ERR_INVALID;
  if (!al16(perm) || !al16(work)) return PPO_ERR_ALIGN;
  if (work_bytes < perm_workspace_bytes(B, 1)) return PPO_ERR_INVALID;
  PPO_CUDA(launch_perm(seed, epoch, 1, B, perm, work, st));
  return PPO_OK;
}

ppo_status ppo_minibatch_loss_grad(ppo_ctx* c, const float* obs, const int32_t* act,
                                   const float* actc, const float* logp_old, const float* adv,
                                   const float* ret, const int32_t* idx, int64_t B, int64_t mb,
                                   const float* adv_stats, float* stats6, cudaStream_t st) {
  TRY(check_minibatch_args(c, obs, act, actc, logp_old, adv, ret, idx, B, mb));
  if ((adv_stats && !al16(adv_stats)) || (stats6 && !al16(stats6))) return PPO_ERR_ALIGN;
  if (c->use_mk) {
    PPO_CUDA(cudaMemsetAsync(c->gbar, 0, 2 * sizeof(unsigned), st));
    return enqueue_minibatch_mk(c, obs, nullptr, act, actc, logp_old, adv, ret, idx, B, mb,
                                adv_stats, stats6, 0, 0.f, st);
  }
  return enqueue_minibatch(c, obs, nullptr, act, actc, logp_old, adv, ret, idx, B, mb, adv_stats,
                           stats6, st);
}

ppo_status ppo_minibatch_loss_grad_fresh(ppo_ctx* c, const float* obs, const int32_t* act,
                                         const float* actc, const float* logp_old,
                                         const float* rew, const float* done, const float* boot,
                                         int64_t T, int64_t N, const int32_t* envs, int64_t ns,
                                         int32_t adv_mode, float gamma, float lambda,
                                         float* stats6, float* adv_out, float* ret_out,
                                         cudaStream_t st) {
  if (!c || !obs || !logp_old || !rew || !done || !boot || !envs) return PPO_ERR_INVALID;
  if (c->s.NH > 0 && !act) return PPO_ERR_INVALID;
  if (c->s.G > 0 && !actc) return PPO_ERR_INVALID;
  if (adv_mode != 1 && adv_mode != 2) return PPO_ERR_INVALID;
  if (c->s.H2 > 512) return PPO_ERR_UNSUPPORTED;
  if (T < 1 || N < 1 || ns < 1 || T * N >= (1ll << 31) || T * ns > c->mbmax)
    return PPO_ERR_INVALID;
  const void* ps[] = {obs, act, actc, logp_old, rew, done, boot, envs, stats6, adv_out, ret_out};
  for (const void* p : ps)
    if (p && !al16(p)) return PPO_ERR_ALIGN;
  const int64_t mb = T * ns;
  const MbRows mr{c->X, c->act_mb, c->actc_mb, c->logp_mb, c->adv_mb, c->ret_mb};
  PPO_CUDA(cudaMemsetAsync(c->fbar, 0, sizeof(unsigned), st));
  PPO_CUDA(enqueue_gather_seg(c, obs, nullptr, act, actc, logp_old, envs, (int)T, (int)ns, N, mb,
                              mr, st));
  c->tr.mark(ST_GATHER, st);
  const FreshSpec fs{rew, done, boot, envs, (int)T, (int)ns, N, gamma, lambda, adv_mode == 2};
  TRY(enqueue_minibatch(c, obs, nullptr, act, actc, logp_old, nullptr, nullptr, nullptr, T * N,
                        mb, nullptr, stats6, st, nullptr, &mr, nullptr, &fs));
  if (adv_out)
    PPO_CUDA(cudaMemcpyAsync(adv_out, c->adv_mb, sizeof(float) * mb, cudaMemcpyDeviceToDevice, st));
  if (ret_out)
    PPO_CUDA(cudaMemcpyAsync(ret_out, c->ret_mb, sizeof(float) * mb, cudaMemcpyDeviceToDevice, st));
  return PPO_OK;
}

ppo_status ppo_policy_act(ppo_ctx* c, const float* obs, int64_t N, uint32_t seed, uint64_t draw0,
                          int32_t* act, float* actc, float* logp, float* value, cudaStream_t st) {
  if (!c || !obs) return PPO_ERR_INVALID;
  const NetShape& s = c->s;
  if ((s.NH > 0 && !act) || (s.G > 0 && !actc)) return PPO_ERR_INVALID;
  if (N < 1 || N > c->mbmax) return PPO_ERR_INVALID;
  if (s.H2 > 512) return PPO_ERR_UNSUPPORTED;
  const void* ps[] = {obs, act, actc, logp, value};
  for (const void* p : ps)
    if (p && !al16(p)) return PPO_ERR_ALIGN;
  const float* P = c->params;
  const int M = (int)N;
  if (c->bf16) {
    auto* X = static_cast<__nv_bfloat16*>(c->X);
    auto* H1 = static_cast<__nv_bfloat16*>(c->H1);
    auto* H2 = static_cast<__nv_bfloat16*>(c->H2);
    PPO_CUDA(launch_pack_obs(obs, N, s.D, s.Dp, X, st));
    c->tr.mark(ST_PACK, st);
    GemmOperands g1{X, s.Dp, c->sh.W1s, s.Dp, M, s.H1, s.Dp};
    PPO_CUDA(tc_gemm_bias_act(g1, P + s.ob1, s.act, H1, s.H1, c->err, kTimeoutNs, c->num_sms, st));
    c->tr.mark(ST_FWD1, st);
    GemmOperands g2{H1, s.H1, c->sh.W2s, s.H1, M, s.H2, s.H1};
    PPO_CUDA(tc_gemm_bias_act(g2, P + s.ob2, s.act, H2, s.H2, c->err, kTimeoutNs, c->num_sms, st));
    c->tr.mark(ST_FWD2, st);
  } else {
    auto* H1 = static_cast<float*>(c->H1);
    auto* H2 = static_cast<float*>(c->H2);
    SimtOperands g1{obs, s.D, 1, P + s.oW1, s.D, 1, M, s.H1, s.D};
    PPO_CUDA(simt_bias_act(g1, P + s.ob1, s.act, H1, s.H1, st));
    c->tr.mark(ST_FWD1, st);
    SimtOperands g2{H1, s.H1, 1, P + s.oW2, s.H1, 1, M, s.H2, s.H1};
    PPO_CUDA(simt_bias_act(g2, P + s.ob2, s.act, H2, s.H2, st));
    c->tr.mark(ST_FWD2, st);
  }
  PolicyActArgs a{};
  a.s = s;
  a.h = c->H2;
  a.h_bf16 = c->bf16;
  a.W3 = c->bf16 ? static_cast<const void*>(c->sh.W3s) : static_cast<const void*>(P + s.oW3);
  a.b3 = P + s.ob3;
  a.logstd = P + s.ologstd;
  a.n = N;
  a.seed = seed;
  a.draw0 = draw0;
  a.act = act;
  a.actc = actc;
  a.logp = logp;
  a.value = value;
  PPO_CUDA(launch_policy_act(a, st));
  c->tr.mark(ST_POLICY_ACT, st);
  return PPO_OK;
}

static ppo_status rnn_check(const ppo_rnn_config* r, NetShape* s, int64_t* P) {
  if (!r) return PPO_ERR_INVALID;
  if (r->obs_dim < 1 || r->hidden < 1 || r->layers < 1) return PPO_ERR_INVALID;
  if (r->n_heads < 0 || r->n_heads > PPO_MAX_HEADS || r->n_gauss < 0 || r->n_gauss > 4)
    return PPO_ERR_INVALID;
  if (r->hidden > 256 || r->layers > 8) return PPO_ERR_UNSUPPORTED;
  if (r->precision != 0 && r->precision != 1) return PPO_ERR_INVALID;
  if (r->precision == 1 && !rnn_tc_supported(r->obs_dim, r->hidden)) return PPO_ERR_UNSUPPORTED;
  std::memset(s, 0, sizeof(*s));
  int C = 0;
  for (int h = 0; h < r->n_heads; ++h) {
    if (r->head_n[h] < 1) return PPO_ERR_INVALID;
    s->head_n[h] = r->head_n[h];
    C += r->head_n[h];
  }
  C += r->n_gauss + 1;
  if (C > 32) return PPO_ERR_UNSUPPORTED;
  s->NH = r->n_heads;
  s->G = r->n_gauss;
  s->C = C;
  s->CP = 32;
  s->D = s->Dp = r->obs_dim;
  s->H1 = s->H2 = r->hidden;
  const int64_t D = r->obs_dim, H = r->hidden, L = r->layers;
  *P = H * D + L * (2 * H * H + 2 * H) + (int64_t)C * H + r->n_gauss;
  return PPO_OK;
}

ppo_status ppo_rnn_param_count(const ppo_rnn_config* cfg, int64_t* n) {
  if (!n) return PPO_ERR_INVALID;
  NetShape s;
  return rnn_check(cfg, &s, n);
}

ppo_status ppo_rnn_workspace_bytes(const ppo_rnn_config* cfg, int64_t T, int64_t ns,
                                   size_t* bytes) {
  NetShape s;
  int64_t P;
  TRY(rnn_check(cfg, &s, &P));
  if (!bytes || T < 1 || ns < 1) return PPO_ERR_INVALID;
  if (cfg->precision == 1) {
    int dev = 0, nsm = 1;
    PPO_CUDA(cudaGetDevice(&dev));
    PPO_CUDA(cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev));
    *bytes = rnn_tc_workspace_bytes(cfg->obs_dim, cfg->hidden, cfg->layers, T, ns, nsm);
    return PPO_OK;
  }
  *bytes = sizeof(float) * rnn_workspace_floats(cfg->obs_dim, cfg->hidden, cfg->layers, T * ns);
  return PPO_OK;
}

ppo_status ppo_rnn_loss_grad(const ppo_rnn_config* cfg, const float* params, int64_t T,
                             int64_t N, const int32_t* envs, int64_t ns, const float* obs,
                             const int32_t* act, const float* actc, const float* logp_old,
                             const float* adv, const float* ret, const float* adv_stats,
                             const float* done, const float* h0, float* grad, float* stats6,
                             void* work, size_t work_bytes, cudaStream_t st) {
  NetShape s;
  int64_t P;
  TRY(rnn_check(cfg, &s, &P));
  if (!params || !envs || !obs || !logp_old || !adv || !ret || !done || !h0 || !grad || !work)
    return PPO_ERR_INVALID;
  if ((s.NH > 0 && !act) || (s.G > 0 && !actc)) return PPO_ERR_INVALID;
  if (T > kGaeMaxT) return PPO_ERR_UNSUPPORTED;
  if (T < 1 || N < 1 || ns < 1 || T * N >= (1ll << 31) || T * ns >= (1ll << 31))
    return PPO_ERR_INVALID;
  size_t need = 0;
  TRY(ppo_rnn_workspace_bytes(cfg, T, ns, &need));
  if (work_bytes < need) return PPO_ERR_INVALID;
  const void* ps[] = {params, envs, obs, act, actc, logp_old, adv, ret, adv_stats, done, h0,
                      grad, stats6, work};
  for (const void* p : ps)
    if (p && !al16(p)) return PPO_ERR_ALIGN;
  RnnLaunch a{};
  a.s = s;
  a.lc = LossCoef{cfg->clip, cfg->vf_coef, cfg->ent_coef};
  a.T = (int)T;
  a.ns = (int)ns;
  a.D = cfg->obs_dim;
  a.H = cfg->hidden;
  a.L = cfg->layers;
  a.N = N;
  a.params = params;
  a.envs = envs;
  a.obs = obs;
  a.act = act;
  a.actc = actc;
  a.logp_old = logp_old;
  a.adv = adv;
  a.ret = ret;
  a.adv_stats = adv_stats;
  a.done = done;
  a.h0 = h0;
  a.grad = grad;
  a.stats6 = stats6;
  a.work = static_cast<float*>(work);
  if (cfg->precision == 1) {
    int dev = 0, nsm = 1;
    PPO_CUDA(cudaGetDevice(&dev));
    PPO_CUDA(cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev));
    PPO_CUDA(tc_prepare());
    PPO_CUDA(launch_rnn_loss_grad_tc(a, nsm, st, nullptr));
    return PPO_OK;
  }
  PPO_CUDA(launch_rnn_loss_grad(a, st));
  return PPO_OK;
}

ppo_status ppo_segment_advantage_workspace_bytes(size_t* bytes) {
  if (!bytes) return PPO_ERR_INVALID;
  *bytes = 16 + sizeof(float) * 3 * (size_t)kFreshMaxGrid;
  return PPO_OK;
}

ppo_status ppo_segment_advantage(const float* rew, const float* done, const float* boot,
                                 int64_t T, int64_t N, const int32_t* envs, int64_t ns,
                                 const float* val, const float* ratio, float gamma, float lambda,
                                 float rho_clip, float c_clip, float* adv, float* ret,
                                 float* adv_norm, float* stats, void* work, size_t work_bytes,
                                 cudaStream_t st) {
  if (!rew || !done || !boot || !envs || !val || !adv || !ret || !work) return PPO_ERR_INVALID;
  if (T > kGaeMaxT) return PPO_ERR_UNSUPPORTED;
  if (T < 1 || N < 1 || ns < 1 || T * N >= (1ll << 31) || T * ns >= (1ll << 31))
    return PPO_ERR_INVALID;
  size_t need = 0;
  ppo_segment_advantage_workspace_bytes(&need);
  if (work_bytes < need) return PPO_ERR_INVALID;
  const void* ps[] = {rew, done, boot, envs, val, ratio, adv, ret, adv_norm, stats, work};
  for (const void* p : ps)
    if (p && !al16(p)) return PPO_ERR_ALIGN;
  PPO_CUDA(fresh_prepare());
  int dev = 0, nsm = 1;
  PPO_CUDA(cudaGetDevice(&dev));
  PPO_CUDA(cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev));
  unsigned* bar = static_cast<unsigned*>(work);
  int* err = reinterpret_cast<int*>(static_cast<uint8_t*>(work) + 4);
  PPO_CUDA(cudaMemsetAsync(work, 0, 16, st));
  FreshAdvArgs f{};
  f.head = 0;
  f.rew = rew;
  f.done = done;
  f.boot = boot;
  f.envs = envs;
  f.T = (int)T;
  f.ns = (int)ns;
  f.N = N;
  f.val = const_cast<float*>(val);
  f.ratio = const_cast<float*>(ratio);
  f.gamma = gamma;
  f.lambda = lambda;
  f.rho_clip = rho_clip;
  f.c_clip = c_clip;
  f.adv = adv;
  f.ret = ret;
  f.adv_norm = adv_norm;
  f.stats = stats;
  f.part = reinterpret_cast<float*>(static_cast<uint8_t*>(work) + 16);
  f.bar = bar;
  f.err = err;
  f.timeout_ns = kTimeoutNs;
  PPO_CUDA(launch_fresh_adv(f, nsm, st));
  return PPO_OK;
}

ppo_status ppo_muon_step(ppo_ctx* c, float lr, float* grad_norm, cudaStream_t st) {
  if (!c) return PPO_ERR_INVALID;
  if (c->cfg.optimizer != 1) return PPO_ERR_INVALID;
  if (grad_norm && !al16(grad_norm)) return PPO_ERR_ALIGN;
  return enqueue_muon(c, lr, grad_norm, st, 0);
}

ppo_status ppo_adam_step(ppo_ctx* c, float lr, float* grad_norm, cudaStream_t st) {
  if (!c) return PPO_ERR_INVALID;
  if (grad_norm && !al16(grad_norm)) return PPO_ERR_ALIGN;
  return enqueue_adam(c, lr, grad_norm, st);
}

static ppo_status check_update_args(ppo_ctx* c, const float* obs, const int32_t* act,
                                    const float* actc, const float* logp_old, const float* val,
                                    const float* rew, const float* done, const float* boot,
                                    int64_t T, int64_t N, int32_t epochs, int32_t minibatches,
                                    const float* stats) {
  if (!c || !val || !rew || !done || !boot) return PPO_ERR_INVALID;
  if (T < 1 || N < 1 || epochs < 1 || minibatches < 1) return PPO_ERR_INVALID;
  if (T > kGaeMaxT) return PPO_ERR_UNSUPPORTED;
  const int64_t B = T * N;
  if (B > c->bmax || epochs > c->emax || B % minibatches != 0) return PPO_ERR_INVALID;
  if (c->cfg.adv_mode != 0 && N % minibatches != 0) return PPO_ERR_INVALID;
  if (c->cfg.adv_mode != 0 && c->s.H2 > 512) return PPO_ERR_UNSUPPORTED;
  if (c->world > 1 && (c->cfg.adv_mode != 0 || c->use_mk)) return PPO_ERR_UNSUPPORTED;
  const int64_t mb = B / minibatches;
  if (mb > c->mbmax || !obs || !logp_old || (c->s.NH > 0 && !act) || (c->s.G > 0 && !actc))
    return PPO_ERR_INVALID;
  const void* ps[] = {obs, act, actc, logp_old, val, rew, done, boot, stats};
  for (const void* p : ps)
    if (p && !al16(p)) return PPO_ERR_ALIGN;
  return PPO_OK;
}

}  // extern "C"

namespace {
// ppo_update with an optional event that part 2 waits for (ppo_update_host)
ppo_status run_update(ppo_ctx* c, const float* obs, const int32_t* act, const float* actc,
                      const float* logp_old, const float* val, const float* rew,
                      const float* done, const float* boot, int64_t T, int64_t N,
                      int32_t epochs, int32_t minibatches, float gamma, float lambda, float lr,
                      uint32_t seed, float* stats, cudaStream_t st,
                      cudaEvent_t wait_before_part2) {
  TRY(check_update_args(c, obs, act, actc, logp_old, val, rew, done, boot, T, N, epochs,
                        minibatches, stats));
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  PPO_CUDA(cudaStreamIsCapturing(st, &cs));
  if (st == nullptr || cs != cudaStreamCaptureStatusNone || c->world > 1) {
    // legacy stream cannot be captured; inside a caller's capture, or with
    // the caller's collectives in the update, just enqueue
    TRY(enqueue_update(c, obs, act, actc, logp_old, val, rew, done, boot, T, N, epochs,
                       minibatches, gamma, lambda, lr, seed, stats, st, 1));
    if (wait_before_part2) PPO_CUDA(cudaStreamWaitEvent(st, wait_before_part2, 0));
    return enqueue_update(c, obs, act, actc, logp_old, val, rew, done, boot, T, N, epochs,
                          minibatches, gamma, lambda, lr, seed, stats, st, 2);
  }
  UpdateKey key{};
  const void* kp[9] = {obs, act, actc, logp_old, val, rew, done, boot, c};
  for (int i = 0; i < 9; ++i) key.p[i] = kp[i];
  key.T = T;
  key.N = N;
  key.epochs = epochs;
  key.minibatches = minibatches;
  key.gamma = gamma;
  key.lambda = lambda;
  key.lr = lr;
  key.seed = seed;
  key.stats = stats;
  key.stream = st;
  GraphEntry* g = nullptr;
  for (GraphEntry& e : c->gc)
    if (e.valid && e.key == key) g = &e;
  if (!g) {
    g = &c->gc[0];
    for (GraphEntry& e : c->gc)
      if (!e.valid || e.used < g->used) g = &e;
    g->reset();
    for (int part = 1; part <= 2; ++part) {
      PPO_CUDA(cudaStreamBeginCapture(st, cudaStreamCaptureModeThreadLocal));
      ppo_status r = enqueue_update(c, obs, act, actc, logp_old, val, rew, done, boot, T, N,
                                    epochs, minibatches, gamma, lambda, lr, seed, stats, st, part);
      cudaGraph_t graph = nullptr;
      cudaError_t e = cudaStreamEndCapture(st, &graph);
      if (r != PPO_OK) {
        if (graph) cudaGraphDestroy(graph);
        return r;
      }
      if (e != cudaSuccess) return PPO_ERR_CUDA;
      e = cudaGraphInstantiate(part == 1 ? &g->pre : &g->main, graph, 0);
      cudaGraphDestroy(graph);
      if (e != cudaSuccess) {
        g->reset();
        return PPO_ERR_CUDA;
      }
    }
    g->key = key;
    g->valid = true;
  }
  g->used = ++c->gclock;
  PPO_CUDA(cudaGraphLaunch(g->pre, st));
  if (wait_before_part2) PPO_CUDA(cudaStreamWaitEvent(st, wait_before_part2, 0));
  PPO_CUDA(cudaGraphLaunch(g->main, st));
  return PPO_OK;
}
}  // namespace

extern "C" {

ppo_status ppo_update(ppo_ctx* c, const float* obs, const int32_t* act, const float* actc,
                      const float* logp_old, const float* val, const float* rew,
                      const float* done, const float* boot, int64_t T, int64_t N,
                      int32_t epochs, int32_t minibatches, float gamma, float lambda, float lr,
                      uint32_t seed, float* stats, cudaStream_t st) {
  return run_update(c, obs, act, actc, logp_old, val, rew, done, boot, T, N, epochs,
                    minibatches, gamma, lambda, lr, seed, stats, st, nullptr);
}

const char* ppo_stage_name(int32_t stage) {
  static const char* names[ST_COUNT] = {
      "pack_obs", "gae_scan", "gae_finalize", "gae_normalize", "perm_hist", "perm_scan",
      "perm_scatter", "gather", "fwd1_gemm", "fwd2_gemm", "head_loss_gemm", "dact2_gemm",
      "dact1_gemm", "wgrad_gemm", "grad_reduce", "grad_sqnorm", "adam", "weight_shadows",
      "minibatch_persistent", "fused_mlp", "grad_reduce_adam", "head_loss_dact2",
      "fresh_advantages", "policy_act", "muon"};
  static const char* phases[kMkPhases] = {
      "phase:gather", "phase:fwd1", "phase:fwd2", "phase:head_loss", "phase:dact2",
      "phase:dact1", "phase:wgrad", "phase:grad_reduce", "phase:adam"};
  if (stage >= ST_COUNT && stage < ST_COUNT + kMkPhases) return phases[stage - ST_COUNT];
  if (stage < 0 || stage >= ST_COUNT) return "unknown";
  return names[stage];
}

static void prof_mark(void* user, int stage, cudaStream_t st) {
  ppo_ctx* c = static_cast<ppo_ctx*>(user);
  const size_t i = c->prof_stages.size();
  if (i + 1 < c->prof_events.size()) {
    // External: inside stream capture this becomes an event-record node
    cudaEventRecordWithFlags(c->prof_events[i + 1], st, cudaEventRecordExternal);
    c->prof_stages.push_back(stage);
  }
}

ppo_status ppo_update_profile(ppo_ctx* c, const float* obs, const int32_t* act,
                              const float* actc, const float* logp_old, const float* val,
                              const float* rew, const float* done, const float* boot, int64_t T,
                              int64_t N, int32_t epochs, int32_t minibatches, float gamma,
                              float lambda, float lr, uint32_t seed, float* stats,
                              float* h_stage_ms, int32_t* h_stage_launches, cudaStream_t st) {
  TRY(check_update_args(c, obs, act, actc, logp_old, val, rew, done, boot, T, N, epochs,
                        minibatches, stats));
  if (!h_stage_ms || !h_stage_launches || st == nullptr) return PPO_ERR_INVALID;
  if (c->world > 1) return PPO_ERR_UNSUPPORTED;
  // launches per minibatch: at most 7 per-stage kernels + 20 of a Muon step
  const size_t need = 8 + 3 * 4 + 40 * (size_t)epochs * minibatches;
  while (c->prof_events.size() < need) {
    cudaEvent_t e;
    PPO_CUDA(cudaEventCreate(&e));
    c->prof_events.push_back(e);
  }
  c->prof_stages.clear();
  PPO_CUDA(cudaMemsetAsync(c->phase_ns, 0, kMkPhases * sizeof(unsigned long long), st));
  c->profiling = true;
  PPO_CUDA(cudaStreamBeginCapture(st, cudaStreamCaptureModeThreadLocal));
  PPO_CUDA(cudaEventRecordWithFlags(c->prof_events[0], st, cudaEventRecordExternal));
  c->tr.fn = prof_mark;
  c->tr.user = c;
  ppo_status r = enqueue_update(c, obs, act, actc, logp_old, val, rew, done, boot, T, N, epochs,
                                minibatches, gamma, lambda, lr, seed, stats, st);
  c->tr = Trace{};
  c->profiling = false;
  cudaGraph_t graph = nullptr;
  cudaError_t e = cudaStreamEndCapture(st, &graph);
  if (r != PPO_OK) {
    if (graph) cudaGraphDestroy(graph);
    return r;
  }
  if (e != cudaSuccess) return PPO_ERR_CUDA;
  cudaGraphExec_t exec = nullptr;
  e = cudaGraphInstantiate(&exec, graph, 0);
  cudaGraphDestroy(graph);
  if (e != cudaSuccess) return PPO_ERR_CUDA;
  e = cudaGraphUpload(exec, st);
  if (e == cudaSuccess) e = cudaGraphLaunch(exec, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  cudaGraphExecDestroy(exec);
  if (e != cudaSuccess) return PPO_ERR_CUDA;
  for (int k = 0; k < ST_COUNT + kMkPhases; ++k) {
    h_stage_ms[k] = 0.f;
    h_stage_launches[k] = 0;
  }
  for (size_t i = 0; i < c->prof_stages.size(); ++i) {
    float ms = 0.f;
    PPO_CUDA(cudaEventElapsedTime(&ms, c->prof_events[i], c->prof_events[i + 1]));
    h_stage_ms[c->prof_stages[i]] += ms;
    h_stage_launches[c->prof_stages[i]] += 1;
  }
  if (c->use_mk) {   // phases of the persistent kernel, as seen by its first CTA
    unsigned long long ns[kMkPhases];
    PPO_CUDA(cudaMemcpy(ns, c->phase_ns, sizeof ns, cudaMemcpyDeviceToHost));
    const int nmb = h_stage_launches[ST_MINIBATCH];
    for (int k = 0; k < kMkPhases; ++k) {
      h_stage_ms[ST_COUNT + k] = (float)(ns[k] * 1e-6);
      h_stage_launches[ST_COUNT + k] = k == kMkPhases - 1 && c->cfg.max_grad_norm < -1.f ? 0 : nmb;
    }
  }
  return PPO_OK;
}

}  // extern "C"

namespace {
// waits (host) for every host update in flight
ppo_status host_wait_all(ppo_ctx* c) {
  if (c->hs_inflight > 0) {
    for (HostSlot& h : c->hs)
      if (h.used) PPO_CUDA(cudaEventSynchronize(h.freed));
    PPO_CUDA(cudaStreamSynchronize(c->cst));
    c->hs_inflight = 0;
  }
  return PPO_OK;
}

// ppo_update_host / ppo_update_host_async: stage the rollout in the next
// slot on the copy stream and enqueue the update and the stats copy-back on
// `st`; returns once everything is enqueued
ppo_status host_update(ppo_ctx* c, const float* h_obs, const int32_t* h_act,
                       const float* h_actc, const float* h_logp_old, const float* h_val,
                       const float* h_rew, const float* h_done, const float* h_boot, int64_t T,
                       int64_t N, int32_t epochs, int32_t minibatches, float gamma,
                       float lambda, float lr, uint32_t seed, float* h_stats, cudaStream_t st) {
  if (!c || !h_obs || !h_logp_old || !h_val || !h_rew || !h_done || !h_boot)
    return PPO_ERR_INVALID;
  if ((c->s.NH > 0 && !h_act) || (c->s.G > 0 && !h_actc)) return PPO_ERR_INVALID;
  if (T < 1 || N < 1 || epochs < 1 || minibatches < 1) return PPO_ERR_INVALID;
  if (T > kGaeMaxT) return PPO_ERR_UNSUPPORTED;
  const int64_t B = T * N;
  if (B > c->bmax) return PPO_ERR_INVALID;
  const NetShape& s = c->s;
  ppo_status r;
  if (!c->cst) PPO_CUDA(cudaStreamCreateWithFlags(&c->cst, cudaStreamNonBlocking));
  HostSlot& h = c->hs[c->hs_next];
  if (!h.obs) {
    const int64_t Bm = c->bmax;
    if ((r = c->alloc_n(&h.obs, Bm * s.D)) != PPO_OK) return r;
    if ((r = c->alloc_n(&h.act, Bm * (s.NH > 0 ? s.NH : 1))) != PPO_OK) return r;
    if ((r = c->alloc_n(&h.actc, Bm * (s.G > 0 ? s.G : 1))) != PPO_OK) return r;
    if ((r = c->alloc_n(&h.logp, Bm)) != PPO_OK) return r;
    if ((r = c->alloc_n(&h.val, Bm)) != PPO_OK) return r;
    if ((r = c->alloc_n(&h.rew, Bm)) != PPO_OK) return r;
    if ((r = c->alloc_n(&h.done, Bm)) != PPO_OK) return r;
    if ((r = c->alloc_n(&h.boot, Bm)) != PPO_OK) return r;
    for (cudaEvent_t* e : {&h.gae_in, &h.rest, &h.freed})
      PPO_CUDA(cudaEventCreateWithFlags(e, cudaEventDisableTiming));
  }
  const int64_t nstats = (int64_t)epochs * minibatches * 6;
  if (h_stats && nstats > c->st_stats_cap) {
    TRY(host_wait_all(c));   // earlier updates may still write the old buffer
    if ((r = c->alloc_n(&c->st_stats, nstats)) != PPO_OK) return r;
    c->st_stats_cap = nstats;
  }
  TRY(check_update_args(c, h.obs, h.act, h.actc, h.logp, h.val, h.rew, h.done, h.boot, T, N,
                        epochs, minibatches, h_stats ? c->st_stats : nullptr));
  // the context's buffers are ordered by one stream: a switch waits first
  if (c->hs_inflight > 0 && st != c->hs_stream) TRY(host_wait_all(c));
  // the call two before this one used this slot: wait until its update and
  // stats copy-back are done, so that on return its results are on the host
  // and its host buffers are no longer read
  if (h.used) PPO_CUDA(cudaEventSynchronize(h.freed));
  auto h2d = [&](void* d, const void* src, size_t bytes) {
    return cudaMemcpyAsync(d, src, bytes, cudaMemcpyHostToDevice, c->cst);
  };
  // GAE's inputs first: part 1 (GAE, moments, permutations) starts as soon
  // as they are in, while observations, actions and old log-probs follow
  PPO_CUDA(h2d(h.val, h_val, sizeof(float) * B));
  PPO_CUDA(h2d(h.rew, h_rew, sizeof(float) * B));
  PPO_CUDA(h2d(h.done, h_done, sizeof(float) * B));
  PPO_CUDA(h2d(h.boot, h_boot, sizeof(float) * N));
  PPO_CUDA(cudaEventRecord(h.gae_in, c->cst));
  PPO_CUDA(h2d(h.obs, h_obs, sizeof(float) * B * s.D));
  if (s.NH > 0) PPO_CUDA(h2d(h.act, h_act, sizeof(int32_t) * B * s.NH));
  if (s.G > 0) PPO_CUDA(h2d(h.actc, h_actc, sizeof(float) * B * s.G));
  PPO_CUDA(h2d(h.logp, h_logp_old, sizeof(float) * B));
  PPO_CUDA(cudaEventRecord(h.rest, c->cst));
  PPO_CUDA(cudaStreamWaitEvent(st, h.gae_in, 0));
  TRY(run_update(c, h.obs, h.act, h.actc, h.logp, h.val, h.rew, h.done, h.boot, T, N, epochs,
                 minibatches, gamma, lambda, lr, seed, h_stats ? c->st_stats : nullptr, st,
                 h.rest));
  if (h_stats)
    PPO_CUDA(cudaMemcpyAsync(h_stats, c->st_stats, sizeof(float) * nstats,
                             cudaMemcpyDeviceToHost, st));
  PPO_CUDA(cudaEventRecord(h.freed, st));
  h.used = true;
  c->hs_next ^= 1;
  c->hs_stream = st;
  ++c->hs_inflight;
  return PPO_OK;
}
}  // namespace

extern "C" {

ppo_status ppo_update_host(ppo_ctx* c, const float* h_obs, const int32_t* h_act,
                           const float* h_actc, const float* h_logp_old, const float* h_val,
                           const float* h_rew, const float* h_done, const float* h_boot,
                           int64_t T, int64_t N, int32_t epochs, int32_t minibatches,
                           float gamma, float lambda, float lr, uint32_t seed, float* h_stats,
                           cudaStream_t st) {
  TRY(host_update(c, h_obs, h_act, h_actc, h_logp_old, h_val, h_rew, h_done, h_boot, T, N,
                  epochs, minibatches, gamma, lambda, lr, seed, h_stats, st));
  return host_wait_all(c);
}

ppo_status ppo_update_host_async(ppo_ctx* c, const float* h_obs, const int32_t* h_act,
                                 const float* h_actc, const float* h_logp_old,
                                 const float* h_val, const float* h_rew, const float* h_done,
                                 const float* h_boot, int64_t T, int64_t N, int32_t epochs,
                                 int32_t minibatches, float gamma, float lambda, float lr,
                                 uint32_t seed, float* h_stats, cudaStream_t st) {
  return host_update(c, h_obs, h_act, h_actc, h_logp_old, h_val, h_rew, h_done, h_boot, T, N,
                     epochs, minibatches, gamma, lambda, lr, seed, h_stats, st);
}

ppo_status ppo_host_wait(ppo_ctx* c) {
  if (!c) return PPO_ERR_INVALID;
  return host_wait_all(c);
}

ppo_status ppo_set_collective(ppo_ctx* c, int32_t world, int32_t rank, ppo_collective_fn fn,
                              void* user) {
  if (!c || world < 1 || rank < 0 || rank >= world || (world > 1 && !fn))
    return PPO_ERR_INVALID;
  if (world > 1 && (c->cfg.adv_mode != 0 || c->use_mk)) return PPO_ERR_UNSUPPORTED;
  if (world > c->mom_cap) {
    ppo_status r = c->alloc_n(&c->mom_all, 3 * (int64_t)world);
    if (r != PPO_OK) return r;
    c->mom_cap = world;
  }
  c->world = world;
  c->rank = rank;
  c->coll = fn;
  c->coll_user = user;
  c->invalidate_graphs();
  return PPO_OK;
}

ppo_status ppo_set_step_trace(ppo_ctx* c, float* d_trace, int64_t max_steps) {
  if (!c || max_steps < 0 || (d_trace == nullptr) != (max_steps == 0)) return PPO_ERR_INVALID;
  if (d_trace && !al16(d_trace)) return PPO_ERR_ALIGN;
  c->trace = d_trace;
  c->trace_cap = max_steps;
  c->invalidate_graphs();   // the cached update graphs do not hold the copies
  return PPO_OK;
}

ppo_status ppo_set_wait_limit(ppo_ctx* c, uint64_t limit_ns) {
  if (!c) return PPO_ERR_INVALID;
  c->wait_ns = limit_ns == 0 ? kTimeoutNs : limit_ns;
  c->invalidate_graphs();   // the limit is a kernel argument inside the cached graphs
  return PPO_OK;
}

ppo_status ppo_sync_status(ppo_ctx* c, cudaStream_t st) {
  if (!c) return PPO_ERR_INVALID;
  PPO_CUDA(cudaStreamSynchronize(st));
  int e = 0;
  PPO_CUDA(cudaMemcpy(&e, c->err, sizeof(int), cudaMemcpyDeviceToHost));
  if (e != 0) {
    PPO_CUDA(cudaMemset(c->err, 0, sizeof(int)));
    return PPO_ERR_TIMEOUT;
  }
  return PPO_OK;
}

}  // extern "C"

// =============================================================================
// Recurrent-policy update ("Teaching Mario to speedrun", sec. 6 "The whole
// algorithm" with sec. 8's MinGRU policy): GAE over the stored values, the
// advantage statistics over all T*N entries, then per epoch the mulberry32
// permutation of the N environments and per minibatch the BPTT loss and
// gradient of its N/minibatches whole segments, clip and Adam.
struct ppo_rnn_ctx {
  ppo_rnn_config cfg;
  NetShape s;
  int64_t P = 0, max_T = 0, max_N = 0;
  int max_epochs = 0, num_sms = 1;
  std::vector<void*> allocs;
  float *params = nullptr, *grad = nullptr, *m = nullptr, *v = nullptr;
  int64_t* step = nullptr;
  double* beta_pow = nullptr;
  unsigned* done_ctr = nullptr;
  double* sq = nullptr;
  float *adv = nullptr, *ret = nullptr, *advstats = nullptr;
  double* gae_part = nullptr;
  int32_t* perm = nullptr;
  void* perm_work = nullptr;
  void* work = nullptr;
  size_t work_bytes = 0;
  int* err = nullptr;   // error word of the bounded device waits (tensor-core path)

  ppo_status alloc(void** p, size_t bytes) {
    void* q = nullptr;
    if (bytes == 0) bytes = 16;
    if (cudaMalloc(&q, bytes) != cudaSuccess) {
      cudaGetLastError();
      return PPO_ERR_NOMEM;
    }
    // zeroed on the legacy stream, which the library's non-blocking streams
    // do not wait for: finish it before any of them writes the buffer
    if (cudaMemset(q, 0, bytes) != cudaSuccess ||
        cudaStreamSynchronize(cudaStreamLegacy) != cudaSuccess) {
      cudaFree(q);
      return PPO_ERR_CUDA;
    }
    allocs.push_back(q);
    *p = q;
    return PPO_OK;
  }
  template <class T>
  ppo_status alloc_n(T** p, int64_t n) {
    return alloc(reinterpret_cast<void**>(p), (size_t)n * sizeof(T));
  }
  ~ppo_rnn_ctx() {
    for (void* p : allocs) cudaFree(p);
  }
};

extern "C" {

ppo_status ppo_rnn_create(const ppo_rnn_config* cfg, const float* h_init_params, int64_t max_T,
                          int64_t max_N, int32_t max_epochs, ppo_rnn_ctx** out) {
  if (!out) return PPO_ERR_INVALID;
  *out = nullptr;
  NetShape s;
  int64_t P;
  TRY(rnn_check(cfg, &s, &P));
  if (max_T < 1 || max_N < 1 || max_epochs < 1 || max_T * max_N >= (1ll << 31))
    return PPO_ERR_INVALID;
  if (max_T > kGaeMaxT) return PPO_ERR_UNSUPPORTED;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return PPO_ERR_CUDA;
  int major = 0, minor = 0;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
    return PPO_ERR_CUDA;
  if (major != 10 || minor != 3) return PPO_ERR_UNSUPPORTED;
  ppo_rnn_ctx* c = new (std::nothrow) ppo_rnn_ctx();
  if (!c) return PPO_ERR_NOMEM;
  c->cfg = *cfg;
  c->s = s;
  c->P = P;
  c->max_T = max_T;
  c->max_N = max_N;
  c->max_epochs = max_epochs;
  cudaDeviceGetAttribute(&c->num_sms, cudaDevAttrMultiProcessorCount, dev);
  if (c->num_sms < 1) c->num_sms = 1;
  auto fail = [&](ppo_status st) {
    delete c;
    return st;
  };
  ppo_status r;
#define A(ptr, n) \
  if ((r = c->alloc_n(&(ptr), (n))) != PPO_OK) return fail(r);
  A(c->params, P);
  A(c->grad, P);
  A(c->m, P);
  A(c->v, P);
  A(c->step, 1);
  A(c->beta_pow, 4);
  A(c->done_ctr, 1);
  A(c->sq, 4096);
  A(c->err, 1);
  const int64_t B = max_T * max_N;
  A(c->adv, B);
  A(c->ret, B);
  A(c->advstats, 4);
  A(c->gae_part, 3 * (int64_t)gae_num_blocks((int)max_N));
  A(c->perm, max_N * max_epochs);
#undef A
  if ((r = c->alloc(&c->perm_work, perm_workspace_bytes(max_N, max_epochs))) != PPO_OK)
    return fail(r);
  // the loss workspace for the largest minibatch (all N environments)
  if ((r = ppo_rnn_workspace_bytes(cfg, max_T, max_N, &c->work_bytes)) != PPO_OK) return fail(r);
  if ((r = c->alloc(&c->work, c->work_bytes)) != PPO_OK) return fail(r);
  if (cfg->precision == 1 && tc_prepare() != cudaSuccess) return fail(PPO_ERR_CUDA);
  if (h_init_params &&
      cudaMemcpy(c->params, h_init_params, sizeof(float) * P, cudaMemcpyHostToDevice) !=
          cudaSuccess)
    return fail(PPO_ERR_CUDA);
  const double one[4] = {1.0, 1.0, 1.0 / (1.0 - cfg->beta1), 1.0 / (1.0 - cfg->beta2)};
  if (cudaMemcpy(c->beta_pow, one, sizeof one, cudaMemcpyHostToDevice) != cudaSuccess)
    return fail(PPO_ERR_CUDA);
  if (cudaDeviceSynchronize() != cudaSuccess) return fail(PPO_ERR_CUDA);
  *out = c;
  return PPO_OK;
}

ppo_status ppo_rnn_destroy(ppo_rnn_ctx* c) {
  if (!c) return PPO_ERR_INVALID;
  cudaDeviceSynchronize();
  delete c;
  return PPO_OK;
}

ppo_status ppo_rnn_buffers(ppo_rnn_ctx* c, float** d_params, float** d_grad, float** d_m,
                           float** d_v) {
  if (!c) return PPO_ERR_INVALID;
  if (d_params) *d_params = c->params;
  if (d_grad) *d_grad = c->grad;
  if (d_m) *d_m = c->m;
  if (d_v) *d_v = c->v;
  return PPO_OK;
}

ppo_status ppo_rnn_update(ppo_rnn_ctx* c, const float* obs, const int32_t* act, const float* actc,
                          const float* logp_old, const float* val, const float* rew,
                          const float* done, const float* boot, const float* h0, int64_t T,
                          int64_t N, int32_t epochs, int32_t minibatches, float gamma,
                          float lambda, float lr, uint32_t seed, float* stats, cudaStream_t st) {
  if (!c || !obs || !logp_old || !val || !rew || !done || !boot || !h0) return PPO_ERR_INVALID;
  if ((c->s.NH > 0 && !act) || (c->s.G > 0 && !actc)) return PPO_ERR_INVALID;
  if (T < 1 || N < 1 || epochs < 1 || minibatches < 1) return PPO_ERR_INVALID;
  if (T > c->max_T || N > c->max_N || epochs > c->max_epochs || N % minibatches != 0)
    return PPO_ERR_INVALID;
  const void* ps[] = {obs, act, actc, logp_old, val, rew, done, boot, h0, stats};
  for (const void* p : ps)
    if (p && !al16(p)) return PPO_ERR_ALIGN;
  const int64_t ns = N / minibatches;
  // judge: GAE, statistics of all T*N advantages; the environment permutations
  PPO_CUDA(cudaMemsetAsync(c->done_ctr, 0, sizeof(unsigned), st));
  const int nb = gae_num_blocks((int)N);
  PPO_CUDA(launch_gae(rew, val, done, boot, (int)T, (int)N, gamma, lambda, c->adv, c->ret,
                      c->gae_part, nb, st));
  PPO_CUDA(launch_gae_finalize(c->gae_part, nb, c->advstats, st));
  PPO_CUDA(launch_perm(seed, 0, epochs, N, c->perm, c->perm_work, st, nullptr));
  // learn
  RnnLaunch a{};
  a.s = c->s;
  a.lc = LossCoef{c->cfg.clip, c->cfg.vf_coef, c->cfg.ent_coef};
  a.T = (int)T;
  a.ns = (int)ns;
  a.D = c->cfg.obs_dim;
  a.H = c->cfg.hidden;
  a.L = c->cfg.layers;
  a.N = N;
  a.params = c->params;
  a.obs = obs;
  a.act = act;
  a.actc = actc;
  a.logp_old = logp_old;
  a.adv = c->adv;
  a.ret = c->ret;
  a.adv_stats = c->advstats;
  a.done = done;
  a.h0 = h0;
  a.grad = c->grad;
  a.work = static_cast<float*>(c->work);
  a.err = c->err;
  AdamArgs aa{};
  aa.p = c->params;
  aa.g = c->grad;
  aa.m = c->m;
  aa.v = c->v;
  aa.P = c->P;
  aa.sq_part = c->sq;
  aa.nsq = 0;   // the norm pass runs before Adam
  aa.max_norm = c->cfg.max_grad_norm;
  aa.lr = lr;
  aa.b1 = c->cfg.beta1;
  aa.b2 = c->cfg.beta2;
  aa.eps = (float)c->cfg.adam_eps;
  aa.omb1 = (float)(1.0 - c->cfg.beta1);
  aa.omb2 = (float)(1.0 - c->cfg.beta2);
  aa.step = c->step;
  aa.beta_pow = c->beta_pow;
  aa.done_ctr = c->done_ctr;
  aa.s = c->s;   // no bf16 shadows: the loss builds its operand forms each minibatch
  for (int e = 0; e < epochs; ++e) {
    for (int k = 0; k < minibatches; ++k) {
      a.envs = c->perm + (int64_t)e * N + (int64_t)k * ns;
      a.stats6 = stats ? stats + ((int64_t)e * minibatches + k) * 6 : nullptr;
      if (c->cfg.precision == 1)
        PPO_CUDA(launch_rnn_loss_grad_tc(a, c->num_sms, st, nullptr));
      else
        PPO_CUDA(launch_rnn_loss_grad(a, st));
      PPO_CUDA(launch_adam(aa, st));
    }
  }
  return PPO_OK;
}

ppo_status ppo_rnn_sync_status(ppo_rnn_ctx* c, cudaStream_t st) {
  if (!c) return PPO_ERR_INVALID;
  PPO_CUDA(cudaStreamSynchronize(st));
  if (c->cfg.precision == 1) {
    int e = 0;
    PPO_CUDA(cudaMemcpy(&e, c->err, sizeof(int), cudaMemcpyDeviceToHost));
    if (e != 0) {
      PPO_CUDA(cudaMemset(c->err, 0, sizeof(int)));
      return PPO_ERR_TIMEOUT;
    }
  }
  return PPO_OK;
}

}  // extern "C"
