// act.cu -- rollout-side policy step: sampled actions, their log-probability
// and the value for every agent of one environment step.
//
// "Teaching Mario to speedrun", sec. 6 "The whole algorithm", step 1, and
// sec. 7 (the trainer's side of a horizon): logits and value from the policy
// for all agents at once, actions sampled from the logits and written
// straight into the action buffer, the probability of the taken action kept
// for the ratio.  The forward GEMMs are the learner's (tensor cores in bf16
// mode); this kernel takes the last hidden layer, one thread per agent (8
// lanes per agent for steps of fewer than 16,384 agents):
//   head outputs z (head_rows.cuh), then per discrete head an inverse-CDF
//   draw (the first category whose cumulative probability exceeds u,
//   compared as u * sum e^(z - max) < running sum), per Gaussian dimension
//   mu + e^s n with n = sqrt(-2 ln(1 - u1)) cos(2 pi u2) (Box-Muller), then
//   log-probability of the stored action and the value column.
// Uniforms: mulberry32 ("PlayTrain", Appendix F.2) as a counter-based
// generator.  Agent i, slot k (head h = slot h; Gaussian dim g = slots
// NH + 2g, NH + 2g + 1; K = NH + 2G slots per agent) takes draw number
// draw0 + i K + k of the stream seeded with `seed`; u = (draw >> 8) 2^-24.
#include "common.cuh"
#include "head_rows.cuh"

namespace ppo {

namespace {

constexpr int kActThreads = 256;

// Draw number `draw` (0-based) of the mulberry32 stream seeded with `seed`:
// the state after draw+1 increments of 0x6D2B79F5, mixed.
__device__ __forceinline__ uint32_t mulberry32_at(uint32_t seed, uint64_t draw) {
  uint32_t t = seed + (uint32_t)(draw + 1) * 0x6D2B79F5u;
  t = (t ^ (t >> 15)) * (t | 1u);
  t ^= t + (t ^ (t >> 7)) * (t | 61u);
  return t ^ (t >> 14);
}

__device__ __forceinline__ float uniform24(uint32_t x) { return (float)(x >> 8) * 5.9604645e-8f; }

// One agent per SPLIT consecutive lanes: SPLIT = 1 for large agent counts;
// SPLIT = 8 spreads a small step (a few thousand agents) over more SMs.
template <int NCOL, int SPLIT>
__global__ void __launch_bounds__(kActThreads)
policy_act_kernel(PolicyActArgs a) {
  extern __shared__ float4 smem_dyn[];
  float* w3t = reinterpret_cast<float*>(smem_dyn);
  pdl_wait();
  const HeadSrc hs{a.h, a.h_bf16, a.W3, a.b3, a.s.H2, a.s.C};
  stage_w3<NCOL>(hs, w3t, kActThreads);
  pdl_trigger();
  const int64_t t = (int64_t)blockIdx.x * kActThreads + threadIdx.x;
  const int64_t i = t / SPLIT;
  const int q = (int)(t % SPLIT);
  const bool valid = i < a.n;
  if (SPLIT == 1 && !valid) return;
  float zr[NCOL];
  if (valid) {
    head_row<NCOL, SPLIT>(hs, w3t, i, zr, q);
  } else {
#pragma unroll
    for (int c = 0; c < NCOL; ++c) zr[c] = 0.f;
  }
  if constexpr (SPLIT > 1) split_sum<NCOL, SPLIT>(zr);   // every lane of the warp
  if (!valid || q != 0) return;
  float z[NCOL];   // dynamically indexed below (local memory)
#pragma unroll
  for (int c = 0; c < NCOL; ++c) z[c] = zr[c];
  const NetShape& s = a.s;
  const int K = s.NH + 2 * s.G;
  const uint64_t d0 = a.draw0 + (uint64_t)i * (uint64_t)K;
  float logp = 0.f;
  int off = 0;
  for (int h = 0; h < s.NH; ++h) {
    const int n = s.head_n[h];
    float m = z[off];
    for (int k = 1; k < n; ++k) m = fmaxf(m, z[off + k]);
    float total = 0.f;
    for (int k = 0; k < n; ++k) total += expf(z[off + k] - m);
    const float thresh = uniform24(mulberry32_at(a.seed, d0 + h)) * total;
    int pick = n - 1;
    float cum = 0.f;
    for (int k = 0; k < n; ++k) {
      cum += expf(z[off + k] - m);
      if (thresh < cum) {
        pick = k;
        break;
      }
    }
    a.act[i * s.NH + h] = pick;
    logp += z[off + pick] - (m + logf(total));
    off += n;
  }
  for (int g = 0; g < s.G; ++g) {
    const float u1 = uniform24(mulberry32_at(a.seed, d0 + s.NH + 2 * g));
    const float u2 = uniform24(mulberry32_at(a.seed, d0 + s.NH + 2 * g + 1));
    const float nrm = sqrtf(-2.f * logf(1.f - u1)) * cospif(2.f * u2);
    const float mu = z[off + g], ls = __ldg(a.logstd + g);
    const float act = mu + expf(ls) * nrm;
    a.actc[i * s.G + g] = act;
    const float d = act - mu;   // the log-density of the action as stored
    logp += -0.5f * d * d * expf(-2.f * ls) - ls - 0.91893853320467274f;   // ln(2 pi) / 2
  }
  if (a.logp) a.logp[i] = logp;
  if (a.value) a.value[i] = z[s.C - 1];
}

// Agent counts below this use 8 lanes per agent.
constexpr int64_t kActSplitBelow = 16384;

int g_act_ready = 0;

template <int NCOL, int SPLIT>
cudaError_t prepare_one() {
  return cudaFuncSetAttribute(policy_act_kernel<NCOL, SPLIT>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize,
                              (int)(w3_floats(NCOL, 512) * sizeof(float)));
}

}  // namespace

cudaError_t policy_act_prepare() {
  if (g_act_ready) return cudaSuccess;
  cudaError_t e = prepare_one<16, 1>();
  if (e == cudaSuccess) e = prepare_one<32, 1>();
  if (e == cudaSuccess) e = prepare_one<16, 8>();
  if (e == cudaSuccess) e = prepare_one<32, 8>();
  if (e == cudaSuccess) g_act_ready = 1;
  return e;
}

cudaError_t launch_policy_act(const PolicyActArgs& a, cudaStream_t st) {
  if (!g_act_ready) return cudaErrorInitializationError;
  if (a.s.H2 > 512) return cudaErrorInvalidValue;
  const int ncol = a.s.C <= 16 ? 16 : 32;
  const bool split = a.n < kActSplitBelow;
  const size_t smem = (size_t)w3_floats(ncol, a.s.H2) * sizeof(float);
  const int64_t threads = a.n * (split ? 8 : 1);
  const dim3 grid((unsigned)((threads + kActThreads - 1) / kActThreads)), block(kActThreads);
  if (ncol == 16)
    return split ? launch_pdl(policy_act_kernel<16, 8>, grid, block, smem, st, a)
                 : launch_pdl(policy_act_kernel<16, 1>, grid, block, smem, st, a);
  return split ? launch_pdl(policy_act_kernel<32, 8>, grid, block, smem, st, a)
               : launch_pdl(policy_act_kernel<32, 1>, grid, block, smem, st, a);
}

}  // namespace ppo
