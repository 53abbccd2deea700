// gather.cu -- observation packing and minibatch gather.
//
// Pack: fp32 observations [B][D] -> bf16 [B][Dp] (zero-padded to the layer-1
// GEMM's K tile) once per update, so each epoch's gathers move 2 bytes per
// element.  Gather: rows idx[0..mb) of the batch ("Teaching Mario to
// speedrun", sec. 6: "for minibatch in shuffle(batch)") into contiguous
// minibatch buffers that the GEMMs' TMA loads can tile; the advantage is
// normalised on the way, (A - mean)/(std + 1e-8).  Segment mode gathers whole
// environment segments (sec. 8, advantages per minibatch from fresh values).
#include "common.cuh"

namespace ppo {

namespace {

constexpr int kPackThreads = 256;

__global__ void __launch_bounds__(kPackThreads)
pack_kernel(const float* __restrict__ obs, int64_t B, int D, int Dp,
            __nv_bfloat16* __restrict__ out) {
  const int vec_per_row = Dp / 8;
  const int64_t total = B * vec_per_row;
  const int64_t stride = (int64_t)gridDim.x * kPackThreads;
  for (int64_t v = (int64_t)blockIdx.x * kPackThreads + threadIdx.x; v < total; v += stride) {
    const int64_t row = v / vec_per_row;
    const int c0 = (int)(v % vec_per_row) * 8;
    const float* src = obs + row * D;
    float f[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) f[j] = (c0 + j < D) ? __ldcs(src + c0 + j) : 0.f;
    uint4 o;
    o.x = pack_bf16x2(f[0], f[1]);
    o.y = pack_bf16x2(f[2], f[3]);
    o.z = pack_bf16x2(f[4], f[5]);
    o.w = pack_bf16x2(f[6], f[7]);
    reinterpret_cast<uint4*>(out + row * Dp)[c0 / 8] = o;
  }
}

constexpr int kGatherThreads = 256;

// One thread per 8-element chunk of a row (bf16 output) or per element (fp32
// output); the thread holding chunk 0 of a row also copies the row's side data.
__global__ void __launch_bounds__(kGatherThreads)
gather_kernel(NetShape s, GatherArgs a, int per_row) {
  pdl_wait();
  pdl_trigger();
  const int64_t t = (int64_t)blockIdx.x * kGatherThreads + threadIdx.x;
  const int64_t r = t / per_row;
  const int c = (int)(t - r * per_row);
  if (r >= a.mb) return;
  int64_t src;
  if (a.seg_envs) {
    const int64_t per = (int64_t)a.seg_T * a.seg_ns;
    const int64_t m = r / per;
    const int64_t rr = r - m * per;
    const int64_t t = rr / a.seg_ns;
    const int64_t j = rr - t * a.seg_ns;
    int64_t e = __ldg(a.seg_envs + m * a.seg_ns + j);
    e = e < 0 ? 0 : (e >= a.seg_N ? a.seg_N - 1 : e);
    src = t * a.seg_N + e;
  } else {
    src = __ldg(a.idx + r);
  }
  src = src < 0 ? 0 : (src >= a.B ? a.B - 1 : src);   // never read outside the batch
  if (a.obs_bf16) {
    const uint4* in = reinterpret_cast<const uint4*>(a.obs_bf16 + src * s.Dp);
    reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(a.X) + r * s.Dp)[c] = __ldg(in + c);
  } else if (a.x_bf16) {
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
  } else {
    static_cast<float*>(a.X)[r * s.D + c] = __ldg(a.obs_f32 + src * s.D + c);
  }
  if (c != 0) return;
  // side data: every load is issued before any store
  int32_t act[PPO_MAX_HEADS];
  float actc[4];
  for (int h = 0; h < s.NH; ++h) act[h] = __ldg(a.act + src * s.NH + h);
  for (int g = 0; g < s.G; ++g) actc[g] = __ldg(a.actc + src * s.G + g);
  const float lp = __ldg(a.logp_old + src);
  float A = 0.f, R = 0.f;
  if (a.adv) {   // no advantages when they are computed per minibatch later
    A = __ldg(a.adv + src);
    R = __ldg(a.ret + src);
    if (a.adv_stats) A = (A - __ldg(a.adv_stats)) / (__ldg(a.adv_stats + 1) + 1e-8f);
  }
  for (int h = 0; h < s.NH; ++h) {
    // an out-of-range action is clamped into its head so the loss never
    // indexes outside the head's logits
    const int n = s.head_n[h];
    a.act_mb[r * s.NH + h] = act[h] < 0 ? 0 : (act[h] >= n ? n - 1 : act[h]);
  }
  for (int g = 0; g < s.G; ++g) a.actc_mb[r * s.G + g] = actc[g];
  a.logp_mb[r] = lp;
  if (a.adv) {
    a.adv_mb[r] = A;
    a.ret_mb[r] = R;
  }
}

}  // namespace

cudaError_t launch_pack_obs(const float* obs, int64_t B, int D, int Dp, __nv_bfloat16* out,
                            cudaStream_t st) {
  const int64_t total = B * (Dp / 8);
  int64_t blocks = (total + kPackThreads - 1) / kPackThreads;
  if (blocks > 152 * 16) blocks = 152 * 16;
  if (blocks < 1) blocks = 1;
  pack_kernel<<<(int)blocks, kPackThreads, 0, st>>>(obs, B, D, Dp, out);
  return cudaGetLastError();
}

cudaError_t launch_gather(const NetShape& s, const GatherArgs& a, cudaStream_t st) {
  const int per_row = (a.obs_bf16 || a.x_bf16) ? s.Dp / 8 : s.D;
  const int64_t threads = a.mb * per_row;
  const int64_t blocks = (threads + kGatherThreads - 1) / kGatherThreads;
  return launch_pdl(gather_kernel, dim3((unsigned)blocks), dim3(kGatherThreads), 0, st, s, a,
                    per_row);
}

}  // namespace ppo
