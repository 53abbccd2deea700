// gather.cu -- observation packing and minibatch gather.
//
// Pack: fp32 observations [B][D] -> bf16 [B][Dp] (zero-padded to the layer-1
// GEMM's K tile) once per update, so each epoch's gathers move 2 bytes per
// element.  Gather: rows idx[0..mb) of the batch ("Teaching Mario to
// speedrun", sec. 6: "for minibatch in shuffle(batch)") into contiguous
// minibatch buffers that the GEMMs' TMA loads can tile; the advantage is
// normalised on the way, (A - mean)/(std + 1e-8).
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
constexpr int kRowsPerBlock = kGatherThreads / kWarp;

__global__ void __launch_bounds__(kGatherThreads)
gather_kernel(NetShape s, GatherArgs a) {
  const int warp = threadIdx.x / kWarp, lane = threadIdx.x % kWarp;
  const int64_t r = (int64_t)blockIdx.x * kRowsPerBlock + warp;
  if (r >= a.mb) return;
  int64_t src = a.idx[r];
  src = src < 0 ? 0 : (src >= a.B ? a.B - 1 : src);   // never read outside the batch
  if (a.obs_bf16) {
    const uint4* in = reinterpret_cast<const uint4*>(a.obs_bf16 + src * s.Dp);
    uint4* out = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(a.X) + r * s.Dp);
    for (int j = lane; j < s.Dp / 8; j += kWarp) out[j] = __ldg(in + j);
  } else if (a.x_bf16) {
    const float* in = a.obs_f32 + src * s.D;
    uint32_t* out = reinterpret_cast<uint32_t*>(static_cast<__nv_bfloat16*>(a.X) + r * s.Dp);
    for (int j = lane; j < s.Dp / 2; j += kWarp) {
      const int c = 2 * j;
      const float x0 = c < s.D ? __ldg(in + c) : 0.f;
      const float x1 = c + 1 < s.D ? __ldg(in + c + 1) : 0.f;
      out[j] = pack_bf16x2(x0, x1);
    }
  } else {
    const float* in = a.obs_f32 + src * s.D;
    float* out = static_cast<float*>(a.X) + r * s.D;
    for (int j = lane; j < s.D; j += kWarp) out[j] = __ldg(in + j);
  }
  if (lane < s.NH) {
    // an out-of-range action is clamped into its head so the loss never
    // indexes outside the head's logits
    int32_t x = a.act[src * s.NH + lane];
    const int n = s.head_n[lane];
    a.act_mb[r * s.NH + lane] = x < 0 ? 0 : (x >= n ? n - 1 : x);
  }
  if (lane < s.G) a.actc_mb[r * s.G + lane] = a.actc[src * s.G + lane];
  if (lane == 0) {
    a.logp_mb[r] = a.logp_old[src];
    float A = a.adv[src];
    if (a.adv_stats) A = (A - a.adv_stats[0]) / (a.adv_stats[1] + 1e-8f);
    a.adv_mb[r] = A;
    a.ret_mb[r] = a.ret[src];
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
  const int64_t blocks = (a.mb + kRowsPerBlock - 1) / kRowsPerBlock;
  gather_kernel<<<(int)blocks, kGatherThreads, 0, st>>>(s, a);
  return cudaGetLastError();
}

}  // namespace ppo
