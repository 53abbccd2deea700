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
constexpr int kGatherRows = 4;   // rows per thread: four independent loads in flight

// Source row of minibatch row r, clamped into the batch.
__device__ __forceinline__ int64_t gather_src(const GatherArgs& a, int64_t r) {
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
  return src < 0 ? 0 : (src >= a.B ? a.B - 1 : src);   // never read outside the batch
}

// One thread per 8-element chunk (bf16 output) or element (fp32 output) of
// kGatherRows consecutive minibatch rows, all loads issued before any store;
// the threads holding chunks 0 .. kGatherRows-1 also copy the rows' side data.
// MODE: 0 packed bf16 observations, 1 fp32 observations to bf16, 2 fp32.
template <int MODE>
__global__ void __launch_bounds__(kGatherThreads)
gather_kernel(NetShape s, GatherArgs a, int per_row) {
  pdl_wait();
  pdl_trigger();
  const int64_t t = (int64_t)blockIdx.x * kGatherThreads + threadIdx.x;
  const int64_t grp = t / per_row;
  const int c = (int)(t - grp * per_row);
  const int64_t r0 = grp * kGatherRows;
  if (r0 >= a.mb) return;
  const int nr = a.mb - r0 < kGatherRows ? (int)(a.mb - r0) : kGatherRows;
  int64_t src[kGatherRows];
#pragma unroll
  for (int k = 0; k < kGatherRows; ++k) src[k] = k < nr ? gather_src(a, r0 + k) : 0;
  if constexpr (MODE == 0) {
    uint4 x[kGatherRows];
#pragma unroll
    for (int k = 0; k < kGatherRows; ++k)
      if (k < nr) x[k] = __ldg(reinterpret_cast<const uint4*>(a.obs_bf16 + src[k] * s.Dp) + c);
#pragma unroll
    for (int k = 0; k < kGatherRows; ++k)
      if (k < nr)
        reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(a.X) + (r0 + k) * s.Dp)[c] = x[k];
  } else if constexpr (MODE == 1) {
    float f[kGatherRows][8];
#pragma unroll
    for (int k = 0; k < kGatherRows; ++k) {
      const float* in = a.obs_f32 + src[k] * s.D;
#pragma unroll
      for (int j = 0; j < 8; ++j) f[k][j] = (k < nr && 8 * c + j < s.D) ? __ldg(in + 8 * c + j) : 0.f;
    }
#pragma unroll
    for (int k = 0; k < kGatherRows; ++k) {
      if (k >= nr) continue;
      uint4 o;
      o.x = pack_bf16x2(f[k][0], f[k][1]);
      o.y = pack_bf16x2(f[k][2], f[k][3]);
      o.z = pack_bf16x2(f[k][4], f[k][5]);
      o.w = pack_bf16x2(f[k][6], f[k][7]);
      reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(a.X) + (r0 + k) * s.Dp)[c] = o;
    }
  } else {
    float x[kGatherRows];
#pragma unroll
    for (int k = 0; k < kGatherRows; ++k) x[k] = k < nr ? __ldg(a.obs_f32 + src[k] * s.D + c) : 0.f;
#pragma unroll
    for (int k = 0; k < kGatherRows; ++k)
      if (k < nr) static_cast<float*>(a.X)[(r0 + k) * s.D + c] = x[k];
  }
  // side data: thread c copies that of row r0 + c (rows taken in turn if a
  // row has fewer than kGatherRows threads), every load before any store
  for (int k = c; k < nr; k += per_row) {
    const int64_t sr = k == 0 ? src[0] : (k == 1 ? src[1] : (k == 2 ? src[2] : src[3]));
    const int64_t r = r0 + k;
    int32_t act[PPO_MAX_HEADS];
    float actc[4];
#pragma unroll
    for (int h = 0; h < PPO_MAX_HEADS; ++h) act[h] = h < s.NH ? __ldg(a.act + sr * s.NH + h) : 0;
#pragma unroll
    for (int g = 0; g < 4; ++g) actc[g] = g < s.G ? __ldg(a.actc + sr * s.G + g) : 0.f;
    const float lp = __ldg(a.logp_old + sr);
    float A = 0.f, R = 0.f;
    if (a.adv) {   // no advantages when they are computed per minibatch later
      A = __ldg(a.adv + sr);
      R = __ldg(a.ret + sr);
      if (a.adv_stats) A = (A - __ldg(a.adv_stats)) / (__ldg(a.adv_stats + 1) + 1e-8f);
    }
#pragma unroll
    for (int h = 0; h < PPO_MAX_HEADS; ++h) {
      // an out-of-range action is clamped into its head so the loss never
      // indexes outside the head's logits
      if (h >= s.NH) break;
      const int n = s.head_n[h];
      a.act_mb[r * s.NH + h] = act[h] < 0 ? 0 : (act[h] >= n ? n - 1 : act[h]);
    }
#pragma unroll
    for (int g = 0; g < 4; ++g)
      if (g < s.G) a.actc_mb[r * s.G + g] = actc[g];
    a.logp_mb[r] = lp;
    if (a.adv) {
      a.adv_mb[r] = A;
      a.ret_mb[r] = R;
    }
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
  const int64_t threads = (a.mb + kGatherRows - 1) / kGatherRows * per_row;
  const int64_t blocks = (threads + kGatherThreads - 1) / kGatherThreads;
  if (a.obs_bf16)
    return launch_pdl(gather_kernel<0>, dim3((unsigned)blocks), dim3(kGatherThreads), 0, st, s, a,
                      per_row);
  if (a.x_bf16)
    return launch_pdl(gather_kernel<1>, dim3((unsigned)blocks), dim3(kGatherThreads), 0, st, s, a,
                      per_row);
  return launch_pdl(gather_kernel<2>, dim3((unsigned)blocks), dim3(kGatherThreads), 0, st, s, a,
                    per_row);
}

}  // namespace ppo
