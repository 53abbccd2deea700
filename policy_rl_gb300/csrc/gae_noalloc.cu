// gae_noalloc.cu -- ppo_gae_noalloc: the GAE scan with advantage moments and
// normalisation, for callers that cannot allocate device memory.
//
// ppo_gae needs a caller-supplied scratch buffer for the per-block moment
// partials.  Some callers cannot obtain one: code that runs between other
// work on a stream that is being captured into a CUDA graph (where
// cudaMalloc is not allowed), latency-critical loops that must never enter
// the device allocator, and hosts whose device memory is owned entirely by
// their own pool.  This entry point keeps its scratch in a fixed-size array
// in the library's own device memory instead.
//
// The array is a file-scope __device__ variable: every GPU that loads the
// library holds it (kNoAllocScratchBytes) until the process exits.  Host code
// cannot use the array's name as a device address, so the first call on each
// device looks the address up with cudaGetSymbolAddress (with that device
// current) and caches it together with the device's current CUDA context;
// that first call should therefore come before any stream capture.  A later
// call that finds another context current on the device (the old one was
// destroyed, e.g. by cudaDeviceReset, and the module loaded again) repeats
// the look-up.  All calls share the array: calls that overlap on the GPU
// (different streams without ordering, or different host threads) race on
// it.  Each call overwrites every partial it reads, so nothing needs clearing.
#include <cudaTypedefs.h>

#include <mutex>

#include "common.cuh"

namespace {

// Largest N (environments) this entry point accepts: one 128-thread block
// per 128 environments, three fp64 moment partials per block.
constexpr int64_t kNoAllocMaxN = 1 << 20;
constexpr int kNoAllocMaxBlocks = (int)(kNoAllocMaxN / 128);
constexpr size_t kNoAllocPartialBytes = (size_t)kNoAllocMaxBlocks * 3 * sizeof(double);
constexpr size_t kNoAllocScratchBytes = kNoAllocPartialBytes + 256;   // + {mean, std}

static __device__ __align__(256) unsigned char g_gae_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mutex;
void* g_scratch_addr[kMaxDevices] = {};
CUcontext g_scratch_ctx[kMaxDevices] = {};
PFN_cuCtxGetCurrent_v4000 g_ctx_get_current = nullptr;

// Device address of g_gae_scratch on the current device: looked up on the
// first call, and again whenever the device's current context has changed.
ppo_status scratch_for_current_device(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return PPO_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return PPO_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  if (g_ctx_get_current == nullptr) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &fn, 4000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess || fn == nullptr) {
      cudaGetLastError();
      return PPO_ERR_CUDA;
    }
    g_ctx_get_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(fn);
  }
  CUcontext cur = nullptr;
  if (g_ctx_get_current(&cur) != CUDA_SUCCESS || cur == nullptr) return PPO_ERR_CUDA;
  if (g_scratch_addr[dev] == nullptr || g_scratch_ctx[dev] != cur) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_gae_scratch) != cudaSuccess || p == nullptr) {
      cudaGetLastError();
      return PPO_ERR_CUDA;
    }
    g_scratch_addr[dev] = p;
    g_scratch_ctx[dev] = cur;
  }
  *out = g_scratch_addr[dev];
  return PPO_OK;
}

bool al16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" ppo_status ppo_gae_noalloc(const float* rew, const float* val, const float* done,
                                      const float* boot, int64_t T, int64_t N, float gamma,
                                      float lambda, float* adv, float* ret, float* adv_norm,
                                      float* stats, cudaStream_t st) {
  if (!rew || !val || !done || !boot || !adv || !ret) return PPO_ERR_INVALID;
  if (T < 1 || N < 1 || T * N >= (1ll << 31)) return PPO_ERR_INVALID;
  if (N > kNoAllocMaxN) return PPO_ERR_UNSUPPORTED;   // beyond the fixed scratch
  if (T > ppo::kGaeMaxT) return PPO_ERR_UNSUPPORTED;
  const void* ps[] = {rew, val, done, boot, adv, ret, adv_norm, stats};
  for (const void* p : ps)
    if (p && !al16(p)) return PPO_ERR_ALIGN;
  const bool need_stats = adv_norm || stats;
  double* part = nullptr;
  float* sbuf = stats;
  if (need_stats) {
    void* scratch = nullptr;
    const ppo_status r = scratch_for_current_device(&scratch);
    if (r != PPO_OK) return r;
    part = static_cast<double*>(scratch);
    if (!sbuf) sbuf = reinterpret_cast<float*>(static_cast<char*>(scratch) + kNoAllocPartialBytes);
  }
  const int nb = ppo::gae_num_blocks((int)N);
  if (ppo::launch_gae(rew, val, done, boot, (int)T, (int)N, gamma, lambda, adv, ret, part, nb,
                      st) != cudaSuccess)
    return PPO_ERR_CUDA;
  if (need_stats) {
    if (ppo::launch_gae_finalize(part, nb, sbuf, st) != cudaSuccess) return PPO_ERR_CUDA;
    if (adv_norm && ppo::launch_normalize(adv, sbuf, adv_norm, T * N, st) != cudaSuccess)
      return PPO_ERR_CUDA;
  }
  return PPO_OK;
}
