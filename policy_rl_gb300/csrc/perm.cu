// perm.cu -- bit-exact minibatch permutation.
//
// "Teaching Mario to speedrun", sec. 6: "for minibatch in shuffle(batch)".
// Key i of epoch e is mulberry32 draw number e*B + i of the stream seeded
// with `seed` ("PlayTrain", Appendix F.2 "seeded RNG"): the generator's state
// is a counter advanced by 0x6D2B79F5 per draw, so draw k is a pure function
// of seed + (k+1)*0x6D2B79F5 and every thread computes its own key.
// The permutation is the index order sorted by (key, index), produced by a
// stable least-significant-digit radix sort: 4 passes of 8 bits, each pass a
// per-tile histogram, one digit-major exclusive scan, and a stable scatter in
// which every warp ranks equal digits with __match_any_sync.
#include "common.cuh"

namespace ppo {

namespace {

constexpr int kSortThreads = 256;
constexpr int kSortWarps = kSortThreads / kWarp;
constexpr int kPerLane = 16;                         // elements per lane
constexpr int kWarpSpan = kWarp * kPerLane;          // 512 elements per warp
constexpr int kTile = kSortWarps * kWarpSpan;        // 4096 elements per block
constexpr int kRadix = 256;
constexpr int kScanThreads = 1024;

__device__ __forceinline__ uint32_t mulberry32_draw(uint32_t seed, uint64_t k) {
  uint32_t t = seed + (uint32_t)(k + 1) * 0x6D2B79F5u;
  uint32_t n = (t ^ (t >> 15)) * (t | 1u);
  n ^= n + (n ^ (n >> 7)) * (n | 61u);
  return n ^ (n >> 14);
}

struct SortIn {
  const uint32_t* keys;   // nullptr: generate from (seed, draw0 + i)
  const int32_t* vals;    // nullptr: value = i
  uint32_t seed;
  uint64_t draw0;
};

__device__ __forceinline__ void load_kv(const SortIn& in, int64_t i, uint32_t& k, int32_t& v) {
  if (in.keys) {
    k = in.keys[i];
    v = in.vals[i];
  } else {
    k = mulberry32_draw(in.seed, in.draw0 + (uint64_t)i);
    v = (int32_t)i;
  }
}

__global__ void __launch_bounds__(kSortThreads)
hist_kernel(SortIn in, int64_t B, int shift, uint32_t* __restrict__ ghist, int num_tiles) {
  __shared__ uint32_t h[kRadix];
  h[threadIdx.x] = 0;
  __syncthreads();
  const int64_t base = (int64_t)blockIdx.x * kTile;
  for (int j = 0; j < kTile / kSortThreads; ++j) {
    const int64_t i = base + j * kSortThreads + threadIdx.x;
    if (i < B) {
      uint32_t k;
      int32_t v;
      load_kv(in, i, k, v);
      atomicAdd(&h[(k >> shift) & 0xFF], 1u);
    }
  }
  __syncthreads();
  ghist[(int64_t)threadIdx.x * num_tiles + blockIdx.x] = h[threadIdx.x];
}

// Exclusive scan of n counts in place (one block, fixed order).
__global__ void __launch_bounds__(kScanThreads) scan_kernel(uint32_t* __restrict__ a, int64_t n) {
  __shared__ uint32_t part[kScanThreads];
  const int64_t per = (n + kScanThreads - 1) / kScanThreads;
  const int64_t lo = threadIdx.x * per;
  const int64_t hi = lo + per < n ? lo + per : n;
  uint32_t s = 0;
  for (int64_t i = lo; i < hi; ++i) s += a[i];
  part[threadIdx.x] = s;
  __syncthreads();
  // Hillis-Steele inclusive scan of the 1024 partial sums
  for (int o = 1; o < kScanThreads; o <<= 1) {
    uint32_t add = threadIdx.x >= o ? part[threadIdx.x - o] : 0u;
    __syncthreads();
    part[threadIdx.x] += add;
    __syncthreads();
  }
  uint32_t run = threadIdx.x > 0 ? part[threadIdx.x - 1] : 0u;
  for (int64_t i = lo; i < hi; ++i) {
    const uint32_t c = a[i];
    a[i] = run;
    run += c;
  }
}

__global__ void __launch_bounds__(kSortThreads)
scatter_kernel(SortIn in, int64_t B, int shift, const uint32_t* __restrict__ gscan, int num_tiles,
               uint32_t* __restrict__ keys_out, int32_t* __restrict__ vals_out) {
  __shared__ uint32_t wofs[kSortWarps][kRadix];
  const int warp = threadIdx.x / kWarp, lane = threadIdx.x % kWarp;
  for (int d = threadIdx.x; d < kSortWarps * kRadix; d += kSortThreads)
    (&wofs[0][0])[d] = 0;
  __syncthreads();

  const int64_t base = (int64_t)blockIdx.x * kTile + (int64_t)warp * kWarpSpan;
  uint32_t k[kPerLane];
  int32_t v[kPerLane];
  uint32_t dig[kPerLane];
#pragma unroll
  for (int r = 0; r < kPerLane; ++r) {
    const int64_t i = base + r * kWarp + lane;
    if (i < B) {
      load_kv(in, i, k[r], v[r]);
      dig[r] = (k[r] >> shift) & 0xFF;
    } else {
      dig[r] = kRadix;   // sentinel: not counted, not written
    }
  }
  // per-warp digit counts
#pragma unroll
  for (int r = 0; r < kPerLane; ++r) {
    const uint32_t peers = __match_any_sync(0xffffffffu, dig[r]);
    const int leader = __ffs(peers) - 1;
    if (lane == leader && dig[r] < kRadix) wofs[warp][dig[r]] += __popc(peers);
    __syncwarp();
  }
  __syncthreads();
  // warp w's first position for digit d: global tile offset + counts of warps < w
  {
    const int d = threadIdx.x;   // kSortThreads == kRadix
    uint32_t run = gscan[(int64_t)d * num_tiles + blockIdx.x];
    for (int w = 0; w < kSortWarps; ++w) {
      const uint32_t c = wofs[w][d];
      wofs[w][d] = run;
      run += c;
    }
  }
  __syncthreads();
  const uint32_t lt_mask = (1u << lane) - 1u;
#pragma unroll
  for (int r = 0; r < kPerLane; ++r) {
    const uint32_t peers = __match_any_sync(0xffffffffu, dig[r]);
    if (dig[r] < kRadix) {
      const uint32_t pos = wofs[warp][dig[r]] + __popc(peers & lt_mask);
      if (keys_out) keys_out[pos] = k[r];
      vals_out[pos] = v[r];
    }
    __syncwarp();
    const int leader = __ffs(peers) - 1;
    if (lane == leader && dig[r] < kRadix) wofs[warp][dig[r]] += __popc(peers);
    __syncwarp();
  }
}

}  // namespace

size_t perm_workspace_bytes(int64_t B, int /*epochs*/) {
  const int64_t tiles = (B + kTile - 1) / kTile;
  const size_t kv = (size_t)B * 4;
  auto al = [](size_t x) { return (x + 255) & ~(size_t)255; };
  return 4 * al(kv) + al((size_t)tiles * kRadix * 4);
}

cudaError_t launch_perm(uint32_t seed, int64_t epoch0, int epochs, int64_t B, int32_t* perm,
                        void* work, cudaStream_t st, const Trace* tr) {
  const int64_t tiles64 = (B + kTile - 1) / kTile;
  const int tiles = (int)tiles64;
  auto al = [](size_t x) { return (x + 255) & ~(size_t)255; };
  char* w = static_cast<char*>(work);
  uint32_t* ka = reinterpret_cast<uint32_t*>(w);
  w += al((size_t)B * 4);
  int32_t* va = reinterpret_cast<int32_t*>(w);
  w += al((size_t)B * 4);
  uint32_t* kb = reinterpret_cast<uint32_t*>(w);
  w += al((size_t)B * 4);
  int32_t* vb = reinterpret_cast<int32_t*>(w);
  w += al((size_t)B * 4);
  uint32_t* ghist = reinterpret_cast<uint32_t*>(w);

  for (int e = 0; e < epochs; ++e) {
    const uint64_t draw0 = (uint64_t)(epoch0 + e) * (uint64_t)B;
    int32_t* out = perm + (int64_t)e * B;
    SortIn in{nullptr, nullptr, seed, draw0};
    for (int pass = 0; pass < 4; ++pass) {
      const int shift = 8 * pass;
      uint32_t* ko;
      int32_t* vo;
      if (pass == 3) {
        ko = nullptr;
        vo = out;
      } else if (pass % 2 == 0) {
        ko = kb;
        vo = vb;
      } else {
        ko = ka;
        vo = va;
      }
      hist_kernel<<<tiles, kSortThreads, 0, st>>>(in, B, shift, ghist, tiles);
      if (tr) tr->mark(ST_PERM_HIST, st);
      scan_kernel<<<1, kScanThreads, 0, st>>>(ghist, (int64_t)tiles * kRadix);
      if (tr) tr->mark(ST_PERM_SCAN, st);
      scatter_kernel<<<tiles, kSortThreads, 0, st>>>(in, B, shift, ghist, tiles, ko, vo);
      if (tr) tr->mark(ST_PERM_SCATTER, st);
      in = SortIn{ko, vo, seed, draw0};
    }
    cudaError_t err = cudaGetLastError();
    if (err != cudaSuccess) return err;
  }
  return cudaSuccess;
}

}  // namespace ppo
