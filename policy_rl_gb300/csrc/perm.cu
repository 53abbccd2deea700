// perm.cu -- bit-exact minibatch permutation.
//
// "Teaching Mario to speedrun", sec. 6: "for minibatch in shuffle(batch)".
// Key i of epoch e is mulberry32 draw number e*B + i of the stream seeded
// with `seed` ("PlayTrain", Appendix F.2 "seeded RNG"): the generator's state
// is a counter advanced by 0x6D2B79F5 per draw, so draw k is a pure function
// of seed + (k+1)*0x6D2B79F5 and every thread computes its own key.
// The permutation is the index order sorted by (key, index), produced by a
// stable least-significant-digit radix sort: 4 passes of 8 bits, each pass a
// per-tile histogram, a per-digit exclusive scan over the tiles (one block per
// digit), and a stable scatter in which every warp ranks equal digits with
// __match_any_sync.
#include "common.cuh"

namespace ppo {

namespace {

constexpr int kSortThreads = 256;
constexpr int kSortWarps = kSortThreads / kWarp;
constexpr int kPerLane = 16;                         // elements per lane
constexpr int kWarpSpan = kWarp * kPerLane;          // 512 elements per warp
constexpr int kTile = kSortWarps * kWarpSpan;        // 4096 elements per block
constexpr int kRadix = 256;

__device__ __forceinline__ uint32_t mulberry32_draw(uint32_t seed, uint64_t k) {
  uint32_t t = seed + (uint32_t)(k + 1) * 0x6D2B79F5u;
  uint32_t n = (t ^ (t >> 15)) * (t | 1u);
  n ^= n + (n ^ (n >> 7)) * (n | 61u);
  return n ^ (n >> 14);
}

// Input of one radix pass for all epochs at once: epoch e = blockIdx.y reads
// keys/vals at offset e*B (or generates draw e*B + i of the stream).
struct SortIn {
  const uint32_t* keys;   // nullptr: generate from (seed, draw0 + e*B + i)
  const int32_t* vals;    // nullptr: value = i
  uint32_t seed;
  uint64_t draw0;
};

__device__ __forceinline__ void load_kv(const SortIn& in, int64_t B, int64_t i, uint32_t& k,
                                        int32_t& v) {
  const int64_t e = blockIdx.y;
  if (in.keys) {
    k = in.keys[e * B + i];
    v = in.vals[e * B + i];
  } else {
    k = mulberry32_draw(in.seed, in.draw0 + (uint64_t)(e * B + i));
    v = (int32_t)i;
  }
}

__global__ void __launch_bounds__(kSortThreads)
hist_kernel(SortIn in, int64_t B, int shift, uint32_t* __restrict__ ghist, int num_tiles) {
  __shared__ uint32_t h[kRadix];
  const int64_t e = blockIdx.y;
  ghist += e * (int64_t)kRadix * num_tiles;
  h[threadIdx.x] = 0;
  __syncthreads();
  const int64_t base = (int64_t)blockIdx.x * kTile;
  for (int j = 0; j < kTile / kSortThreads; ++j) {
    const int64_t i = base + j * kSortThreads + threadIdx.x;
    if (i < B) {
      const uint32_t k = in.keys ? in.keys[e * B + i]
                                 : mulberry32_draw(in.seed, in.draw0 + (uint64_t)(e * B + i));
      atomicAdd(&h[(k >> shift) & 0xFF], 1u);
    }
  }
  __syncthreads();
  ghist[(int64_t)threadIdx.x * num_tiles + blockIdx.x] = h[threadIdx.x];
}

// Exclusive scan over 256 threads (fixed order); returns the exclusive prefix
// of x and writes the block total to *total.
__device__ __forceinline__ uint32_t block_excl_scan256(uint32_t x, uint32_t* wsum,
                                                       uint32_t* total) {
  const int lane = threadIdx.x % kWarp, warp = threadIdx.x / kWarp;
  uint32_t incl = x;
#pragma unroll
  for (int o = 1; o < kWarp; o <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == kWarp - 1) wsum[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    uint32_t v = lane < kSortWarps ? wsum[lane] : 0u;
#pragma unroll
    for (int o = 1; o < kSortWarps; o <<= 1) {
      const uint32_t y = __shfl_up_sync(0xffffffffu, v, o);
      if (lane >= o) v += y;
    }
    if (lane < kSortWarps) wsum[lane] = v;
  }
  __syncthreads();
  const uint32_t excl = incl - x + (warp > 0 ? wsum[warp - 1] : 0u);
  *total = wsum[kSortWarps - 1];
  __syncthreads();
  return excl;
}

// One block per digit: exclusive scan of that digit's per-tile counts (in
// place) and the digit's total count.
constexpr int kScanPer = 8;
__global__ void __launch_bounds__(kSortThreads)
digit_scan_kernel(uint32_t* __restrict__ ghist, int num_tiles, uint32_t* __restrict__ dtotal) {
  __shared__ uint32_t wsum[kSortWarps];
  ghist += (int64_t)blockIdx.y * kRadix * num_tiles;
  dtotal += (int64_t)blockIdx.y * kRadix;
  uint32_t* row = ghist + (int64_t)blockIdx.x * num_tiles;
  uint32_t carry = 0;
  for (int base = 0; base < num_tiles; base += kSortThreads * kScanPer) {
    const int i0 = base + threadIdx.x * kScanPer;
    uint32_t c[kScanPer];
    uint32_t sum = 0;
#pragma unroll
    for (int j = 0; j < kScanPer; ++j) {
      c[j] = (i0 + j < num_tiles) ? row[i0 + j] : 0u;
      sum += c[j];
    }
    uint32_t chunk_total;
    uint32_t run = carry + block_excl_scan256(sum, wsum, &chunk_total);
#pragma unroll
    for (int j = 0; j < kScanPer; ++j)
      if (i0 + j < num_tiles) {
        row[i0 + j] = run;
        run += c[j];
      }
    carry += chunk_total;
  }
  if (threadIdx.x == 0) dtotal[blockIdx.x] = carry;
}

__global__ void __launch_bounds__(kSortThreads)
scatter_kernel(SortIn in, int64_t B, int shift, const uint32_t* __restrict__ gscan, int num_tiles,
               const uint32_t* __restrict__ dtotal, uint32_t* __restrict__ keys_out,
               int32_t* __restrict__ vals_out) {
  __shared__ uint32_t wofs[kSortWarps][kRadix];
  __shared__ uint32_t dbase[kRadix];
  __shared__ uint32_t wsum[kSortWarps];
  const int warp = threadIdx.x / kWarp, lane = threadIdx.x % kWarp;
  {
    const int64_t e = blockIdx.y;
    gscan += e * (int64_t)kRadix * num_tiles;
    dtotal += e * kRadix;
    if (keys_out) keys_out += e * B;
    vals_out += e * B;
  }
  {
    // first output position of each digit: exclusive scan of the digit totals
    uint32_t tot;
    dbase[threadIdx.x] = block_excl_scan256(dtotal[threadIdx.x], wsum, &tot);
  }
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
      load_kv(in, B, i, k[r], v[r]);
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
    uint32_t run = dbase[d] + gscan[(int64_t)d * num_tiles + blockIdx.x];
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

size_t perm_workspace_bytes(int64_t B, int epochs) {
  const int64_t tiles = (B + kTile - 1) / kTile;
  const size_t kv = (size_t)B * 4 * epochs;
  auto al = [](size_t x) { return (x + 255) & ~(size_t)255; };
  return 4 * al(kv) + al((size_t)tiles * kRadix * 4 * epochs) + al((size_t)kRadix * 4 * epochs);
}

cudaError_t launch_perm(uint32_t seed, int64_t epoch0, int epochs, int64_t B, int32_t* perm,
                        void* work, cudaStream_t st, const Trace* tr) {
  const int tiles = (int)((B + kTile - 1) / kTile);
  auto al = [](size_t x) { return (x + 255) & ~(size_t)255; };
  const size_t kv = (size_t)B * 4 * epochs;
  char* w = static_cast<char*>(work);
  uint32_t* ka = reinterpret_cast<uint32_t*>(w);
  w += al(kv);
  int32_t* va = reinterpret_cast<int32_t*>(w);
  w += al(kv);
  uint32_t* kb = reinterpret_cast<uint32_t*>(w);
  w += al(kv);
  int32_t* vb = reinterpret_cast<int32_t*>(w);
  w += al(kv);
  uint32_t* ghist = reinterpret_cast<uint32_t*>(w);
  w += al((size_t)tiles * kRadix * 4 * epochs);
  uint32_t* dtotal = reinterpret_cast<uint32_t*>(w);

  // all epochs sorted together: epoch e = blockIdx.y, output perm + e*B
  const uint64_t draw0 = (uint64_t)epoch0 * (uint64_t)B;
  SortIn in{nullptr, nullptr, seed, draw0};
  for (int pass = 0; pass < 4; ++pass) {
    const int shift = 8 * pass;
    uint32_t* ko;
    int32_t* vo;
    if (pass == 3) {
      ko = nullptr;
      vo = perm;
    } else if (pass % 2 == 0) {
      ko = kb;
      vo = vb;
    } else {
      ko = ka;
      vo = va;
    }
    hist_kernel<<<dim3(tiles, epochs), kSortThreads, 0, st>>>(in, B, shift, ghist, tiles);
    if (tr) tr->mark(ST_PERM_HIST, st);
    digit_scan_kernel<<<dim3(kRadix, epochs), kSortThreads, 0, st>>>(ghist, tiles, dtotal);
    if (tr) tr->mark(ST_PERM_SCAN, st);
    scatter_kernel<<<dim3(tiles, epochs), kSortThreads, 0, st>>>(in, B, shift, ghist, tiles,
                                                                  dtotal, ko, vo);
    if (tr) tr->mark(ST_PERM_SCATTER, st);
    in = SortIn{ko, vo, seed, draw0};
  }
  return cudaGetLastError();
}

}  // namespace ppo
