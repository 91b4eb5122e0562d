// Routing: histogram of the top-k expert ids, exclusive prefix sum, and the
// stable permutation of the T*k flat rows into expert buckets
// ("Strata #3752", commits "moe_ws wiring" and "swiglu_quant landed":
// quantize_scatter, the group bounds uploaded with the layer).
//
// All integer and bit-exact.  Up to 2^14 entries (T*k) one kernel does it all
// in one CTA (route_fused: 32 warps, each counting and then placing a
// contiguous 1/32 of the entries with its counts in shared memory); a launch
// saved matters more there than parallelism.  Beyond that, three kernels:
//   1. route_hist    -- one warp per chunk of 1024 flat entries counts the
//                       chunk's rows per expert (shared-memory histogram);
//                       the CTA then writes, per expert, each of its chunks'
//                       first row within the CTA and the CTA's total;
//   2. route_scan    -- one CTA turns the [CTA][expert] totals into the base
//                       row of every (CTA, expert), the expert counts,
//                       their exclusive prefix sum (group bounds), the
//                       largest-first expert order, and the product kernels'
//                       work list: every expert's rows cut into 128-row
//                       tiles, largest expert first, a short remainder cut
//                       into 32-row tiles for the small-row tier;
//   3. route_scatter -- each warp walks its chunk again, 32 entries at a
//                       time; __match_any_sync groups lanes of equal expert,
//                       a lane's rank among them keeps flat order, so rows of
//                       a bucket come out in increasing flat index t*k + r.
#include <atomic>

#include "common.cuh"

namespace moe {
namespace {

__global__ void __launch_bounds__(kRouteWarps * 32)
route_hist_kernel(const int32_t* __restrict__ ids, int64_t n, int E, int nchunks,
                  int32_t* __restrict__ hist, int32_t* __restrict__ status) {
  extern __shared__ int32_t sh[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int chunk = blockIdx.x * kRouteWarps + warp;
  int32_t* h = sh + warp * E;
  for (int e = lane; e < E; e += 32) h[e] = 0;
  __syncwarp();
  if (chunk < nchunks) {
    const int64_t beg = (int64_t)chunk * kRouteChunk;
    const int64_t end = min(n, beg + kRouteChunk);
    // all of this lane's ids first (independent loads), then the counts
    int v[kRouteChunk / 32];
#pragma unroll
    for (int j = 0; j < kRouteChunk / 32; j++) {
      const int64_t i = beg + lane + 32 * j;
      v[j] = i < end ? __ldg(ids + i) : 0;
    }
    bool bad = false;
#pragma unroll
    for (int j = 0; j < kRouteChunk / 32; j++) {
      if (beg + lane + 32 * j >= end) break;
      if ((unsigned)v[j] < (unsigned)E)
        atomicAdd(&h[v[j]], 1);
      else
        bad = true;
    }
    if (bad) atomicOr(status, MOE_STATUS_BAD_EXPERT_ID);
  }
  __syncthreads();
  // per expert, the CTA's chunks in order: each chunk's first row within the
  // CTA (hist rows 0 .. nchunks-1) and the CTA's total (row nchunks + CTA)
  for (int e = threadIdx.x; e < E; e += kRouteWarps * 32) {
    int run = 0;
#pragma unroll
    for (int w = 0; w < kRouteWarps; w++) {
      const int c = blockIdx.x * kRouteWarps + w;
      const int v = sh[w * E + e];
      if (c < nchunks) hist[(int64_t)c * E + e] = run;
      run += v;
    }
    hist[(int64_t)(nchunks + blockIdx.x) * E + e] = run;
  }
}

// Exclusive prefix sum over the 1024 threads of the CTA (one value each).
__device__ __forceinline__ int block_excl_scan(int v, int32_t* s_warp) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  __syncthreads();  // s_warp free for reuse
  if (lane == 31) s_warp[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    const int w = s_warp[lane];
    int wi = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, wi, o);
      if (lane >= o) wi += y;
    }
    s_warp[lane] = wi - w;
  }
  __syncthreads();
  return s_warp[warp] + incl - v;
}

// Per-expert lists, run by one CTA of 1024 threads, thread e standing for
// expert e (E <= 1024) with run = its row count: counts, the group bounds
// (returned: the expert's first routed row), the largest-first order and
// the work list of tiles with its split count.
struct ScanShared {
  __align__(16) int32_t cnt[1024];  // rows of expert e (0 past E), or its rank key
  int32_t tiles[1024];              // tcgen05 tiles of the expert at rank r, then their first
  int32_t small[1024];              // small-row tiles of the expert at rank r, then their first
  int32_t warp[32];
  int32_t tot[2];                   // tcgen05 tiles, small-row tiles
};
__device__ __forceinline__ int expert_lists(int run, int E, int32_t* __restrict__ counts,
                                            int32_t* __restrict__ offsets,
                                            int32_t* __restrict__ order, int4* __restrict__ tiles,
                                            int32_t* __restrict__ ntiles, ScanShared& sh) {
  const int tid = threadIdx.x;
  if (tid < E) counts[tid] = run;
  // experts rank by (count descending, id ascending).  While every count
  // fits in 22 bits the pair is one unsigned key, the count above 1023 - id,
  // and an expert's rank is the number of larger keys (one compare and one
  // add per expert instead of four tests: the ranking was most of the
  // routing step's time)
  const bool wide = __syncthreads_or(run >= (1 << 22));
  const uint32_t key = ((uint32_t)run << 10) | (uint32_t)(1023 - tid);
  sh.cnt[tid] = wide ? run : (int32_t)key;
  sh.tiles[tid] = 0;
  sh.small[tid] = 0;
  const int excl = block_excl_scan(run, sh.warp);  // also orders the writes above
  int rank = 0;
  // this expert's tiles: full 128-row tiles, then the remainder -- one more
  // tcgen05 tile, or 32-row small-row tiles when it is at most kSmallSplit rows
  const int nfull = run / kTileRows, rem = run - nfull * kTileRows;
  const bool rem_small = rem > 0 && rem <= kSmallSplit;
  const int nbig = nfull + (rem > 0 && !rem_small ? 1 : 0);
  const int nsm = rem_small ? (rem + kSmallTileRows - 1) / kSmallTileRows : 0;
  if (tid < E) {
    offsets[tid] = excl;
    if (tid == E - 1) offsets[E] = excl + run;
    // past E the entries are those of count 0 with ids above every
    // expert's, so whole 16-byte reads count nothing extra (E <= 1024)
    if (!wide) {
      int r0 = 0, r1 = 0;
      for (int e2 = 0; e2 < E; e2 += 8) {
        const uint4 a = *reinterpret_cast<const uint4*>(sh.cnt + e2);
        const uint4 b = *reinterpret_cast<const uint4*>(sh.cnt + e2 + 4);
        r0 += (a.x > key) + (a.y > key) + (a.z > key) + (a.w > key);
        r1 += (b.x > key) + (b.y > key) + (b.z > key) + (b.w > key);
      }
      rank = r0 + r1;
    } else {
      for (int e2 = 0; e2 < E; e2 += 4) {
        const int4 c4 = *reinterpret_cast<const int4*>(sh.cnt + e2);
        rank += (c4.x > run) || (c4.x == run && e2 < tid);
        rank += (c4.y > run) || (c4.y == run && e2 + 1 < tid);
        rank += (c4.z > run) || (c4.z == run && e2 + 2 < tid);
        rank += (c4.w > run) || (c4.w == run && e2 + 3 < tid);
      }
    }
    order[rank] = tid;
    sh.tiles[rank] = nbig;
    sh.small[rank] = nsm;
  }
  __syncthreads();
  // first tile of each rank in each list (thread tid stands for rank tid here)
  const int nt = sh.tiles[tid], ns = sh.small[tid];
  const int tbase = block_excl_scan(nt, sh.warp);
  const int sbase = block_excl_scan(ns, sh.warp);
  if (tid == 1023) {
    sh.tot[0] = tbase + nt;
    sh.tot[1] = sbase + ns;
    ntiles[0] = tbase + nt + sbase + ns;
    ntiles[1] = tbase + nt;  // the tcgen05 tiles come first
    // the small-row launches' work counters ({next item, CTAs done} for
    // gate/up, then for down) start at zero
    ntiles[3] = ntiles[4] = ntiles[5] = ntiles[6] = 0;
  }
  __syncthreads();
  sh.tiles[tid] = tbase;
  sh.small[tid] = sh.tot[0] + sbase;
  __syncthreads();
  if (tid < E) {
    const int first = sh.tiles[rank];
    for (int i = 0; i < nbig; i++)
      tiles[first + i] = make_int4(tid, excl + i * kTileRows, min(kTileRows, run - i * kTileRows), 0);
    const int sfirst = sh.small[rank];
    const int r0 = excl + nfull * kTileRows;
    for (int j = 0; j < nsm; j++)
      tiles[sfirst + j] = make_int4(tid, r0 + j * kSmallTileRows,
                                    min(kSmallTileRows, rem - j * kSmallTileRows), 0);
  }
  return excl;
}

// One CTA of 1024 threads; thread e owns expert e (E <= 1024).  It walks the
// per-CTA totals (hist rows nchunks ..), not the chunks: each becomes the
// expert's first routed row for that CTA's chunks.
__global__ void __launch_bounds__(1024)
route_scan_kernel(int32_t* __restrict__ hist, int nchunks, int E,
                  int32_t* __restrict__ counts, int32_t* __restrict__ offsets,
                  int32_t* __restrict__ order, int4* __restrict__ tiles,
                  int32_t* __restrict__ ntiles) {
  __shared__ ScanShared sh;
  const int tid = threadIdx.x;
  const int nctas = (nchunks + kRouteWarps - 1) / kRouteWarps;
  int32_t* ctot = hist + (int64_t)nchunks * E;
  int run = 0;
  if (tid < E) {
#pragma unroll 8
    for (int b = 0; b < nctas; b++) {
      const int64_t idx = (int64_t)b * E + tid;
      const int v = ctot[idx];
      ctot[idx] = run;  // rows of expert tid in CTAs before b
      run += v;
    }
  }
  const int excl = expert_lists(run, E, counts, offsets, order, tiles, ntiles, sh);
  if (tid < E) {
#pragma unroll 8
    for (int b = 0; b < nctas; b++) ctot[(int64_t)b * E + tid] += excl;
  }
}

// Stable placement of entries [beg, end) of ids, 32 at a time in index
// order: lanes of equal expert are grouped with __match_any_sync and a
// lane's rank among them keeps flat order; h[e] is the next routed row of
// expert e for this range.
__device__ __forceinline__ void scatter_range(const int32_t* __restrict__ ids, int64_t beg,
                                              int64_t end, int E, int32_t* h,
                                              int32_t* __restrict__ row_src,
                                              int32_t* __restrict__ dst_of) {
  const int lane = threadIdx.x & 31;
  const unsigned lt = (1u << lane) - 1u;
  for (int64_t b0 = beg; b0 < end; b0 += 32 * 8) {
    int v[8];  // this lane's next 8 ids first (independent loads)
#pragma unroll
    for (int j = 0; j < 8; j++) {
      const int64_t i = b0 + 32 * j + lane;
      v[j] = i < end ? __ldg(ids + i) : -1;
    }
#pragma unroll
    for (int j = 0; j < 8; j++) {
      const int64_t base = b0 + 32 * j;
      if (base >= end) break;
      const int64_t i = base + lane;
      const bool act = i < end;
      const int e = v[j];
      const bool valid = act && (unsigned)e < (unsigned)E;
      const unsigned peers = __match_any_sync(0xffffffffu, valid ? e : -1);
      const int rank = __popc(peers & lt);
      const int pos = valid ? h[e] + rank : -1;
      __syncwarp();
      if (valid && rank == 0) h[e] += __popc(peers);
      __syncwarp();
      if (valid) row_src[pos] = (int32_t)i;
      if (act) dst_of[i] = pos;
    }
  }
}

// The whole routing step in one CTA of 1024 threads (n <= kFusedMaxEntries):
// warp w owns the contiguous range [w*S, (w+1)*S) of flat entries (S =
// ceil(n/32) rounded up to 32) and a shared-memory count per expert.  Counts,
// then the per-expert lists (with every warp's base for every expert), then
// the stable scatter -- one launch, the histograms never leave the SM.
constexpr int kFusedWarps = 32;
constexpr int64_t kFusedMaxEntries = 1 << 14;
__global__ void __launch_bounds__(1024)
route_fused_kernel(const int32_t* __restrict__ ids, int64_t n, int E,
                   int32_t* __restrict__ counts, int32_t* __restrict__ offsets,
                   int32_t* __restrict__ order, int4* __restrict__ tiles,
                   int32_t* __restrict__ ntiles, int32_t* __restrict__ row_src,
                   int32_t* __restrict__ dst_of, int32_t* __restrict__ status,
                   int zero_status) {
  extern __shared__ int32_t hw[];  // [kFusedWarps][E]
  __shared__ ScanShared sh;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (zero_status && tid == 0) *status = 0;  // before any bit below is set
  const int64_t S = ((n + kFusedWarps - 1) / kFusedWarps + 31) & ~(int64_t)31;
  const int64_t beg = min(n, (int64_t)warp * S), end = min(n, beg + S);
  int32_t* h = hw + warp * E;
  for (int e = lane; e < E; e += 32) h[e] = 0;
  __syncthreads();  // (orders the status reset above before any atomicOr)
  bool bad = false;
  for (int64_t b0 = beg; b0 < end; b0 += 32 * 8) {
    int v[8];
#pragma unroll
    for (int j = 0; j < 8; j++) {
      const int64_t i = b0 + 32 * j + lane;
      v[j] = i < end ? __ldg(ids + i) : 0;
    }
#pragma unroll
    for (int j = 0; j < 8; j++) {
      if (b0 + 32 * j + lane >= end) break;
      if ((unsigned)v[j] < (unsigned)E)
        atomicAdd(&h[v[j]], 1);
      else
        bad = true;
    }
  }
  if (bad) atomicOr(status, MOE_STATUS_BAD_EXPERT_ID);
  __syncthreads();
  int run = 0;
  if (tid < E) {
#pragma unroll 8
    for (int w = 0; w < kFusedWarps; w++) {
      const int v = hw[w * E + tid];
      hw[w * E + tid] = run;  // rows of expert tid in ranges before warp w's
      run += v;
    }
  }
  const int excl = expert_lists(run, E, counts, offsets, order, tiles, ntiles, sh);
  if (tid < E) {
#pragma unroll 8
    for (int w = 0; w < kFusedWarps; w++) hw[w * E + tid] += excl;
  }
  __syncthreads();
  scatter_range(ids, beg, end, E, h, row_src, dst_of);
}

__global__ void __launch_bounds__(kRouteWarps * 32)
route_scatter_kernel(const int32_t* __restrict__ ids, int64_t n, int E, int nchunks,
                     const int32_t* __restrict__ hist, int32_t* __restrict__ row_src,
                     int32_t* __restrict__ dst_of) {
  extern __shared__ int32_t sh[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int chunk = blockIdx.x * kRouteWarps + warp;
  int32_t* h = sh + warp * E;
  if (chunk >= nchunks) return;
  const int32_t* cbase = hist + (int64_t)(nchunks + blockIdx.x) * E;  // this CTA's chunks
  for (int e = lane; e < E; e += 32) h[e] = hist[(int64_t)chunk * E + e] + cbase[e];
  __syncwarp();
  const int64_t beg = (int64_t)chunk * kRouteChunk;
  scatter_range(ids, beg, min(n, beg + kRouteChunk), E, h, row_src, dst_of);
}

}  // namespace

cudaError_t launch_route(const int32_t* ids, int64_t n, int E, int32_t* hist,
                         int32_t* counts, int32_t* offsets, int32_t* order,
                         int32_t* row_src, int32_t* dst_of, int4* tiles, int32_t* ntiles,
                         int32_t* status, bool zero_status, cudaStream_t st) {
  if (n <= kFusedMaxEntries) {
    // one launch; its per-warp counts take 32*E int32 of shared memory
    const size_t fsmem = sizeof(int32_t) * kFusedWarps * E;
    // the shared-memory attribute is set once per device and context
    static std::atomic<uint64_t> ready[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    const uint64_t ctx = current_context_id();
    if (ctx == 0 || ready[dev].load(std::memory_order_acquire) != ctx) {
      const cudaError_t e = cudaFuncSetAttribute(
          route_fused_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
          (int)(sizeof(int32_t) * kFusedWarps * 1024));
      if (e != cudaSuccess) return e;
      ready[dev].store(ctx, std::memory_order_release);
    }
    route_fused_kernel<<<1, 1024, fsmem, st>>>(ids, n, E, counts, offsets, order, tiles, ntiles,
                                               row_src, dst_of, status, zero_status ? 1 : 0);
    count_launch();
    return cudaGetLastError();
  }
  if (zero_status) {
    const cudaError_t e = cudaMemsetAsync(status, 0, sizeof(int32_t), st);
    if (e != cudaSuccess) return e;
  }
  const int nchunks = route_chunks(n);
  const int grid = (nchunks + kRouteWarps - 1) / kRouteWarps;
  const size_t smem = sizeof(int32_t) * kRouteWarps * E;
  if (grid > 0) {
    route_hist_kernel<<<grid, kRouteWarps * 32, smem, st>>>(ids, n, E, nchunks, hist, status);
    count_launch();
  }
  route_scan_kernel<<<1, 1024, 0, st>>>(hist, nchunks, E, counts, offsets, order, tiles,
                                        ntiles);
  count_launch();
  if (grid > 0) {
    route_scatter_kernel<<<grid, kRouteWarps * 32, smem, st>>>(ids, n, E, nchunks, hist,
                                                                row_src, dst_of);
    count_launch();
  }
  return cudaGetLastError();
}


// ------------------------------------------------------------------------
// Routing without caller-provided scratch (moe_route_noalloc).
//
// Some callers cannot allocate device memory at the point where they route
// a batch: code running inside another framework's allocator-free region,
// or a host that only hands over its own input and output buffers.  For
// them the routing step's scratch (the per-chunk histogram, the expert order
// and the tile list) lives in this fixed array instead of in a workspace.
// Every GPU that loads the library keeps it (1 MiB) until the process exits.
// All calls share it, so calls whose work overlaps on the GPU race.
namespace {

constexpr int64_t kNoAllocScratchInts = 1 << 18;  // 1 MiB of int32
static __device__ __align__(256) int32_t g_route_scratch[kNoAllocScratchInts];

// layout in ints: [0] status bits, [1..2] the tile counts ([4..7] zeroed with
// them), [64..] expert order, then the tile list (int4), then the chunk
// histogram
struct NoAllocLayout {
  int64_t order, tiles, hist, total;
};
NoAllocLayout noalloc_layout(int64_t n, int E) {
  NoAllocLayout L;
  L.order = 64;
  L.tiles = (L.order + E + 3) & ~(int64_t)3;  // 16-byte aligned
  L.hist = L.tiles + 4 * max_tiles(n, E);
  L.total = L.hist + route_hist_rows(n) * E;
  return L;
}

// Device address of the scratch array in the current device's context,
// looked up on every call with that device current (a lookup is cheap, and
// an address kept from an earlier context would dangle after
// cudaDeviceReset).  The host-side name of the array is only a stand-in and
// must never be handed to a kernel.
int32_t* noalloc_scratch(int* err) {
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_route_scratch) != cudaSuccess || !p) {
    cudaGetLastError();
    *err = MOE_ERR_LAUNCH;
    return nullptr;
  }
  return static_cast<int32_t*>(p);
}

}  // namespace
}  // namespace moe

extern "C" int moe_route_noalloc(const MoeLayerDesc* desc, const int32_t* topk_ids,
                                 int32_t* counts, int32_t* offsets, int32_t* row_src,
                                 int32_t* dst_of, moe_stream_t stream) {
  using namespace moe;
  if (!desc) return MOE_ERR_NULL;
  if (desc->T < 0 || desc->E < 1 || desc->E > 1024 || desc->k < 1 || desc->k > desc->E ||
      (int64_t)desc->T * desc->k >= ((int64_t)1 << 24))
    return MOE_ERR_SHAPE;
  const int64_t n = (int64_t)desc->T * desc->k;
  if (!counts || !offsets || (n > 0 && (!topk_ids || !row_src || !dst_of))) return MOE_ERR_NULL;
  const NoAllocLayout L = noalloc_layout(n, desc->E);
  if (L.total > kNoAllocScratchInts) return MOE_ERR_SCRATCH;
  int major = 0, minor = 0, dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
      major != 10 || minor != 3)
    return MOE_ERR_DEVICE;
  int err = MOE_OK;
  int32_t* scratch = noalloc_scratch(&err);
  if (!scratch) return err;
  cudaStream_t st = (cudaStream_t)stream;
  // the status word is accumulated with atomics: start it at zero
  if (cudaMemsetAsync(scratch, 0, sizeof(int32_t), st) != cudaSuccess) return MOE_ERR_LAUNCH;
  const cudaError_t e =
      launch_route(topk_ids, n, desc->E, scratch + L.hist, counts, offsets, scratch + L.order,
                   row_src, dst_of, reinterpret_cast<int4*>(scratch + L.tiles), scratch + 1,
                   scratch, false, st);
  return e == cudaSuccess ? MOE_OK : MOE_ERR_LAUNCH;
}
