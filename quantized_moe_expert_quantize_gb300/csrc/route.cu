// Routing: histogram of the top-k expert ids, exclusive prefix sum, and the
// stable permutation of the T*k flat rows into expert buckets
// ("Strata #3752", commits "moe_ws wiring" and "swiglu_quant landed":
// quantize_scatter, the group bounds uploaded with the layer).
//
// Three small kernels, all integer and bit-exact:
//   1. route_hist    -- one warp per chunk of 1024 flat entries counts the
//                       chunk's rows per expert (shared-memory histogram);
//   2. route_scan    -- one CTA turns the [chunk][expert] counts into the
//                       base row of every (chunk, expert), the expert counts,
//                       their exclusive prefix sum (group bounds), the
//                       largest-first expert order, and the product kernels'
//                       work list: every expert's rows cut into 128-row
//                       tiles, largest expert first, a short remainder cut
//                       into 32-row tiles for the small-row tier;
//   3. route_scatter -- each warp walks its chunk again, 32 entries at a
//                       time; __match_any_sync groups lanes of equal expert,
//                       a lane's rank among them keeps flat order, so rows of
//                       a bucket come out in increasing flat index t*k + r.
#include <mutex>

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
  if (chunk >= nchunks) return;  // whole warp; no CTA barrier below
  for (int e = lane; e < E; e += 32) h[e] = 0;
  __syncwarp();
  const int64_t beg = (int64_t)chunk * kRouteChunk;
  const int64_t end = min(n, beg + kRouteChunk);
  bool bad = false;
  for (int64_t i = beg + lane; i < end; i += 32) {
    const int e = ids[i];
    if ((unsigned)e < (unsigned)E)
      atomicAdd(&h[e], 1);
    else
      bad = true;
  }
  if (bad) atomicOr(status, MOE_STATUS_BAD_EXPERT_ID);
  __syncwarp();
  for (int e = lane; e < E; e += 32) hist[(int64_t)chunk * E + e] = h[e];
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

// One CTA of 1024 threads; thread e owns expert e (E <= 1024).
__global__ void __launch_bounds__(1024)
route_scan_kernel(int32_t* __restrict__ hist, int nchunks, int E,
                  int32_t* __restrict__ counts, int32_t* __restrict__ offsets,
                  int32_t* __restrict__ order, int4* __restrict__ tiles,
                  int32_t* __restrict__ ntiles) {
  __shared__ int32_t s_cnt[1024];    // rows of expert e
  __shared__ int32_t s_tiles[1024];  // tcgen05 tiles of the expert at rank r
  __shared__ int32_t s_small[1024];  // small-row tiles of the expert at rank r
  __shared__ int32_t s_warp[32];
  __shared__ int32_t s_tot[2];       // tcgen05 tiles, small-row tiles
  const int tid = threadIdx.x;
  int run = 0;
  if (tid < E) {
    for (int c = 0; c < nchunks; c++) {
      const int64_t idx = (int64_t)c * E + tid;
      const int v = hist[idx];
      hist[idx] = run;  // rows of expert tid in chunks before c
      run += v;
    }
    counts[tid] = run;
  }
  s_cnt[tid] = run;
  s_tiles[tid] = 0;
  s_small[tid] = 0;
  const int excl = block_excl_scan(run, s_warp);  // also orders s_cnt / s_tiles writes
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
    for (int c = 0; c < nchunks; c++) hist[(int64_t)c * E + tid] += excl;
    // rank by (count descending, id ascending)
    for (int e2 = 0; e2 < E; e2++) {
      const int c2 = s_cnt[e2];
      rank += (c2 > run) || (c2 == run && e2 < tid);
    }
    order[rank] = tid;
    s_tiles[rank] = nbig;
    s_small[rank] = nsm;
  }
  __syncthreads();
  // first tile of each rank in each list (thread tid stands for rank tid here)
  const int nt = s_tiles[tid], ns = s_small[tid];
  const int tbase = block_excl_scan(nt, s_warp);
  const int sbase = block_excl_scan(ns, s_warp);
  if (tid == 1023) {
    s_tot[0] = tbase + nt;
    s_tot[1] = sbase + ns;
    ntiles[0] = tbase + nt + sbase + ns;
    ntiles[1] = tbase + nt;  // the tcgen05 tiles come first
  }
  __syncthreads();
  s_tiles[tid] = tbase;
  s_small[tid] = s_tot[0] + sbase;
  __syncthreads();
  if (tid < E) {
    const int first = s_tiles[rank];
    for (int i = 0; i < nbig; i++)
      tiles[first + i] = make_int4(tid, excl + i * kTileRows, min(kTileRows, run - i * kTileRows), 0);
    const int sfirst = s_small[rank];
    const int r0 = excl + nfull * kTileRows;
    for (int j = 0; j < nsm; j++)
      tiles[sfirst + j] = make_int4(tid, r0 + j * kSmallTileRows,
                                    min(kSmallTileRows, rem - j * kSmallTileRows), 0);
  }
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
  for (int e = lane; e < E; e += 32) h[e] = hist[(int64_t)chunk * E + e];
  __syncwarp();
  const unsigned lt = (1u << lane) - 1u;
  const int64_t beg = (int64_t)chunk * kRouteChunk;
  const int64_t end = min(n, beg + kRouteChunk);
  for (int64_t base = beg; base < end; base += 32) {
    const int64_t i = base + lane;
    const bool act = i < end;
    const int e = act ? ids[i] : -1;
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

}  // namespace

cudaError_t launch_route(const int32_t* ids, int64_t n, int E, int32_t* hist,
                         int32_t* counts, int32_t* offsets, int32_t* order,
                         int32_t* row_src, int32_t* dst_of, int4* tiles, int32_t* ntiles,
                         int32_t* status, cudaStream_t st) {
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

// layout in ints: [0] status bits, [1] tile count, [64..] expert order,
// then the tile list (int4), then the chunk histogram
struct NoAllocLayout {
  int64_t order, tiles, hist, total;
};
NoAllocLayout noalloc_layout(int64_t n, int E) {
  NoAllocLayout L;
  L.order = 64;
  L.tiles = (L.order + E + 3) & ~(int64_t)3;  // 16-byte aligned
  L.hist = L.tiles + 4 * max_tiles(n, E);
  L.total = L.hist + (int64_t)route_chunks(n) * E;
  return L;
}

// Device address of the scratch array on the current device, found once per
// device with that device current.  The host-side name of the array is only
// a stand-in and must never be handed to a kernel.
int32_t* noalloc_scratch(int* err) {
  static std::mutex mu;
  static int32_t* addr[64] = {nullptr};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
    *err = MOE_ERR_DEVICE;
    return nullptr;
  }
  std::lock_guard<std::mutex> lock(mu);
  if (!addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_route_scratch) != cudaSuccess || !p) {
      *err = MOE_ERR_LAUNCH;
      return nullptr;
    }
    addr[dev] = static_cast<int32_t*>(p);
  }
  return addr[dev];
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
                   scratch, st);
  return e == cudaSuccess ? MOE_OK : MOE_ERR_LAUNCH;
}
