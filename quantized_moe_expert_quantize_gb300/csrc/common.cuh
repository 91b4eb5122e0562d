// Shared device/host helpers of the CUDA library (not of the oracle).
#pragma once
#include <cstdint>
#include <cstddef>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "moe_prefill.h"

namespace moe {

// ---------------------------------------------------------------- formats
constexpr int kBlockBytes = 18;       // W2 and W4NL blocks are 18 bytes
constexpr int kQ8Bytes = 34;          // Q8_0 blocks: fp16 d + 32 int8 codes
constexpr int kW2Values = 64;         // values per W2 block
constexpr int kW4Values = 32;         // values per W4NL (and Q8_0) block
constexpr int kQBlock = 32;           // q8 block of activations

// Row stride (in floats) of a q8 scale matrix [rows x K/32]: padded to a
// multiple of 4 so every row starts 16-byte aligned (tensor-map rule).
__host__ __device__ inline int scale_stride(int K) { return ((K / 32) + 3) & ~3; }

__host__ __device__ constexpr int block_values(int fmt) { return fmt == MOE_FMT_W2 ? kW2Values : kW4Values; }
__host__ __device__ constexpr int block_bytes(int fmt) { return fmt == MOE_FMT_Q8_0 ? kQ8Bytes : kBlockBytes; }
__host__ __device__ constexpr int code_bytes(int fmt) { return block_bytes(fmt) - 2; }
// Blocks per chunk of the tiled pack: a 256-row chunk stays within 18 KB.
__host__ __device__ constexpr int chunk_blocks(int fmt) { return fmt == MOE_FMT_Q8_0 ? 2 : 4; }
__host__ __device__ inline int64_t row_bytes(int fmt, int K) {
  return (int64_t)(K / block_values(fmt)) * block_bytes(fmt);
}

// fp16 bit patterns of the integers -2..1 (W2 codes 0..3 minus 2).
constexpr uint64_t kW2HalfLut = 0x3C000000BC00C000ull;

// fp16 bit patterns of the W4NL table {-127,-104,-83,-65,-49,-35,-22,-10,
// 1,13,25,38,53,69,89,113} (exact: every entry has at most 7 significant bits).
__constant__ const uint16_t c_nl4_half[16] = {
    0xD7F0, 0xD680, 0xD530, 0xD410, 0xD220, 0xD060, 0xCD80, 0xC900,
    0x3C00, 0x4A80, 0x4E40, 0x50C0, 0x52A0, 0x5450, 0x5590, 0x5710};

// ------------------------------------------------------------- launch count
void count_launch(int n = 1);

// -------------------------------------------------------------- route
constexpr int kRouteChunk = 1024;  // flat entries per warp
constexpr int kRouteWarps = 8;     // warps per CTA
inline int route_chunks(int64_t n) { return (int)((n + kRouteChunk - 1) / kRouteChunk); }
// rows of E int32 the multi-launch routing keeps: one per chunk (the chunk's
// first row in each expert within its CTA), then one per CTA of chunks
inline int64_t route_hist_rows(int64_t n) {
  const int c = route_chunks(n);
  return (int64_t)c + (c + kRouteWarps - 1) / kRouteWarps;
}

// Routed-row tiles of the product kernels.  Every expert's rows are cut
// into tiles of kTileRows rows for the tcgen05 kernel; what is left after
// its full tiles (rows % kTileRows) goes to the small-row tier in tiles of
// at most kSmallTileRows rows when it is at most kSmallSplit rows, else it is
// one more (partial) tcgen05 tile.  A partial tcgen05 tile costs as much as a
// full one; a small-row tile costs about in proportion to its rows.
constexpr int kTileRows = 128;
constexpr int kSmallTileRows = 32;
constexpr int kSmallSplit = 32;
static_assert(kSmallSplit % kSmallTileRows == 0 && kSmallSplit < kTileRows, "split rule");
__host__ __device__ inline int64_t max_tiles(int64_t rows, int E) {
  return rows / kTileRows + (int64_t)E * (1 + kSmallSplit / kSmallTileRows) + 1;
}

// tiles: int4 {expert, first routed row, rows, 0} [max_tiles]; ntiles: int32
// [2] = {all tiles, tcgen05 tiles}.  The tcgen05 tiles come first, experts in
// largest-first order; the small-row tiles are the tail [ntiles[1], ntiles[0]).
// zero_status: the status word starts at zero (inside the one-launch routing,
// a memset before the multi-launch one).
cudaError_t launch_route(const int32_t* ids, int64_t n, int E, int32_t* hist,
                         int32_t* counts, int32_t* offsets, int32_t* order,
                         int32_t* row_src, int32_t* dst_of, int4* tiles, int32_t* ntiles,
                         int32_t* status, bool zero_status, cudaStream_t st);

// ---------------------------------------------------- elementwise kernels
// q8 of x [T x K], scattered to routed rows: q [rows_max x K],
// d [rows_max x scale_stride(K)]
cudaError_t launch_quant_q8(const float* x, int64_t T, int K, int k, const int32_t* dst_of,
                            int64_t rows_max, __half* q, float* d, cudaStream_t st);
// swiglu + q8 of GU [rows x 2 n_ff] (gate/up columns in layout gu_layout):
// hq [rows_max x n_ff], dh [rows_max x scale_stride(n_ff)]
cudaError_t launch_swiglu_quant(const float* gu, const int32_t* nrows_dev, int64_t rows_max,
                                int n_ff, int gu_layout, __half* hq, float* dh, cudaStream_t st);
// tokens [t0, t0 + T) of the combine; rows_max bounds dst_of's row indices
cudaError_t launch_combine(const float* topk_w, const int32_t* dst_of, const float* dm,
                           int64_t t0, int64_t T, int k, int d, int64_t rows_max, float* out,
                           cudaStream_t st);

// ------------------------------------------------------------ products
// The combine fused into the down product's epilogue (when out is set): the
// last of a token's rows to finish a 32-column group of Dm sums the token's
// k rows in rank order into out [T x N_out].
struct CombineArgs {
  float* out;
  const float* topk_w;       // [T x k]
  const int32_t* dst_of;     // [T*k] flat entry -> routed row (-1: dropped)
  const int32_t* row_src;    // [rows] routed row -> flat entry
  int32_t* cnt;              // [T x N_out/32] arrivals per (token, group)
  int k;
};

struct GemmArgs {
  const uint8_t* pack;       // device-tiled weight pack
  const int64_t* eoff;       // [E][2] byte offsets in the tiled pack
  int which;                 // 0 = gate/up, 1 = down
  int fmt;                   // MOE_FMT_*
  int64_t pack_bytes;
  const int4* tiles;         // routed-row tiles, largest expert first
  const int32_t* ntiles;
  int E;
  const __half* act;         // activation values [rows_max x K] (exact fp16 integers, routed-row order)
  const float* act_d;        // activation scales [rows_max x scale_stride(K)]
  int K;                     // reduction length
  int N_out;                 // output columns (weight rows)
  float* out;                // [rows x N_out] (unused when hq is set); gate/up
                             //   columns in layout gu_layout
  int gu_layout;             // MOE_GU_*
  __half* hq;                // gate/up only: if set, swiglu_quant is fused and Hq / dh
  float* dh;                 //   are written instead of GU
  int64_t rows_max;          // capacity of the routed-row buffers (T*k)
  int32_t* status;
  int32_t* sched;            // small-row launch: {next item, CTAs done}, zeroed by routing
  CombineArgs comb;          // down only: the combine fused into the epilogue
};

// The fused combine's per-(token, 32-column group) arrival counters start
// at the token's count of dropped ranks, so that the last of its valid rows
// is the one that sees k - 1.
cudaError_t launch_combine_init(const int32_t* dst_of, int64_t T, int k, int groups,
                                int32_t* cnt, cudaStream_t st);

// Sum of a token's k rows of Dm over one 32-column group in rank order (one
// fma per rank, from 0), into out: the combine's arithmetic, run by the last
// row to arrive.  Dm is read through L2 (other SMs wrote it).
__device__ __forceinline__ void combine_group32(const float* __restrict__ dm, int64_t rows_max,
                                                int N_out, const float* __restrict__ topk_w,
                                                const int32_t* __restrict__ dst_of, int64_t t, int k,
                                                int col0, float* __restrict__ out) {
  float4 acc[8];
#pragma unroll
  for (int j = 0; j < 8; j++) acc[j] = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int r = 0; r < k; r++) {
    const int32_t pos = __ldcg(dst_of + t * k + r);
    if (pos < 0 || pos >= rows_max) continue;  // dropped row
    const float w = __ldcg(topk_w + t * k + r);
    const float4* src = reinterpret_cast<const float4*>(dm + (int64_t)pos * N_out + col0);
#pragma unroll
    for (int j = 0; j < 8; j++) {
      const float4 v = __ldcg(src + j);
      acc[j].x = fmaf(w, v.x, acc[j].x);
      acc[j].y = fmaf(w, v.y, acc[j].y);
      acc[j].z = fmaf(w, v.z, acc[j].z);
      acc[j].w = fmaf(w, v.w, acc[j].w);
    }
  }
  float4* dst = reinterpret_cast<float4*>(out + t * N_out + col0);
#pragma unroll
  for (int j = 0; j < 8; j++) dst[j] = acc[j];
}

// A routed row's arrival for its token's 32-column group starting at col0
// of Dm [rows_max x N_out], after its values of the group are stored (by
// this thread, or by its warp before a __syncwarp): fence, count in, and
// combine the group if it is the last of the token's rows.
__device__ __forceinline__ void combine_arrive(const CombineArgs& c, const float* dm,
                                               int64_t rows_max, int N_out, int64_t row, int col0) {
  const int32_t src = __ldcg(c.row_src + row);
  if (src < 0 || src >= rows_max) return;
  const int64_t t = src / c.k;
  __threadfence();
  const int old = atomicAdd(c.cnt + t * (N_out / 32) + col0 / 32, 1);
  if (old == c.k - 1) {
    __threadfence();
    combine_group32(dm, rows_max, N_out, c.topk_w, c.dst_of, t, c.k, col0, c.out);
  }
}
bool tc_supported(const MoeLayerDesc& d);
// tcgen05 kernel: the tiles [0, ntiles[1])
cudaError_t launch_gemm_tc(const GemmArgs& a, cudaStream_t st);
// small-row tier: the tiles [ntiles[1], ntiles[0]) (<= kSmallTileRows rows each)
cudaError_t launch_gemm_small(const GemmArgs& a, cudaStream_t st);

// ------------------------------------------------------- tiled weight pack
int64_t tiled_matrix_bytes(int fmt, int N_out, int K);
int64_t tiled_pack_bytes(const MoeLayerDesc& d);
cudaError_t launch_tile_weights(const MoeLayerDesc& d, const uint8_t* src, int64_t src_bytes,
                                const int64_t* src_eoff, uint8_t* dst, int64_t* dst_eoff,
                                int32_t* status, cudaStream_t st);

int device_sm_count();

// Identity of the current CUDA context (cuCtxGetId), 0 if there is none.
// One-time set-up per device (kernel attributes, the side stream) is keyed
// on it, so that it is redone in a new context after cudaDeviceReset.
uint64_t current_context_id();

}  // namespace moe
