// Device-tiled weight pack: a byte permutation of the row-major pack that
// lets the product kernel stage one (256-row tile, 4-block K chunk) with a
// single bulk copy and read each block's codes as an aligned 16-byte word.
//
// Tiled matrix [N_out x K], bpr = K / values-per-block blocks per row:
//   tile t holds NW = min(256, N_out - 256t) rows, at byte 256 * t * bpr * 18:
//     down: rows 256t .. 256t+NW-1;
//     gate/up: gate rows 128t .. 128t+NW/2-1, then the up rows
//     n_ff+128t .. n_ff+128t+NW/2-1 (a tile yields whole blocks of H) --
//     gate row g is row g of the source matrix and up row g is row n_ff+g
//     (split layout), or rows 2g and 2g+1 (interleaved layout);
//   chunk c of a tile covers blocks cb*c .. cb*c+nbc-1 (cb = 4 blocks, 2 for
//     Q8_0), nbc = min(cb, bpr - cb*c), at byte cb * c * NW * BB of the tile
//     (BB = 18 bytes a block, 34 for Q8_0; the tile at 256 * t * bpr * BB);
//   inside a chunk: the CB code bytes (16, or 32 for Q8_0) of (row r, block
//     j) at (j*NW + r)*CB, then the fp16 scales at nbc*NW*CB + (j*NW + r)*2.
// Expert e's gate/up matrix starts at e*(gu_bytes + down_bytes), its down
// matrix gu_bytes later.  Every chunk starts 16-byte aligned.
#include <algorithm>

#include "common.cuh"

namespace moe {
namespace {

struct TileJob {
  const uint8_t* src;
  int64_t src_bytes;
  const int64_t* src_eoff;  // [E][2]
  uint8_t* dst;
  int64_t* dst_eoff;        // [E][2]
  int32_t* status;          // may be null
  int E;
  int gu_layout;            // MOE_GU_*
  int fmt[2];
  int N[2], K[2], bpr[2];
  int64_t mbytes[2];        // bytes of one matrix
};

__global__ void tile_weights_kernel(const TileJob j) {
  const int e = blockIdx.z >> 1, which = blockIdx.z & 1;
  const int bpr = j.bpr[which];
  const int64_t per_expert = j.mbytes[0] + j.mbytes[1];
  const int64_t dbase = (int64_t)e * per_expert + (which ? j.mbytes[0] : 0);
  if (blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0)
    j.dst_eoff[2 * e + which] = dbase;
  const int64_t soff = j.src_eoff[2 * e + which];
  const bool ok = soff >= 0 && (soff & 15) == 0 && soff + j.mbytes[which] <= j.src_bytes;
  if (!ok && blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0 && j.status)
    atomicOr(j.status, MOE_STATUS_BAD_OFFSET);
  // one thread per (row, block)
  const int64_t n = (int64_t)j.N[which] * bpr;
  for (int64_t i = (int64_t)blockIdx.y * blockDim.x * gridDim.x + (int64_t)blockIdx.x * blockDim.x +
                   threadIdx.x;
       i < n; i += (int64_t)blockDim.x * gridDim.x * gridDim.y) {
    const int row = (int)(i / bpr), blk = (int)(i % bpr);
    int t, r;
    if (which == 1) {
      t = row >> 8;
      r = row & 255;
    } else {
      // gate/up: tile t pairs gate rows 128t.. with the up rows n_ff + 128t..
      const int n_ff = j.N[0] >> 1;
      const bool inter = j.gu_layout == MOE_GU_INTERLEAVED;
      const bool up = inter ? (row & 1) : row >= n_ff;
      const int gr = inter ? row >> 1 : (up ? row - n_ff : row);  // gate/up output
      t = gr >> 7;
      r = (gr & 127) + (up ? min(128, n_ff - 128 * t) : 0);
    }
    const int fmt = j.fmt[which];
    const int bb = block_bytes(fmt), cbytes = code_bytes(fmt), cb = chunk_blocks(fmt);
    const int nw = min(256, j.N[which] - 256 * t);
    const int c = blk / cb, jj = blk - c * cb, nbc = min(cb, bpr - cb * c);
    const int64_t chunk = dbase + (int64_t)256 * t * bpr * bb + (int64_t)cb * c * nw * bb;
    uint8_t* codes = j.dst + chunk + ((int64_t)jj * nw + r) * cbytes;
    uint16_t* scale = reinterpret_cast<uint16_t*>(j.dst + chunk + (int64_t)nbc * nw * cbytes +
                                                  ((int64_t)jj * nw + r) * 2);
    // the block's 2-byte words: scale, then the codes (8 or 16 words)
    const uint16_t* s = reinterpret_cast<const uint16_t*>(
        j.src + soff + ((int64_t)row * bpr + blk) * bb);
    *scale = ok ? s[0] : 0;
    for (int q = 0; q < cbytes / 16; q++) {
      uint32_t w[4];
#pragma unroll
      for (int k = 0; k < 4; k++)
        w[k] = ok ? ((uint32_t)s[1 + 8 * q + 2 * k] | ((uint32_t)s[2 + 8 * q + 2 * k] << 16)) : 0u;
      reinterpret_cast<uint4*>(codes)[q] = make_uint4(w[0], w[1], w[2], w[3]);
    }
  }
}

}  // namespace

int64_t tiled_matrix_bytes(int fmt, int N_out, int K) { return (int64_t)N_out * row_bytes(fmt, K); }

int64_t tiled_pack_bytes(const MoeLayerDesc& d) {
  return (int64_t)d.E * (tiled_matrix_bytes(d.gu_fmt, 2 * d.n_ff, d.d) +
                         tiled_matrix_bytes(d.down_fmt, d.d, d.n_ff));
}

cudaError_t launch_tile_weights(const MoeLayerDesc& d, const uint8_t* src, int64_t src_bytes,
                                const int64_t* src_eoff, uint8_t* dst, int64_t* dst_eoff,
                                int32_t* status, cudaStream_t st) {
  TileJob j{};
  j.src = src;
  j.src_bytes = src_bytes;
  j.src_eoff = src_eoff;
  j.dst = dst;
  j.dst_eoff = dst_eoff;
  j.status = status;
  j.E = d.E;
  j.gu_layout = d.gu_layout;
  j.fmt[0] = d.gu_fmt;
  j.fmt[1] = d.down_fmt;
  j.N[0] = 2 * d.n_ff;
  j.K[0] = d.d;
  j.N[1] = d.d;
  j.K[1] = d.n_ff;
  j.bpr[0] = d.d / block_values(d.gu_fmt);
  j.bpr[1] = d.n_ff / block_values(d.down_fmt);
  j.mbytes[0] = tiled_matrix_bytes(d.gu_fmt, j.N[0], j.K[0]);
  j.mbytes[1] = tiled_matrix_bytes(d.down_fmt, j.N[1], j.K[1]);
  const int64_t most = std::max((int64_t)j.N[0] * j.bpr[0], (int64_t)j.N[1] * j.bpr[1]);
  const int threads = 256;
  const int gx = (int)std::min<int64_t>((most + threads - 1) / threads, 64);
  dim3 grid(gx, 1, 2 * d.E);
  tile_weights_kernel<<<grid, threads, 0, st>>>(j);
  count_launch();
  return cudaGetLastError();
}

}  // namespace moe
