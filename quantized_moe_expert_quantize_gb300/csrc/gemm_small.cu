// Small-row tier of the grouped expert products: tiles of at most
// kSmallTileRows (32) routed rows -- experts with few rows, and the short
// remainder of every expert after its full 128-row tiles.
//
// Same arithmetic as the tcgen05 kernel -- per 32-value K block the exact
// integer sum of w_int * q, then the fp32 epilogue in K order ("Strata #3752",
// commit "moe_ws kernels") -- on a different tile shape.  With a handful of
// rows per expert the work is a weight stream: each expert's weight tile is
// read for a few rows (the pages tune a separate tier by rows per expert,
// "Strata #3752", addendum).  A 128-row tcgen05 tile would compute mostly
// padding at the cost of a full one; here the weights are the M side of
// mma.sync.m16n8k16, decoded into fp16 fragments in registers, and the routed
// rows are its N side (1 to 4 fragments of 8), with fp32 accumulators in
// registers.  The A values are exact fp16 integers (W2: c-2, or 256*(c-2)
// against B values pre-scaled by 1/256; W4NL: the table; Q8_0: the code) and
// the B values the q8 integers, so every product and every 32-value block
// sum is exact in fp32; the weight scale enters in the epilogue, where
// d_w * isum is exact for W2.
//
// Item: one small-row tile of the work list against one 256-row tile of the
// tiled weight pack.  8 warps own 32 tile rows each (2 m16 fragments; for
// gate/up, 16 gate rows and the matching up rows).  Two CTAs run on each
// multiprocessor.  A 3-slot ring holds per slot one weight chunk (one bulk
// copy) and the tile's activation rows and scales (2-D TMA boxes of 16 rows);
// lane 0 of warp 0 refills a slot once all 8 warps have released it.
//
// The routed rows' activations are stored pair-interleaved in every 16-value
// group (position 2i holds value i, 2i+1 holds value i+8).  Taking the MMA's
// k as the stored position, a lane's A-fragment pairs are the weights of
// values (c, c+8) and (c+4, c+12) of a group -- pairs that one code word
// yields with one mask each -- and its B fragments come from ldmatrix on the
// 128-byte-swizzled activation boxes.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
#include <mutex>

#include "common.cuh"
#include "sm100_ptx.cuh"

namespace moe {
namespace {

using namespace ptx;

constexpr int kTN = 256;           // weight rows per item (one tile of the tiled pack)
constexpr int kWarps = 8;          // warps, 32 tile rows each (warp 0 also loads the ring)
constexpr int kThreads = kWarps * 32;
constexpr int kSlots = 3;
constexpr int kRows = kSmallTileRows;  // routed rows per small tile (MMA N: up to 4 n8 fragments)
constexpr int kBoxRows = 16;           // rows per activation box (one or two boxes per tile)
// weight blocks per chunk of the tiled pack: chunk_blocks(format) -- 4, or 2
// for Q8_0; a 256-row chunk stays within 18 KB
constexpr int kChunkVals = 256;    // K values per activation box (a W2 chunk; a W4NL chunk uses 128)
constexpr int kRawBytes = 4 * kTN * kBlockBytes;              // 18,432
static_assert(chunk_blocks(MOE_FMT_Q8_0) * kTN * kQ8Bytes <= kRawBytes, "Q8_0 chunk fits a slot");
// scales per row of an activation-scale box: a chunk's q8 blocks, at least 4
// (a TMA box row is a multiple of 16 bytes and starts 16-byte aligned: a
// 2-block Q8_0 chunk takes the aligned box of 4 holding its two scales)
__host__ __device__ constexpr int dx_width(int fmt) {
  return chunk_blocks(fmt) * block_values(fmt) / 32 > 4 ? chunk_blocks(fmt) * block_values(fmt) / 32
                                                        : 4;
}
constexpr int kActBytes = kRows * kChunkVals * 2;       // 16,384: 32 rows x 256 fp16
constexpr int kDxBytes = kRows * (kChunkVals / 32) * 4;  // 1,024: 32 rows x 8 scales
// slots 1024-byte aligned: the activation boxes use the 128-byte swizzle
constexpr int kSlotBytes = (kRawBytes + kActBytes + kDxBytes + 1023) & ~1023;
constexpr int kActBox = 64;                                  // values per activation box (128 B)
constexpr int kOffBar = kSlots * kSlotBytes;  // full[kSlots] mbarriers
constexpr int kOffRel = kOffBar + kSlots * 8;  // per slot: warps done with it (int, 8 B apart)
constexpr int kOffMisc = kOffBar + 2 * kSlots * 8;
// misc: abort flag (+0), W4NL table (+64), warp-pair barriers [2][kWarps/2]
// (+128), the ring producer's state (+192); then the warp-pair amax exchange
// [2][kWarps][kRows] fp32
constexpr int kOffAmax = kOffMisc + 256;
// the dp4a path (W2 tiles of at most kDp4aRows rows, see item_dp4a): the
// chunk's activations as int8 words [2 buffers][kDp4aRows rows][64 words],
// their 32-value sums [2][kDp4aRows][8], the up rows of the fused
// swiglu_quant [kDp4aRows][128] fp32, and its mbarriers (chunk buffers [2],
// up exchange)
constexpr int kDp4aRows = 4;
constexpr int kOffConv = kOffAmax + 2 * kWarps * kRows * 4;
constexpr int kOffConvSum = kOffConv + 2 * kDp4aRows * 64 * 4;
constexpr int kOffUp = kOffConvSum + 2 * kDp4aRows * 8 * 4;
constexpr int kOffDbar = kOffUp + kDp4aRows * (kTN / 2) * 4;
// per slot, written by the ring producer with the slot's item: {first routed
// row, rows, weight tile, its rows}
constexpr int kOffInfo = kOffDbar + 64;
constexpr int kSmemBytes = kOffInfo + kSlots * 16 + 1024;  // + alignment slack
constexpr uint64_t kTimeoutNs = 1000000000ull;
constexpr int kModeGU = 0, kModeSwiglu = 1, kModeDown = 2;
static_assert(kSlotBytes % 1024 == 0 && kRawBytes % 1024 == 0, "swizzled boxes 1024-byte aligned");
static_assert(kRows == 2 * kBoxRows && kRows == 32, "a tile is one or two activation boxes");
// two CTAs a multiprocessor: 16 warps, 4 per sub-partition, 128 registers each
static_assert(kSmemBytes + 1024 <= 233472 / 2, "two CTAs a multiprocessor");
constexpr int kMaxRegs = 65536 / (2 * kThreads);
static_assert(kMaxRegs == 128, "register cap");

struct SmArgs {
  const uint8_t* pack;
  const int64_t* eoff;
  int which;
  int64_t pack_bytes;
  const int4* tiles;
  const int32_t* ntiles;  // {tiles, big-expert tiles}
  int E;
  int K, N_out, bpr, bb;  // bb: bytes per weight block
  float* out;
  int gu_layout;
  __half* hq;
  float* dh;
  int64_t rows_max;
  int32_t* status;
  int32_t* sched;    // {next item, CTAs done}: zero at launch (see prod_seek)
  CombineArgs comb;  // down: the combine fused into the epilogue (comb.out set)
};

__device__ __forceinline__ uint32_t hsub2_u32(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}
__device__ __forceinline__ uint32_t hmul2_u32(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}
// Four 8x8 b16 matrices from shared memory; lanes 8m..8m+7 give the row
// addresses of matrix m, and lane (g, cq) receives row g, pair cq of each.
__device__ __forceinline__ void ldsm_x4(uint32_t saddr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(saddr));
}
// D = A(16x16, row) * B(16x8, col) + D, fp16 operands, fp32 accumulate.
__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
// D = A * B + C.
__device__ __forceinline__ void mma16816c(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                          uint32_t b1, const float (&c)[4]) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%10,%11,%12,%13};"
      : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(c[0]), "f"(c[1]),
        "f"(c[2]), "f"(c[3]));
}

// W2 fragments.  ws is a code word shifted right by 2*cq (codes of values
// cq, cq+4, cq+8, cq+12 of the group at bits 0, 8, 16, 24).  Pair lo:
// (c_cq - 2, c_{cq+8} - 2); pair hi: 256 * (c_{cq+4} - 2, c_{cq+12} - 2) --
// the codes dropped into the mantissas of 1024 (one logic op) and the offset
// subtracted, exact.  The B pairs facing pair hi are pre-scaled by 1/256
// (exact for |q| <= 127), so every product is the integer (c - 2) * q.
__device__ __forceinline__ uint32_t w2_pair_lo(uint32_t ws) {
  return hsub2_u32((ws & 0x00030003u) | 0x64006400u, 0x64026402u);  // (1024 + c) - 1026
}
__device__ __forceinline__ uint32_t w2_pair_hi(uint32_t ws) {
  return hsub2_u32((ws & 0x03000300u) | 0x64006400u, 0x66006600u);  // (1024 + 256c) - 1536
}
constexpr uint32_t kHalfInv256 = 0x1C001C00u;  // fp16 pair (1/256, 1/256)
// Q8_0: the fp16 pair (q_n, q_{n+8}) of two code words: byte sel selects code
// n of lo and code n+8 of hi into bytes 0 and 2; each byte, sign bit flipped,
// becomes the low mantissa byte of 1024 + 128 + q, and 1152 comes off: exact.
__device__ __forceinline__ uint32_t q8_pair(uint32_t lo, uint32_t hi, uint32_t sel) {
  const uint32_t t = __byte_perm(lo, hi, sel);
  return hsub2_u32((t & 0x00FF00FFu) ^ 0x64806480u, 0x64806480u);
}
// W4NL: the fp16 pair (T[idx_i], T[idx_{i+8}]) from the group's two words.
__device__ __forceinline__ uint32_t w4_pair(uint32_t wlo, uint32_t whi, int i,
                                            const uint16_t* lut) {
  return (uint32_t)lut[(wlo >> (4 * i)) & 15u] | ((uint32_t)lut[(whi >> (4 * i)) & 15u] << 16);
}

// Shared-memory loads at 32-bit shared addresses (volatile: they read bytes
// that a TMA wrote after the mbarrier wait before them).
__device__ __forceinline__ uint2 lds64(uint32_t a) {
  uint2 v;
  asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(a));
  return v;
}
__device__ __forceinline__ uint4 lds128(uint32_t a) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(a));
  return v;
}
__device__ __forceinline__ float lds_f32(uint32_t a) {
  float v;
  asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(a));
  return v;
}
__device__ __forceinline__ float lds_half_as_f32(uint32_t a) {
  unsigned short h;
  asm volatile("ld.shared.u16 %0, [%1];" : "=h"(h) : "r"(a));
  return __half2float(__ushort_as_half(h));
}

// One item's products: every chunk of the item's weight tile against its
// (up to 8 * NNT) routed rows, accumulated per 32-value block in K order into
// acc (m16 fragment mt = tile rows rbase[mt]..+15, n8 fragment nt).  Tile
// rows past the tile's end compute garbage from in-slot bytes and are never
// stored.  Every shared-memory address is a per-lane offset, fixed for the
// item, plus a per-chunk base advanced once a block.
template <int FMT, int NNT, typename Refill>
__device__ __forceinline__ bool consume_item(const uint8_t* smem, uint64_t* full,
                                             volatile int* s_abort, uint32_t& cc, int nchunks,
                                             int bpr, int nw, const int (&rbase)[2],
                                             const uint16_t* s_lut, int lane,
                                             float (&acc)[2][4][4], Refill&& refill) {
  constexpr bool kW2 = (FMT == MOE_FMT_W2);
  constexpr int kBv = kW2 ? 64 : 32;        // values per weight block
  constexpr int kCB = chunk_blocks(FMT);     // weight blocks per chunk
  constexpr int kCode = code_bytes(FMT);     // code bytes per (row, block)
  constexpr int kVals = kCB * kBv;           // K values per chunk
  constexpr int kDxW = dx_width(FMT);        // scales per dx row in the slot
  constexpr int kQpb = kBv / 32;             // q8 blocks per weight block
  constexpr uint32_t kBoxBytes = kRows * kActBox * 2;  // one 64-value activation box
  const int g = lane >> 2, cq = lane & 3;
  // ldmatrix: lanes 8m..8m+7 give rows 0..7 of matrix m; matrix 2ks + hf is
  // stored positions 8hf..8hf+7 of group 2qb + ks: 16-byte chunk m + 4(qb&1)
  // of the row in box qb/2, before the 128-byte swizzle
  const int lm = lane >> 3, lr = lane & 7;
  const uint32_t bsw0 = (uint32_t)(lr * 128 + ((lm ^ lr) << 4));
  const uint32_t bsw1 = (uint32_t)(lr * 128 + (((lm + 4) ^ lr) << 4));
  // this lane's tile rows rbase[mt] + g (+8 for h = 1): code and scale offsets
  const uint32_t rc0 = (uint32_t)((rbase[0] + g) * kCode), rc1 = (uint32_t)((rbase[1] + g) * kCode);
  const uint32_t rs0 = (uint32_t)((rbase[0] + g) * 2), rs1 = (uint32_t)((rbase[1] + g) * 2);
  const uint32_t dxl = (uint32_t)(2 * cq * kDxW * 4);  // routed row 2cq of the dx box
  const uint32_t codes_step = (uint32_t)(nw * kCode), scales_step = (uint32_t)(nw * 2);
  const uint32_t smem_s = smem_u32(smem);
  const float zero[4] = {0.0f, 0.0f, 0.0f, 0.0f};
  for (int c = 0; c < nchunks; c++, cc++) {
    const uint32_t slot = cc % kSlots;
    if (!mbar_wait(&full[slot], (cc / kSlots) & 1, s_abort, kTimeoutNs, false)) return false;
    const uint32_t sp = smem_s + slot * kSlotBytes;
    const int nbc = min(kCB, bpr - c * kCB);
    const int dxo = (c * (kVals / 32)) & 3;  // this chunk's first scale in the dx box
    uint32_t cj = sp;                                        // block j's code records
    uint32_t sj = sp + (uint32_t)(nbc * nw * kCode);         // and fp16 scales
    const uint32_t act = sp + kRawBytes;                     // [box][32 rows][128 B], swizzled
    uint32_t dxj = sp + kRawBytes + kActBytes + dxl + (uint32_t)(dxo * 4);  // q8 block j*kQpb
#pragma unroll 1
    for (int j = 0; j < nbc; j++, cj += codes_step, sj += scales_step, dxj += 4 * kQpb) {
      float dw[2][2];  // scale of weight block j, tile rows rbase+g / +8
      dw[0][0] = lds_half_as_f32(sj + rs0);
      dw[0][1] = lds_half_as_f32(sj + rs0 + 16);
      dw[1][0] = lds_half_as_f32(sj + rs1);
      dw[1][1] = lds_half_as_f32(sj + rs1 + 16);
#pragma unroll
      for (int qq = 0; qq < kQpb; qq++) {
        const int qb = j * kQpb + qq;  // q8 block within the chunk
        // B fragments, one ldmatrix.x4 per n8 fragment (routed rows
        // 8nt..8nt+7): lane (g, cq) receives b[ks][nt][hf]
        uint32_t b[2][NNT][2];
        float dx[NNT][2];  // activation scales of routed rows 8nt + 2cq, +1
        const uint32_t bsrc =
            kQpb == 2 ? act + (uint32_t)j * kBoxBytes + (qq ? bsw1 : bsw0)
                      : act + (uint32_t)(qb >> 1) * kBoxBytes + ((qb & 1) ? bsw1 : bsw0);
#pragma unroll
        for (int nt = 0; nt < NNT; nt++) {
          ldsm_x4(bsrc + nt * 8 * 128, b[0][nt][0], b[0][nt][1], b[1][nt][0], b[1][nt][1]);
          if (kW2) {
            b[0][nt][1] = hmul2_u32(b[0][nt][1], kHalfInv256);
            b[1][nt][1] = hmul2_u32(b[1][nt][1], kHalfInv256);
          }
          dx[nt][0] = lds_f32(dxj + 4 * qq + nt * 8 * kDxW * 4);
          dx[nt][1] = lds_f32(dxj + 4 * qq + nt * 8 * kDxW * 4 + kDxW * 4);
        }
#pragma unroll
        for (int mt = 0; mt < 2; mt++) {
          // A fragments of both 16-value groups of the block
          uint32_t af[2][4];
          const uint32_t wrow = cj + (mt ? rc1 : rc0);
#pragma unroll
          for (int h = 0; h < 2; h++) {
            const uint32_t wr = wrow + h * 8 * kCode;
            if (kW2) {
              // code words of groups 2qq, 2qq+1 of the block
              const uint2 w = lds64(wr + 8 * qq);
              const uint32_t ws0 = w.x >> (2 * cq), ws1 = w.y >> (2 * cq);
              af[0][h] = w2_pair_lo(ws0);
              af[0][2 + h] = w2_pair_hi(ws0);
              af[1][h] = w2_pair_lo(ws1);
              af[1][2 + h] = w2_pair_hi(ws1);
            } else if (FMT == MOE_FMT_Q8_0) {
              // group ks = words 4ks..4ks+3: values cq, cq+8 in words 4ks, 4ks+2
              // and cq+4, cq+12 in words 4ks+1, 4ks+3, byte cq of each
              const uint4 w0 = lds128(wr), w1 = lds128(wr + 16);
              const uint32_t sel = (uint32_t)(cq | (cq << 4) | ((4 + cq) << 8) | ((4 + cq) << 12));
              af[0][h] = q8_pair(w0.x, w0.z, sel);
              af[0][2 + h] = q8_pair(w0.y, w0.w, sel);
              af[1][h] = q8_pair(w1.x, w1.z, sel);
              af[1][2 + h] = q8_pair(w1.y, w1.w, sel);
            } else {
              const uint4 w = lds128(wr);
              af[0][h] = w4_pair(w.x, w.y, cq, s_lut);
              af[0][2 + h] = w4_pair(w.x, w.y, cq + 4, s_lut);
              af[1][h] = w4_pair(w.z, w.w, cq, s_lut);
              af[1][2 + h] = w4_pair(w.z, w.w, cq + 4, s_lut);
            }
          }
#pragma unroll
          for (int nt = 0; nt < NNT; nt++) {
            float p[4];  // the block's integer sums
            mma16816c(p, af[0], b[0][nt][0], b[0][nt][1], zero);
            mma16816(p, af[1], b[1][nt][0], b[1][nt][1]);
            // epilogue of the block, in K order: acc += d_x * (d_w * isum)
            // (W2, d_w * isum exact) or acc += (d_w * d_x) * isum (W4NL)
#pragma unroll
            for (int i = 0; i < 4; i++) {
              const float dxi = dx[nt][i & 1];
              const float dwr = dw[mt][i >> 1];
              acc[mt][nt][i] = kW2 ? __fmaf_rn(dxi, __fmul_rn(dwr, p[i]), acc[mt][nt][i])
                                   : __fmaf_rn(__fmul_rn(dwr, dxi), p[i], acc[mt][nt][i]);
            }
          }
        }
      }
    }
    refill(cc);
  }
  return true;
}

__device__ __forceinline__ void sts32(uint32_t a, uint32_t v) {
  asm volatile("st.shared.u32 [%0], %1;" ::"r"(a), "r"(v) : "memory");
}
__device__ __forceinline__ uint32_t lds32(uint32_t a) {
  uint32_t v;
  asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(a));
  return v;
}
__device__ __forceinline__ uint32_t hadd2_u32(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("add.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

// One W2 item of U <= kDp4aRows routed rows on the integer dot-product
// units instead of the tensor cores.  With so few rows an m16n8k16 MMA is at
// most half used (its N side is 8 rows) and each lane still decodes its
// share of every weight value into fp16; dp4a takes four 2-bit codes, each
// in a byte, against four int8 activations, so a code word decodes with a
// shift and a mask per four values and no fp16 step.
//
// Thread tid owns tile row tid (gate/up: gate rows below nw/2, the matching
// up rows above; down: output column 256*wt + tid).  Per chunk the CTA first
// turns the U activation rows of the slot (fp16 integers, stored
// pair-interleaved and 128-byte swizzled) into int8 words in the order the
// codes come out of a word -- word s of group G holds values 16G + s, +4, +8,
// +12 -- together with each 32-value block's sum of q (one word per thread,
// all warps, an mbarrier of all warps publishes them; two buffers by chunk).
// Then each thread, per 64-value W2 block of its row: the four code words,
// each shifted by 2s and masked to bytes (c in 0..3), dp4a against the
// activation words of every row; per 32-value block the exact integer
// isum = sum(c q) - 2 sum(q) = sum((c - 2) q), and the same epilogue as the
// tensor-core paths, acc += d_x * (d_w * isum) with d_w * isum exact: the
// bits equal the m16n8k16 path's.
template <int MODE, int U, typename Refill>
__device__ __forceinline__ bool item_dp4a(const SmArgs& a, const uint8_t* smem, uint64_t* full,
                                          uint64_t* cbar, uint64_t* ubar,
                                          volatile int* s_abort, uint32_t& cc, uint32_t& dc,
                                          uint32_t& uc, int nchunks, int nw, int4 t, int wt,
                                          Refill&& refill) {
  constexpr int kCB = chunk_blocks(MOE_FMT_W2);  // 4 W2 blocks (256 values) a chunk
  constexpr int kCode = code_bytes(MOE_FMT_W2);  // 16
  constexpr int kDxW = dx_width(MOE_FMT_W2);     // 8 scales a row of the dx box
  constexpr uint32_t kBoxBytes = kRows * kActBox * 2;
  static_assert(kCB * 64 == kChunkVals && kDxW == 8, "a W2 chunk is 8 q8 blocks");
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const uint32_t smem_s = smem_u32(smem);
  const uint32_t conv_s = smem_s + kOffConv, csum_s = smem_s + kOffConvSum;
  float acc[U];
#pragma unroll
  for (int r = 0; r < U; r++) acc[r] = 0.0f;
  for (int c = 0; c < nchunks; c++, cc++, dc++) {
    const uint32_t slot = cc % kSlots;
    if (!mbar_wait(&full[slot], (cc / kSlots) & 1, s_abort, kTimeoutNs, false)) return false;
    const uint32_t sp = smem_s + slot * kSlotBytes;
    const int nbc = min(kCB, a.bpr - c * kCB);
    const uint32_t buf = dc & 1;
    const uint32_t words = conv_s + buf * (kDp4aRows * 64 * 4);  // [row][64]
    const uint32_t sums = csum_s + buf * (kDp4aRows * 8 * 4);    // [row][8]
    // this thread's first code words and scale, read now: they run under the
    // conversion and its wait (the next block's are read under each block)
    uint32_t cj = sp + (uint32_t)(tid * kCode);                             // codes of (block j, row tid)
    uint32_t sj = sp + (uint32_t)(nbc * nw * kCode) + (uint32_t)(tid * 2);  // its fp16 scale
    uint4 w4 = lds128(cj);
    float dw = lds_half_as_f32(sj);
    // ---- the chunk's activation words: thread tid < 64U makes word tid
    // (row tid/64, group G, shift s) from stored words 8G+s (values s, s+8)
    // and 8G+s+4 (values s+4, s+12); 1536 + q in fp16 has q's two's
    // complement in its low byte
    {
      int qsum = 0;
      if (tid < 64 * U) {  // whole warps
        const int r = tid >> 6, jj = tid & 63, G = jj >> 2, sh = jj & 3;
        const int w0 = 8 * G + sh, w1 = w0 + 4;
        const uint32_t row = sp + kRawBytes + (uint32_t)(r * 128);
        const uint32_t x = lds32(row + (uint32_t)(w0 >> 5) * kBoxBytes +
                                 ((((w0 & 31) >> 2) ^ (r & 7)) << 4) + (w0 & 3) * 4);
        const uint32_t y = lds32(row + (uint32_t)(w1 >> 5) * kBoxBytes +
                                 ((((w1 & 31) >> 2) ^ (r & 7)) << 4) + (w1 & 3) * 4);
        const uint32_t word = __byte_perm(hadd2_u32(x, 0x66006600u), hadd2_u32(y, 0x66006600u),
                                          0x6240);
        sts32(words + (uint32_t)(r * 256 + jj * 4), word);
        qsum = __dp4a((int)word, 0x01010101, 0);
      }
      // a q8 block is 8 consecutive words: lanes 8m .. 8m+7
      qsum += __shfl_xor_sync(0xffffffffu, qsum, 1);
      qsum += __shfl_xor_sync(0xffffffffu, qsum, 2);
      qsum += __shfl_xor_sync(0xffffffffu, qsum, 4);
      if (tid < 64 * U && (tid & 7) == 0)
        sts32(sums + (uint32_t)((tid >> 6) * 32 + ((tid & 63) >> 3) * 4), (uint32_t)qsum);
      __syncwarp();
      if (lane == 0) mbar_arrive(&cbar[buf]);
      if (!mbar_wait(&cbar[buf], (dc >> 1) & 1, s_abort, kTimeoutNs, false)) return false;
    }
    // ---- this thread's row against the U rows
    const uint32_t dxs = sp + kRawBytes + kActBytes;  // [32 rows][8] fp32 (this chunk's 8 blocks)
#pragma unroll 1
    for (int j = 0; j < nbc; j++) {
      const uint32_t wv[4] = {w4.x, w4.y, w4.z, w4.w};  // groups 4j .. 4j+3
      uint32_t cw[4][4];                                 // [group][shift]: codes as bytes
#pragma unroll
      for (int g = 0; g < 4; g++)
#pragma unroll
        for (int sh = 0; sh < 4; sh++) cw[g][sh] = (wv[g] >> (2 * sh)) & 0x03030303u;
      const float dwj = dw;
      if (j + 1 < nbc) {
        cj += nw * kCode;
        sj += nw * 2;
        w4 = lds128(cj);
        dw = lds_half_as_f32(sj);
      }
#pragma unroll
      for (int r = 0; r < U; r++) {
        int isum[2] = {0, 0};  // q8 blocks 2j, 2j+1
#pragma unroll
        for (int g = 0; g < 4; g++) {
          const uint4 av = lds128(words + (uint32_t)(r * 256 + 64 * j + 16 * g));
          isum[g >> 1] = __dp4a((int)cw[g][0], (int)av.x, isum[g >> 1]);
          isum[g >> 1] = __dp4a((int)cw[g][1], (int)av.y, isum[g >> 1]);
          isum[g >> 1] = __dp4a((int)cw[g][2], (int)av.z, isum[g >> 1]);
          isum[g >> 1] = __dp4a((int)cw[g][3], (int)av.w, isum[g >> 1]);
        }
#pragma unroll
        for (int qq = 0; qq < 2; qq++) {
          const int qb = 2 * j + qq;
          const int qs = (int)lds32(sums + (uint32_t)(r * 32 + qb * 4));
          const float dx = lds_f32(dxs + (uint32_t)((r * kDxW + qb) * 4));
          acc[r] = __fmaf_rn(dx, __fmul_rn(dwj, (float)(isum[qq] - 2 * qs)), acc[r]);
        }
      }
    }
    refill(cc);
  }

  // ---- the item's outputs
  if (MODE == kModeDown) {
    if (tid < nw) {
#pragma unroll
      for (int r = 0; r < U; r++) a.out[(int64_t)(t.y + r) * a.N_out + wt * kTN + tid] = acc[r];
    }
    if (a.comb.out && 32 * warp < nw) {
      // the warp stored the 32-column group 32w .. 32w+31 of every routed
      // row of the tile; one lane per row counts it in
      __syncwarp();
      if (lane < U)
        combine_arrive(a.comb, a.out, a.rows_max, a.N_out, (int64_t)t.y + lane, wt * kTN + 32 * warp);
    }
    return true;
  }
  const int n_ff = a.N_out >> 1, nwg = nw >> 1;
  if (MODE == kModeGU) {
    if (tid < nw) {
      const bool up = tid >= nwg;
      const int o = wt * (kTN / 2) + (up ? tid - nwg : tid);
      const int col = a.gu_layout == MOE_GU_INTERLEAVED ? 2 * o + (up ? 1 : 0) : (up ? n_ff : 0) + o;
#pragma unroll
      for (int r = 0; r < U; r++) a.out[(int64_t)(t.y + r) * a.N_out + col] = acc[r];
    }
    return true;
  }
  // swiglu_quant fused: the up threads hand their rows to the gate threads
  // through shared memory; a gate warp then holds 32 consecutive outputs of
  // H, one q8 block, per routed row
  float* s_up = reinterpret_cast<float*>(const_cast<uint8_t*>(smem) + kOffUp);
  if (tid >= nwg && tid < nw) {
#pragma unroll
    for (int r = 0; r < U; r++) s_up[r * (kTN / 2) + tid - nwg] = acc[r];
  }
  __syncwarp();
  if (lane == 0) mbar_arrive(ubar);
  if (!mbar_wait(ubar, uc & 1, s_abort, kTimeoutNs, false)) return false;
  uc++;
  if (tid < nwg) {  // whole warps: nwg is a multiple of 32
    const int o = wt * (kTN / 2) + tid;
    // stored position of output o in its 16-value group (pair-interleaved)
    const int i16 = o & 15;
    const int pos = (o & ~15) + (i16 < 8 ? 2 * i16 : 2 * (i16 - 8) + 1);
#pragma unroll
    for (int r = 0; r < U; r++) {
      const float gv = acc[r], uv = s_up[r * (kTN / 2) + tid];
      const float hv = __fmul_rn(__fdiv_rn(gv, __fadd_rn(1.0f, expf(-gv))), uv);
      float amax = fabsf(hv);
#pragma unroll
      for (int m = 1; m < 32; m <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, m));
      const float d = __fdiv_rn(amax, 127.0f);
      const float q = (d == 0.0f) ? 0.0f : rintf(__fdiv_rn(hv, d));
      a.hq[(int64_t)(t.y + r) * n_ff + pos] = __float2half_rn(q);
      if (lane == 0) a.dh[(int64_t)(t.y + r) * scale_stride(n_ff) + (o >> 5)] = d;
    }
  }
  return true;
}

// One item (small-row tile x 256-row weight tile) of the work list, checked.
struct ItemInfo {
  int4 t;        // {expert, first routed row, rows, -}
  int wt, nw;    // weight tile, its rows
  int64_t off;   // byte offset of the expert's matrix in the tiled pack
  bool ok;
};
__device__ __forceinline__ ItemInfo item_info(const SmArgs& a, int first, int n_wtiles,
                                              int64_t mbytes, int item) {
  ItemInfo I;
  I.t = __ldg(a.tiles + first + item / n_wtiles);
  I.wt = item % n_wtiles;
  I.nw = min(kTN, a.N_out - I.wt * kTN);
  const bool rows_ok = (unsigned)I.t.x < (unsigned)a.E && I.t.y >= 0 && I.t.z > 0 &&
                       I.t.z <= kRows && (int64_t)I.t.y + I.t.z <= a.rows_max;
  I.off = rows_ok ? __ldg(a.eoff + 2 * I.t.x + a.which) : -1;
  I.ok = rows_ok && I.off >= 0 && (I.off & 15) == 0 && I.off + mbytes <= a.pack_bytes;
  return I;
}

// Work distribution: the producer of every CTA takes the next item of the
// work list from a counter in global memory (a.sched[0]), so a CTA that
// drew cheap items draws more.  Items differ in cost several times over (an
// m16n8k16 item of 17-32 rows against a dp4a item of one row), and with a
// fixed round-robin deal the multiprocessors sat idle a fifth of the time
// at 128 tokens.  The producer writes each chunk's item into s_item[slot],
// and the item's rows and weight tile into the slot's info record, before it
// arms the slot (the consumers take them from there, not from the work list
// in global memory); after the list it arms one more slot with no copies and
// item -1, which ends the consumers' loop.  routing zeroes the counters, and
// the last CTA to finish zeroes them again for the next launch.
//
// The load side of the ring (run by whichever warp releases a slot last):
// the next (item, chunk) to load, in the order the warps consume them.  Per
// chunk: one bulk copy of the raw weight chunk and the tile's activation
// rows and scales in 2-D TMA boxes of 16 rows (rows past the tile land in
// rows that are never read).
struct Producer {
  int item, c;  // next item (>= total: nothing left) and chunk
  const uint8_t* wbase;
  int row0, nw, nbox;
  uint32_t issued;
  int ended;    // the closing slot is armed
  int rows, wt;  // the item's routed rows and weight tile
};
__device__ __forceinline__ void prod_seek(Producer& p, const SmArgs& a, int first, int total,
                                          int n_wtiles, int64_t mbytes) {
  for (;;) {
    p.item = atomicAdd(a.sched, 1);
    if (p.item >= total) {
      p.item = total;
      return;
    }
    const ItemInfo I = item_info(a, first, n_wtiles, mbytes, p.item);
    if (!I.ok) {
      atomicOr(a.status, MOE_STATUS_BAD_OFFSET);
      continue;
    }
    p.c = 0;
    p.row0 = I.t.y;
    p.nw = I.nw;
    p.rows = I.t.z;
    p.wt = I.wt;
    p.nbox = I.t.z > kBoxRows ? 2 : 1;
    p.wbase = a.pack + I.off + (int64_t)I.wt * kTN * a.bpr * a.bb;
    return;
  }
}
static_assert(sizeof(Producer) <= 48 && alignof(Producer) <= 16, "producer state fits its slot");
template <int FMT>
__device__ __forceinline__ void prod_issue(Producer& p, uint8_t* smem, uint64_t* full,
                                           const SmArgs& a, const CUtensorMap* tmap,
                                           const CUtensorMap* tmap_d, int first, int total,
                                           int n_wtiles, int64_t mbytes, int nchunks) {
  constexpr int kCB = chunk_blocks(FMT), kBB = block_bytes(FMT);
  constexpr int kVals = kCB * block_values(FMT);
  constexpr int kDxW = dx_width(FMT);
  const uint32_t slot = p.issued % kSlots;
  volatile int* s_item = reinterpret_cast<volatile int*>(smem + kOffMisc + 240);
  if (p.item >= total) {  // the closing slot: no copies, item -1
    s_item[slot] = -1;
    mbar_arrive(&full[slot]);
    p.ended = 1;
    p.issued++;
    return;
  }
  asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(smem_u32(smem) + kOffInfo + 16 * slot),
               "r"(p.row0), "r"(p.rows), "r"(p.wt), "r"(p.nw)
               : "memory");
  s_item[slot] = p.item;
  uint8_t* sp = smem + slot * kSlotBytes;
  const int nbc = min(kCB, a.bpr - p.c * kCB);
  const uint32_t raw = (uint32_t)(nbc * p.nw * kBB);
  mbar_arrive_expect_tx(&full[slot], raw + (uint32_t)(p.nbox * kBoxRows * kVals * 2) +
                                         (uint32_t)(p.nbox * kBoxRows * kDxW * 4));
  bulk_g2s(sp, p.wbase + (int64_t)p.c * kCB * p.nw * kBB, raw, &full[slot]);
  for (int hb = 0; hb < p.nbox; hb++) {
#pragma unroll
    for (int bx = 0; bx < kVals / kActBox; bx++)
      tma_load_2d(sp + kRawBytes + bx * (kRows * kActBox * 2) + hb * (kBoxRows * 128), tmap,
                  p.c * kVals + bx * kActBox, p.row0 + kBoxRows * hb, &full[slot]);
    tma_load_2d(sp + kRawBytes + kActBytes + hb * (kBoxRows * kDxW * 4), tmap_d,
                (p.c * (kVals / 32)) & ~3, p.row0 + kBoxRows * hb, &full[slot]);
  }
  p.issued++;
  if (++p.c == nchunks) prod_seek(p, a, first, total, n_wtiles, mbytes);
}

template <int FMT, int MODE>
__global__ void __launch_bounds__(kThreads, 2)
gemm_small_kernel(const SmArgs a, const __grid_constant__ CUtensorMap tmap,
                  const __grid_constant__ CUtensorMap tmap_d) {
  constexpr bool kW2 = (FMT == MOE_FMT_W2);
  constexpr bool kDown = (MODE == kModeDown);

  extern __shared__ uint8_t smem_raw[];
  // 1024-byte aligned base, offset from the shared array itself (an integer
  // round trip would hide the shared address space from the compiler)
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kOffBar);
  int* s_rel = reinterpret_cast<int*>(smem + kOffRel);
  volatile int* s_abort = reinterpret_cast<volatile int*>(smem + kOffMisc);
  uint16_t* s_lut = reinterpret_cast<uint16_t*>(smem + kOffMisc + 64);
  uint64_t* pairbar = reinterpret_cast<uint64_t*>(smem + kOffMisc + 128);
  float* s_amax = reinterpret_cast<float*>(smem + kOffAmax);
  uint64_t* cbar = reinterpret_cast<uint64_t*>(smem + kOffDbar);  // [2], then the up exchange

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    for (int i = 0; i < kSlots; i++) {
      mbar_init(&full[i], 1);
      s_rel[2 * i] = 0;
    }
    for (int i = 0; i < kWarps; i++) mbar_init(&pairbar[i], 64);  // both warps of a pair
    for (int i = 0; i < 3; i++) mbar_init(&cbar[i], kWarps);      // lane 0 of every warp
    *s_abort = 0;
    fence_mbar_init();
  }
  if (FMT == MOE_FMT_W4NL && tid < 16) s_lut[tid] = c_nl4_half[tid];
  __syncthreads();

  const int n_wtiles = (a.N_out + kTN - 1) / kTN;
  const int nt_all = max(0, min(a.ntiles[0], (int)max_tiles(a.rows_max, a.E)));
  const int first = max(0, min(a.ntiles[1], nt_all));
  const int total = (nt_all - first) * n_wtiles;
  const int nchunks = (a.bpr + chunk_blocks(FMT) - 1) / chunk_blocks(FMT);
  const int64_t mbytes = (int64_t)a.N_out * a.bpr * a.bb;

  // ring: thread 0 prefills every slot; then lane 0 of the last warp to
  // release a slot refills it, so no warp waits for the others to finish a
  // chunk (with warp 0 waiting on a release barrier instead, 128 tokens took
  // 2 % longer).  The producer state lives in shared memory: one thread at a
  // time touches it, and as registers it would be held by every thread.
  Producer& prod = *reinterpret_cast<Producer*>(smem + kOffMisc + 192);
  volatile int* s_item = reinterpret_cast<volatile int*>(smem + kOffMisc + 240);
  if (tid == 0) {
    prod.issued = 0;
    prod.ended = 0;
    prefetch_tmap(&tmap);
    prefetch_tmap(&tmap_d);
    prod_seek(prod, a, first, total, n_wtiles, mbytes);
    for (int s = 0; s < kSlots && !prod.ended; s++)
      prod_issue<FMT>(prod, smem, full, a, &tmap, &tmap_d, first, total, n_wtiles, mbytes, nchunks);
  }
  auto refill = [&](uint32_t done) {  // chunk `done` was consumed by this warp
    __syncwarp();
    if (lane == 0) {
      // the last warp to release chunk `done`'s slot loads the chunk kSlots
      // ahead into it; the chunks are released in order, so the loads are
      // issued in order, one at a time
      int* rel = s_rel + 2 * (done % kSlots);
      __threadfence_block();
      if (atomicAdd(rel, 1) == kWarps - 1) {
        *rel = 0;
        __threadfence_block();
        if (!*reinterpret_cast<volatile int*>(&prod.ended))
          prod_issue<FMT>(prod, smem, full, a, &tmap, &tmap_d, first, total, n_wtiles, mbytes,
                          nchunks);
        __threadfence_block();
      }
    }
    __syncwarp();
  };

  const int g = lane >> 2, cq = lane & 3;
  uint32_t cc = 0;
  uint32_t xc = 0;  // amax exchanges of this warp's pair so far
  uint32_t dc = 0;  // chunks of dp4a items so far (their conversion buffers)
  uint32_t uc = 0;  // up-row exchanges of dp4a items so far
  bool alive = true;
  while (alive) {
    // the next item is the one the producer put in the next slot
    if (!(alive = mbar_wait(&full[cc % kSlots], (cc / kSlots) & 1, s_abort, kTimeoutNs, false)))
      break;
    const int item = s_item[cc % kSlots];
    if (item < 0) break;  // the closing slot
    // the item's rows and weight tile, as the producer found them
    const uint4 inf = lds128(smem_u32(smem) + kOffInfo + 16 * (cc % kSlots));
    const int4 t = make_int4(0, (int)inf.x, (int)inf.y, 0);
    const int wt = (int)inf.z, nw = (int)inf.w;
    if constexpr (kW2) {
      if (t.z <= kDp4aRows) {
#define MOE_SMALL_DP4A(N)                                                                       \
  item_dp4a<MODE, N>(a, smem, full, cbar, cbar + 2, s_abort, cc, dc, uc, nchunks, nw, t, wt, \
                     refill)
        alive = t.z == 1   ? MOE_SMALL_DP4A(1)
                : t.z == 2 ? MOE_SMALL_DP4A(2)
                : t.z == 3 ? MOE_SMALL_DP4A(3)
                           : MOE_SMALL_DP4A(4);
#undef MOE_SMALL_DP4A
        if (!alive) break;
        continue;
      }
    }
    {
      const int u = t.z;
      const int nnt = (u + 7) >> 3;  // n8 fragments of routed rows (1 to 4)
      // tile rows of m16 fragment mt: down 32w + 16mt; gate/up (tile = nwg
      // gate rows then the matching nwg up rows) gate 16w (mt 0), up nwg + 16w
      // (mt 1) -- the warp holds both halves of outputs 16w .. 16w+15
      const int nwg = nw >> 1;
      const int rbase[2] = {kDown ? 32 * warp : 16 * warp, kDown ? 32 * warp + 16 : nwg + 16 * warp};
      const bool active = kDown ? 32 * warp < nw : 16 * warp < nwg;  // warp-uniform
      float acc[2][4][4];
#pragma unroll
      for (int mt = 0; mt < 2; mt++)
#pragma unroll
        for (int nt = 0; nt < 4; nt++)
#pragma unroll
          for (int i = 0; i < 4; i++) acc[mt][nt][i] = 0.0f;
#define MOE_SMALL_CONSUME(N)                                                                  \
  consume_item<FMT, N>(smem, full, s_abort, cc, nchunks, a.bpr, nw, rbase, s_lut, lane, \
                       acc, refill)
      alive = nnt == 1   ? MOE_SMALL_CONSUME(1)
              : nnt == 2 ? MOE_SMALL_CONSUME(2)
              : nnt == 3 ? MOE_SMALL_CONSUME(3)
                         : MOE_SMALL_CONSUME(4);
#undef MOE_SMALL_CONSUME
      if (!alive) break;

      // ---- store.  C fragment: rows g, g+8 of the m16 tile, routed rows
      // 8nt + 2cq, +1 (only rows < u are real)
      if (kDown) {
        if (!active) continue;
#pragma unroll
        for (int mt = 0; mt < 2; mt++) {
#pragma unroll
          for (int nt = 0; nt < 4; nt++) {
            if (nt >= nnt) break;
#pragma unroll
            for (int i = 0; i < 4; i++) {
              const int rr = 8 * nt + 2 * cq + (i & 1);
              const int r = rbase[mt] + g + 8 * (i >> 1);
              if (rr < u && r < nw) a.out[(int64_t)(t.y + rr) * a.N_out + wt * kTN + r] = acc[mt][nt][i];
            }
          }
        }
        if (a.comb.out) {
          // the warp stored the 32-column group 32w .. 32w+31 of every routed
          // row of the tile; one lane per row counts it in
          __syncwarp();
          if (lane < u)
            combine_arrive(a.comb, a.out, a.rows_max, a.N_out, (int64_t)t.y + lane, wt * kTN + 32 * warp);
        }
      } else if (MODE == kModeGU) {
        if (!active) continue;
        const int n_ff = a.N_out >> 1;
        // gate and up outputs 128t + 16w + g (+8): columns o and n_ff + o
        // (split), or 2o and 2o + 1 (interleaved)
        const int o = wt * (kTN / 2) + 16 * warp + g;
        const bool inter = a.gu_layout == MOE_GU_INTERLEAVED;
#pragma unroll
        for (int nt = 0; nt < 4; nt++)
#pragma unroll
          for (int i = 0; i < 4; i++) {
            const int rr = 8 * nt + 2 * cq + (i & 1);
            if (nt < nnt && rr < u) {
              const int oo = o + 8 * (i >> 1);
              float* orow = a.out + (int64_t)(t.y + rr) * a.N_out;
              if (inter) {
                *reinterpret_cast<float2*>(orow + 2 * oo) =
                    make_float2(acc[0][nt][i], acc[1][nt][i]);
              } else {
                orow[oo] = acc[0][nt][i];
                orow[n_ff + oo] = acc[1][nt][i];
              }
            }
          }
      } else {
        // swiglu_quant fused: the warp holds outputs 128t + 16w .. +15 (one
        // 16-value group; the q8 block of H is this warp's group and its pair
        // warp's), 2 values a thread per routed row: outputs g and g+8, exactly
        // the stored pair (positions 2g, 2g+1) of the group.  The pair's amax
        // goes through shared memory, double-buffered by exchange parity
        // (a warp cannot run two exchanges ahead of its pair).  Warps are
        // active in pairs: nwg is a multiple of 64.
        if (!active) continue;
        const int n_ff = a.N_out >> 1;
        const int o = wt * (kTN / 2) + 16 * warp;
        const uint32_t xb = xc & 1;
        float* am_own = s_amax + (xb * kWarps + warp) * kRows;
        const float* am_pair = s_amax + (xb * kWarps + (warp ^ 1)) * kRows;
        float hv[4][2][2];  // [nt][col][output g / g+8]
        float am[4][2];
#pragma unroll
        for (int nt = 0; nt < 4; nt++) {
          if (nt >= nnt) break;
#pragma unroll
          for (int col = 0; col < 2; col++) {
            float amax = 0.0f;
#pragma unroll
            for (int e = 0; e < 2; e++) {
              const int i = 2 * e + col;
              const float gv = acc[0][nt][i], uv = acc[1][nt][i];
              hv[nt][col][e] = __fmul_rn(__fdiv_rn(gv, __fadd_rn(1.0f, expf(-gv))), uv);
              amax = fmaxf(amax, fabsf(hv[nt][col][e]));
            }
            amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 4));
            amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 8));
            amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 16));
            am[nt][col] = amax;
            if (g == 0) am_own[8 * nt + 2 * cq + col] = amax;
          }
        }
        uint64_t* pb = &pairbar[xb * (kWarps / 2) + (warp >> 1)];
        mbar_arrive(pb);
        if (!(alive = mbar_wait(pb, (xc >> 1) & 1, s_abort, kTimeoutNs, false))) break;
        xc++;
#pragma unroll
        for (int nt = 0; nt < 4; nt++) {
          if (nt >= nnt) break;
#pragma unroll
          for (int col = 0; col < 2; col++) {
            const int rr = 8 * nt + 2 * cq + col;
            const float d = __fdiv_rn(fmaxf(am[nt][col], am_pair[rr]), 127.0f);
            if (rr < u) {
              const float q0 = (d == 0.0f) ? 0.0f : rintf(__fdiv_rn(hv[nt][col][0], d));
              const float q1 = (d == 0.0f) ? 0.0f : rintf(__fdiv_rn(hv[nt][col][1], d));
              __half* hrow = a.hq + (int64_t)(t.y + rr) * n_ff + o;
              *reinterpret_cast<__half2*>(hrow + 2 * g) = __floats2half2_rn(q0, q1);
              if (g == 0 && (warp & 1) == 0)
                a.dh[(int64_t)(t.y + rr) * scale_stride(n_ff) + (o >> 5)] = d;
            }
          }
        }
      }
    }
  }
  // copies still in flight after an abort land before the CTA exits (every
  // warp has issued its last load)
  __syncthreads();
  if (tid == 0)
    for (uint32_t i = cc; i < prod.issued; i++)
      if (!mbar_wait(&full[i % kSlots], (i / kSlots) & 1, s_abort, kTimeoutNs, false)) break;
  if (*s_abort && tid == 0) atomicOr(a.status, MOE_STATUS_PIPE_TIMEOUT);
  // the last CTA to finish (every producer has taken its last item) zeroes
  // the work counter for the next launch
  if (tid == 0) {
    __threadfence();
    if (atomicAdd(a.sched + 1, 1) == (int)gridDim.x - 1) {
      a.sched[0] = 0;
      a.sched[1] = 0;
      __threadfence();
    }
  }
}

PFN_cuTensorMapEncodeTiled_v12000 get_encode_small() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// Resident CTAs a multiprocessor (two by design), found once per device and
// context together with the kernel's attributes.
template <int FMT, int MODE>
cudaError_t launch_small(const SmArgs& a, const CUtensorMap& tm, const CUtensorMap& td,
                         int64_t items, cudaStream_t st) {
  static std::atomic<uint64_t> ready[64];
  static std::atomic<int> per_sm[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  const uint64_t ctx = current_context_id();
  if (ctx == 0 || ready[dev].load(std::memory_order_acquire) != ctx) {
    // two CTAs a multiprocessor: the full shared-memory carveout
    cudaError_t e = cudaFuncSetAttribute(
        gemm_small_kernel<FMT, MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(gemm_small_kernel<FMT, MODE>,
                               cudaFuncAttributePreferredSharedMemoryCarveout,
                               (int)cudaSharedmemCarveoutMaxShared);
    int n = 0;
    if (e == cudaSuccess)
      e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, gemm_small_kernel<FMT, MODE>, kThreads,
                                                         kSmemBytes);
    if (e != cudaSuccess) return e;
    if (n < 1) return cudaErrorInvalidConfiguration;
    per_sm[dev].store(n, std::memory_order_relaxed);
    ready[dev].store(ctx, std::memory_order_release);
  }
  const int grid =
      (int)std::max<int64_t>(
          1, std::min<int64_t>(items, (int64_t)per_sm[dev].load(std::memory_order_relaxed) *
                                          device_sm_count()));
  gemm_small_kernel<FMT, MODE><<<grid, kThreads, kSmemBytes, st>>>(a, tm, td);
  return cudaSuccess;
}

}  // namespace

cudaError_t launch_gemm_small(const GemmArgs& g, cudaStream_t st) {
  if (g.rows_max == 0) return cudaSuccess;
  SmArgs a{};
  a.pack = g.pack;
  a.eoff = g.eoff;
  a.which = g.which;
  a.pack_bytes = g.pack_bytes;
  a.tiles = g.tiles;
  a.ntiles = g.ntiles;
  a.E = g.E;
  a.K = g.K;
  a.N_out = g.N_out;
  a.bpr = g.K / block_values(g.fmt);
  a.bb = block_bytes(g.fmt);
  a.out = g.out;
  a.gu_layout = g.gu_layout;
  a.hq = g.hq;
  a.dh = g.dh;
  a.rows_max = g.rows_max;
  a.status = g.status;
  a.sched = g.sched;
  a.comb = g.comb;

  auto encode = get_encode_small();
  if (!encode) return cudaErrorNotSupported;
  // activations: [rows_max x K] fp16, boxes of 64 values (128 B, 128-byte
  // swizzle) x 16 rows, one chunk's worth per chunk
  const int vals = chunk_blocks(g.fmt) * block_values(g.fmt);
  CUtensorMap tm, td;
  const cuuint64_t dims[2] = {(cuuint64_t)g.K, (cuuint64_t)g.rows_max};
  const cuuint64_t strides[1] = {(cuuint64_t)g.K * 2};
  const cuuint32_t box[2] = {(cuuint32_t)kActBox, (cuuint32_t)kBoxRows};
  const cuuint32_t estr[2] = {1, 1};
  if (encode(&tm, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<__half*>(g.act), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;
  // their scales: [rows_max x scale_stride(K)] fp32, boxes of dx_width (8 for
  // W2, 4 otherwise) x 16 rows
  const int ss = scale_stride(g.K);
  const cuuint64_t ddims[2] = {(cuuint64_t)ss, (cuuint64_t)g.rows_max};
  const cuuint64_t dstrides[1] = {(cuuint64_t)ss * 4};
  const cuuint32_t dbox[2] = {(cuuint32_t)dx_width(g.fmt), (cuuint32_t)kBoxRows};
  if (encode(&td, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float*>(g.act_d), ddims, dstrides,
             dbox, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;

  // one item per (small-row tile, 256-row weight tile)
  const int64_t n_wtiles = (g.N_out + kTN - 1) / kTN;
  const int64_t items_max =
      (int64_t)std::min<int64_t>((int64_t)g.E * (kSmallSplit / kSmallTileRows), g.rows_max) * n_wtiles;
  const int mode = g.which == 1 ? kModeDown : (g.hq ? kModeSwiglu : kModeGU);
  cudaError_t e;
  if (g.fmt == MOE_FMT_W2) {
    e = mode == kModeDown     ? launch_small<MOE_FMT_W2, kModeDown>(a, tm, td, items_max, st)
        : mode == kModeSwiglu ? launch_small<MOE_FMT_W2, kModeSwiglu>(a, tm, td, items_max, st)
                              : launch_small<MOE_FMT_W2, kModeGU>(a, tm, td, items_max, st);
  } else if (g.fmt == MOE_FMT_W4NL) {
    e = mode == kModeDown     ? launch_small<MOE_FMT_W4NL, kModeDown>(a, tm, td, items_max, st)
        : mode == kModeSwiglu ? launch_small<MOE_FMT_W4NL, kModeSwiglu>(a, tm, td, items_max, st)
                              : launch_small<MOE_FMT_W4NL, kModeGU>(a, tm, td, items_max, st);
  } else {
    e = mode == kModeDown     ? launch_small<MOE_FMT_Q8_0, kModeDown>(a, tm, td, items_max, st)
        : mode == kModeSwiglu ? launch_small<MOE_FMT_Q8_0, kModeSwiglu>(a, tm, td, items_max, st)
                              : launch_small<MOE_FMT_Q8_0, kModeGU>(a, tm, td, items_max, st);
  }
  if (e != cudaSuccess) return e;
  count_launch();
  return cudaGetLastError();
}

}  // namespace moe
