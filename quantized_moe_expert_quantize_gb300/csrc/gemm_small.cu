// Small-expert tier of the grouped expert products: experts with at most
// kSmallRows (16) routed rows.
//
// Same arithmetic as the tcgen05 kernel -- per 32-value K block the exact
// integer sum of w_int * q, then the fp32 epilogue in K order ("Strata #3752",
// commit "moe_ws kernels") -- on a different tile shape.  With a handful of
// rows per expert the layer streams weights: each expert's whole weight matrix
// is read for a few rows, so the time is the weight bytes (the pages tune a
// separate tier by rows per expert, "Strata #3752", addendum).  A 128-row
// tcgen05 tile would compute mostly padding; here the weights are the MMA's
// M side, decoded straight into mma.sync.m16n8k16 fp16 fragments in
// registers, and the few routed rows are its N side (8 per fragment), with
// fp32 accumulators in registers.  Operands are exact fp16 integers (|w|,
// |q| <= 127; W2 with its scale folded, d*(c-2) exact), so each 16-value
// MMA step and each 32-value block sum is exact in fp32.
//
// Item: one small expert's rows (one tile of the work list) against one
// 256-row tile of the tiled weight pack.  4 compute warps own 64 tile rows
// each (4 m16 fragments); warp 4 produces: per 4-block weight chunk one bulk
// copy of the raw chunk and one 2-D TMA box each of the 16 activation rows
// and their scales, into a ring of 4 slots.
//
// The routed rows' activations are stored pair-interleaved in every 16-value
// group (position 2i holds value i, 2i+1 holds value i+8).  Taking the MMA's
// k as the stored position, a thread's A-fragment pairs are the weights of
// values (c, c+8) and (c+4, c+12) of a group -- exactly the pairs one code
// word yields with one mask per pair -- and its B-fragment pairs are single
// 32-bit words of the stored rows.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <mutex>

#include "common.cuh"
#include "sm100_ptx.cuh"

namespace moe {
namespace {

using namespace ptx;

constexpr int kTN = 256;           // weight rows per item (one tile of the tiled pack)
constexpr int kWarps = 4;          // compute warps, 64 tile rows each
constexpr int kThreads = (kWarps + 1) * 32;
constexpr int kSlots = 4;
constexpr int kChunkBlocks = 4;    // weight blocks per chunk of the tiled pack
constexpr int kChunkVals = 256;    // K values per activation box (a W2 chunk; a W4NL chunk uses 128)
constexpr int kRawBytes = kChunkBlocks * kTN * kBlockBytes;  // 18,432
constexpr int kActBytes = kSmallRows * kChunkVals * 2;       // 8,192: 16 rows x 256 fp16
constexpr int kDxBytes = kSmallRows * (kChunkVals / 32) * 4;  // 512: 16 rows x 8 scales
// slots 1024-byte aligned: the activation boxes use the 128-byte swizzle
constexpr int kSlotBytes = (kRawBytes + kActBytes + kDxBytes + 1023) & ~1023;
constexpr int kActBox = 64;                                  // values per activation box (128 B)
constexpr int kOffBar = kSlots * kSlotBytes;
constexpr int kOffMisc = kOffBar + 2 * kSlots * 8;
constexpr int kSmemBytes = kOffMisc + 128 + 1024;  // abort flag, W4NL table; + alignment slack
constexpr uint64_t kTimeoutNs = 1000000000ull;
constexpr int kModeGU = 0, kModeSwiglu = 1, kModeDown = 2;
static_assert(kSlotBytes % 1024 == 0 && kRawBytes % 1024 == 0, "swizzled boxes 1024-byte aligned");
static_assert(kSmemBytes <= 232448 / 2, "two CTAs a multiprocessor");

struct SmArgs {
  const uint8_t* pack;
  const int64_t* eoff;
  int which;
  int64_t pack_bytes;
  const int4* tiles;
  const int32_t* ntiles;  // {tiles, big-expert tiles}
  int E;
  int K, N_out, bpr;
  float* out;
  __half* hq;
  float* dh;
  int64_t rows_max;
  int32_t* status;
};

__device__ __forceinline__ uint32_t hmul2_u32(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
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

// W2 fragments without arithmetic.  ws is a code word shifted right by 2*cq
// (codes of values cq, cq+4, cq+8, cq+12 of the group at bits 0, 8, 16, 24).
// Pair a: (1024 + c_cq, 1024 + c_{cq+8}); pair b: (1024 + 256 c_{cq+4},
// 1024 + 256 c_{cq+12}) -- the codes dropped into fp16 mantissas, exact.  The
// B pairs facing pair b are pre-scaled by 1/256 (exact for |q| <= 127), so
// every product is an integer: (1024 + c) q on the low half of the group's
// MMA k and 4q + c q on the high half.  The 1024 / 4 offsets and the code
// bias 2 are taken out by starting each block's accumulation at
// -(1026 sum_lo q + 6 sum_hi q), itself one MMA of the constant A below
// against the same B.  All partial sums are integers below 2^23, so the
// block sum sum (c-2) q comes out exact.
__device__ __forceinline__ uint32_t w2_pair_lo(uint32_t ws) { return (ws & 0x00030003u) | 0x64006400u; }
__device__ __forceinline__ uint32_t w2_pair_hi(uint32_t ws) { return (ws & 0x03000300u) | 0x64006400u; }
constexpr uint32_t kHalfInv256 = 0x1C001C00u;  // fp16 pair (1/256, 1/256)
constexpr uint32_t kCorrLo = 0xE402E402u;      // fp16 pair (-1026, -1026)
constexpr uint32_t kCorrHi = 0xE600E600u;      // fp16 pair (-1536, -1536) = -6 * 256
// W4NL: the fp16 pair (T[idx_i], T[idx_{i+8}]) from the group's two words.
__device__ __forceinline__ uint32_t w4_pair(uint32_t wlo, uint32_t whi, int i,
                                            const uint16_t* lut) {
  return (uint32_t)lut[(wlo >> (4 * i)) & 15u] | ((uint32_t)lut[(whi >> (4 * i)) & 15u] << 16);
}

// One item's products: every chunk of the item's weight tile against its
// (up to 8 * NNT) routed rows, accumulated per 32-value block in K order into
// acc (fragment mt of tile rows rbase[mt]..+15, n8 fragment nt).  Tile rows
// past the tile's end compute garbage from in-slot bytes and are never stored.
template <int FMT, int NNT>
__device__ __forceinline__ bool consume_item(const uint8_t* smem, uint64_t* full, uint64_t* empty,
                                             volatile int* s_abort, uint32_t& cc, int nchunks,
                                             int bpr, int nw, const int (&rbase)[4],
                                             const uint16_t* s_lut, int lane,
                                             float (&acc)[4][2][4]) {
  constexpr bool kW2 = (FMT == MOE_FMT_W2);
  constexpr int kBv = kW2 ? 64 : 32;        // values per weight block
  constexpr int kVals = kChunkBlocks * kBv;  // K values per chunk
  constexpr int kQpb = kBv / 32;             // q8 blocks per weight block
  const int g = lane >> 2, cq = lane & 3;
  const uint32_t ca[4] = {kCorrLo, kCorrLo, kCorrHi, kCorrHi};
  const float zero[4] = {0.0f, 0.0f, 0.0f, 0.0f};
  for (int c = 0; c < nchunks; c++, cc++) {
    const uint32_t slot = cc % kSlots;
    if (!mbar_wait(&full[slot], (cc / kSlots) & 1, s_abort, kTimeoutNs, false)) return false;
    const uint8_t* sp = smem + slot * kSlotBytes;
    const int nbc = min(kChunkBlocks, bpr - c * kChunkBlocks);
    const uint16_t* scl = reinterpret_cast<const uint16_t*>(sp + nbc * nw * 16);
    const uint8_t* act = sp + kRawBytes;  // [box][16 rows][128 B], 128-byte swizzle
    const float* dxs = reinterpret_cast<const float*>(sp + kRawBytes + kActBytes);
#pragma unroll
    for (int j = 0; j < kChunkBlocks; j++) {
      if (j >= nbc) break;
      float dw[4][2];   // scale of weight block j, tile rows rbase+g / +8
#pragma unroll
      for (int mt = 0; mt < 4; mt++)
#pragma unroll
        for (int h = 0; h < 2; h++)
          dw[mt][h] = __half2float(__ushort_as_half(scl[j * nw + rbase[mt] + g + 8 * h]));
#pragma unroll
      for (int qq = 0; qq < kQpb; qq++) {
        const int qb = j * kQpb + qq;  // q8 block within the chunk
        // the block's code words for this q8 block (two 16-value groups), rows
        // rbase+g / +8: W2 words 2qq, 2qq+1; W4NL all four
        uint2 cw[4][2][2 / kQpb];
#pragma unroll
        for (int mt = 0; mt < 4; mt++)
#pragma unroll
          for (int h = 0; h < 2; h++) {
            const uint2* src =
                reinterpret_cast<const uint2*>(sp + (j * nw + rbase[mt] + g + 8 * h) * 16);
#pragma unroll
            for (int e = 0; e < 2 / kQpb; e++) cw[mt][h][e] = src[qq + e];
          }
        // B fragments: routed row n = 8nt + g, stored positions 2cq,+1 (16-byte
        // chunk 2*(grp%4)) and 2cq+8,+9 (chunk 2*(grp%4)+1) of box grp/4
        uint32_t b[2][NNT][2];
#pragma unroll
        for (int ks = 0; ks < 2; ks++) {
          const int grp = 2 * qb + ks;
          const uint8_t* box = act + (grp >> 2) * (kSmallRows * kActBox * 2);
#pragma unroll
          for (int nt = 0; nt < NNT; nt++) {
            const int n = 8 * nt + g;
            const uint8_t* row = box + n * 128;
            const int ch = 2 * (grp & 3);
            b[ks][nt][0] = *reinterpret_cast<const uint32_t*>(row + ((ch ^ (n & 7)) << 4) + 4 * cq);
            b[ks][nt][1] =
                *reinterpret_cast<const uint32_t*>(row + (((ch + 1) ^ (n & 7)) << 4) + 4 * cq);
            if (kW2) b[ks][nt][1] = hmul2_u32(b[ks][nt][1], kHalfInv256);
          }
        }
        float ci[NNT][4];  // accumulation start of the block
#pragma unroll
        for (int nt = 0; nt < NNT; nt++) {
          if (kW2) {
            mma16816c(ci[nt], ca, b[0][nt][0], b[0][nt][1], zero);
            mma16816(ci[nt], ca, b[1][nt][0], b[1][nt][1]);
          } else {
#pragma unroll
            for (int i = 0; i < 4; i++) ci[nt][i] = 0.0f;
          }
        }
        float p[4][NNT][4];  // the block's integer sums
#pragma unroll
        for (int ks = 0; ks < 2; ks++) {
#pragma unroll
          for (int mt = 0; mt < 4; mt++) {
            uint32_t af[4];
#pragma unroll
            for (int h = 0; h < 2; h++) {
              if (kW2) {
                // code word of group 2qq + ks of the block
                const uint32_t w = ks ? cw[mt][h][0].y : cw[mt][h][0].x;
                const uint32_t ws = w >> (2 * cq);
                af[h] = w2_pair_lo(ws);
                af[2 + h] = w2_pair_hi(ws);
              } else {
                const uint2 q2 = cw[mt][h][ks];
                const uint32_t wlo = q2.x, whi = q2.y;
                af[h] = w4_pair(wlo, whi, cq, s_lut);
                af[2 + h] = w4_pair(wlo, whi, cq + 4, s_lut);
              }
            }
#pragma unroll
            for (int nt = 0; nt < NNT; nt++) {
              if (ks == 0)
                mma16816c(p[mt][nt], af, b[0][nt][0], b[0][nt][1], ci[nt]);
              else
                mma16816(p[mt][nt], af, b[1][nt][0], b[1][nt][1]);
            }
          }
        }
        // epilogue of the block, in K order: acc += d_x * (d_w * isum) (W2,
        // d_w * isum exact) or acc += (d_w * d_x) * isum (W4NL)
#pragma unroll
        for (int nt = 0; nt < NNT; nt++) {
          const float dx0 = dxs[(8 * nt + 2 * cq) * (kVals / 32) + qb];
          const float dx1 = dxs[(8 * nt + 2 * cq + 1) * (kVals / 32) + qb];
#pragma unroll
          for (int mt = 0; mt < 4; mt++) {
#pragma unroll
            for (int i = 0; i < 4; i++) {
              const float dx = (i & 1) ? dx1 : dx0;
              const float dwr = dw[mt][i >> 1];
              acc[mt][nt][i] = kW2 ? __fmaf_rn(dx, __fmul_rn(dwr, p[mt][nt][i]), acc[mt][nt][i])
                                   : __fmaf_rn(__fmul_rn(dwr, dx), p[mt][nt][i], acc[mt][nt][i]);
            }
          }
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[slot]);
  }
  return true;
}

template <int FMT, int MODE>
__global__ void __maxnreg__(200)
gemm_small_kernel(const SmArgs a, const __grid_constant__ CUtensorMap tmap,
                  const __grid_constant__ CUtensorMap tmap_d) {
  constexpr bool kW2 = (FMT == MOE_FMT_W2);
  constexpr bool kDown = (MODE == kModeDown);
  constexpr int kBv = kW2 ? 64 : 32;                  // values per weight block
  constexpr int kVals = kChunkBlocks * kBv;           // K values per chunk

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kOffBar);
  uint64_t* empty = full + kSlots;
  volatile int* s_abort = reinterpret_cast<volatile int*>(smem + kOffMisc);
  uint16_t* s_lut = reinterpret_cast<uint16_t*>(smem + kOffMisc + 64);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    for (int i = 0; i < kSlots; i++) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], kWarps);
    }
    *s_abort = 0;
    fence_mbar_init();
  }
  if (!kW2 && tid < 16) s_lut[tid] = c_nl4_half[tid];
  __syncthreads();

  const int n_wtiles = (a.N_out + kTN - 1) / kTN;
  const int nt_all = max(0, min(a.ntiles[0], (int)max_tiles(a.rows_max, a.E)));
  const int first = max(0, min(a.ntiles[1], nt_all));
  const int total = (nt_all - first) * n_wtiles;
  const int nchunks = (a.bpr + kChunkBlocks - 1) / kChunkBlocks;
  const int64_t mbytes = (int64_t)a.N_out * a.bpr * kBlockBytes;

  if (warp == kWarps) {
    // ================================================== producer
    if (lane == 0) {
      prefetch_tmap(&tmap);
      prefetch_tmap(&tmap_d);
      uint32_t cc = 0;
      bool alive = true;
      for (int item = blockIdx.x; item < total && alive; item += gridDim.x) {
        const int4 t = __ldg(a.tiles + first + item / n_wtiles);
        const int wt = item % n_wtiles;
        const int nw = min(kTN, a.N_out - wt * kTN);
        const bool rows_ok = (unsigned)t.x < (unsigned)a.E && t.y >= 0 && t.z > 0 &&
                             t.z <= kSmallRows && (int64_t)t.y + t.z <= a.rows_max;
        const int64_t off = rows_ok ? __ldg(a.eoff + 2 * t.x + a.which) : -1;
        if (!(rows_ok && off >= 0 && (off & 15) == 0 && off + mbytes <= a.pack_bytes)) continue;
        const uint8_t* wbase = a.pack + off + (int64_t)wt * kTN * a.bpr * kBlockBytes;
        for (int c = 0; c < nchunks; c++, cc++) {
          const uint32_t slot = cc % kSlots;
          if (!(alive = mbar_wait(&empty[slot], ((cc / kSlots) & 1) ^ 1, s_abort, kTimeoutNs)))
            break;
          uint8_t* sp = smem + slot * kSlotBytes;
          const int nbc = min(kChunkBlocks, a.bpr - c * kChunkBlocks);
          const uint32_t raw = (uint32_t)(nbc * nw * kBlockBytes);
          mbar_arrive_expect_tx(&full[slot], raw + (uint32_t)(kSmallRows * kVals * 2) +
                                                 (uint32_t)(kSmallRows * (kVals / 32) * 4));
          bulk_g2s(sp, wbase + (int64_t)c * kChunkBlocks * nw * kBlockBytes, raw, &full[slot]);
          // the expert's (up to 16) activation rows and their scales; rows
          // past the expert land in rows that are never read
#pragma unroll
          for (int bx = 0; bx < kVals / kActBox; bx++)
            tma_load_2d(sp + kRawBytes + bx * (kSmallRows * kActBox * 2), &tmap,
                        c * kVals + bx * kActBox, t.y, &full[slot]);
          tma_load_2d(sp + kRawBytes + kActBytes, &tmap_d, c * (kVals / 32), t.y, &full[slot]);
        }
      }
    }
    __syncwarp();
  } else {
    // ================================================== compute warps
    const int g = lane >> 2, cq = lane & 3;
    uint32_t cc = 0;
    bool alive = true;
    for (int item = blockIdx.x; item < total && alive; item += gridDim.x) {
      const int4 t = __ldg(a.tiles + first + item / n_wtiles);
      const int wt = item % n_wtiles;
      const int nw = min(kTN, a.N_out - wt * kTN);
      const bool rows_ok = (unsigned)t.x < (unsigned)a.E && t.y >= 0 && t.z > 0 &&
                           t.z <= kSmallRows && (int64_t)t.y + t.z <= a.rows_max;
      const int64_t off = rows_ok ? __ldg(a.eoff + 2 * t.x + a.which) : -1;
      if (!(rows_ok && off >= 0 && (off & 15) == 0 && off + mbytes <= a.pack_bytes)) {
        if (tid == 0) atomicOr(a.status, MOE_STATUS_BAD_OFFSET);
        continue;
      }
      const int u = t.z;
      const int nnt = (u + 7) >> 3;  // n8 fragments of routed rows (1 or 2)
      // tile rows of m16 fragment mt: down 64w + 16mt; gate/up (tile = nwg
      // gate rows then the matching nwg up rows) gate 32w + 16mt (mt 0,1),
      // up nwg + 32w + 16(mt-2) (mt 2,3)
      const int nwg = nw >> 1;
      int rbase[4];
      bool mact[4];
#pragma unroll
      for (int mt = 0; mt < 4; mt++) {
        rbase[mt] = kDown ? 64 * warp + 16 * mt
                          : (mt < 2 ? 32 * warp + 16 * mt : nwg + 32 * warp + 16 * (mt - 2));
        mact[mt] = kDown ? rbase[mt] < nw : 32 * warp + 16 * (mt & 1) < nwg;
      }
      float acc[4][2][4];
#pragma unroll
      for (int mt = 0; mt < 4; mt++)
#pragma unroll
        for (int nt = 0; nt < 2; nt++)
#pragma unroll
          for (int i = 0; i < 4; i++) acc[mt][nt][i] = 0.0f;
      alive = nnt == 1 ? consume_item<FMT, 1>(smem, full, empty, s_abort, cc, nchunks, a.bpr, nw,
                                              rbase, s_lut, lane, acc)
                       : consume_item<FMT, 2>(smem, full, empty, s_abort, cc, nchunks, a.bpr, nw,
                                              rbase, s_lut, lane, acc);
      if (!alive) break;

      // ---- store.  C fragment: rows g, g+8 of the m16 tile, routed rows
      // 8nt + 2cq, +1 (only rows < u are real)
      if (kDown) {
#pragma unroll
        for (int mt = 0; mt < 4; mt++) {
          if (!mact[mt]) continue;
#pragma unroll
          for (int nt = 0; nt < 2; nt++) {
#pragma unroll
            for (int i = 0; i < 4; i++) {
              const int rr = 8 * nt + 2 * cq + (i & 1);
              const int o = wt * kTN + rbase[mt] + g + 8 * (i >> 1);
              if (nt < nnt && rr < u) a.out[(int64_t)(t.y + rr) * a.N_out + o] = acc[mt][nt][i];
            }
          }
        }
      } else if (MODE == kModeGU) {
        const int n_ff = a.N_out >> 1;
#pragma unroll
        for (int mt = 0; mt < 4; mt++) {
          if (!mact[mt]) continue;
          // gate and up outputs 128t + 32w + 16(mt&1) + g (+8)
          const int o = wt * (kTN / 2) + 32 * warp + 16 * (mt & 1) + (mt < 2 ? 0 : n_ff);
#pragma unroll
          for (int nt = 0; nt < 2; nt++)
#pragma unroll
            for (int i = 0; i < 4; i++) {
              const int rr = 8 * nt + 2 * cq + (i & 1);
              if (nt < nnt && rr < u)
                a.out[(int64_t)(t.y + rr) * a.N_out + o + g + 8 * (i >> 1)] = acc[mt][nt][i];
            }
        }
      } else {
        // swiglu_quant fused: the warp holds outputs 128t + 32w .. + 31 (one
        // q8 block of H) for each routed row: 4 values a thread (fragments
        // 0,1 x rows g, g+8), the block across the 8 lanes of equal cq
        const int n_ff = a.N_out >> 1;
        const int o = wt * (kTN / 2) + 32 * warp;
        if (32 * warp < nwg) {
#pragma unroll
          for (int nt = 0; nt < 2; nt++) {
            if (nt >= nnt) continue;
#pragma unroll
            for (int col = 0; col < 2; col++) {
              float h[4];  // (fragment 0 row g, fragment 0 row g+8, fragment 1 row g, row g+8)
              float amax = 0.0f;
#pragma unroll
              for (int k = 0; k < 4; k++) {
                const int mt = k >> 1, i = 2 * (k & 1) + col;
                const float gv = acc[mt][nt][i], uv = acc[mt + 2][nt][i];
                h[k] = __fmul_rn(__fdiv_rn(gv, __fadd_rn(1.0f, expf(-gv))), uv);
                amax = fmaxf(amax, fabsf(h[k]));
              }
              amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 4));
              amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 8));
              amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 16));
              const float d = __fdiv_rn(amax, 127.0f);
              const int rr = 8 * nt + 2 * cq + col;
              if (rr < u) {
                __half* hrow = a.hq + (int64_t)(t.y + rr) * n_ff + o;
#pragma unroll
                for (int mt = 0; mt < 2; mt++) {
                  // 16-value group mt: position 2g holds value g, 2g+1 value g+8
                  const float q0 = (d == 0.0f) ? 0.0f : rintf(__fdiv_rn(h[2 * mt], d));
                  const float q1 = (d == 0.0f) ? 0.0f : rintf(__fdiv_rn(h[2 * mt + 1], d));
                  *reinterpret_cast<__half2*>(hrow + 16 * mt + 2 * g) = __floats2half2_rn(q0, q1);
                }
                if (g == 0) a.dh[(int64_t)(t.y + rr) * scale_stride(n_ff) + (o >> 5)] = d;
              }
            }
          }
        }
      }
    }
  }
  if (*s_abort && tid == 0) atomicOr(a.status, MOE_STATUS_PIPE_TIMEOUT);
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

template <int FMT, int MODE>
cudaError_t launch_small(const SmArgs& a, const CUtensorMap& tm, const CUtensorMap& td, int grid,
                         cudaStream_t st) {
  static bool done[64] = {false};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && !done[dev]) {
    const cudaError_t e = cudaFuncSetAttribute(
        gemm_small_kernel<FMT, MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) return e;
    done[dev] = true;
  }
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
  a.out = g.out;
  a.hq = g.hq;
  a.dh = g.dh;
  a.rows_max = g.rows_max;
  a.status = g.status;

  auto encode = get_encode_small();
  if (!encode) return cudaErrorNotSupported;
  // activations: [rows_max x K] fp16, boxes of 64 values (128 B, 128-byte
  // swizzle) x 16 rows, one chunk's worth per chunk
  const int vals = kChunkBlocks * block_values(g.fmt);
  CUtensorMap tm, td;
  const cuuint64_t dims[2] = {(cuuint64_t)g.K, (cuuint64_t)g.rows_max};
  const cuuint64_t strides[1] = {(cuuint64_t)g.K * 2};
  const cuuint32_t box[2] = {(cuuint32_t)kActBox, (cuuint32_t)kSmallRows};
  const cuuint32_t estr[2] = {1, 1};
  if (encode(&tm, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<__half*>(g.act), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;
  // their scales: [rows_max x scale_stride(K)] fp32, boxes of 8 (W2) or 4 blocks x 16 rows
  const int ss = scale_stride(g.K);
  const cuuint64_t ddims[2] = {(cuuint64_t)ss, (cuuint64_t)g.rows_max};
  const cuuint64_t dstrides[1] = {(cuuint64_t)ss * 4};
  const cuuint32_t dbox[2] = {(cuuint32_t)(vals / 32), (cuuint32_t)kSmallRows};
  if (encode(&td, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float*>(g.act_d), ddims, dstrides,
             dbox, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;

  // one item per (small expert, 256-row weight tile); two CTAs a multiprocessor
  const int64_t n_wtiles = (g.N_out + kTN - 1) / kTN;
  const int64_t items_max = (int64_t)std::min<int64_t>(g.E, g.rows_max) * n_wtiles;
  const int grid = (int)std::max<int64_t>(1, std::min<int64_t>(items_max, 2 * device_sm_count()));
  const int mode = g.which == 1 ? kModeDown : (g.hq ? kModeSwiglu : kModeGU);
  cudaError_t e;
  if (g.fmt == MOE_FMT_W2) {
    e = mode == kModeDown     ? launch_small<MOE_FMT_W2, kModeDown>(a, tm, td, grid, st)
        : mode == kModeSwiglu ? launch_small<MOE_FMT_W2, kModeSwiglu>(a, tm, td, grid, st)
                              : launch_small<MOE_FMT_W2, kModeGU>(a, tm, td, grid, st);
  } else {
    e = mode == kModeDown     ? launch_small<MOE_FMT_W4NL, kModeDown>(a, tm, td, grid, st)
        : mode == kModeSwiglu ? launch_small<MOE_FMT_W4NL, kModeSwiglu>(a, tm, td, grid, st)
                              : launch_small<MOE_FMT_W4NL, kModeGU>(a, tm, td, grid, st);
  }
  if (e != cudaSuccess) return e;
  count_launch();
  return cudaGetLastError();
}

}  // namespace moe
