// Grouped expert products on the 5th-generation tensor cores (tcgen05).
//
// For one expert e, output row o (a weight row) and routed row r:
//   out[r, o] = sum over 32-value K blocks b, in increasing b, of
//               d_w[o,b] * d_x[r,b] * isum_b(o, r)
// with isum_b the exact integer sum of w_int * q over the block, and the
// fp32 accumulation carried block by block in K order ("Strata #3752",
// commit "moe_ws kernels": MMQ's int8 values, scales and per-32-value
// epilogue in K order; the block's integer sum is exact, so only the float
// epilogue's order matters).
//
// Exact block sums on fp16 tensor cores.  Both operands are small integers
// held exactly in fp16 and accumulated in fp32: every product is below 2^14
// and every partial sum of a 32-value block is below 2^24.  On sm_103a the
// int8 MMA (mma.sync s8; tcgen05 kind::i8 does not exist there) runs at
// about 150 TOPS against 1.9 PFLOP/s for fp16, so fp16 is the exact route.
//
// W2 weights: the fp16 scale is folded into the operand (d*(c-2), exact in
// fp16 since c-2 is in {-2,-1,0,1}), so the tensor core returns d_w*isum
// exactly and the epilogue is one fma per (output, block):
//     acc = fma(d_x, d_w*isum, acc)
// -- one rounding where the plain statement rounds d_w*d_x first; the two
// differ by at most an ulp per block.  W4NL and Q8_0 weights (T[idx]*d and
// q*d are not exact in fp16) keep the integer operand and the two-step
// epilogue
//     acc = fma(d_w*d_x, isum, acc).
//
// Tiles: up to 128 routed rows of one expert (MMA M, the TMEM lanes; each
// expert runs its own row count, no padding to a group maximum) against 256
// weight rows (MMA N, the TMEM columns: a 128 x 256 x 16 MMA runs at the
// full tensor rate, 128 x 128 at half), K in stages of 64 values.  Experts
// are scheduled largest first over a persistent grid of one CTA per SM.
// Every 32-value block's 128 x 256 fp32 result is read back from TMEM by 16
// epilogue warps (a warp can only reach its own quarter of the lanes; four
// warps per quarter keep enough TMEM loads in flight), scaled and added into
// fp32 registers; two TMEM buffers of 256 columns let the MMA of block b+1
// run while block b is read.
//
// Warp roles (768 threads):
//   warps 0-15  epilogue: warp w owns rows 32*(w%4).. and weight-row columns
//               64*(w/4)..+63; TMEM -> registers, per-block fp32 epilogue,
//               store
//   warps 16-19 weight decode: raw blocks (bulk-copied to shared memory)
//               -> fp16 operand tile in the 128-byte swizzle layout
//   warp 20     producer: one 2-D TMA box of the tile's 128 activation rows
//               per stage
//   warp 21     MMA issue (one thread) and TMEM allocation
//   warp 22     producer: one 2-D TMA box of the tile's activation scales
//               per 4 blocks, up to 8 boxes ahead of the epilogue
//   warp 23     producer: raw weight chunks of the tiled pack (one bulk copy
//               per 256-row x 4-block chunk), one chunk ahead of the decode
// Each stream has its own ring and its own warp, so none of them waits
// behind another's barrier.
// Activations arrive in routed-row order (the q8 and swiglu_quant steps
// scatter each row to its routed slot), so a tile's rows are one contiguous
// range, and pair-interleaved within each 16-value group (position 2i holds
// value i, position 2i+1 holds value i+8), which lets the W2 decode turn a
// 32-bit code word into fp16 pairs with one logic op.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
#include <cstring>
#include <mutex>

#include "common.cuh"
#include "sm100_ptx.cuh"

namespace moe {
namespace {

using namespace ptx;

constexpr int kTM = 128;          // routed rows per tile (MMA M, TMEM lanes)
constexpr int kTN = 256;          // weight rows per tile (MMA N, TMEM columns)
constexpr int kSK = 64;           // K values per stage (one 128-byte swizzle row of fp16)
constexpr int kStages = 3;
constexpr int kTBufs = 2;         // TMEM accumulator buffers of kTN columns
constexpr int kRawSlot = 4 * kTN * kBlockBytes;  // one raw chunk of the tiled pack: 18 KB
static_assert(chunk_blocks(MOE_FMT_Q8_0) * kTN * kQ8Bytes <= kRawSlot, "Q8_0 chunk fits a slot");
constexpr int kDxRing = 8;        // activation-scale entries of 4 blocks x 128 rows
constexpr int kDwRing = 16;       // W4NL / Q8_0 weight scales, one entry per 32-value block
constexpr int kScaleBox = 4;      // scale columns per TMA box: 16 bytes a row
constexpr int kEpiWarps = 16;
constexpr int kWarpDecode = 16;   // warps 16..19
constexpr int kWarpProducer = 20;  // activations
constexpr int kWarpMma = 21;
constexpr int kWarpScales = 22;    // activation scales
constexpr int kWarpRaw = 23;       // raw weight chunks
constexpr int kThreads = 768;
// Register split.  The kernel launches at 80 registers a thread (24 warps);
// setmaxnreg then moves registers from the other roles to the epilogue.  The
// shares may not add up to more than the launch allocation (768 * 80), or
// the epilogue's increase would wait forever.
constexpr int kLaunchRegs = 80;
template <int FMT>
struct Regs {
  // epilogue 96: 64 accumulators + 16 loaded values + addressing; every
  // other warp 40.  The sum stays below the launch allocation (59392 of
  // 61440), so the increase never depends on an exact count.
  static constexpr int epi = 96;
  static constexpr int other = 40;
  static_assert(kEpiWarps * 32 * epi + (kThreads - kEpiWarps * 32) * other <
                    kThreads * kLaunchRegs,
                "register split exceeds the launch allocation");
};
constexpr uint32_t kTmemCols = kTBufs * kTN;
constexpr uint64_t kTimeoutNs = 1000000000ull;
constexpr int kMaxGrid = 1024;

constexpr int kABytes = kTM * kSK * 2;          // activation operand per stage: 16 KB
constexpr int kBBytes = kTN * kSK * 2;          // weight operand per stage: 32 KB
constexpr int kDxBytes = kTM * kScaleBox * 4;   // one scale entry: 2 KB

// shared memory layout (offsets from a 1024-aligned base)
constexpr int kOffA = 0;
constexpr int kOffB = kOffA + kStages * kABytes;
constexpr int kOffRaw = kOffB + kStages * kBBytes;
constexpr int kOffDx = kOffRaw + 2 * kRawSlot;
constexpr int kOffDw = kOffDx + kDxRing * kDxBytes;
constexpr int kOffBar = kOffDw + kDwRing * kTN * 4;
constexpr int kNumBars = 3 * kStages + 2 * kTBufs + 4 + 2 * kDxRing + 2 * kDwRing + 1;
constexpr int kOffEoff = kOffBar + kNumBars * 8;  // int64 [E] weight offsets of this product
constexpr int kOffMisc = kOffEoff + 1024 * 8;
constexpr int kSmemBytes = kOffMisc + 128 + 1024;  // + alignment slack
static_assert(kSmemBytes <= 232448, "exceeds the 227 KB of shared memory a CTA can have");
static_assert(kOffBar % 8 == 0 && kOffEoff % 8 == 0 && kOffRaw % 16 == 0 && kOffDx % 128 == 0,
              "alignment");

// What the epilogue writes: GU rows (gate/up), Hq and its scales (gate/up
// with swiglu_quant fused), Dm rows (down), or Dm rows with the combine
// fused (a mode of its own, so that the plain down kernel carries none of
// its code).
constexpr int kModeGU = 0, kModeSwiglu = 1, kModeDown = 2, kModeDownComb = 3;

struct TcArgs {
  const uint8_t* pack;  // tiled weight pack
  const int64_t* eoff;
  int which;            // 0 gate/up, 1 down
  int64_t pack_bytes;
  const int4* tiles;    // {expert, first routed row, rows, 0}, largest expert first
  const int32_t* ntiles;
  int E;
  int K;
  int N_out;
  int bpr;              // weight blocks per row
  float* out;           // GU [rows x N_out] (gate/up columns in layout gu_layout) or Dm
  int gu_layout;        // MOE_GU_*
  __half* hq;           // fused swiglu_quant: Hq [rows x N_out/2], pair-interleaved
  float* dh;            // fused swiglu_quant: scales [rows x scale_stride(N_out/2)]
  int64_t rows_max;
  int32_t* status;
};

struct Item {
  int e, row0, nrows, NW, o0;
  bool ok;
  const uint8_t* wbase;  // the 256-row weight tile in the tiled pack
};

// One work item: routed-row tile g = item / n_wtiles of the work list
// against weight-row tile item % n_wtiles.  Everything read from the work
// list is bounds-checked: a list not written by the routing step (stage API
// misuse) is skipped, never followed.
template <int FMT>
__device__ __forceinline__ Item make_item(const TcArgs& a, const int64_t* s_eoff, int4 t,
                                          int wtile) {
  constexpr int kBB = block_bytes(FMT);
  Item it;
  it.e = t.x;
  it.row0 = t.y;
  it.nrows = t.z;
  it.o0 = wtile * kTN;
  it.NW = min(kTN, a.N_out - it.o0);
  const bool rows_ok = (unsigned)it.e < (unsigned)a.E && it.row0 >= 0 && it.nrows > 0 &&
                       it.nrows <= kTM && (int64_t)it.row0 + it.nrows <= a.rows_max;
  const int64_t off = rows_ok ? s_eoff[it.e] : -1;
  const int64_t mbytes = (int64_t)a.N_out * a.bpr * kBB;
  it.ok = rows_ok && off >= 0 && (off & 15) == 0 && off + mbytes <= a.pack_bytes;
  it.wbase = it.ok ? a.pack + off + (int64_t)it.o0 * a.bpr * kBB : nullptr;
  return it;
}

__device__ __forceinline__ int4 load_tile(const TcArgs& a, int64_t item, int64_t total,
                                          int n_wtiles) {
  return item < total ? __ldg(a.tiles + item / n_wtiles) : make_int4(-1, 0, 0, 0);
}

// ---------------------------------------------------------------- decode
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

// Store 8 consecutive fp16 pairs (16 bytes) as 16-byte chunk j of row r of a
// 128-byte-swizzled K-major tile.
__device__ __forceinline__ void st_swizzled(uint8_t* tile, int r, int j, uint32_t a0, uint32_t a1,
                                            uint32_t a2, uint32_t a3) {
  uint8_t* p = tile + (r >> 3) * 1024 + (r & 7) * 128 + ((j ^ (r & 7)) << 4);
  *reinterpret_cast<uint4*>(p) = make_uint4(a0, a1, a2, a3);
}

// Decode one W2 block (64 values; code word q holds codes 16q..16q+15 at
// bits 2i) into the 128-byte row r of the stage's operand tile: fp16 pairs in
// pair-interleaved order, scale folded: pair i of word q holds
// (d*(c_{16q+i}-2), d*(c_{16q+i+8}-2)).
__device__ __forceinline__ void decode_w2_store(uint4 codes, uint16_t dh, uint8_t* tile, int r) {
  const uint32_t d2 = (uint32_t)dh | ((uint32_t)dh << 16);
  const uint32_t cw[4] = {codes.x, codes.y, codes.z, codes.w};
#pragma unroll
  for (int q = 0; q < 4; q++) {
#pragma unroll
    for (int half = 0; half < 2; half++) {
      uint32_t o[4];
#pragma unroll
      for (int i = 0; i < 4; i++) {
        // (1024 + c_i, 1024 + c_{i+8}): the codes placed in the fp16 mantissas
        const uint32_t pr = ((cw[q] >> (2 * (4 * half + i))) & 0x00030003u) | 0x64006400u;
        o[i] = hmul2_u32(hsub2_u32(pr, 0x64026402u), d2);  // (c - 2) * d, exact
      }
      st_swizzled(tile, r, 2 * q + half, o[0], o[1], o[2], o[3]);
    }
  }
}

// Decode one W4NL block (32 values; word 2g holds indices 16g..16g+7, word
// 2g+1 indices 16g+8..16g+15, nibble i at bits 4i) into 16-byte chunks
// 4*kb .. 4*kb+3 of operand row r: fp16 pairs of the integers T[idx]
// (exact), pair-interleaved.
__device__ __forceinline__ void decode_w4_store(uint4 codes, const uint16_t* lut, uint8_t* tile,
                                                int r, int kb) {
  const uint32_t cw[4] = {codes.x, codes.y, codes.z, codes.w};
#pragma unroll
  for (int g = 0; g < 2; g++) {
#pragma unroll
    for (int half = 0; half < 2; half++) {
      uint32_t o[4];
#pragma unroll
      for (int i = 0; i < 4; i++) {
        const int n = 4 * half + i;
        o[i] = (uint32_t)lut[(cw[2 * g] >> (4 * n)) & 15u] |
               ((uint32_t)lut[(cw[2 * g + 1] >> (4 * n)) & 15u] << 16);
      }
      st_swizzled(tile, r, 4 * kb + 2 * g + half, o[0], o[1], o[2], o[3]);
    }
  }
}

// fp16 pair (q_n, q_{n+8}) of two Q8_0 code words: byte sel selects code n
// of lo and code n+8 of hi into bytes 0 and 2; each byte, sign bit flipped,
// becomes the low mantissa byte of 1024 + 128 + q, and 1152 comes off: exact.
__device__ __forceinline__ uint32_t q8_pair(uint32_t lo, uint32_t hi, uint32_t sel) {
  const uint32_t t = __byte_perm(lo, hi, sel);
  return hsub2_u32((t & 0x00FF00FFu) ^ 0x64806480u, 0x64806480u);
}

// Decode one Q8_0 block (32 int8 codes; word w holds codes 4w..4w+3) into
// 16-byte chunks 4*kb .. 4*kb+3 of operand row r: fp16 integers,
// pair-interleaved like the other formats.
__device__ __forceinline__ void decode_q8_store(const uint4* codes, uint8_t* tile, int r, int kb) {
  const uint4 a = codes[0], b = codes[1];
  const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
  for (int g = 0; g < 2; g++) {
#pragma unroll
    for (int half = 0; half < 2; half++) {
      uint32_t o[4];
#pragma unroll
      for (int i = 0; i < 4; i++) {
        // values n = 4*half + i and n + 8 of group g: byte i of words
        // 4g + half and 4g + 2 + half
        const uint32_t sel = (uint32_t)(i | (i << 4) | ((4 + i) << 8) | ((4 + i) << 12));
        o[i] = q8_pair(w[4 * g + half], w[4 * g + 2 + half], sel);
      }
      st_swizzled(tile, r, 4 * kb + 2 * g + half, o[0], o[1], o[2], o[3]);
    }
  }
}

// ------------------------------------------------------------- epilogue
// 32-byte store of 8 consecutive fp32 values (4 packed pairs); p 32-byte aligned.
__device__ __forceinline__ void st_global_v8(float* p, const float2* v) {
  asm volatile("st.global.v8.f32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(p), "f"(v[0].x),
               "f"(v[0].y), "f"(v[1].x), "f"(v[1].y), "f"(v[2].x), "f"(v[2].y), "f"(v[3].x),
               "f"(v[3].y)
               : "memory");
}
__device__ __forceinline__ void st_global_v8_u32(void* p, const uint32_t* v) {
  asm volatile("st.global.v8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(p), "r"(v[0]), "r"(v[1]),
               "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7])
               : "memory");
}

// One q8 block of H from a thread's 32 gate values (acc[0..15]) and the
// matching 32 up values (acc[16..31]): H = silu(g)*u, each step rounded to
// fp32 ("Strata #3752", commit "swiglu_quant"), then d = amax/127 and
// q = rint(h/d) (d = 0 gives q = 0), stored as exact fp16 integers,
// pair-interleaved in each 16-value group, with the block's scale.
__device__ __forceinline__ void swiglu_q8_block_store(float2* acc, __half* hq, float* dh) {
  float amax = 0.0f;
#pragma unroll
  for (int j = 0; j < 16; j++) {
    const float2 g = acc[j], u = acc[16 + j];
    const float h0 = __fmul_rn(__fdiv_rn(g.x, __fadd_rn(1.0f, expf(-g.x))), u.x);
    const float h1 = __fmul_rn(__fdiv_rn(g.y, __fadd_rn(1.0f, expf(-g.y))), u.y);
    acc[j] = make_float2(h0, h1);
    amax = fmaxf(amax, fmaxf(fabsf(h0), fabsf(h1)));
  }
  const float d = __fdiv_rn(amax, 127.0f);
  uint32_t w[16];
#pragma unroll
  for (int g = 0; g < 2; g++) {
#pragma unroll
    for (int i = 0; i < 8; i++) {
      // values 16g+i and 16g+i+8 (acc holds value pairs 2j, 2j+1 in acc[j])
      const int lo = 16 * g + i, hi = lo + 8;
      const float vlo = (lo & 1) ? acc[lo >> 1].y : acc[lo >> 1].x;
      const float vhi = (hi & 1) ? acc[hi >> 1].y : acc[hi >> 1].x;
      const float q0 = (d == 0.0f) ? 0.0f : rintf(__fdiv_rn(vlo, d));
      const float q1 = (d == 0.0f) ? 0.0f : rintf(__fdiv_rn(vhi, d));
      const __half2 hq2 = __floats2half2_rn(q0, q1);  // exact: |q| <= 127
      w[8 * g + i] = *reinterpret_cast<const uint32_t*>(&hq2);
    }
  }
  st_global_v8_u32(hq, w);
  st_global_v8_u32(hq + 16, w + 8);
  *dh = d;
}

// Exit drain of a producer's ring: `issued` copies were armed on the full
// barriers full[i % n] (phase parity (i / n) & 1); the consumers waited for
// all but possibly the last n of them.  Waits for those with the polling
// wait, bounded by its count alone (not cut short by the abort flag), so no
// bulk or tensor copy is still writing shared memory when the CTA exits.
__device__ __forceinline__ void drain_ring(uint64_t* full, uint32_t n, uint32_t issued,
                                           volatile int* abort) {
  for (uint32_t i = issued > n ? issued - n : 0; i < issued; i++)
    if (!mbar_wait(&full[i % n], (i / n) & 1, abort, kTimeoutNs, false)) break;
}

// ---------------------------------------------------------------- kernel
template <int FMT, int MODE>
__global__ void __launch_bounds__(kThreads, 1)
gemm_tc_kernel(const TcArgs a, const __grid_constant__ CUtensorMap tmap,
               const __grid_constant__ CUtensorMap tmap_d, const CombineArgs comb) {
  constexpr bool kFold = (FMT == MOE_FMT_W2);
  constexpr bool kDown = (MODE == kModeDown || MODE == kModeDownComb);
  constexpr int kBps = kFold ? 1 : 2;                  // weight blocks per stage
  constexpr int kCB = chunk_blocks(FMT);               // weight blocks per raw chunk
  constexpr int kCode = code_bytes(FMT);               // code bytes per (row, block)
  constexpr int kBB = block_bytes(FMT);
  constexpr int kSpc = kCB / kBps;                     // stages per raw chunk

  extern __shared__ uint8_t smem_raw[];
  // 1024-byte aligned base, offset from the shared array itself (an integer
  // round trip would hide the shared address space from the compiler)
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint8_t* sA = smem + kOffA;
  uint8_t* sB = smem + kOffB;
  uint8_t* sRaw = smem + kOffRaw;
  float* sDx = reinterpret_cast<float*>(smem + kOffDx);  // [kDxRing][kTM rows][4 blocks]
  float* sDw = reinterpret_cast<float*>(smem + kOffDw);  // [kDwRing][kTN]
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kOffBar);
  uint64_t* full_tma = bars;                  // [kStages] activation bytes landed
  uint64_t* full_dec = bars + kStages;        // [kStages] decode warps
  uint64_t* empty = bars + 2 * kStages;       // [kStages] MMA commit
  uint64_t* tfull = bars + 3 * kStages;       // [kTBufs]  MMA commit
  uint64_t* tempty = tfull + kTBufs;          // [kTBufs]  epilogue warps
  uint64_t* rfull = tempty + kTBufs;          // [2]       raw bytes landed
  uint64_t* rempty = rfull + 2;               // [2]       decode warps done with the slot
  uint64_t* dfull = rempty + 2;               // [kDxRing] scale bytes landed
  uint64_t* dempty = dfull + kDxRing;         // [kDxRing] epilogue warps
  uint64_t* wfull = dempty + kDxRing;         // [kDwRing] decode warps (W4NL / Q8_0 scales)
  uint64_t* wempty = wfull + kDwRing;         // [kDwRing] epilogue warps
  uint64_t* fin = wempty + kDwRing;           // MMA drain at exit
  int64_t* s_eoff = reinterpret_cast<int64_t*>(smem + kOffEoff);
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(smem + kOffMisc);
  volatile int* s_abort = reinterpret_cast<volatile int*>(smem + kOffMisc + 4);
  uint16_t* s_lut = reinterpret_cast<uint16_t*>(smem + kOffMisc + 64);  // W4NL table

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  if (tid == 0) {
    for (int s = 0; s < kStages; s++) {
      mbar_init(&full_tma[s], 1);   // the producer's expect-tx arrival
      mbar_init(&full_dec[s], 4);   // one arrival per decode warp
      mbar_init(&empty[s], 1);      // MMA commit
    }
    for (int b = 0; b < kTBufs; b++) {
      mbar_init(&tfull[b], 1);
      mbar_init(&tempty[b], kEpiWarps);
    }
    for (int b = 0; b < 2; b++) {
      mbar_init(&rfull[b], 1);
      mbar_init(&rempty[b], 4);
    }
    for (int j = 0; j < kDxRing; j++) {
      mbar_init(&dfull[j], 1);
      mbar_init(&dempty[j], kEpiWarps);
    }
    for (int j = 0; j < kDwRing; j++) {
      mbar_init(&wfull[j], 4);
      mbar_init(&wempty[j], kEpiWarps);
    }
    mbar_init(fin, 1);
    *s_abort = 0;
    fence_mbar_init();
  }
  if (warp == kWarpMma) {
    tmem_alloc(s_tmem, kTmemCols);
    tmem_relinquish();
    tc_fence_before();
  }
  for (int e = tid; e < a.E; e += kThreads) s_eoff[e] = a.eoff[2 * e + a.which];
  if (FMT == MOE_FMT_W4NL && tid < 16) s_lut[tid] = c_nl4_half[tid];
  __syncthreads();
  tc_fence_after();

  const int n_wtiles = (a.N_out + kTN - 1) / kTN;
  // the big experts' tiles [0, ntiles[1]); the small-expert tier takes the rest
  const int64_t total =
      (int64_t)max(0, min(min(a.ntiles[1], a.ntiles[0]), (int)max_tiles(a.rows_max, a.E))) *
      n_wtiles;
  const int nstages = a.K / kSK;
  const int nb = 2 * nstages;  // 32-value blocks of the reduction
  const uint32_t tmem = *s_tmem;
  const int64_t stride = gridDim.x;

  if (warp < kEpiWarps) {
    // ================================================== epilogue
    // (kept lean in registers: 64 accumulators and 16 loaded values leave
    // little room, and a spill reload inside the block loop costs more than
    // recomputing a value)
    setmaxnreg_inc<Regs<FMT>::epi>();
    const int q = warp & 3, h = warp >> 2;
    const int trow = 32 * q + lane;  // routed row within the tile (TMEM lane)
    const float* dxrow = sDx + trow * kScaleBox;
    uint32_t gb = 0;  // 32-value blocks consumed so far (TMEM buffer gb & 1)
    uint32_t gd = 0;  // activation-scale entries consumed so far
    bool alive = true;
    // the next item's tile entry is loaded one item ahead (its global-memory
    // latency then runs under the current item)
    int4 tnext = load_tile(a, blockIdx.x, total, n_wtiles);
    for (int item = blockIdx.x; item < (int)total && alive; item += (int)stride) {
      const int wtile = item % n_wtiles;
      const Item I = make_item<FMT>(a, s_eoff, tnext, wtile);
      tnext = load_tile(a, item + stride, total, n_wtiles);
      if (!I.ok) {
        if (lane == 0 && warp == 0) atomicOr(a.status, MOE_STATUS_BAD_OFFSET);
        continue;
      }
      // This warp's 64 TMEM columns, 16 per load: down, columns 64h..64h+63
      // of the tile; gate/up (tile = NWg gate rows, then the matching NWg up
      // rows), gate columns 32h..32h+31 and the up columns NWg + 32h.. of the
      // same outputs.  tc0 covers loads 0-1, tc1 loads 2-3.
      const int nwg = I.NW >> 1;
      const uint32_t tc0 = tmem + ((uint32_t)(32 * q) << 16) + (kDown ? 64 * h : 32 * h);
      const uint32_t tc1 = kDown ? tc0 + 32 : tc0 + nwg;
      // warp-uniform: this warp's rows and columns hold results
      const bool active = 32 * q < I.nrows && (kDown ? 64 * h < I.NW : 32 * h < nwg);
      float2 acc[32];  // columns of load c, pair j in acc[8c + j]
#pragma unroll
      for (int i = 0; i < 32; i++) acc[i] = make_float2(0.0f, 0.0f);
      for (int b = 0; b < nb; b++, gb++) {
        const uint32_t buf = gb & 1, de = gd % kDxRing;
        if ((b & 3) == 0 &&
            !(alive = mbar_wait(&dfull[de], (gd / kDxRing) & 1, s_abort, kTimeoutNs, false)))
          break;
        // the block's activation scale, read before the wait for its product:
        // under the MMAs' operand traffic a shared-memory read takes hundreds
        // of cycles, and here it runs under that wait
        const float dx = dxrow[de * (kTM * kScaleBox) + (b & 3)];
        if (!kFold && !(alive = mbar_wait(&wfull[gb % kDwRing], (gb / kDwRing) & 1, s_abort,
                                          kTimeoutNs, false)))
          break;
        if (!(alive = mbar_wait(&tfull[buf], (gb >> 1) & 1, s_abort, kTimeoutNs, false))) break;
        tc_fence_after();
        if (active) {
          const float2 dx2 = make_float2(dx, dx);
#pragma unroll
          for (int c = 0; c < 4; c++) {
            // 16 columns per TMEM load; the buffer is handed back once the
            // last load of the block has landed
            const uint32_t taddr = (c < 2 ? tc0 : tc1) + buf * kTN + 16 * (c & 1);
            float2 v[8];
            tmem_ld16x2(taddr, v);
            tmem_wait_ld();
            if (c == 3) {
              tc_fence_before();
              __syncwarp();
              if (lane == 0) mbar_arrive(&tempty[buf]);
            }
            if (kFold) {
#pragma unroll
              for (int j = 0; j < 8; j++) acc[8 * c + j] = __ffma2_rn(dx2, v[j], acc[8 * c + j]);
            } else {
              // weight scales of the same columns (tile rows)
              const float* dws = sDw + (gb % kDwRing) * kTN + (taddr & 0xFFFFu) - (buf * kTN) -
                                 (uint32_t)(tmem & 0xFFFFu);
#pragma unroll
              for (int j = 0; j < 4; j++) {
                // 16-byte loads: the 16 columns start 64-byte aligned
                const float4 w4 = *reinterpret_cast<const float4*>(dws + 4 * j);
                acc[8 * c + 2 * j] = __ffma2_rn(__fmul2_rn(make_float2(w4.x, w4.y), dx2),
                                                v[2 * j], acc[8 * c + 2 * j]);
                acc[8 * c + 2 * j + 1] = __ffma2_rn(__fmul2_rn(make_float2(w4.z, w4.w), dx2),
                                                    v[2 * j + 1], acc[8 * c + 2 * j + 1]);
              }
            }
          }
        } else {
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&tempty[buf]);
        }
        // this block's scales are read: release the entries
        const bool last_of_entry = (b & 3) == 3 || b == nb - 1;
        if (last_of_entry || !kFold) {
          __syncwarp();
          if (lane == 0) {
            if (last_of_entry) mbar_arrive(&dempty[de]);
            if (!kFold) mbar_arrive(&wempty[gb % kDwRing]);
          }
        }
        if (last_of_entry) gd++;
      }
      if (!alive) break;
      if (!active || trow >= I.nrows) continue;
      const int64_t row = I.row0 + trow;  // routed row
      if (kDown) {
        // Dm row, outputs o0 + 64h .. + 63: 32-byte stores
        float* outp = a.out + row * a.N_out + I.o0 + 64 * h;
#pragma unroll
        for (int j = 0; j < 8; j++) st_global_v8(outp + 8 * j, acc + 4 * j);
        if (MODE == kModeDownComb) {
          // this thread stored both 32-column groups of its row (the combine
          // fused into the epilogue: a parameter of its own, so that the
          // other products' arguments keep their layout)
          combine_arrive(comb, a.out, a.rows_max, a.N_out, row, I.o0 + 64 * h);
          combine_arrive(comb, a.out, a.rows_max, a.N_out, row, I.o0 + 64 * h + 32);
        }
      } else if (MODE == kModeGU) {
        // gate outputs 128t + 32h .. + 31, and the matching up outputs
        const int o = (I.o0 >> 1) + 32 * h;
        if (a.gu_layout == MOE_GU_INTERLEAVED) {
          // gate j at column 2j, up j at 2j+1: 8 floats = outputs 4m .. 4m+3
          float* p = a.out + row * a.N_out + 2 * o;
#pragma unroll
          for (int m = 0; m < 8; m++) {
            const float2 g0 = acc[2 * m], g1 = acc[2 * m + 1];
            const float2 u0 = acc[16 + 2 * m], u1 = acc[16 + 2 * m + 1];
            const float2 v[4] = {make_float2(g0.x, u0.x), make_float2(g0.y, u0.y),
                                 make_float2(g1.x, u1.x), make_float2(g1.y, u1.y)};
            st_global_v8(p + 8 * m, v);
          }
        } else {
          float* gp = a.out + row * a.N_out + o;
          float* up = gp + (a.N_out >> 1);
#pragma unroll
          for (int j = 0; j < 4; j++) {
            st_global_v8(gp + 8 * j, acc + 4 * j);
            st_global_v8(up + 8 * j, acc + 16 + 4 * j);
          }
        }
      } else {
        // swiglu_quant fused: H = silu(g) * u for the 32 outputs
        // o .. o+31 (one q8 block of H), quantized to q8 in registers
        const int o = (I.o0 >> 1) + 32 * h;
        swiglu_q8_block_store(acc, a.hq + row * (a.N_out >> 1) + o,
                              a.dh + row * scale_stride(a.N_out >> 1) + (o >> 5));
      }
    }
  } else if (warp < kWarpDecode + 4) {
    // ================================================== weight decode
    setmaxnreg_dec<Regs<FMT>::other>();
    const int t = tid - kWarpDecode * 32;  // rows t and t + 128 of the weight tile
    uint32_t it = 0, cc = 0, gw = 0;
    bool alive = true;
    for (int64_t item = blockIdx.x; item < total && alive; item += stride) {
      // (this role runs ahead of the MMA; its per-item load latency is hidden)
      const Item I = make_item<FMT>(a, s_eoff, load_tile(a, item, total, n_wtiles),
                               (int)(item % n_wtiles));
      if (!I.ok) continue;
      const uint8_t* raw = nullptr;
      uint32_t slot = 0;
      int nbc = 0;
      for (int s = 0; s < nstages; s++, it++) {
        const int sc = s % kSpc;
        if (sc == 0) {
          slot = cc & 1;
          if (!(alive = mbar_wait(&rfull[slot], (cc >> 1) & 1, s_abort, kTimeoutNs))) break;
          raw = sRaw + slot * kRawSlot;
          nbc = min(kCB, a.bpr - (s / kSpc) * kCB);
        }
        const int st = it % kStages;
        const uint8_t* codes = raw;
        const uint16_t* scales = reinterpret_cast<const uint16_t*>(raw + nbc * I.NW * kCode);
        // W2: this thread's two rows' codes and scales, read before the wait
        // for the stage (the raw slot is already full; the reads run under it)
        uint4 wc[2];
        uint16_t wd[2];
        if (kFold) {
#pragma unroll
          for (int rr = 0; rr < 2; rr++) {
            const int idx = sc * I.NW + min(t + 128 * rr, I.NW - 1);
            wc[rr] = *reinterpret_cast<const uint4*>(codes + idx * 16);
            wd[rr] = scales[idx];
          }
        }
        if (!(alive = mbar_wait(&empty[st], ((it / kStages) & 1) ^ 1, s_abort, kTimeoutNs))) break;
        uint8_t* tileB = sB + st * kBBytes;
        if (kFold) {
#pragma unroll
          for (int rr = 0; rr < 2; rr++) {
            const int r = t + 128 * rr;
            if (r < I.NW) decode_w2_store(wc[rr], wd[rr], tileB, r);
          }
        } else {
          // two blocks per stage, each with its own scale slot in the ring
#pragma unroll
          for (int kb = 0; kb < 2; kb++) {
            const uint32_t w = gw + kb;
            if (!(alive = mbar_wait(&wempty[w % kDwRing], ((w / kDwRing) & 1) ^ 1, s_abort,
                                    kTimeoutNs)))
              break;
#pragma unroll
            for (int rr = 0; rr < 2; rr++) {
              const int r = t + 128 * rr;
              if (r < I.NW) {
                const int idx = (2 * sc + kb) * I.NW + r;
                if (FMT == MOE_FMT_W4NL)
                  decode_w4_store(*reinterpret_cast<const uint4*>(codes + idx * kCode), s_lut,
                                  tileB, r, kb);
                else
                  decode_q8_store(reinterpret_cast<const uint4*>(codes + idx * kCode), tileB, r,
                                  kb);
                sDw[(w % kDwRing) * kTN + r] = __half2float(__ushort_as_half(scales[idx]));
              }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&wfull[w % kDwRing]);
          }
          if (!alive) break;
          gw += 2;
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&full_dec[st]);
        if (sc == kSpc - 1 || s == nstages - 1) {
          if (lane == 0) mbar_arrive(&rempty[slot]);
          cc++;
        }
      }
    }
  } else if (warp == kWarpProducer) {
    // ================================================== activation producer
    setmaxnreg_dec<Regs<FMT>::other>();
    if (lane == 0) {
      prefetch_tmap(&tmap);
      uint32_t it = 0;
      bool alive = true;
      for (int64_t item = blockIdx.x; item < total && alive; item += stride) {
        const Item I = make_item<FMT>(a, s_eoff, load_tile(a, item, total, n_wtiles),
                                 (int)(item % n_wtiles));
        if (!I.ok) continue;
        for (int s = 0; s < nstages; s++, it++) {
          const int st = it % kStages;
          if (!(alive = mbar_wait(&empty[st], ((it / kStages) & 1) ^ 1, s_abort, kTimeoutNs)))
            break;
          // the tile's 128 activation rows (rows past the tile, or past the
          // buffer: zero fill, land on TMEM lanes never read)
          mbar_arrive_expect_tx(&full_tma[st], (uint32_t)kABytes);
          tma_load_2d(sA + st * kABytes, &tmap, s * kSK, I.row0, &full_tma[st]);
        }
      }
      // exit drain: copies the MMA never waited for (after an abort) land
      // before the CTA exits; only the last kStages can still be in flight
      drain_ring(full_tma, kStages, it, s_abort);
    }
    __syncwarp();
  } else if (warp == kWarpScales) {
    // ================================================== activation-scale producer
    // runs up to kDxRing entries (4 blocks each) ahead of the epilogue
    setmaxnreg_dec<Regs<FMT>::other>();
    if (lane == 0) {
      prefetch_tmap(&tmap_d);
      uint32_t gd = 0;
      bool alive = true;
      for (int64_t item = blockIdx.x; item < total && alive; item += stride) {
        const Item I = make_item<FMT>(a, s_eoff, load_tile(a, item, total, n_wtiles),
                                 (int)(item % n_wtiles));
        if (!I.ok) continue;
        for (int j = 0; j < (nb + 3) / 4; j++, gd++) {
          // scales of blocks 4j .. 4j+3 of the tile's 128 rows
          const uint32_t de = gd % kDxRing;
          if (!(alive = mbar_wait(&dempty[de], ((gd / kDxRing) & 1) ^ 1, s_abort, kTimeoutNs)))
            break;
          mbar_arrive_expect_tx(&dfull[de], (uint32_t)kDxBytes);
          tma_load_2d(sDx + de * (kTM * kScaleBox), &tmap_d, 4 * j, I.row0, &dfull[de]);
        }
      }
      drain_ring(dfull, kDxRing, gd, s_abort);
    }
    __syncwarp();
  } else if (warp == kWarpRaw) {
    // ================================================== raw weight producer
    // one bulk copy per (256-row tile, 4-block chunk), into two slots
    setmaxnreg_dec<Regs<FMT>::other>();
    if (lane == 0) {
      const int chunks_per_item = (a.bpr + kCB - 1) / kCB;
      uint32_t issued = 0;
      bool alive = true;
      for (int64_t item = blockIdx.x; item < total && alive; item += stride) {
        const Item I = make_item<FMT>(a, s_eoff, load_tile(a, item, total, n_wtiles),
                                 (int)(item % n_wtiles));
        if (!I.ok) continue;
        for (int c = 0; c < chunks_per_item; c++, issued++) {
          const uint32_t slot = issued & 1;
          if (!(alive = mbar_wait(&rempty[slot], ((issued >> 1) & 1) ^ 1, s_abort, kTimeoutNs)))
            break;
          const int nbc = min(kCB, a.bpr - c * kCB);
          const uint32_t bytes = (uint32_t)(nbc * I.NW * kBB);
          mbar_arrive_expect_tx(&rfull[slot], bytes);
          bulk_g2s(sRaw + slot * kRawSlot, I.wbase + (int64_t)c * kCB * I.NW * kBB,
                   bytes, &rfull[slot]);
        }
      }
      drain_ring(rfull, 2, issued, s_abort);
    }
    __syncwarp();
  } else if (warp == kWarpMma) {
    // ================================================== MMA issue
    setmaxnreg_dec<Regs<FMT>::other>();
    if (lane == 0) {
      uint32_t it = 0, bc = 0;
      bool alive = true;
      int4 tnext = load_tile(a, blockIdx.x, total, n_wtiles);
      for (int64_t item = blockIdx.x; item < total && alive; item += stride) {
        const Item I = make_item<FMT>(a, s_eoff, tnext, (int)(item % n_wtiles));
        tnext = load_tile(a, item + stride, total, n_wtiles);
        if (!I.ok) continue;
        const uint32_t idesc = idesc_f16_f32(kTM, I.NW);  // M = routed rows, N = weight rows
        for (int s = 0; s < nstages && alive; s++, it++) {
          const int st = it % kStages;
          const uint32_t ph = (it / kStages) & 1;
          if (!mbar_wait(&full_tma[st], ph, s_abort, kTimeoutNs, false) ||
              !mbar_wait(&full_dec[st], ph, s_abort, kTimeoutNs, false)) {
            alive = false;
            break;
          }
          tc_fence_after();
          const uint32_t xaddr = smem_u32(sA + st * kABytes);  // routed rows: MMA A operand
          const uint32_t waddr = smem_u32(sB + st * kBBytes);  // weights: MMA B operand
          for (int kb = 0; kb < 2; kb++) {
            const uint32_t buf = bc & 1;
            if (!mbar_wait(&tempty[buf], ((bc >> 1) & 1) ^ 1, s_abort, kTimeoutNs, false)) {
              alive = false;
              break;
            }
            tc_fence_after();
            const uint32_t d_tmem = tmem + buf * kTN;
#pragma unroll
            for (int k16 = 0; k16 < 2; k16++) {
              const uint32_t koff = kb * 64 + k16 * 32;  // bytes along the 128-byte row
              mma_f16(d_tmem, smem_desc_sw128(xaddr + koff), smem_desc_sw128(waddr + koff),
                      idesc, k16);
            }
            mma_commit(&tfull[buf]);
            bc++;
          }
          if (!alive) break;
          mma_commit(&empty[st]);
        }
      }
      // drain: every MMA issued above has completed once this arrives (a
      // polling wait, bounded by its count alone: it does not give up early
      // when another role has set the abort flag, so TMEM is never freed
      // under a running MMA)
      mma_commit(fin);
      mbar_wait(fin, 0, s_abort, kTimeoutNs, false);
    }
    __syncwarp();
  }

  if (*s_abort && tid == 0) atomicOr(a.status, MOE_STATUS_PIPE_TIMEOUT);
  tc_fence_before();
  __syncthreads();
  if (warp == kWarpMma) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// ------------------------------------------------------------ host side
PFN_cuTensorMapEncodeTiled_v12000 get_encode() {
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

// Shared-memory size attribute, and a check that the kernel was built with
// the register count the role split assumes (a smaller launch allocation
// would leave the epilogue's register increase waiting forever).
template <int FMT, int MODE>
cudaError_t prepare_kernel() {
  // once per device and context (the attribute does not outlive the context)
  static std::atomic<uint64_t> ready[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  const uint64_t ctx = current_context_id();
  if (ctx != 0 && ready[dev].load(std::memory_order_acquire) == ctx) return cudaSuccess;
  cudaFuncAttributes attr;
  cudaError_t e = cudaFuncGetAttributes(&attr, gemm_tc_kernel<FMT, MODE>);
  if (e != cudaSuccess) return e;
  if (attr.numRegs != kLaunchRegs) return cudaErrorInvalidKernelImage;
  e = cudaFuncSetAttribute(gemm_tc_kernel<FMT, MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           kSmemBytes);
  if (e == cudaSuccess) ready[dev].store(ctx, std::memory_order_release);
  return e;
}

}  // namespace

bool tc_supported(const MoeLayerDesc& d) {
  // K of both products a multiple of one 64-value stage, outputs a multiple
  // of 128 rows (one 128- or 256-row weight tile at the end)
  return d.d % kSK == 0 && d.n_ff % kSK == 0 && d.d % 128 == 0 && (2 * d.n_ff) % 128 == 0;
}

cudaError_t launch_gemm_tc(const GemmArgs& g, cudaStream_t st) {
  if (g.rows_max == 0) return cudaSuccess;
  TcArgs a{};
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
  a.gu_layout = g.gu_layout;
  a.rows_max = g.rows_max;
  a.status = g.status;

  auto encode = get_encode();
  if (!encode) return cudaErrorNotSupported;
  CUtensorMap tmap;
  const cuuint64_t dims[2] = {(cuuint64_t)g.K, (cuuint64_t)g.rows_max};
  const cuuint64_t strides[1] = {(cuuint64_t)g.K * 2};
  const cuuint32_t box[2] = {(cuuint32_t)kSK, (cuuint32_t)kTM};
  const cuuint32_t estr[2] = {1, 1};
  if (encode(&tmap, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<__half*>(g.act), dims, strides,
             box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;
  CUtensorMap tmap_d;
  const int ss = scale_stride(g.K);
  const cuuint64_t ddims[2] = {(cuuint64_t)ss, (cuuint64_t)g.rows_max};
  const cuuint64_t dstrides[1] = {(cuuint64_t)ss * 4};
  const cuuint32_t dbox[2] = {(cuuint32_t)kScaleBox, (cuuint32_t)kTM};
  if (encode(&tmap_d, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float*>(g.act_d), ddims,
             dstrides, dbox, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;

  const int64_t tiles_max = max_tiles(g.rows_max, g.E) * (int64_t)((g.N_out + kTN - 1) / kTN);
  const int grid = (int)std::min<int64_t>(std::min<int64_t>(tiles_max, device_sm_count()),
                                          kMaxGrid);
  const int mode = g.which == 1 ? (g.comb.out ? kModeDownComb : kModeDown)
                                : (g.hq ? kModeSwiglu : kModeGU);
  cudaError_t e = cudaSuccess;
#define MOE_LAUNCH_TC(F, M)                                                             \
  if ((e = prepare_kernel<F, M>()) != cudaSuccess) return e;                            \
  gemm_tc_kernel<F, M><<<grid, kThreads, kSmemBytes, st>>>(a, tmap, tmap_d, g.comb);
  if (g.fmt == MOE_FMT_W2) {
    if (mode == kModeDown) { MOE_LAUNCH_TC(MOE_FMT_W2, kModeDown) }
    else if (mode == kModeDownComb) { MOE_LAUNCH_TC(MOE_FMT_W2, kModeDownComb) }
    else if (mode == kModeSwiglu) { MOE_LAUNCH_TC(MOE_FMT_W2, kModeSwiglu) }
    else { MOE_LAUNCH_TC(MOE_FMT_W2, kModeGU) }
  } else if (g.fmt == MOE_FMT_W4NL) {
    if (mode == kModeDown) { MOE_LAUNCH_TC(MOE_FMT_W4NL, kModeDown) }
    else if (mode == kModeDownComb) { MOE_LAUNCH_TC(MOE_FMT_W4NL, kModeDownComb) }
    else if (mode == kModeSwiglu) { MOE_LAUNCH_TC(MOE_FMT_W4NL, kModeSwiglu) }
    else { MOE_LAUNCH_TC(MOE_FMT_W4NL, kModeGU) }
  } else {
    if (mode == kModeDown) { MOE_LAUNCH_TC(MOE_FMT_Q8_0, kModeDown) }
    else if (mode == kModeDownComb) { MOE_LAUNCH_TC(MOE_FMT_Q8_0, kModeDownComb) }
    else if (mode == kModeSwiglu) { MOE_LAUNCH_TC(MOE_FMT_Q8_0, kModeSwiglu) }
    else { MOE_LAUNCH_TC(MOE_FMT_Q8_0, kModeGU) }
  }
#undef MOE_LAUNCH_TC
  count_launch();
  return cudaGetLastError();
}

}  // namespace moe
