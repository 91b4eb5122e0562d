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
// differ by at most an ulp per block.  W4NL weights (T[idx]*d is not exact
// in fp16) keep the integer operand and the two-step epilogue
//     acc = fma(d_w*d_x, isum, acc).
//
// Tiles: up to 128 routed rows of one expert (MMA M, the TMEM lanes; each
// expert runs its own row count, no padding to a group maximum) against 128
// weight rows (MMA N, the TMEM columns), K in stages of 64 values.  Experts
// are scheduled largest first over a persistent grid of one CTA per SM.
// With routed rows on the lanes, a thread owns one row and its activation
// scale is a single register per block: the epilogue is packed fp32 fmas
// (two per issue slot) on values read from TMEM.  Four TMEM accumulator
// buffers let the epilogue load block b+1 while it computes block b.
//
// Warp roles (512 threads):
//   warps 0-7   epilogue: warp w owns rows 32*(w%4).. and weight-row columns
//               64*(w/4)..+63; TMEM -> registers, per-block fp32 epilogue,
//               store
//   warps 8-11  weight decode: raw blocks (bulk-copied to shared memory)
//               -> fp16 operand tile in the 128-byte swizzle layout, once
//               per tile
//   warp 12     producer: raw weight bytes by TMA (a tensor map retargeted
//               per expert on the device: one 2-D box of 128 rows x 8 blocks
//               per chunk, or one bulk copy of a whole small tile), one 2-D
//               TMA box of the tile's 128 activation rows (routed-row order)
//               and one of their scales per stage
//   warp 13     MMA issue (one thread) and TMEM allocation
//   warps 14-15 idle
// Activations arrive in routed-row order (the q8 and swiglu_quant steps
// scatter each row to its routed slot), so a tile's rows are one contiguous
// range, and pair-interleaved within each 16-value group (position 2i holds
// value i, position 2i+1 holds value i+8), which lets the W2 decode turn a
// 32-bit code word into fp16 pairs with one logic op.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstring>
#include <mutex>

#include "common.cuh"
#include "sm100_ptx.cuh"

namespace moe {
namespace {

using namespace ptx;

constexpr int kM = 128;          // weight rows per tile (MMA N, TMEM columns)
constexpr int kNmax = 128;       // routed rows per tile (MMA M, TMEM lanes)
constexpr int kSub = 128;
constexpr int kTBufs = 4;        // TMEM accumulator buffers of 128 columns
constexpr int kSK = 64;          // K values per stage (one 128-byte swizzle row of fp16)
constexpr int kStages = 4;
constexpr int kRawSlot = 23040;  // bytes per raw-weight slot (128 rows x 180 B)
constexpr int kThreads = 512;
constexpr int kWarpProducer = 12;
constexpr int kWarpMma = 13;
constexpr uint32_t kTmemCols = 512;  // four buffers x 128 fp32 columns
constexpr uint64_t kTimeoutNs = 1000000000ull;
constexpr int kMaxGrid = 1024;   // CTAs; each owns two 128-byte tensor-map slots

constexpr int kScaleBox = 4;    // scale columns (32-value blocks) per TMA box: 16 bytes a row
constexpr int kABytes = kM * kSK * 2;     // weight operand per stage: 16 KB
constexpr int kBBytes = kNmax * kSK * 2;  // activation operand per stage: 16 KB

// shared memory layout (offsets from a 1024-aligned base)
constexpr int kOffA = 0;
constexpr int kOffB = kOffA + kStages * kABytes;
constexpr int kOffRaw = kOffB + kStages * kBBytes;
constexpr int kOffDx = kOffRaw + 2 * kRawSlot;
constexpr int kOffDw = kOffDx + kStages * kScaleBox * kNmax * 4;
constexpr int kOffBar = kOffDw + kStages * 2 * kM * 4;
constexpr int kNumBars = 3 * kStages + 2 * kTBufs + 2 + 2 + 1;
constexpr int kOffEoff = kOffBar + kNumBars * 8;  // int64 [E] weight offsets of this product
constexpr int kOffMisc = kOffEoff + 1024 * 8;
constexpr int kOffTmap = (kOffMisc + 256 + 127) & ~127;  // two 128-byte weight tensor maps
constexpr int kSmemBytes = kOffTmap + 256 + 1024;  // + alignment slack
static_assert(kSmemBytes <= 232448, "exceeds the 227 KB of shared memory a CTA can have");
static_assert(kOffTmap % 128 == 0 && kOffBar % 8 == 0 && kOffEoff % 8 == 0, "alignment");

struct TcArgs {
  const uint8_t* pack;
  const int64_t* eoff;
  int which;            // 0 gate/up, 1 down
  int64_t pack_bytes;
  const int4* tiles;    // {expert, first routed row, rows, 0}, largest expert first
  const int32_t* ntiles;
  int E;
  const float* act_d;   // activation scales [rows_max x scale_stride(K)]
  int K;
  int N_out;
  int64_t pitch;        // weight row bytes
  int chunk_row_bytes;  // raw bytes per row per chunk
  int stages_per_chunk;
  int raw_slots;        // 2 (ping-pong) or 1 (one tile fills both slots)
  bool rows_mode;       // raw chunks are per-row copies (else one copy of the tile)
  float* out;
  int64_t rows_max;
  int32_t* status;
  uint8_t* tmap_slots;  // per CTA: two 128-byte global slots for the weight tensor map
};

struct Item {
  int e, row0, nrows, N, o0;
  bool ok;
  const uint8_t* wbase;
};

// One work item: routed-row tile g = item / n_wtiles of the work list
// against weight-row tile item % n_wtiles.  Everything read from the work
// list is bounds-checked: a list not written by the routing step (stage API
// misuse) is skipped, never followed.
__device__ __forceinline__ Item make_item(const TcArgs& a, const int64_t* s_eoff, int4 t,
                                          int wtile) {
  Item it;
  it.e = t.x;
  it.row0 = t.y;
  it.nrows = t.z;
  it.N = (it.nrows + 15) & ~15;
  it.o0 = wtile * kM;
  const bool rows_ok = (unsigned)it.e < (unsigned)a.E && it.row0 >= 0 && it.nrows > 0 &&
                       it.nrows <= kNmax && (int64_t)it.row0 + it.nrows <= a.rows_max;
  const int64_t off = rows_ok ? s_eoff[it.e] : -1;
  it.ok = rows_ok && off >= 0 && (off & 15) == 0 && off + a.pitch * a.N_out <= a.pack_bytes;
  it.wbase = it.ok ? a.pack + off + (int64_t)it.o0 * a.pitch : nullptr;
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

// Decode one W2 block (64 values) of weight row r into the 128-byte row of
// the stage's operand tile: fp16 pairs in pair-interleaved order, scale
// folded: pair i of code word q holds (d*(c_{16q+i}-2), d*(c_{16q+i+8}-2)).
// Code words are read one at a time from the 2-byte-aligned block (a funnel
// shift of two aligned words) and each 16-byte chunk is stored as soon as it
// is built, to keep the decode warps' registers few.
__device__ __forceinline__ void decode_w2_store(const uint8_t* blk, uint8_t* tile, int r) {
  const uint16_t dh = *reinterpret_cast<const uint16_t*>(blk);
  const uint32_t d2 = (uint32_t)dh | ((uint32_t)dh << 16);
  const uintptr_t ca = reinterpret_cast<uintptr_t>(blk + 2);
  const uint32_t* cw = reinterpret_cast<const uint32_t*>(ca & ~(uintptr_t)3);
  const uint32_t sh = (uint32_t)(ca & 3) * 8;
  uint32_t prev = cw[0];
#pragma unroll
  for (int q = 0; q < 4; q++) {
    const uint32_t next = cw[q + 1];
    const uint32_t w = __funnelshift_r(prev, next, sh);
    prev = next;
#pragma unroll
    for (int half = 0; half < 2; half++) {
      uint32_t o[4];
#pragma unroll
      for (int i = 0; i < 4; i++) {
        // (1024 + c_i, 1024 + c_{i+8}): the codes placed in the fp16 mantissas
        const uint32_t pr = ((w >> (2 * (4 * half + i))) & 0x00030003u) | 0x64006400u;
        o[i] = hmul2_u32(hsub2_u32(pr, 0x64026402u), d2);  // (c - 2) * d, exact
      }
      st_swizzled(tile, r, 2 * q + half, o[0], o[1], o[2], o[3]);
    }
  }
}

// Decode one W4NL block (32 values) of weight row r into 16-byte chunks
// 4*kb .. 4*kb+3 of the operand row: fp16 pairs of the integers T[idx]
// (exact), pair-interleaved.  Returns the block scale.
__device__ __forceinline__ float decode_w4_store(const uint8_t* blk, const uint16_t* lut,
                                                 uint8_t* tile, int r, int kb) {
  const uint16_t dh = *reinterpret_cast<const uint16_t*>(blk);
  const uintptr_t ca = reinterpret_cast<uintptr_t>(blk + 2);
  const uint32_t* cw = reinterpret_cast<const uint32_t*>(ca & ~(uintptr_t)3);
  const uint32_t sh = (uint32_t)(ca & 3) * 8;
  // word 2g: values 16g..16g+7, word 2g+1: 16g+8..16g+15
#pragma unroll
  for (int g = 0; g < 2; g++) {
    const uint32_t wlo = __funnelshift_r(cw[2 * g], cw[2 * g + 1], sh);
    const uint32_t whi = __funnelshift_r(cw[2 * g + 1], cw[2 * g + 2], sh);
#pragma unroll
    for (int half = 0; half < 2; half++) {
      uint32_t o[4];
#pragma unroll
      for (int i = 0; i < 4; i++) {
        const int n = 4 * half + i;
        o[i] = (uint32_t)lut[(wlo >> (4 * n)) & 15u] | ((uint32_t)lut[(whi >> (4 * n)) & 15u] << 16);
      }
      st_swizzled(tile, r, 4 * kb + 2 * g + half, o[0], o[1], o[2], o[3]);
    }
  }
  return __half2float(__ushort_as_half(dh));
}

// ---------------------------------------------------------------- kernel
template <int FMT>
__global__ void __launch_bounds__(kThreads, 1)
gemm_tc_kernel(const TcArgs a, const __grid_constant__ CUtensorMap tmap,
               const __grid_constant__ CUtensorMap tmap_d,
               const __grid_constant__ CUtensorMap tmap_w) {
  constexpr bool kFold = (FMT == MOE_FMT_W2);

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  uint8_t* sA = smem + kOffA;
  uint8_t* sB = smem + kOffB;
  uint8_t* sRaw = smem + kOffRaw;
  float* sDx = reinterpret_cast<float*>(smem + kOffDx);  // [stage][kNmax rows][4 blocks]
  float* sDw = reinterpret_cast<float*>(smem + kOffDw);  // [stage][2][kM]
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kOffBar);
  uint64_t* full_tma = bars;                // [kStages] producer + scale copies + TMA bytes
  uint64_t* full_dec = bars + kStages;      // [kStages] decode warps
  uint64_t* empty = bars + 2 * kStages;     // [kStages] MMA commit + epilogue warps
  uint64_t* tfull = bars + 3 * kStages;     // [kTBufs]  MMA commit
  uint64_t* tempty = tfull + kTBufs;        // [kTBufs]  epilogue warps
  uint64_t* rfull = tempty + kTBufs;        // [2]       raw bytes landed
  uint64_t* rempty = rfull + 2;             // [2]       decode warps done with the slot
  uint64_t* fin = rempty + 2;               // MMA drain at exit
  int64_t* s_eoff = reinterpret_cast<int64_t*>(smem + kOffEoff);
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(smem + kOffMisc);
  volatile int* s_abort = reinterpret_cast<volatile int*>(smem + kOffMisc + 4);
  uint16_t* s_lut = reinterpret_cast<uint16_t*>(smem + kOffMisc + 64);  // W4NL table

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  if (tid == 0) {
    for (int s = 0; s < kStages; s++) {
      mbar_init(&full_tma[s], 1);   // the producer's expect-tx arrival
      mbar_init(&full_dec[s], 4);     // one arrival per decode warp
      mbar_init(&empty[s], 1 + 8);    // MMA commit + one arrival per epilogue warp
    }
    for (int b = 0; b < kTBufs; b++) {
      mbar_init(&tfull[b], 1);
      mbar_init(&tempty[b], 8);       // one arrival per epilogue warp
    }
    for (int b = 0; b < 2; b++) {
      mbar_init(&rfull[b], 1);
      mbar_init(&rempty[b], 4);       // one arrival per decode warp
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
  if (FMT != MOE_FMT_W2 && tid < 16) s_lut[tid] = c_nl4_half[tid];
  __syncthreads();
  tc_fence_after();

  const int n_wtiles = a.N_out / kM;
  const int64_t total = (int64_t)max(0, min(*a.ntiles, (int)max_tiles(a.rows_max, a.E))) * n_wtiles;
  const int nstages = a.K / kSK;
  const uint32_t tmem = *s_tmem;
  const int64_t stride = gridDim.x;

  if (warp < 8) {
    // ================================================== epilogue
    setmaxnreg_inc<216>();  // 256 x 216 + 256 x 40 = 512 x 128 registers
    const int q = warp & 3, h = warp >> 2;
    const int trow = 32 * q + lane;  // routed row within the tile (TMEM lane)
    const uint32_t tlane = tmem + ((uint32_t)(32 * q) << 16) + 64 * h;
    uint32_t it = 0, bc = 0;
    bool alive = true;
    int4 tnext = load_tile(a, blockIdx.x, total, n_wtiles);
    for (int64_t item = blockIdx.x; item < total && alive; item += stride) {
      const Item I = make_item(a, s_eoff, tnext, (int)(item % n_wtiles));
      tnext = load_tile(a, item + stride, total, n_wtiles);  // prefetch
      if (!I.ok) {
        if (lane == 0 && warp == 0) atomicOr(a.status, MOE_STATUS_BAD_OFFSET);
        continue;
      }
      const bool active = 32 * q < I.nrows;  // warp-uniform
      const int nb = 2 * nstages;            // 32-value blocks of the item
      float2 acc[32];  // columns 2i, 2i+1 of this warp's 64
#pragma unroll
      for (int i = 0; i < 32; i++) acc[i] = make_float2(0.0f, 0.0f);
      float2 va[32], vb[32];
      // Block b of the item: stage it + b/2, TMEM buffer (bc + b) % 4.
      // EPI_LOAD: wait until the MMA filled block b's buffer (and, at a
      // stage's first block, until the stage's scales landed), start the
      // TMEM read.  EPI_RELEASE: the read is in registers, hand the buffer
      // back.  EPI_COMPUTE: acc += d_x * (d_w*isum)  (W2, scale folded) or
      // acc += (d_w*d_x) * isum  (W4NL); after a stage's second block the
      // stage's scales are no longer read.
#define EPI_LOAD(b, v)                                                                   \
  {                                                                                      \
    const uint32_t st_ = (it + (b) / 2) % kStages, ph_ = ((it + (b) / 2) / kStages) & 1; \
    if (((b) & 1) == 0) {                                                                \
      alive = mbar_wait(&full_tma[st_], ph_, s_abort, kTimeoutNs, false);                       \
      if (!kFold && alive) alive = mbar_wait(&full_dec[st_], ph_, s_abort, kTimeoutNs, false); \
    }                                                                                    \
    const uint32_t n_ = bc + (b), buf_ = n_ % kTBufs;                                     \
    if (alive) alive = mbar_wait(&tfull[buf_], (n_ / kTBufs) & 1, s_abort, kTimeoutNs, false);  \
    tc_fence_after();                                                                    \
    if (alive && active) {                                                               \
      tmem_ld32x2(tlane + buf_ * kM, (v));                                               \
      tmem_ld32x2(tlane + buf_ * kM + 32, (v) + 16);                                     \
    }                                                                                    \
  }
#define EPI_RELEASE(b)                                              \
  {                                                                 \
    tmem_wait_ld();                                                 \
    tc_fence_before();                                              \
    __syncwarp();                                                   \
    if (lane == 0) mbar_arrive(&tempty[(bc + (b)) % kTBufs]);       \
  }
#define EPI_COMPUTE(b, v)                                                                 \
  {                                                                                       \
    const uint32_t st_ = (it + (b) / 2) % kStages;                                        \
    const int kb_ = (b) & 1;                                                              \
    if (active) {                                                                         \
      const float dx = sDx[(st_ * kNmax + trow) * kScaleBox + ((2 * ((b) / 2)) & 2) + kb_]; \
      const float2 dx2 = make_float2(dx, dx);                                             \
      if (kFold) {                                                                        \
        _Pragma("unroll") for (int j = 0; j < 32; j++)                                    \
            acc[j] = __ffma2_rn(dx2, (v)[j], acc[j]);                                     \
      } else {                                                                            \
        const float* dws = sDw + (st_ * 2 + kb_) * kM + 64 * h;                           \
        _Pragma("unroll") for (int j = 0; j < 32; j += 2) {                               \
          const float4 w4 = *reinterpret_cast<const float4*>(dws + 2 * j);                \
          const float2 s01 = __fmul2_rn(make_float2(w4.x, w4.y), dx2);                    \
          const float2 s23 = __fmul2_rn(make_float2(w4.z, w4.w), dx2);                    \
          acc[j] = __ffma2_rn(s01, (v)[j], acc[j]);                                       \
          acc[j + 1] = __ffma2_rn(s23, (v)[j + 1], acc[j + 1]);                           \
        }                                                                                 \
      }                                                                                   \
    }                                                                                     \
    if (kb_ == 1) {                                                                       \
      __syncwarp();                                                                       \
      if (lane == 0) mbar_arrive(&empty[st_]);                                            \
    }                                                                                     \
  }
      EPI_LOAD(0, va);
      if (!alive) break;
      EPI_RELEASE(0);
      for (int b = 0; b < nb; b += 2) {
        // even block in va, odd block in vb; the next read is in flight
        // while the current block is computed
        EPI_LOAD(b + 1, vb);
        if (!alive) break;
        EPI_COMPUTE(b, va);
        EPI_RELEASE(b + 1);
        if (b + 2 < nb) {
          EPI_LOAD(b + 2, va);
          if (!alive) break;
        }
        EPI_COMPUTE(b + 1, vb);
        if (b + 2 < nb) EPI_RELEASE(b + 2);
      }
#undef EPI_LOAD
#undef EPI_RELEASE
#undef EPI_COMPUTE
      if (!alive) break;
      it += nstages;
      bc += nb;
      // store: routed row row0 + trow, outputs o0 + 64h .. + 63
      if (trow < I.nrows) {
        float4* outp = reinterpret_cast<float4*>(a.out + (int64_t)(I.row0 + trow) * a.N_out +
                                                 I.o0 + 64 * h);
#pragma unroll
        for (int j = 0; j < 16; j++)
          outp[j] = make_float4(acc[2 * j].x, acc[2 * j].y, acc[2 * j + 1].x, acc[2 * j + 1].y);
      }
    }
  } else if (warp < 12) {
    // ================================================== weight decode
    setmaxnreg_dec<40>();
    const int r = tid - 256;  // weight row within the tile
    uint32_t it = 0, cc = 0;
    bool alive = true;
    for (int64_t item = blockIdx.x; item < total && alive; item += stride) {
      // (this role runs ahead of the MMA; its per-item load latency is hidden)
      const Item I = make_item(a, s_eoff, load_tile(a, item, total, n_wtiles),
                               (int)(item % n_wtiles));
      if (!I.ok) continue;
      const uint8_t* raw = nullptr;
      uint32_t slot = 0;
      for (int s = 0; s < nstages; s++, it++) {
        const int sc = s % a.stages_per_chunk;
        if (sc == 0) {
          slot = cc % a.raw_slots;
          if (!mbar_wait(&rfull[slot], (cc / a.raw_slots) & 1, s_abort, kTimeoutNs)) { alive = false; break; }
          raw = sRaw + slot * kRawSlot + (int64_t)r * a.chunk_row_bytes;
        }
        const int st = it % kStages;
        const uint32_t ph = (it / kStages) & 1;
        if (!mbar_wait(&empty[st], ph ^ 1, s_abort, kTimeoutNs)) { alive = false; break; }
        uint8_t* tileA = sA + st * kABytes;
        if (FMT == MOE_FMT_W2) {
          decode_w2_store(raw + sc * kBlockBytes, tileA, r);
        } else {
#pragma unroll
          for (int kb = 0; kb < 2; kb++)
            sDw[(st * 2 + kb) * kM + r] =
                decode_w4_store(raw + (sc * 2 + kb) * kBlockBytes, s_lut, tileA, r, kb);
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&full_dec[st]);
        if (sc == a.stages_per_chunk - 1 || s == nstages - 1) {
          if (lane == 0) mbar_arrive(&rempty[slot]);
          cc++;
        }
      }
    }
  } else if (warp == kWarpProducer) {
    // ================================================== producer
    setmaxnreg_dec<40>();
    prefetch_tmap(&tmap);
    prefetch_tmap(&tmap_d);
    // Raw weight chunks form one stream over this CTA's items; chunk q of an
    // item covers stages [q*spc, (q+1)*spc).  With two raw slots the next
    // chunk is issued while the current one is decoded; with one slot (a
    // tile that fills both) only once the previous one is fully decoded.
    const int spc = a.stages_per_chunk;
    const int chunks_per_item = (nstages + spc - 1) / spc;
    const int bps = (FMT == MOE_FMT_W2) ? 1 : 2;  // blocks per stage
    int64_t r_item = blockIdx.x;
    int r_chunk = 0;
    uint32_t issued = 0, r_items = 0;  // raw chunks issued, items whose raw stream began
    uint8_t* s_tmap = smem + kOffTmap;  // two copies of the weight tensor-map template
    if (a.rows_mode) {
      for (int i = lane; i < 64; i += 32)
        reinterpret_cast<uint32_t*>(s_tmap)[i] = reinterpret_cast<const uint32_t*>(&tmap_w)[i & 31];
      __syncwarp();
    }
    Item RI;
    auto seek_raw = [&]() -> bool {
      while (r_item < total) {
        RI = make_item(a, s_eoff, load_tile(a, r_item, total, n_wtiles), (int)(r_item % n_wtiles));
        if (RI.ok) return true;
        r_item += stride;
      }
      return false;
    };
    bool r_valid = seek_raw();
    auto issue_raw = [&]() -> bool {
      if (!r_valid) return true;
      const uint32_t slot = issued % a.raw_slots;
      if (!mbar_wait(&rempty[slot], ((issued / a.raw_slots) & 1) ^ 1, s_abort, kTimeoutNs))
        return false;
      const int s0 = r_chunk * spc;
      const int row_bytes = a.rows_mode ? a.chunk_row_bytes : (int)a.pitch;
      const uint32_t bytes = (uint32_t)(row_bytes * kM);
      uint8_t* dst = sRaw + slot * kRawSlot;
      uint8_t* gslot = a.tmap_slots + ((int64_t)blockIdx.x * 2 + (r_items & 1)) * 128;
      if (a.rows_mode && r_chunk == 0) {
        // point this item's weight tensor map (slots ping-pong per item) at
        // the expert's matrix; its previous user, two items back, has landed
        uint8_t* sm = s_tmap + 128 * (r_items & 1);
        if (lane == 0) tmap_replace_address(sm, RI.wbase - (int64_t)RI.o0 * a.pitch);
        __syncwarp();
        tmap_publish(gslot, sm);
      }
      if (lane == 0) {
        mbar_arrive_expect_tx(&rfull[slot], bytes);
        if (a.rows_mode)  // 128 weight rows x one chunk of 8 blocks: one 2-D box
          tma_load_2d(dst, gslot, s0 * bps * kBlockBytes, RI.o0, &rfull[slot]);
        else  // the whole contiguous 128-row tile: one bulk copy
          bulk_g2s(dst, RI.wbase, bytes, &rfull[slot]);
      }
      __syncwarp();
      issued++;
      if (++r_chunk == chunks_per_item) {
        r_chunk = 0;
        r_items++;
        r_item += stride;
        r_valid = seek_raw();
      }
      return true;
    };
    bool alive = true;
    const bool ahead = a.raw_slots == 2;
    if (ahead) alive = issue_raw();  // chunk 0
    uint32_t it = 0;
    for (int64_t item = blockIdx.x; item < total && alive; item += stride) {
      const Item I = make_item(a, s_eoff, load_tile(a, item, total, n_wtiles),
                               (int)(item % n_wtiles));
      if (!I.ok) continue;
      for (int s = 0; s < nstages; s++, it++) {
        if (s % spc == 0) {
          if (!(alive = issue_raw())) break;  // the next chunk (ahead) or this one
        }
        const int st = it % kStages;
        const uint32_t ph = (it / kStages) & 1;
        if (!mbar_wait(&empty[st], ph ^ 1, s_abort, kTimeoutNs)) { alive = false; break; }
        if (lane == 0) {
          // the tile's 128 activation rows (rows past the tile, or past the
          // buffer: zero fill, land on TMEM lanes never read) and their
          // scales: blocks (2s & ~3) .. +3, of which 2s and 2s+1 are used
          mbar_arrive_expect_tx(&full_tma[st], (uint32_t)(kBBytes + kNmax * kScaleBox * 4));
          tma_load_2d(sB + st * kBBytes, &tmap, s * kSK, I.row0, &full_tma[st]);
          tma_load_2d(sDx + st * kNmax * kScaleBox, &tmap_d, (2 * s) & ~3, I.row0, &full_tma[st]);
        }
      }
    }
  } else if (warp == kWarpMma) {
    // ================================================== MMA issue
    setmaxnreg_dec<40>();
    if (lane == 0) {
      uint32_t it = 0, bc = 0;
      bool alive = true;
      int4 tnext = load_tile(a, blockIdx.x, total, n_wtiles);
      for (int64_t item = blockIdx.x; item < total && alive; item += stride) {
        const Item I = make_item(a, s_eoff, tnext, (int)(item % n_wtiles));
        tnext = load_tile(a, item + stride, total, n_wtiles);
        if (!I.ok) continue;
        const uint32_t idesc = idesc_f16_f32(kNmax, kM);  // M = 128 routed rows, N = 128 weight rows
        for (int s = 0; s < nstages && alive; s++, it++) {
          const int st = it % kStages;
          const uint32_t ph = (it / kStages) & 1;
          if (!mbar_wait(&full_tma[st], ph, s_abort, kTimeoutNs, false) ||
              !mbar_wait(&full_dec[st], ph, s_abort, kTimeoutNs, false)) {
            alive = false;
            break;
          }
          tc_fence_after();
          const uint32_t waddr = smem_u32(sA + st * kABytes);  // weights: MMA B operand
          const uint32_t xaddr = smem_u32(sB + st * kBBytes);  // routed rows: MMA A operand
          for (int kb = 0; kb < 2; kb++) {
            const uint32_t buf = bc % kTBufs;
            if (!mbar_wait(&tempty[buf], ((bc / kTBufs) & 1) ^ 1, s_abort, kTimeoutNs, false)) {
              alive = false;
              break;
            }
            tc_fence_after();
            const uint32_t d_tmem = tmem + buf * kM;
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
      // drain: every MMA issued above has completed once this arrives
      mma_commit(fin);
      mbar_wait(fin, 0, s_abort, kTimeoutNs);
    }
    __syncwarp();
  } else {
    setmaxnreg_dec<40>();
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

template <int FMT>
cudaError_t set_smem_attr() {
  static bool done[64] = {false};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && done[dev]) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(gemm_tc_kernel<FMT>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (e == cudaSuccess && dev >= 0 && dev < 64) done[dev] = true;
  return e;
}

}  // namespace

// Raw-staging plan for one weight matrix [N_out x K]: false if unsupported.
bool tc_raw_plan(int fmt, int K, int64_t* pitch, int* chunk_row_bytes, int* stages_per_chunk,
                 int* raw_slots, bool* rows_mode) {
  const int bpr = K / block_values(fmt);  // blocks per row
  const int64_t p = (int64_t)bpr * kBlockBytes;
  const int bps = fmt == MOE_FMT_W2 ? 1 : 2;  // blocks per 64-value stage
  *pitch = p;
  if (kM * p <= 2 * kRawSlot) {  // whole tile in one chunk
    *rows_mode = false;
    *chunk_row_bytes = (int)p;
    *stages_per_chunk = K / kSK;
    *raw_slots = kM * p <= kRawSlot ? 2 : 1;
    return true;
  }
  // per-row chunks of 8 blocks (144 B): rows must start 16-byte aligned
  if (p % 16 == 0 && bpr % 8 == 0) {
    *rows_mode = true;
    *chunk_row_bytes = 8 * kBlockBytes;
    *stages_per_chunk = 8 / bps;
    *raw_slots = 2;
    return true;
  }
  return false;
}

bool tc_supported(const MoeLayerDesc& d) {
  int64_t p;
  int crb, spc, rs;
  bool rm;
  return d.d % 128 == 0 && tc_raw_plan(d.gu_fmt, d.d, &p, &crb, &spc, &rs, &rm) &&
         tc_raw_plan(d.down_fmt, d.n_ff, &p, &crb, &spc, &rs, &rm);
}

cudaError_t launch_gemm_tc(const GemmArgs& g, const void* act, uint8_t* tmap_slots,
                           cudaStream_t st) {
  if (g.rows_max == 0) return cudaSuccess;
  TcArgs a{};
  a.pack = g.pack;
  a.eoff = g.eoff;
  a.which = g.which;
  a.pack_bytes = g.pack_bytes;
  a.tiles = g.tiles;
  a.ntiles = g.ntiles;
  a.E = g.E;
  a.act_d = g.act_d;
  a.K = g.K;
  a.N_out = g.N_out;
  a.out = g.out;
  a.rows_max = g.rows_max;
  a.status = g.status;
  if (!tc_raw_plan(g.fmt, g.K, &a.pitch, &a.chunk_row_bytes, &a.stages_per_chunk, &a.raw_slots,
                   &a.rows_mode))
    return cudaErrorInvalidValue;

  auto encode = get_encode();
  if (!encode) return cudaErrorNotSupported;
  CUtensorMap tmap;
  const cuuint64_t dims[2] = {(cuuint64_t)g.K, (cuuint64_t)g.rows_max};
  const cuuint64_t strides[1] = {(cuuint64_t)g.K * 2};
  const cuuint32_t box[2] = {(cuuint32_t)kSK, (cuuint32_t)kNmax};
  const cuuint32_t estr[2] = {1, 1};
  if (encode(&tmap, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void*>(act), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;
  CUtensorMap tmap_d;
  const int ss = scale_stride(g.K);
  const cuuint64_t ddims[2] = {(cuuint64_t)ss, (cuuint64_t)g.rows_max};
  const cuuint64_t dstrides[1] = {(cuuint64_t)ss * 4};
  const cuuint32_t dbox[2] = {(cuuint32_t)kScaleBox, (cuuint32_t)kNmax};
  if (encode(&tmap_d, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float*>(g.act_d), ddims,
             dstrides, dbox, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;

  // weight tensor-map template for rows mode: [N_out rows x pitch bytes],
  // boxes of 128 rows x one chunk; the kernel retargets its base per expert
  CUtensorMap tmap_w;
  std::memset(&tmap_w, 0, sizeof(tmap_w));
  if (a.rows_mode) {
    const cuuint64_t wdims[2] = {(cuuint64_t)a.pitch, (cuuint64_t)g.N_out};
    const cuuint64_t wstrides[1] = {(cuuint64_t)a.pitch};
    const cuuint32_t wbox[2] = {(cuuint32_t)a.chunk_row_bytes, (cuuint32_t)kM};
    if (encode(&tmap_w, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(g.pack), wdims,
               wstrides, wbox, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  a.tmap_slots = tmap_slots;

  const int64_t tiles_max = max_tiles(g.rows_max, g.E) * (int64_t)(g.N_out / kM);
  const int grid = (int)std::min<int64_t>(std::min<int64_t>(tiles_max, device_sm_count()),
                                          kMaxGrid);
  cudaError_t e;
  if (g.fmt == MOE_FMT_W2) {
    if ((e = set_smem_attr<MOE_FMT_W2>()) != cudaSuccess) return e;
    gemm_tc_kernel<MOE_FMT_W2><<<grid, kThreads, kSmemBytes, st>>>(a, tmap, tmap_d, tmap_w);
  } else {
    if ((e = set_smem_attr<MOE_FMT_W4NL>()) != cudaSuccess) return e;
    gemm_tc_kernel<MOE_FMT_W4NL><<<grid, kThreads, kSmemBytes, st>>>(a, tmap, tmap_d, tmap_w);
  }
  count_launch();
  return cudaGetLastError();
}

}  // namespace moe
