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
// Tiles: 128 weight rows (MMA M, TMEM lanes) x up to 256 routed rows of one
// expert (MMA N, 16-row granularity: each expert runs its own row count,
// no padding to a group maximum), K in stages of 64 values.  Experts are
// scheduled largest first over a persistent grid of one CTA per SM.
//
// Warp roles (512 threads):
//   warps 0-7   epilogue: TMEM -> registers, per-block fp32 epilogue, store
//   warps 8-11  weight decode: raw blocks (bulk-copied to shared memory)
//               -> fp16 operand tile in the 128-byte swizzle layout, once
//               per tile
//   warp 12     producer: bulk TMA of raw weight bytes, TMA gather4 of the
//               tile's activation rows, activation scales
//   warp 13     MMA issue (one thread) and TMEM allocation
//   warps 14-15 idle
// Activations are stored pair-interleaved within each 16-value group
// (position 2i holds value i, position 2i+1 holds value i+8), which lets the
// W2 decode turn a 32-bit code word into fp16 pairs with one logic op.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <mutex>

#include "common.cuh"
#include "sm100_ptx.cuh"

namespace moe {
namespace {

using namespace ptx;

constexpr int kM = 128;          // weight rows per tile
constexpr int kNmax = 256;       // routed rows per tile
constexpr int kSK = 64;          // K values per stage (one 128-byte swizzle row of fp16)
constexpr int kStages = 3;
constexpr int kRawSlot = 23040;  // bytes per raw-weight slot (128 rows x 180 B)
constexpr int kThreads = 512;
constexpr int kWarpProducer = 12;
constexpr int kWarpMma = 13;
constexpr uint32_t kTmemCols = 512;  // two accumulators of 256 fp32 columns
constexpr uint64_t kTimeoutNs = 1000000000ull;

constexpr int kABytes = kM * kSK * 2;     // 16 KB
constexpr int kBBytes = kNmax * kSK * 2;  // 32 KB

// shared memory layout (offsets from a 1024-aligned base)
constexpr int kOffA = 0;
constexpr int kOffB = kOffA + kStages * kABytes;
constexpr int kOffRaw = kOffB + kStages * kBBytes;
constexpr int kOffDx = kOffRaw + 2 * kRawSlot;
constexpr int kOffDw = kOffDx + kStages * 2 * kNmax * 4;
constexpr int kOffTok = kOffDw + kStages * 2 * kM * 4;
constexpr int kOffBar = kOffTok + kNmax * 4;
constexpr int kNumBars = 3 * kStages + 2 + 2 + 2 + 2 + 1;
constexpr int kOffPrefix = kOffBar + kNumBars * 8;
constexpr int kOffMisc = kOffPrefix + 1025 * 4;
constexpr int kSmemBytes = kOffMisc + 256 + 1024;  // misc words + alignment slack

struct TcArgs {
  const uint8_t* pack;
  const int64_t* eoff;
  int which;            // 0 gate/up, 1 down
  int64_t pack_bytes;
  const int32_t* counts;
  const int32_t* offsets;
  const int32_t* order;
  int E;
  const float* act_d;   // activation scales [act_rows x K/32]
  const int32_t* row_src;  // gate/up: routed row -> flat entry (token = entry / k_top)
  int k_top;
  int64_t act_rows;     // rows of the activation tensor map
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
};

struct Item {
  int e, row0, nrows, N, o0;
  bool ok;
  const uint8_t* wbase;
};

// Tile prefix over experts in largest-first order: s_prefix[j] = number of
// routed-row tiles of experts order[0..j-1].
__device__ void build_prefix(const TcArgs& a, int32_t* s_prefix, int32_t* s_warp) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int per = (a.E + kThreads - 1) / kThreads;  // <= 2 for E <= 1024
  int loc[2];
  int sum = 0;
#pragma unroll
  for (int i = 0; i < 2; i++) {
    const int j = tid * per + i;
    int v = 0;
    if (i < per && j < a.E) {
      const int c = a.counts[a.order[j]];
      v = c > 0 ? (c + kNmax - 1) / kNmax : 0;
    }
    loc[i] = v;
    sum += v;
  }
  int incl = sum;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) s_warp[warp] = incl;
  __syncthreads();
  int base = 0;
  for (int w = 0; w < warp; w++) base += s_warp[w];
  int run = base + incl - sum;
#pragma unroll
  for (int i = 0; i < 2; i++) {
    const int j = tid * per + i;
    if (i < per && j < a.E) s_prefix[j] = run;
    run += loc[i];
  }
  if (tid == kThreads - 1) s_prefix[a.E] = run;
  __syncthreads();
}

__device__ __forceinline__ Item get_item(const TcArgs& a, const int32_t* s_prefix, int n_wtiles,
                                         int64_t item) {
  Item it;
  const int gtile = (int)(item / n_wtiles);
  const int wtile = (int)(item - (int64_t)gtile * n_wtiles);
  int lo = 0, hi = a.E - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (s_prefix[mid] <= gtile) lo = mid; else hi = mid - 1;
  }
  it.e = a.order[lo];
  const int ttile = gtile - s_prefix[lo];
  const int n_e = a.counts[it.e];
  it.row0 = a.offsets[it.e] + ttile * kNmax;
  it.nrows = min(kNmax, n_e - ttile * kNmax);
  it.N = (it.nrows + 15) & ~15;
  it.o0 = wtile * kM;
  const bool rows_ok = (unsigned)it.e < (unsigned)a.E && a.offsets[it.e] >= 0 &&
                       (int64_t)a.offsets[it.e] + n_e <= a.rows_max && it.nrows > 0;
  const int64_t off = rows_ok ? a.eoff[2 * it.e + a.which] : -1;
  it.ok = rows_ok && off >= 0 && (off & 15) == 0 && off + a.pitch * a.N_out <= a.pack_bytes;
  it.wbase = it.ok ? a.pack + off + (int64_t)it.o0 * a.pitch : nullptr;
  return it;
}

// ---------------------------------------------------------------- decode
// Little-endian 32-bit word of code bytes starting at a 2-byte-aligned
// shared address p (p may be 2 mod 4).
__device__ __forceinline__ void load_words(const uint8_t* p, int nwords, uint32_t* w) {
  const uintptr_t a = reinterpret_cast<uintptr_t>(p);
  const uint32_t* q = reinterpret_cast<const uint32_t*>(a & ~(uintptr_t)3);
  const uint32_t sh = (uint32_t)(a & 3) * 8;
  uint32_t prev = q[0];
  for (int i = 0; i < nwords; i++) {
    const uint32_t next = q[i + 1];
    w[i] = __funnelshift_r(prev, next, sh);
    prev = next;
  }
}

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

// One W2 block (64 values) of one row -> 32 fp16 pairs in pair-interleaved
// order, scale folded: pair i of code word w holds (d*(c_{16w+i}-2),
// d*(c_{16w+i+8}-2)).
__device__ __forceinline__ void decode_w2_block(const uint8_t* blk, uint32_t (&out)[32],
                                                float& dsc) {
  const uint16_t dh = *reinterpret_cast<const uint16_t*>(blk);
  dsc = __half2float(__ushort_as_half(dh));
  uint32_t w[4];
  load_words(blk + 2, 4, w);
  const uint32_t d2 = (uint32_t)dh | ((uint32_t)dh << 16);
  const uint32_t k1026 = 0x64026402u;  // fp16 pair (1026, 1026)
#pragma unroll
  for (int q = 0; q < 4; q++) {
#pragma unroll
    for (int i = 0; i < 8; i++) {
      // (1024 + c_i, 1024 + c_{i+8}) by placing the codes in the mantissas
      const uint32_t pr = ((w[q] >> (2 * i)) & 0x00030003u) | 0x64006400u;
      out[q * 8 + i] = hmul2_u32(hsub2_u32(pr, k1026), d2);  // exact
    }
  }
}

// One W4NL block (32 values) of one row -> 16 fp16 pairs of T[idx]
// (integers, exact), pair-interleaved.
__device__ __forceinline__ void decode_w4_block(const uint8_t* blk, const uint16_t* lut,
                                                uint32_t (&out)[16], float& dsc) {
  const uint16_t dh = *reinterpret_cast<const uint16_t*>(blk);
  dsc = __half2float(__ushort_as_half(dh));
  uint32_t w[4];
  load_words(blk + 2, 4, w);  // word 2g: values 16g..16g+7, word 2g+1: 16g+8..16g+15
#pragma unroll
  for (int g = 0; g < 2; g++) {
#pragma unroll
    for (int i = 0; i < 8; i++) {
      const uint32_t lo = lut[(w[2 * g] >> (4 * i)) & 15u];
      const uint32_t hi = lut[(w[2 * g + 1] >> (4 * i)) & 15u];
      out[g * 8 + i] = lo | (hi << 16);
    }
  }
}

// Store 8 consecutive fp16 pairs (16 bytes) as 16-byte chunk j of row r of a
// 128-byte-swizzled K-major tile.
__device__ __forceinline__ void st_swizzled(uint8_t* tile, int r, int j, uint32_t a0, uint32_t a1,
                                            uint32_t a2, uint32_t a3) {
  uint8_t* p = tile + (r >> 3) * 1024 + (r & 7) * 128 + ((j ^ (r & 7)) << 4);
  *reinterpret_cast<uint4*>(p) = make_uint4(a0, a1, a2, a3);
}

// ---------------------------------------------------------------- kernel
template <int FMT>
__global__ void __launch_bounds__(kThreads, 1)
gemm_tc_kernel(const TcArgs a, const __grid_constant__ CUtensorMap tmap) {
  constexpr bool kFold = (FMT == MOE_FMT_W2);
  constexpr int kBlocksPerStage = (FMT == MOE_FMT_W2) ? 1 : 2;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  uint8_t* sA = smem + kOffA;
  uint8_t* sB = smem + kOffB;
  uint8_t* sRaw = smem + kOffRaw;
  float* sDx = reinterpret_cast<float*>(smem + kOffDx);  // [stage][2][kNmax]
  float* sDw = reinterpret_cast<float*>(smem + kOffDw);  // [stage][2][kM]
  int32_t* sTok = reinterpret_cast<int32_t*>(smem + kOffTok);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kOffBar);
  uint64_t* full_tma = bars;                // [kStages]  producer arrivals + TMA bytes
  uint64_t* full_dec = bars + kStages;      // [kStages]  decode threads
  uint64_t* empty = bars + 2 * kStages;     // [kStages]  MMA commit + epilogue threads
  uint64_t* tfull = bars + 3 * kStages;     // [2]        MMA commit
  uint64_t* tempty = tfull + 2;             // [2]        epilogue threads
  uint64_t* rfull = tempty + 2;             // [2]        raw bytes landed
  uint64_t* rempty = rfull + 2;             // [2]        decode threads done with the slot
  uint64_t* fin = rempty + 2;               // MMA drain at exit
  int32_t* s_prefix = reinterpret_cast<int32_t*>(smem + kOffPrefix);
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(smem + kOffMisc);
  volatile int* s_abort = reinterpret_cast<volatile int*>(smem + kOffMisc + 4);
  int32_t* s_warp = reinterpret_cast<int32_t*>(smem + kOffMisc + 8);  // 16 ints
  uint16_t* s_lut = reinterpret_cast<uint16_t*>(smem + kOffMisc + 8 + 64);  // not used by W2

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  if (tid == 0) {
    for (int s = 0; s < kStages; s++) {
      mbar_init(&full_tma[s], 32);
      mbar_init(&full_dec[s], 128);
      mbar_init(&empty[s], 1 + 256);
    }
    for (int b = 0; b < 2; b++) {
      mbar_init(&tfull[b], 1);
      mbar_init(&tempty[b], 256);
      mbar_init(&rfull[b], 1);
      mbar_init(&rempty[b], 128);
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
  build_prefix(a, s_prefix, s_warp);  // contains __syncthreads (barriers, TMEM address visible)
  tc_fence_after();

  const int n_wtiles = a.N_out / kM;
  const int64_t total = (int64_t)s_prefix[a.E] * n_wtiles;
  const int nstages = a.K / kSK;
  const uint32_t tmem = *s_tmem;
  const int kblocks = a.K / 32;

  if (warp < 8) {
    // ================================================== epilogue
    setmaxnreg_inc<200>();
    const int q = warp & 3, h = warp >> 2;
    const int r = 32 * q + lane;  // weight row within the tile
    uint32_t it = 0, bc = 0;
    bool alive = true;
    for (int64_t item = blockIdx.x; item < total && alive; item += gridDim.x) {
      const Item I = get_item(a, s_prefix, n_wtiles, item);
      if (!I.ok) {
        if (lane == 0 && warp == 0) atomicOr(a.status, MOE_STATUS_BAD_OFFSET);
        continue;
      }
      const int ncols = min(128, max(0, I.N - 128 * h));  // columns of this warp, multiple of 16
      float acc[128];
#pragma unroll
      for (int i = 0; i < 128; i++) acc[i] = 0.0f;
      for (int s = 0; s < nstages && alive; s++, it++) {
        const int st = it % kStages;
        const uint32_t ph = (it / kStages) & 1;
        alive = mbar_wait(&full_tma[st], ph, s_abort, kTimeoutNs);
        if (!kFold && alive) alive = mbar_wait(&full_dec[st], ph, s_abort, kTimeoutNs);
        if (!alive) break;
#pragma unroll
        for (int kb = 0; kb < 2; kb++) {
          const uint32_t buf = bc & 1;
          if (!mbar_wait(&tfull[buf], (bc >> 1) & 1, s_abort, kTimeoutNs)) { alive = false; break; }
          tc_fence_after();
          const float* dxs = sDx + (st * 2 + kb) * kNmax + 128 * h;
          float dws = 0.0f;
          if (!kFold) dws = sDw[(st * 2 + kb) * kM + r];
          const uint32_t tbase = tmem + ((uint32_t)(32 * q) << 16) + buf * 256 + 128 * h;
#pragma unroll
          for (int c = 0; c < 4; c++) {
            if (32 * c < ncols) {
              float v[32];
              tmem_ld32(tbase + 32 * c, v);
              tmem_wait_ld();
#pragma unroll
              for (int j4 = 0; j4 < 8; j4++) {
                const float4 dx4 = *reinterpret_cast<const float4*>(dxs + 32 * c + 4 * j4);
                const float dxv[4] = {dx4.x, dx4.y, dx4.z, dx4.w};
#pragma unroll
                for (int u = 0; u < 4; u++) {
                  const int j = 4 * j4 + u;
                  if (kFold)
                    acc[32 * c + j] = fmaf(dxv[u], v[j], acc[32 * c + j]);
                  else
                    acc[32 * c + j] = fmaf(__fmul_rn(dws, dxv[u]), v[j], acc[32 * c + j]);
                }
              }
            }
          }
          tc_fence_before();
          mbar_arrive(&tempty[buf]);
          bc++;
        }
        if (!alive) break;
        mbar_arrive(&empty[st]);
      }
      if (!alive) break;
      // store: column = routed row row0 + col, row = output o0 + r
      float* outp = a.out + (int64_t)I.row0 * a.N_out + I.o0 + r;
#pragma unroll
      for (int c = 0; c < 4; c++)
#pragma unroll
        for (int j = 0; j < 32; j++) {
          const int col = 128 * h + 32 * c + j;
          if (col < I.nrows) outp[(int64_t)col * a.N_out] = acc[32 * c + j];
        }
    }
  } else if (warp < 12) {
    // ================================================== weight decode
    setmaxnreg_dec<56>();
    const int r = tid - 256;  // weight row within the tile
    if (FMT != MOE_FMT_W2) {
      // fp16 bit patterns of the W4NL table, from the constant bank
      if (r < 16) s_lut[r] = c_nl4_half[r];
      asm volatile("bar.sync 1, 128;" ::: "memory");
    }
    uint32_t it = 0, cc = 0;
    bool alive = true;
    for (int64_t item = blockIdx.x; item < total && alive; item += gridDim.x) {
      const Item I = get_item(a, s_prefix, n_wtiles, item);
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
          uint32_t v[32];
          float dsc;
          decode_w2_block(raw + sc * kBlockBytes, v, dsc);
#pragma unroll
          for (int j = 0; j < 8; j++)
            st_swizzled(tileA, r, j, v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
          sDw[(st * 2 + 0) * kM + r] = dsc;
          sDw[(st * 2 + 1) * kM + r] = dsc;
        } else {
#pragma unroll
          for (int kb = 0; kb < 2; kb++) {
            uint32_t v[16];
            float dsc;
            decode_w4_block(raw + (sc * 2 + kb) * kBlockBytes, s_lut, v, dsc);
#pragma unroll
            for (int j = 0; j < 4; j++)
              st_swizzled(tileA, r, 4 * kb + j, v[4 * j], v[4 * j + 1], v[4 * j + 2],
                          v[4 * j + 3]);
            sDw[(st * 2 + kb) * kM + r] = dsc;
          }
        }
        fence_proxy_async_smem();
        mbar_arrive(&full_dec[st]);
        if (sc == a.stages_per_chunk - 1 || s == nstages - 1) {
          mbar_arrive(&rempty[slot]);
          cc++;
        }
      }
    }
  } else if (warp == kWarpProducer) {
    // ================================================== producer
    setmaxnreg_dec<56>();
    prefetch_tmap(&tmap);
    // Raw chunks run one chunk ahead of the stages.  The chunk stream covers
    // this CTA's items in order; chunk q of an item = stages
    // [q*spc, (q+1)*spc).
    const int spc = a.stages_per_chunk;
    const int chunks_per_item = (nstages + spc - 1) / spc;
    int64_t r_item = blockIdx.x;  // item of the next raw chunk to issue
    int r_chunk = 0;
    uint32_t issued = 0;          // raw chunks issued
    Item RI;
    bool r_valid = false;
    auto next_raw_item = [&]() {
      while (r_item < total) {
        RI = get_item(a, s_prefix, n_wtiles, r_item);
        if (RI.ok) return true;
        r_item += gridDim.x;
      }
      return false;
    };
    r_valid = next_raw_item();
    bool alive = true;
    auto issue_raw = [&]() -> bool {
      if (!r_valid) return true;
      const uint32_t slot = issued % a.raw_slots;
      if (!mbar_wait(&rempty[slot], ((issued / a.raw_slots) & 1) ^ 1, s_abort, kTimeoutNs))
        return false;
      const int s0 = r_chunk * spc;
      const int ns = min(spc, nstages - s0);
      const int blocks_per_stage = (FMT == MOE_FMT_W2) ? 1 : 2;
      const int row_bytes = a.rows_mode ? ns * blocks_per_stage * kBlockBytes : (int)a.pitch;
      const uint32_t bytes = (uint32_t)(row_bytes * kM);
      uint8_t* dst = sRaw + slot * kRawSlot;
      if (lane == 0) mbar_arrive_expect_tx(&rfull[slot], bytes);
      __syncwarp();
      if (a.rows_mode) {
        const uint8_t* src = RI.wbase + (int64_t)s0 * blocks_per_stage * kBlockBytes;
        for (int row = lane; row < kM; row += 32)
          bulk_g2s(dst + row * a.chunk_row_bytes, src + row * a.pitch, (uint32_t)row_bytes,
                   &rfull[slot]);
      } else if (lane == 0) {
        bulk_g2s(dst, RI.wbase, bytes, &rfull[slot]);
      }
      issued++;
      if (++r_chunk == chunks_per_item) {
        r_chunk = 0;
        r_item += gridDim.x;
        r_valid = next_raw_item();
      }
      return true;
    };
    // With two raw slots the next chunk is issued while the current one is
    // decoded; with one slot (a tile that fills both) a chunk can only be
    // issued once the previous one is fully decoded, i.e. just in time.
    const bool ahead = a.raw_slots == 2;
    if (ahead) alive = issue_raw();  // chunk 0
    uint32_t it = 0;
    for (int64_t item = blockIdx.x; item < total && alive; item += gridDim.x) {
      const Item I = get_item(a, s_prefix, n_wtiles, item);
      if (!I.ok) continue;
      // token (activation row) of each tile column; padding columns repeat column 0
      for (int col = lane; col < kNmax; col += 32) {
        int t = 0;
        if (col < I.N) {
          const int cc = col < I.nrows ? col : 0;
          const int rr = I.row0 + cc;
          t = a.row_src ? a.row_src[rr] / a.k_top : rr;
          if ((uint64_t)t >= (uint64_t)a.act_rows) {
            atomicOr(a.status, MOE_STATUS_BAD_ROUTING);
            t = 0;
          }
        }
        sTok[col] = t;
      }
      __syncwarp();
      for (int s = 0; s < nstages; s++, it++) {
        if (s % spc == 0) {
          if (!(alive = issue_raw())) break;  // the next chunk (ahead) or this one
        }
        const int st = it % kStages;
        const uint32_t ph = (it / kStages) & 1;
        if (!mbar_wait(&empty[st], ph ^ 1, s_abort, kTimeoutNs)) { alive = false; break; }
        // activation scales of the stage's two 32-value blocks
        for (int col = lane; col < I.N; col += 32) {
          const int t = sTok[col];
          const float* dp = a.act_d + (int64_t)t * kblocks + 2 * s;
          const bool valid = col < I.nrows;
          sDx[(st * 2 + 0) * kNmax + col] = valid ? dp[0] : 0.0f;
          sDx[(st * 2 + 1) * kNmax + col] = valid ? dp[1] : 0.0f;
        }
        if (lane == 0) mbar_arrive_expect_tx(&full_tma[st], (uint32_t)I.N * 128u);
        __syncwarp();
        if (lane != 0) mbar_arrive(&full_tma[st]);
        uint8_t* tileB = sB + st * kBBytes;
        for (int g = lane; g < I.N / 4; g += 32)
          tma_gather4(tileB + g * 512, &tmap, s * kSK, sTok[4 * g], sTok[4 * g + 1],
                      sTok[4 * g + 2], sTok[4 * g + 3], &full_tma[st]);
      }
    }
    (void)r_valid;
  } else if (warp == kWarpMma) {
    // ================================================== MMA issue
    setmaxnreg_dec<56>();
    if (lane == 0) {
      uint32_t it = 0, bc = 0;
      bool alive = true;
      for (int64_t item = blockIdx.x; item < total && alive; item += gridDim.x) {
        const Item I = get_item(a, s_prefix, n_wtiles, item);
        if (!I.ok) continue;
        const uint32_t idesc = idesc_f16_f32(kM, I.N);
        for (int s = 0; s < nstages && alive; s++, it++) {
          const int st = it % kStages;
          const uint32_t ph = (it / kStages) & 1;
          if (!mbar_wait(&full_tma[st], ph, s_abort, kTimeoutNs) ||
              !mbar_wait(&full_dec[st], ph, s_abort, kTimeoutNs)) {
            alive = false;
            break;
          }
          tc_fence_after();
          const uint32_t aaddr = smem_u32(sA + st * kABytes);
          const uint32_t baddr = smem_u32(sB + st * kBBytes);
          for (int kb = 0; kb < 2; kb++) {
            const uint32_t buf = bc & 1;
            if (!mbar_wait(&tempty[buf], ((bc >> 1) & 1) ^ 1, s_abort, kTimeoutNs)) {
              alive = false;
              break;
            }
            tc_fence_after();
            const uint32_t d_tmem = tmem + buf * 256;
#pragma unroll
            for (int k16 = 0; k16 < 2; k16++) {
              const uint32_t koff = kb * 64 + k16 * 32;  // bytes along the 128-byte row
              mma_f16(d_tmem, smem_desc_sw128(aaddr + koff), smem_desc_sw128(baddr + koff),
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
    setmaxnreg_dec<56>();
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

cudaError_t launch_gemm_tc(const GemmArgs& g, const void* act, int64_t act_rows,
                           cudaStream_t st) {
  if (g.rows_max == 0 || act_rows == 0) return cudaSuccess;
  TcArgs a{};
  a.pack = g.pack;
  a.eoff = g.eoff;
  a.which = g.which;
  a.pack_bytes = g.pack_bytes;
  a.counts = g.counts;
  a.offsets = g.offsets;
  a.order = g.order;
  a.E = g.E;
  a.act_d = g.act_d;
  a.row_src = g.row_src;
  a.k_top = g.k_top;
  a.act_rows = act_rows;
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
  const cuuint64_t dims[2] = {(cuuint64_t)g.K, (cuuint64_t)act_rows};
  const cuuint64_t strides[1] = {(cuuint64_t)g.K * 2};
  const cuuint32_t box[2] = {64, 1};
  const cuuint32_t estr[2] = {1, 1};
  if (encode(&tmap, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void*>(act), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;

  const int64_t tiles_max = (g.rows_max / kNmax + g.E) * (int64_t)(g.N_out / kM);
  const int grid = (int)std::min<int64_t>(tiles_max, device_sm_count());
  cudaError_t e;
  if (g.fmt == MOE_FMT_W2) {
    if ((e = set_smem_attr<MOE_FMT_W2>()) != cudaSuccess) return e;
    gemm_tc_kernel<MOE_FMT_W2><<<grid, kThreads, kSmemBytes, st>>>(a, tmap);
  } else {
    if ((e = set_smem_attr<MOE_FMT_W4NL>()) != cudaSuccess) return e;
    gemm_tc_kernel<MOE_FMT_W4NL><<<grid, kThreads, kSmemBytes, st>>>(a, tmap);
  }
  count_launch();
  return cudaGetLastError();
}

}  // namespace moe
