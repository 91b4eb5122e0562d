// Grouped expert products (gate/up and down) -- first, simple version.
//
// For one expert e with n_e routed rows, output column o and routed row r:
//   out[r, o] = sum over 32-value K blocks b, in increasing b, of
//               acc = fma(d_w[o,b] * d_x[r,b], isum_b(o, r), acc)
// with isum_b the exact integer sum of w_int * q over the block
// ("Strata #3752", commit "moe_ws kernels": MMQ's int8 values, scales and
// per-32-value epilogue in K order; the integer block sum is exact, so only
// the float epilogue's order matters).
//
// Integer sums on the tensor cores: both operands are small integers held
// exactly in fp16 (|w_int| <= 127, |q| <= 127), every product is below 2^14
// and every partial sum of a 32-value block below 2^24, so fp16 MMA with fp32
// accumulation returns the block sum exactly.  (On sm_103a the int8 MMA runs
// at a quarter of the fp16 rate, so fp16 is the faster exact route.)
//
// Work: tiles of 64 weight rows x 64 routed rows of one expert, experts in
// largest-first order, each expert only as many row tiles as it has rows
// (no padding to a group maximum).  Weight blocks are decoded into shared
// memory once per tile.  This version uses the legacy warp-level mma.sync;
// it is the reference point for the tcgen05 kernel.
#include <algorithm>

#include "common.cuh"

namespace moe {
namespace {

constexpr int kTW = 64;           // weight rows per tile
constexpr int kTT = 64;           // routed rows per tile
constexpr int kSK = 64;           // K values per stage
constexpr int kPitch = kSK + 8;   // fp16 per smem row: 144 bytes, conflict-free fragments
constexpr int kThreads = 128;


__device__ __forceinline__ void mma_f16_16816(float (&d)[4], const uint32_t (&a)[4],
                                              const uint32_t (&b)[2]) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}

__device__ __forceinline__ float half_bits_to_float(uint16_t h) {
  return __half2float(__ushort_as_half(h));
}

// Tile prefix over experts in largest-first order: s_prefix[j] = number of
// row tiles of experts order[0..j-1].  Whole CTA.
__device__ void build_tile_prefix(const int32_t* __restrict__ counts,
                                  const int32_t* __restrict__ order, int E,
                                  int32_t* s_prefix, int32_t* s_warp) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int per = (E + blockDim.x - 1) / blockDim.x;
  int loc[8];  // per <= 8 for E <= 1024 and 128 threads
  int sum = 0;
#pragma unroll
  for (int i = 0; i < 8; i++) {
    const int j = tid * per + i;
    int v = 0;
    if (i < per && j < E) v = (counts[order[j]] + kTT - 1) / kTT;
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
  int wbase = 0;
  for (int w = 0; w < warp; w++) wbase += s_warp[w];
  int run = wbase + incl - sum;
#pragma unroll
  for (int i = 0; i < 8; i++) {
    const int j = tid * per + i;
    if (i < per && j < E) s_prefix[j] = run;
    run += loc[i];
  }
  if (tid == blockDim.x - 1) s_prefix[E] = run;
  __syncthreads();
}

__global__ void __launch_bounds__(kThreads)
gemm_mma_kernel(GemmArgs a) {
  __shared__ __align__(16) __half s_w[kTW][kPitch];
  __shared__ __align__(16) __half s_x[kTT][kPitch];
  __shared__ float s_dw[kTW][2];
  __shared__ float s_dx[kTT][2];
  __shared__ int32_t s_prefix[1025];
  __shared__ int32_t s_warp[32];
  __shared__ int32_t s_arow[kTT];

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = lane >> 2, c = lane & 3;
  const int wm = warp >> 1, wn = warp & 1;  // 2 x 2 warps, 32 x 32 each

  build_tile_prefix(a.counts, a.order, a.E, s_prefix, s_warp);
  const int n_wtiles = a.N_out / kTW;
  const int64_t total = (int64_t)s_prefix[a.E] * n_wtiles;
  const int64_t rb = row_bytes(a.fmt, a.K);
  const int nstages = a.K / kSK;

  for (int64_t item = blockIdx.x; item < total; item += gridDim.x) {
    const int gtile = (int)(item / n_wtiles);
    const int wtile = (int)(item - (int64_t)gtile * n_wtiles);
    // expert slot j with s_prefix[j] <= gtile < s_prefix[j+1]
    int lo = 0, hi = a.E - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (s_prefix[mid] <= gtile) lo = mid; else hi = mid - 1;
    }
    const int e = a.order[lo];
    const int ttile = gtile - s_prefix[lo];
    const int n_e = a.counts[e];
    const int row0 = a.offsets[e] + ttile * kTT;
    const int nrows = min(kTT, n_e - ttile * kTT);
    const int o0 = wtile * kTW;

    // A workspace not written by the routing step (misuse of the stage API)
    // is caught here instead of being followed out of bounds.
    const bool rows_ok = (unsigned)e < (unsigned)a.E && a.offsets[e] >= 0 &&
                         (int64_t)a.offsets[e] + n_e <= a.rows_max;
    const int64_t off = rows_ok ? a.eoff[2 * e + a.which] : -1;
    const bool off_ok = off >= 0 && (off & 15) == 0 && off + rb * a.N_out <= a.pack_bytes;
    if (!rows_ok || !off_ok) {
      if (tid == 0) atomicOr(a.status, rows_ok ? MOE_STATUS_BAD_OFFSET : MOE_STATUS_BAD_ROUTING);
      continue;  // uniform over the CTA
    }
    const uint8_t* wmat = a.pack + off;

    if (tid < kTT) {
      int arow = -1;
      if (tid < nrows) {
        const int r = row0 + tid;
        arow = a.row_src ? a.row_src[r] / a.k_top : r;
        if ((uint64_t)arow >= (uint64_t)a.act_rows) {
          atomicOr(a.status, MOE_STATUS_BAD_ROUTING);
          arow = -1;
        }
      }
      s_arow[tid] = arow;
    }
    __syncthreads();

    float acc[2][4][4];
#pragma unroll
    for (int mi = 0; mi < 2; mi++)
#pragma unroll
      for (int ni = 0; ni < 4; ni++)
#pragma unroll
        for (int q = 0; q < 4; q++) acc[mi][ni][q] = 0.0f;

    for (int s = 0; s < nstages; s++) {
      // ---- decode 64 weight rows x 64 values into fp16 integers
      {
        const int wr = tid >> 1, half = tid & 1;
        const uint8_t* row = wmat + (int64_t)(o0 + wr) * rb;
        uint32_t out[16];
        float dsc;
        if (a.fmt == MOE_FMT_W2) {
          const uint8_t* blk = row + (int64_t)s * kBlockBytes;
          dsc = half_bits_to_float((uint16_t)(blk[0] | (blk[1] << 8)));
#pragma unroll
          for (int bi = 0; bi < 8; bi++) {
            const uint32_t byte = blk[2 + half * 8 + bi];
            const uint32_t h0 = (uint32_t)(kW2HalfLut >> (16 * (byte & 3))) & 0xFFFFu;
            const uint32_t h1 = (uint32_t)(kW2HalfLut >> (16 * ((byte >> 2) & 3))) & 0xFFFFu;
            const uint32_t h2 = (uint32_t)(kW2HalfLut >> (16 * ((byte >> 4) & 3))) & 0xFFFFu;
            const uint32_t h3 = (uint32_t)(kW2HalfLut >> (16 * ((byte >> 6) & 3))) & 0xFFFFu;
            out[2 * bi] = h0 | (h1 << 16);
            out[2 * bi + 1] = h2 | (h3 << 16);
          }
        } else {
          const uint8_t* blk = row + (int64_t)(2 * s + half) * kBlockBytes;
          dsc = half_bits_to_float((uint16_t)(blk[0] | (blk[1] << 8)));
#pragma unroll
          for (int bi = 0; bi < 16; bi++) {
            const uint32_t byte = blk[2 + bi];
            out[bi] = (uint32_t)c_nl4_half[byte & 15] | ((uint32_t)c_nl4_half[byte >> 4] << 16);
          }
        }
        uint4* dst = reinterpret_cast<uint4*>(&s_w[wr][half * 32]);
#pragma unroll
        for (int v = 0; v < 4; v++)
          dst[v] = make_uint4(out[4 * v], out[4 * v + 1], out[4 * v + 2], out[4 * v + 3]);
        s_dw[wr][half] = dsc;
      }
      // ---- activations: 64 rows x 64 values (gathered rows)
      {
        const int tr = tid >> 1, half = tid & 1;
        const int arow = s_arow[tr];
        uint4* dst = reinterpret_cast<uint4*>(&s_x[tr][half * 32]);
        if (arow >= 0) {
          const uint4* src = reinterpret_cast<const uint4*>(
              a.act + (int64_t)arow * a.K + s * kSK + half * 32);
#pragma unroll
          for (int v = 0; v < 4; v++) dst[v] = src[v];
          s_dx[tr][half] = a.act_d[(int64_t)arow * (a.K / kQBlock) + 2 * s + half];
        } else {
#pragma unroll
          for (int v = 0; v < 4; v++) dst[v] = make_uint4(0, 0, 0, 0);
          s_dx[tr][half] = 0.0f;
        }
      }
      __syncthreads();

#pragma unroll
      for (int kb = 0; kb < 2; kb++) {
        uint32_t af[2][2][4], bf[4][2][2];
#pragma unroll
        for (int mi = 0; mi < 2; mi++)
#pragma unroll
          for (int ks = 0; ks < 2; ks++) {
            const int r = wm * 32 + mi * 16 + g;
            const int k0 = kb * 32 + ks * 16 + 2 * c;
            af[mi][ks][0] = *reinterpret_cast<const uint32_t*>(&s_w[r][k0]);
            af[mi][ks][1] = *reinterpret_cast<const uint32_t*>(&s_w[r + 8][k0]);
            af[mi][ks][2] = *reinterpret_cast<const uint32_t*>(&s_w[r][k0 + 8]);
            af[mi][ks][3] = *reinterpret_cast<const uint32_t*>(&s_w[r + 8][k0 + 8]);
          }
#pragma unroll
        for (int ni = 0; ni < 4; ni++)
#pragma unroll
          for (int ks = 0; ks < 2; ks++) {
            const int t = wn * 32 + ni * 8 + g;
            const int k0 = kb * 32 + ks * 16 + 2 * c;
            bf[ni][ks][0] = *reinterpret_cast<const uint32_t*>(&s_x[t][k0]);
            bf[ni][ks][1] = *reinterpret_cast<const uint32_t*>(&s_x[t][k0 + 8]);
          }
#pragma unroll
        for (int mi = 0; mi < 2; mi++) {
          const int r0 = wm * 32 + mi * 16 + g;
          const float dw0 = s_dw[r0][kb], dw1 = s_dw[r0 + 8][kb];
#pragma unroll
          for (int ni = 0; ni < 4; ni++) {
            const int t0 = wn * 32 + ni * 8 + 2 * c;
            const float dx0 = s_dx[t0][kb], dx1 = s_dx[t0 + 1][kb];
            float isum[4] = {0.f, 0.f, 0.f, 0.f};
            mma_f16_16816(isum, af[mi][0], bf[ni][0]);
            mma_f16_16816(isum, af[mi][1], bf[ni][1]);
            acc[mi][ni][0] = fmaf(__fmul_rn(dw0, dx0), isum[0], acc[mi][ni][0]);
            acc[mi][ni][1] = fmaf(__fmul_rn(dw0, dx1), isum[1], acc[mi][ni][1]);
            acc[mi][ni][2] = fmaf(__fmul_rn(dw1, dx0), isum[2], acc[mi][ni][2]);
            acc[mi][ni][3] = fmaf(__fmul_rn(dw1, dx1), isum[3], acc[mi][ni][3]);
          }
        }
      }
      __syncthreads();
    }

    // ---- store: row r of the tile is weight row o0 + r, column t routed row row0 + t
#pragma unroll
    for (int mi = 0; mi < 2; mi++)
#pragma unroll
      for (int ni = 0; ni < 4; ni++)
#pragma unroll
        for (int q = 0; q < 4; q++) {
          const int r = wm * 32 + mi * 16 + g + (q >= 2 ? 8 : 0);
          const int t = wn * 32 + ni * 8 + 2 * c + (q & 1);
          if (t < nrows) a.out[(int64_t)(row0 + t) * a.N_out + o0 + r] = acc[mi][ni][q];
        }
  }
}

}  // namespace

cudaError_t launch_gemm(const GemmArgs& a, cudaStream_t st) {
  const int64_t rows_max = a.rows_max;
  if (rows_max == 0) return cudaSuccess;
  const int64_t tiles_max = (rows_max / kTT + a.E) * (int64_t)(a.N_out / kTW);
  const int64_t grid = std::min<int64_t>(tiles_max, (int64_t)device_sm_count() * 8);
  gemm_mma_kernel<<<(unsigned)grid, kThreads, 0, st>>>(a);
  count_launch();
  return cudaGetLastError();
}

}  // namespace moe
