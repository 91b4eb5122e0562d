// Bandwidth-bound steps of the layer:
//   quant_q8      -- x -> q8 per 32-value block ("Strata #3752", commit
//                    "swiglu_quant": quantize_mmq_q8_1; layer spec, tiny
//                    configuration: d = amax/127, q = rint(x/d), d = 0 -> 0),
//                    scattered to the token's k routed rows (quantize_scatter,
//                    "Strata #3752" commits "moe_ws wiring"), so the product
//                    kernels read contiguous per-expert row ranges;
//   swiglu_quant  -- H = silu(g)*u and its q8 in one pass, H never stored
//                    ("Strata #3752", commit "swiglu_quant");
//   combine       -- out[t] = sum over ranks r = 0..k-1 of w[t,r]*Dm[row]
//                    (layer spec, tiny configuration).
//
// Quantised values are stored as exact fp16 integers (|q| <= 127): that is
// the operand type of the fp16 tensor-core products, and it carries the same
// information as the int8 code.  Within each 16-value group they are stored
// pair-interleaved (position 2i holds value i, 2i+1 holds value i+8), the
// order the product kernel's weight decode produces; a permutation inside a
// 32-value block leaves every block sum unchanged.
//
// Every division is IEEE (__fdiv_rn), rounding to integer is rintf (half to
// even), and the q8 decisions are taken in fp32 exactly as the method states.
// This file must not be compiled with fast-math.
#include "common.cuh"

namespace moe {
namespace {

// Quantise 8 consecutive values held by one thread; four consecutive lanes
// hold one 32-value block.  Returns the block scale.
__device__ __forceinline__ float q8_group8(const float (&v)[8], uint4& packed) {
  float amax = 0.0f;
#pragma unroll
  for (int i = 0; i < 8; i++) amax = fmaxf(amax, fabsf(v[i]));
  amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
  amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
  const float d = __fdiv_rn(amax, 127.0f);
  uint32_t w[4];
#pragma unroll
  for (int i = 0; i < 4; i++) {
    const float q0 = (d == 0.0f) ? 0.0f : rintf(__fdiv_rn(v[2 * i], d));
    const float q1 = (d == 0.0f) ? 0.0f : rintf(__fdiv_rn(v[2 * i + 1], d));
    const __half2 h = __floats2half2_rn(q0, q1);  // exact: |q| <= 127
    w[i] = *reinterpret_cast<const uint32_t*>(&h);
  }
  // Pair-interleave within each 16-value group: this thread (8 values) and
  // its partner lane (the other 8 values of the group) swap halves so that
  // stored position 2i holds value i and 2i+1 holds value i+8.
  const bool first = (threadIdx.x & 1) == 0;  // values 0..7 of the group
  const uint32_t s0 = first ? w[2] : w[0];
  const uint32_t s1 = first ? w[3] : w[1];
  const uint32_t r0 = __shfl_xor_sync(0xffffffffu, s0, 1);
  const uint32_t r1 = __shfl_xor_sync(0xffffffffu, s1, 1);
  const uint32_t l0 = first ? w[0] : r0, l1 = first ? w[1] : r1;  // values 0-3 / 4-7 pairs
  const uint32_t h0 = first ? r0 : w[2], h1 = first ? r1 : w[3];  // values 8-11 / 12-15 pairs
  packed = make_uint4(__byte_perm(l0, h0, 0x5410), __byte_perm(l0, h0, 0x7632),
                      __byte_perm(l1, h1, 0x5410), __byte_perm(l1, h1, 0x7632));
  return d;
}

// Routed-row layout of the product inputs: values [R x K] fp16 (row r =
// routed row r), scales [R x scale_stride(K)] (rows padded to 16 bytes), so
// a product tile's rows are one contiguous range of both.
__global__ void __launch_bounds__(256)
quant_q8_kernel(const float* __restrict__ x, int64_t groups, int K, int k,
                const int32_t* __restrict__ dst_of, int64_t rows_max,
                __half* __restrict__ q, float* __restrict__ d) {
  const int64_t g = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const bool ok = g < groups;  // groups is a multiple of 4: quads are whole
  float v[8];
  if (ok) {
    const float4 a = __ldcs(reinterpret_cast<const float4*>(x) + 2 * g);
    const float4 b = __ldcs(reinterpret_cast<const float4*>(x) + 2 * g + 1);
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
    v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
  } else {
#pragma unroll
    for (int i = 0; i < 8; i++) v[i] = 0.0f;
  }
  uint4 packed;
  const float db = q8_group8(v, packed);
  if (ok) {
    const int per_row = K / 8;
    const int64_t t = g / per_row;
    const int c = (int)(g - t * per_row);
    const int blk = c >> 2;
    for (int r = 0; r < k; r++) {
      const int32_t dst = dst_of[t * k + r];
      if (dst < 0 || dst >= rows_max) continue;  // dropped (bad expert id)
      reinterpret_cast<uint4*>(q + (int64_t)dst * K)[c] = packed;
      if ((c & 3) == 0) d[(int64_t)dst * scale_stride(K) + blk] = db;
    }
  }
}

__global__ void __launch_bounds__(256)
swiglu_quant_kernel(const float* __restrict__ gu, const int32_t* __restrict__ nrows_dev,
                    int64_t rows_max, int n_ff, int gu_layout, __half* __restrict__ hq,
                    float* __restrict__ dh) {
  const int per_row = n_ff / 8;
  // rows actually routed, clamped to the buffers (a stale count cannot overrun)
  const int64_t nrows = min((int64_t)max(*nrows_dev, 0), rows_max);
  const int64_t groups = nrows * per_row;
  const int64_t g = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const bool ok = g < groups;
  float v[8];
  if (ok) {
    const int64_t row = g / per_row;
    const int c = (int)(g - row * per_row);
    float gv[8], uv[8];
    if (gu_layout == MOE_GU_INTERLEAVED) {
      // outputs 8c..8c+7: gate j at column 2j, up j at 2j+1
      const float4* p = reinterpret_cast<const float4*>(gu + row * 2 * n_ff + c * 16);
#pragma unroll
      for (int q = 0; q < 4; q++) {
        const float4 f = __ldcs(p + q);
        gv[2 * q] = f.x;
        uv[2 * q] = f.y;
        gv[2 * q + 1] = f.z;
        uv[2 * q + 1] = f.w;
      }
    } else {
      const float4* gp = reinterpret_cast<const float4*>(gu + row * 2 * n_ff + c * 8);
      const float4* up = reinterpret_cast<const float4*>(gu + row * 2 * n_ff + n_ff + c * 8);
      const float4 g0 = __ldcs(gp), g1 = __ldcs(gp + 1), u0 = __ldcs(up), u1 = __ldcs(up + 1);
      gv[0] = g0.x; gv[1] = g0.y; gv[2] = g0.z; gv[3] = g0.w;
      gv[4] = g1.x; gv[5] = g1.y; gv[6] = g1.z; gv[7] = g1.w;
      uv[0] = u0.x; uv[1] = u0.y; uv[2] = u0.z; uv[3] = u0.w;
      uv[4] = u1.x; uv[5] = u1.y; uv[6] = u1.z; uv[7] = u1.w;
    }
#pragma unroll
    for (int i = 0; i < 8; i++) {
      // silu(g) * u = (g / (1 + exp(-g))) * u, each step rounded to fp32
      const float den = __fadd_rn(1.0f, expf(-gv[i]));
      v[i] = __fmul_rn(__fdiv_rn(gv[i], den), uv[i]);
    }
  } else {
#pragma unroll
    for (int i = 0; i < 8; i++) v[i] = 0.0f;
  }
  uint4 packed;
  const float db = q8_group8(v, packed);
  if (ok) {
    reinterpret_cast<uint4*>(hq)[g] = packed;
    if ((g & 3) == 0) {
      const int64_t row = g / per_row;
      const int blk = (int)(g - row * per_row) >> 2;
      dh[row * scale_stride(n_ff) + blk] = db;
    }
  }
}

__global__ void __launch_bounds__(256)
combine_kernel(const float* __restrict__ topk_w, const int32_t* __restrict__ dst_of,
               const float4* __restrict__ dm, int64_t T, int k, int d4, int64_t rows_max,
               float4* __restrict__ out) {
  const int64_t g = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (g >= T * d4) return;
  const int64_t t = g / d4;
  const int c = (int)(g - t * d4);
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int r = 0; r < k; r++) {
    const int32_t pos = dst_of[t * k + r];
    if (pos < 0 || pos >= rows_max) continue;  // dropped row (bad expert id)
    const float w = topk_w[t * k + r];
    const float4 v = __ldcs(dm + (int64_t)pos * d4 + c);
    acc.x = fmaf(w, v.x, acc.x);
    acc.y = fmaf(w, v.y, acc.y);
    acc.z = fmaf(w, v.z, acc.z);
    acc.w = fmaf(w, v.w, acc.w);
  }
  out[g] = acc;
}

// Arrival counters of the fused combine: cnt[t][g] = the count of token t's
// dropped ranks (dst_of < 0), for every 32-column group g.
__global__ void __launch_bounds__(256)
combine_init_kernel(const int32_t* __restrict__ dst_of, int64_t T, int k, int groups,
                    int32_t* __restrict__ cnt) {
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= T * groups) return;
  const int64_t t = i / groups;
  int dropped = 0;
  for (int r = 0; r < k; r++) dropped += dst_of[t * k + r] < 0;
  cnt[i] = dropped;
}

inline unsigned blocks_for(int64_t threads, int per_block) {
  return (unsigned)((threads + per_block - 1) / per_block);
}

}  // namespace

cudaError_t launch_quant_q8(const float* x, int64_t T, int K, int k, const int32_t* dst_of,
                            int64_t rows_max, __half* q, float* d, cudaStream_t st) {
  const int64_t groups = T * (K / 8);
  if (groups == 0) return cudaSuccess;
  quant_q8_kernel<<<blocks_for(groups, 256), 256, 0, st>>>(x, groups, K, k, dst_of, rows_max, q,
                                                            d);
  count_launch();
  return cudaGetLastError();
}

cudaError_t launch_swiglu_quant(const float* gu, const int32_t* nrows_dev, int64_t rows_max,
                                int n_ff, int gu_layout, __half* hq, float* dh, cudaStream_t st) {
  const int64_t groups = rows_max * (n_ff / 8);
  if (groups == 0) return cudaSuccess;
  swiglu_quant_kernel<<<blocks_for(groups, 256), 256, 0, st>>>(gu, nrows_dev, rows_max, n_ff,
                                                                gu_layout, hq, dh);
  count_launch();
  return cudaGetLastError();
}

cudaError_t launch_combine_init(const int32_t* dst_of, int64_t T, int k, int groups,
                                int32_t* cnt, cudaStream_t st) {
  const int64_t n = T * groups;
  if (n == 0) return cudaSuccess;
  combine_init_kernel<<<blocks_for(n, 256), 256, 0, st>>>(dst_of, T, k, groups, cnt);
  count_launch();
  return cudaGetLastError();
}

cudaError_t launch_combine(const float* topk_w, const int32_t* dst_of, const float* dm,
                           int64_t t0, int64_t T, int k, int d, int64_t rows_max, float* out,
                           cudaStream_t st) {
  const int64_t n = T * (d / 4);
  if (n == 0) return cudaSuccess;
  combine_kernel<<<blocks_for(n, 256), 256, 0, st>>>(
      topk_w + t0 * k, dst_of + t0 * k, reinterpret_cast<const float4*>(dm), T, k, d / 4,
      rows_max, reinterpret_cast<float4*>(out + t0 * d));
  count_launch();
  return cudaGetLastError();
}

}  // namespace moe
