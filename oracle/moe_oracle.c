/*
 * CPU oracle of the quantized MoE prefill layer -- TEST INFRASTRUCTURE ONLY.
 *
 * Only the tests, the smoke check and the benchmark's CPU-baseline leg use
 * this file.  It shares no code, header, table or helper with the CUDA
 * library; the two meet only through the seeded inputs of the `synth`
 * module.  It is deliberately plain and slow: loops written in the order
 * the method states, fp32 arithmetic with every rounding explicit (compile
 * with -ffp-contract=off so no multiply-add is fused behind our back).
 *
 * The method (the pages are three pull requests of the "Strata" inference
 * engine):
 *
 *   route      -- bucket the T*k (token, expert) rows by expert: counts,
 *                 exclusive prefix sum, stable permutation ("Strata #3752",
 *                 commits "moe_ws wiring" and "swiglu_quant landed":
 *                 quantize_scatter, group bounds).  Inside a bucket rows keep
 *                 increasing flat index i = t*k + r (the pages do not fix the
 *                 order; this is the plain stable reading).
 *   q8         -- per 32-value block: amax, d = amax/127, q = rint(x/d),
 *                 d == 0 gives q = 0 (the layer spec's tiny configuration;
 *                 "Strata #3752", commit "swiglu_quant": quantize_mmq_q8_1).
 *                 d is kept in fp32.
 *   products   -- gate/up and down: for each output, over the 32-value K
 *                 blocks in increasing order, isum = exact int32 sum of
 *                 w_int*q, then acc = fma(d_w*d_x, isum, acc) with the
 *                 product d_w*d_x rounded to fp32 first ("Strata #3752",
 *                 commit "moe_ws kernels": per-32-value epilogue in K order,
 *                 the block's integer sum is exact so only the float order
 *                 matters; "Strata #2145", Descricao: MAGIC C operand).
 *   swiglu_q   -- H = silu(g)*u with g the gate half and u the up half of a
 *                 GU row, then q8 of H per 32-value block; H never stored
 *                 ("Strata #3752", commit "swiglu_quant").  The gate/up
 *                 rows are "split" (gate j at j, up j at n_ff + j) or
 *                 "interleaved" (gate j at 2j, up j at 2j + 1): the commit's
 *                 test runs both; it names the layouts without defining
 *                 them, and these are the plain readings.  The GU row's
 *                 columns follow the weight rows, so only this step sees
 *                 the layout.
 *   combine    -- out[t] = sum over the token's top-k ranks r = 0..k-1, in
 *                 that order, of w[t,r]*Dm[row(t,r)] with one fma per rank
 *                 (the layer spec's tiny configuration).
 *
 * Weight formats: see the byte layouts in the `synth` module (W2: 64-value
 * blocks, fp16 d, 2-bit codes c, value d*(c-2); W4NL: 32-value blocks, fp16
 * d, 4-bit index into a 16-entry table, value d*T[idx]; Q8_0: 32-value
 * blocks of 34 bytes, fp16 d then 32 int8 codes q, value d*q -- the pages
 * name Q8_0 as a down type of the swiglu_quant test ("Strata #3752") without
 * laying it out, and this is the common layout of that name).
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_W2 1
#define ORC_W4NL 2
#define ORC_Q8_0 3

static const int ORC_NL4[16] = {-127, -104, -83, -65, -49, -35, -22, -10,
                                1,    13,   25,  38,  53,  69,  89,  113};

/* IEEE binary16 -> binary32, written from the format's definition. */
static float orc_half(uint16_t h) {
  int sign = (h >> 15) & 1;
  int ex = (h >> 10) & 31;
  int man = h & 1023;
  float v;
  if (ex == 0)
    v = ldexpf((float)man, -24); /* zero or subnormal */
  else if (ex == 31)
    v = man ? NAN : INFINITY;
  else
    v = ldexpf((float)(1024 + man), ex - 25);
  return sign ? -v : v;
}

static int orc_block_values(int fmt) { return fmt == ORC_W2 ? 64 : 32; }
static int orc_block_bytes(int fmt) { return fmt == ORC_Q8_0 ? 34 : 18; }

int64_t orc_row_bytes(int fmt, int K) {
  return (int64_t)(K / orc_block_values(fmt)) * orc_block_bytes(fmt);
}

/* Integer weight value (c-2, T[idx] or q) of element j of a row. */
static int orc_w_int(int fmt, const uint8_t *row, int j) {
  int bv = orc_block_values(fmt);
  const uint8_t *blk = row + (int64_t)(j / bv) * orc_block_bytes(fmt);
  int jj = j % bv;
  if (fmt == ORC_Q8_0) return (int)(int8_t)blk[2 + jj];
  if (fmt == ORC_W2) {
    int c = (blk[2 + jj / 4] >> (2 * (jj % 4))) & 3;
    return c - 2;
  }
  int idx = (blk[2 + jj / 2] >> (4 * (jj % 2))) & 15;
  return ORC_NL4[idx];
}

/* fp16 scale of the block holding element j of a row, as fp32. */
static float orc_w_scale(int fmt, const uint8_t *row, int j) {
  int bv = orc_block_values(fmt);
  const uint8_t *blk = row + (int64_t)(j / bv) * orc_block_bytes(fmt);
  return orc_half((uint16_t)(blk[0] | (blk[1] << 8)));
}

/* Dequantized element, for tests only: scale * integer value, in double. */
double orc_w_value(int fmt, const uint8_t *row, int j) {
  return (double)orc_w_scale(fmt, row, j) * (double)orc_w_int(fmt, row, j);
}

/* ---------------------------------------------------------------- route */
/* Histogram, exclusive prefix sum (group bounds) and stable bucketing of the
 * T*k flat rows ("Strata #3752", commits "moe_ws wiring" and "swiglu_quant
 * landed": quantize_scatter and the group bounds).
 * Returns the number of entries whose expert id is out of range; those get
 * dst_of = -1 and no row. */
int64_t orc_route(int64_t T, int k, int E, const int32_t *ids, int32_t *counts,
                  int32_t *offsets, int32_t *row_src, int32_t *dst_of) {
  int64_t n = T * k, bad = 0;
  int32_t *fill = (int32_t *)malloc(sizeof(int32_t) * (E > 0 ? E : 1));
  for (int e = 0; e < E; e++) counts[e] = 0;
  for (int64_t i = 0; i < n; i++) {
    int32_t e = ids[i];
    if (e < 0 || e >= E) {
      bad++;
      continue;
    }
    counts[e]++;
  }
  offsets[0] = 0;
  for (int e = 0; e < E; e++) offsets[e + 1] = offsets[e] + counts[e];
  for (int e = 0; e < E; e++) fill[e] = offsets[e];
  for (int64_t i = 0; i < n; i++) {
    int32_t e = ids[i];
    if (e < 0 || e >= E) {
      dst_of[i] = -1;
      continue;
    }
    int32_t pos = fill[e]++;
    row_src[pos] = (int32_t)i;
    dst_of[i] = pos;
  }
  free(fill);
  return bad;
}

/* ------------------------------------------------------------------- q8 */
/* q8 of one row, block by block: amax, d = amax/127, q = rint(x/d), d = 0
 * gives q = 0 (the layer spec's tiny configuration; "Strata #3752", commit
 * "swiglu_quant": quantize_mmq_q8_1 on 32-value blocks). */
static void orc_q8_row(int K, const float *x, int8_t *q, float *d) {
  for (int b = 0; b < K / 32; b++) {
    const float *xb = x + 32 * b;
    float amax = 0.0f;
    for (int i = 0; i < 32; i++) {
      float a = fabsf(xb[i]);
      if (a > amax) amax = a;
    }
    float db = amax / 127.0f;
    d[b] = db;
    for (int i = 0; i < 32; i++)
      q[32 * b + i] = (db == 0.0f) ? 0 : (int8_t)rintf(xb[i] / db);
  }
}

void orc_quant_q8(int64_t rows, int K, const float *x, int8_t *q, float *d) {
  for (int64_t r = 0; r < rows; r++)
    orc_q8_row(K, x + r * K, q + r * K, d + r * (K / 32));
}

/* ------------------------------------------------------------- products */
/* The per-32-value epilogue in K order ("Strata #3752", commit "moe_ws
 * kernels"): acc = fma(d_w*d_x, isum, acc) block by block, isum exact.
 * One activation row (q, dq) against every row of one expert's weight
 * matrix [n_out x K]. */
static void orc_product_row(int fmt, int K, int n_out, const uint8_t *wmat,
                            const int8_t *q, const float *dq, float *out) {
  int64_t rb = orc_row_bytes(fmt, K);
  int nb = K / 32;
  int *wi = (int *)malloc(sizeof(int) * K);
  float *ws = (float *)malloc(sizeof(float) * nb);
  for (int o = 0; o < n_out; o++) {
    const uint8_t *wrow = wmat + (int64_t)o * rb;
    for (int j = 0; j < K; j++) wi[j] = orc_w_int(fmt, wrow, j);
    for (int b = 0; b < nb; b++) ws[b] = orc_w_scale(fmt, wrow, 32 * b);
    float acc = 0.0f;
    for (int b = 0; b < nb; b++) {
      int32_t isum = 0;
      for (int i = 0; i < 32; i++) isum += wi[32 * b + i] * (int32_t)q[32 * b + i];
      float s = ws[b] * dq[b];
      acc = fmaf(s, (float)isum, acc);
    }
    out[o] = acc;
  }
  free(wi);
  free(ws);
}

/* Per-block integer sums of one (weight row, activation row) pair; for the
 * block-sum invariants in the tests. */
void orc_block_sums(int fmt, int K, const uint8_t *wrow, const int8_t *q,
                    int32_t *isum) {
  for (int b = 0; b < K / 32; b++) {
    int32_t s = 0;
    for (int i = 0; i < 32; i++) s += orc_w_int(fmt, wrow, 32 * b + i) * (int32_t)q[32 * b + i];
    isum[b] = s;
  }
}

/* rows activation rows against one expert matrix: out [rows x n_out]. */
void orc_expert_rows(int fmt, int K, int n_out, const uint8_t *wmat,
                     int64_t rows, const int8_t *q, const float *dq, float *out) {
  for (int64_t r = 0; r < rows; r++)
    orc_product_row(fmt, K, n_out, wmat, q + r * K, dq + r * (K / 32),
                    out + r * n_out);
}

/* ------------------------------------------------------- swiglu + quant */
/* gate/up row layouts */
#define ORC_GU_SPLIT 0
#define ORC_GU_INTERLEAVED 1

/* H = silu(g)*u then q8 of H, H never kept beyond this row's scratch
 * ("Strata #3752", commit "swiglu_quant"). */
static void orc_swiglu_quant_row(int n_ff, int layout, const float *gu,
                                 int8_t *hq, float *dh, float *hbuf) {
  for (int j = 0; j < n_ff; j++) {
    float g = gu[j];
    float u = gu[n_ff + j];
    if (layout == ORC_GU_INTERLEAVED) {
      g = gu[2 * j];
      u = gu[2 * j + 1];
    }
    hbuf[j] = (g / (1.0f + expf(-g))) * u;
  }
  orc_q8_row(n_ff, hbuf, hq, dh);
}

void orc_swiglu_quant(int64_t rows, int n_ff, int layout, const float *gu,
                      int8_t *hq, float *dh) {
  float *h = (float *)malloc(sizeof(float) * n_ff);
  for (int64_t r = 0; r < rows; r++)
    orc_swiglu_quant_row(n_ff, layout, gu + r * 2 * n_ff, hq + r * n_ff,
                         dh + r * (n_ff / 32), h);
  free(h);
}

/* --------------------------------------------------------------- combine */
/* out[t] = sum over ranks r = 0..k-1, in that order, of w[t,r]*Dm[row(t,r)],
 * one fma per rank (the layer spec's tiny configuration); dropped rows add
 * nothing. */
void orc_combine(int64_t T, int k, int d, const float *w, const int32_t *dst_of,
                 const float *dm, float *out) {
  for (int64_t t = 0; t < T; t++)
    for (int j = 0; j < d; j++) {
      float acc = 0.0f;
      for (int r = 0; r < k; r++) {
        int32_t pos = dst_of[t * k + r];
        if (pos < 0) continue;
        acc = fmaf(w[t * k + r], dm[(int64_t)pos * d + j], acc);
      }
      out[t * d + j] = acc;
    }
}

/* ------------------------------------------------------------ full layer */
typedef struct {
  int d, n_ff, k, gu_fmt, down_fmt, gu_layout;
  const uint8_t *pack;
  const int64_t *eoff;
  const int32_t *ids, *row_src;
  const int8_t *xq;
  const float *dx;
  float *gu;
  int8_t *hq;
  float *dh;
  float *dm;
  int64_t r0, r1;
} orc_job;

static void *orc_rows_worker(void *p) {
  orc_job *j = (orc_job *)p;
  int nff2 = 2 * j->n_ff;
  float *hbuf = (float *)malloc(sizeof(float) * j->n_ff);
  for (int64_t r = j->r0; r < j->r1; r++) {
    int32_t src = j->row_src[r];
    int64_t t = src / j->k;
    int e = j->ids[src];
    const uint8_t *wgu = j->pack + j->eoff[2 * e];
    const uint8_t *wdn = j->pack + j->eoff[2 * e + 1];
    float *gu = j->gu + r * nff2;
    int8_t *hq = j->hq + r * j->n_ff;
    float *dh = j->dh + r * (j->n_ff / 32);
    orc_product_row(j->gu_fmt, j->d, nff2, wgu, j->xq + t * j->d,
                    j->dx + t * (j->d / 32), gu);
    orc_swiglu_quant_row(j->n_ff, j->gu_layout, gu, hq, dh, hbuf);
    orc_product_row(j->down_fmt, j->n_ff, j->d, wdn, hq, dh, j->dm + r * j->d);
  }
  free(hbuf);
  return NULL;
}

/*
 * The whole layer.  Every intermediate is written to caller memory:
 * counts[E], offsets[E+1], row_src[R], dst_of[T*k], xq[T*d], dx[T*d/32],
 * gu[R*2*n_ff], hq[R*n_ff], dh[R*n_ff/32], dm[R*d], out[T*d], R = valid
 * rows.  The routed rows are split over `threads` POSIX threads; each row's
 * arithmetic is the same whatever the split.  Returns the count of
 * out-of-range expert ids.
 */
int64_t orc_layer(int64_t T, int d, int n_ff, int E, int k, int gu_fmt,
                  int down_fmt, int gu_layout, const float *x, const int32_t *ids,
                  const float *w, const uint8_t *pack, const int64_t *eoff,
                  int32_t *counts, int32_t *offsets, int32_t *row_src,
                  int32_t *dst_of, int8_t *xq, float *dx, float *gu,
                  int8_t *hq, float *dh, float *dm, float *out, int threads) {
  int64_t bad = orc_route(T, k, E, ids, counts, offsets, row_src, dst_of);
  int64_t R = offsets[E];
  orc_quant_q8(T, d, x, xq, dx);
  if (threads < 1) threads = 1;
  pthread_t *th = (pthread_t *)malloc(sizeof(pthread_t) * threads);
  orc_job *jobs = (orc_job *)malloc(sizeof(orc_job) * threads);
  for (int i = 0; i < threads; i++) {
    orc_job j = {d, n_ff, k, gu_fmt, down_fmt, gu_layout, pack, eoff, ids, row_src,
                 xq, dx, gu, hq, dh, dm, R * i / threads, R * (i + 1) / threads};
    jobs[i] = j;
    pthread_create(&th[i], NULL, orc_rows_worker, &jobs[i]);
  }
  for (int i = 0; i < threads; i++) pthread_join(th[i], NULL);
  free(th);
  free(jobs);
  orc_combine(T, k, d, w, dst_of, dm, out);
  return bad;
}
