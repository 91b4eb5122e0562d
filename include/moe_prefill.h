/*
 * moe_prefill.h -- C ABI of libmoeprefill.so: the prompt-path (prefill)
 * routed-expert FFN of a quantized mixture-of-experts layer on one GB300
 * (sm_103a).
 *
 * The layer, as the "Strata" pull requests describe it:
 *   route   : bucket the T*k (token, expert) rows by expert -- histogram,
 *             exclusive prefix sum, stable permutation ("Strata #3752",
 *             commits "moe_ws wiring" and "swiglu_quant landed":
 *             quantize_scatter and the group bounds);
 *   q8      : activations to int8 per 32-value block, d = amax/127,
 *             q = rint(x/d), d = 0 gives q = 0 ("Strata #3752", commit
 *             "swiglu_quant": quantize_mmq_q8_1; the layer spec's tiny
 *             configuration);
 *   gate/up : per routed row, GU = sum over 32-value K blocks, in K order,
 *             of d_w*d_x*isum, isum the exact integer block sum
 *             ("Strata #3752", commit "moe_ws kernels");
 *   swiglu_quant : H = silu(g)*u, requantized to q8 per 32-value block in
 *             the same pass, H never stored ("Strata #3752", commit
 *             "swiglu_quant");
 *   down    : Dm = the same per-block product of the down weights with Hq;
 *   combine : out[t] = sum over the token's top-k ranks in rank order of
 *             w[t,r]*Dm[row(t,r)] (the layer spec's tiny configuration).
 *
 * Conventions for every entry point:
 *   - Every pointer argument named d_* or documented "device" is device
 *     memory of the current CUDA device, owned by the caller.  The library
 *     allocates no device memory and keeps no state between calls except a
 *     launch counter and, per device, three CUDA streams and seven events
 *     (created on the first product call that is not being captured, kept
 *     until the process exits): the products' small-row launches run on one
 *     stream, forked from `stream` by an event and joined back before the
 *     call returns (once per stage in the stage entry points, once for both
 *     products in the whole-layer calls), so the work stays ordered on
 *     `stream` (under stream capture, as graph edges); the host-buffer
 *     layer's copies run on the other two.  All work is enqueued with no host
 *     synchronisation, unless the entry point says otherwise.
 *   - Arguments are validated on the host before anything is launched; a
 *     negative MOE_ERR_* code is returned and nothing is enqueued.
 *   - Conditions only the device can see (an expert id outside [0, E), an
 *     expert offset that is misaligned or runs past weight_pack_bytes, a
 *     pipeline wait that timed out) set bits of a device status word in the
 *     workspace (moe_read_status); the offending rows or experts are skipped,
 *     never accessed out of bounds.
 *   - The stream is a cudaStream_t (0 = legacy default stream).
 */
#ifndef MOE_PREFILL_H
#define MOE_PREFILL_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *moe_stream_t; /* == cudaStream_t */

/* Weight formats.
 * MOE_FMT_W2  : 64 values per 18-byte block: fp16 scale d (little endian,
 *               bytes 0-1), then 16 bytes of 2-bit codes c; code j sits in
 *               byte 2 + j/4 at bit 2*(j%4).  Value = d*(c-2).
 * MOE_FMT_W4NL: 32 values per 18-byte block: fp16 d, then 16 bytes of 4-bit
 *               indices; index j sits in byte 2 + j/2, low nibble for even j.
 *               Value = d*T[idx], T = {-127,-104,-83,-65,-49,-35,-22,-10,1,
 *               13,25,38,53,69,89,113}.
 * MOE_FMT_Q8_0: 32 values per 34-byte block: fp16 d, then 32 int8 codes q;
 *               code j sits in byte 2 + j.  Value = d*q.  ("Strata #3752",
 *               commit "swiglu_quant", names Q8_0 as a down type of its test
 *               without laying it out; this is the common layout of that
 *               name.)
 * A weight matrix [rows x K] is row-major, each row its blocks back to back. */
enum { MOE_FMT_W2 = 1, MOE_FMT_W4NL = 2, MOE_FMT_Q8_0 = 3 };

/* Row order of a gate/up matrix [2*n_ff x d] ("Strata #3752", commit
 * "swiglu_quant": its test runs "split and interleaved gate/up rows"; the
 * page names the two without defining them -- these are the plain readings):
 *   MOE_GU_SPLIT        gate rows 0..n_ff-1, then up rows n_ff..2*n_ff-1
 *   MOE_GU_INTERLEAVED  gate row j at row 2j, up row j at row 2j+1
 * H = silu(gate)*up pairs gate j with up j either way. */
enum { MOE_GU_SPLIT = 0, MOE_GU_INTERLEAVED = 1 };

/* Layer flags (MoeLayerDesc.flags).
 *   MOE_FLAG_FUSED_COMBINE  moe_prefill_layer runs the combine inside the
 *     down product's epilogue instead of as a pass of its own: after a
 *     routed row's Dm values of a 32-column group are stored, the row counts
 *     itself in for its token and group (a device-scope atomic after a
 *     fence); the last of the token's k rows to arrive sums the k rows of
 *     the group in rank order, one fma per rank -- the same arithmetic as
 *     moe_combine, so out is bit-identical either way ("Strata #3752",
 *     Validation: the prompt path's combine fused with the write).  Dm is
 *     still written (a row cannot know it is the last before it has
 *     published its values).
 *   MOE_FLAG_HOST_OUT_DEFERRED  moe_prefill_layer_host does not make `stream`
 *     wait for out's copy back to the host: in a run of calls, one call's
 *     out goes back while the next call computes.  Every out copied by the
 *     host-buffer calls so far is complete once moe_host_out_join(stream)
 *     has been enqueued and `stream` has been synchronised.  Each call's
 *     combine waits for the previous call's copy before it writes the
 *     staging buffer.  Under stream capture, and with MOE_FLAG_FUSED_COMBINE,
 *     out's copy runs on `stream` and the flag changes nothing.  Other entry
 *     points ignore it. */
enum { MOE_FLAG_FUSED_COMBINE = 1, MOE_FLAG_HOST_OUT_DEFERRED = 2 };

enum {
  MOE_OK = 0,
  MOE_ERR_NULL = -1,        /* a required pointer is NULL                  */
  MOE_ERR_SHAPE = -2,       /* T, d, n_ff, E or k out of the supported set */
  MOE_ERR_FORMAT = -3,      /* unknown weight format or gate/up layout     */
  MOE_ERR_ALIGN = -4,       /* a pointer is not aligned as documented      */
  MOE_ERR_WORKSPACE = -5,   /* workspace smaller than moe_prefill_workspace_bytes */
  MOE_ERR_DEVICE = -6,      /* no sm_103 device is current                 */
  MOE_ERR_LAUNCH = -7,      /* a CUDA call failed while enqueueing         */
  MOE_ERR_DEVICE_STATUS = -8, /* moe_read_status found device-side errors  */
  MOE_ERR_SCRATCH = -9       /* too large for moe_route_noalloc's fixed scratch */
};

/* Device status bits (moe_read_status). */
enum {
  MOE_STATUS_BAD_EXPERT_ID = 1,   /* a topk id outside [0, E): row dropped  */
  MOE_STATUS_BAD_OFFSET = 2,      /* an expert offset misaligned or past the pack: expert skipped */
  MOE_STATUS_PIPE_TIMEOUT = 4,    /* a bounded pipeline wait gave up        */
  MOE_STATUS_BAD_ROUTING = 8      /* a stage found routing data that moe_route
                                     did not write (stage API misuse): skipped */
};

/* Supported shapes: T >= 0; d a multiple of 128, 128 <= d <= 8192; n_ff a
 * multiple of 64, 64 <= n_ff <= 4096; 1 <= E <= 1024; 1 <= k <= E;
 * T*k < 2^24.  Other shapes return MOE_ERR_SHAPE. */
typedef struct MoeLayerDesc {
  int32_t T;        /* tokens                                        */
  int32_t d;        /* hidden size (gate/up K, down output rows)      */
  int32_t n_ff;     /* expert width (down K)                          */
  int32_t E;        /* experts                                        */
  int32_t k;        /* experts per token (top-k)                      */
  int32_t gu_fmt;   /* MOE_FMT_* of the gate/up matrices              */
  int32_t down_fmt; /* MOE_FMT_* of the down matrices                 */
  int32_t gu_layout;/* MOE_GU_SPLIT or MOE_GU_INTERLEAVED            */
  uint32_t flags;   /* MOE_FLAG_* bits (0 = none)                     */
  int32_t reserved; /* must be 0                                      */
  int64_t weight_pack_bytes; /* size of the tiled weight pack; expert matrices must lie inside */
} MoeLayerDesc;

/* Device pointers into a workspace, as laid out by this library.  Every
 * region is 256-byte aligned.  R = T*k (rows of entries with a valid id come
 * first; offsets[E] is the number of valid rows).
 *   counts  int32 [E]        rows per expert
 *   offsets int32 [E+1]      exclusive prefix sum of counts
 *   order   int32 [E]        expert ids by count, largest first, ties by id
 *   row_src int32 [R]        routed row -> flat entry t*k+r
 *   dst_of  int32 [R]        flat entry -> routed row (-1 if its id is bad)
 *   xq      fp16  [R*d]      q8 values of x as exact fp16 integers, one row
 *                            per routed row (row r holds token row_src[r]/k:
 *                            quantize and scatter), stored pair-interleaved in
 *                            every 16-value group: position 2i holds value i,
 *                            2i+1 holds value i+8
 *   dx      fp32  [R*sd]     q8 scales of x per routed row, rows padded to
 *                            sd = d/32 rounded up to a multiple of 4
 *   gu      fp32  [R*2*n_ff] gate/up rows, columns in the weight rows' order:
 *                            gate j at j and up j at n_ff+j (MOE_GU_SPLIT)
 *                            or at 2j and 2j+1 (MOE_GU_INTERLEAVED); the
 *                            same bytes as dm (gu == dm): the down product
 *                            overwrites it, the fused layer never writes it
 *   hq      fp16  [R*n_ff]   q8 values of H as exact fp16 integers, stored
 *                            pair-interleaved like xq
 *   dh      fp32  [R*sf]     q8 scales of H, rows padded to sf = n_ff/32
 *                            rounded up to a multiple of 4
 *   dm      fp32  [R*d]      down rows
 *   status  int32 [1]        MOE_STATUS_* bits */
typedef struct MoeWorkspaceView {
  int32_t *counts, *offsets, *order, *row_src, *dst_of;
  uint16_t *xq;
  float *dx, *gu;
  uint16_t *hq;
  float *dh, *dm;
  int32_t *status;
} MoeWorkspaceView;

/* Bytes of device workspace the layer and the stage entry points need for
 * `desc` (0 if desc is invalid).  Host only. */
size_t moe_prefill_workspace_bytes(const MoeLayerDesc *desc);

/* Fill `view` with the device addresses of the workspace regions.  Host
 * only; returns MOE_OK or an error code. */
int moe_workspace_view(const MoeLayerDesc *desc, void *workspace,
                       size_t workspace_bytes, MoeWorkspaceView *view);

/* Device-tiled weight pack.  The product kernels read the weights in a
 * tiled byte order, a permutation of the row-major pack made once per layer
 * (at load time) by moe_tile_weights.  For each weight matrix [N_out x K] of
 * bpr = K / (values per block) blocks per row, BB bytes a block (18; 34 for
 * Q8_0), CB code bytes a block (BB - 2) and cb blocks a chunk (4; 2 for
 * Q8_0):
 *   tile t holds NW = min(256, N_out - 256t) rows and starts at byte
 *     256*t*bpr*BB of the matrix.  Down: rows 256t .. 256t+NW-1.  Gate/up:
 *     gate rows 128t .. 128t+NW/2-1, then the matching up rows (tile row
 *     r < NW/2 is gate output 128t+r, tile row NW/2+r is up output
 *     128t+r); gate output g is row g of the row-major matrix and up output
 *     g row n_ff+g (MOE_GU_SPLIT), or rows 2g and 2g+1 (MOE_GU_INTERLEAVED);
 *   chunk c of a tile covers blocks cb*c .. cb*c+nbc-1, nbc = min(cb,
 *     bpr - cb*c), and starts at byte cb*c*NW*BB of the tile;
 *   inside a chunk, the CB code bytes (block bytes 2..BB-1) of (tile row r,
 *     chunk block j) lie at (j*NW + r)*CB, then the fp16 scales (block bytes
 *     0..1) at nbc*NW*CB + (j*NW + r)*2.
 * A tiled matrix has the row-major matrix's size.  Expert e's gate/up matrix
 * starts at e*(G + D) and its down matrix at e*(G + D) + G, G and D the
 * matrices' sizes; moe_tiled_pack_bytes(desc) = E*(G + D). */
int64_t moe_tiled_pack_bytes(const MoeLayerDesc *desc);

/* Tile a row-major weight pack (the block layouts of the MOE_FMT_* formats
 * above: expert e's gate/up matrix [2*n_ff x d] at expert_offsets[2e], its
 * down matrix [d x n_ff] at expert_offsets[2e+1], each offset a multiple of
 * 16 and each matrix inside weight_pack_bytes).
 *   weight_pack    device bytes [weight_pack_bytes], 16-byte aligned
 *   expert_offsets device int64 [E x 2] (row-major pack offsets)
 *   tiled_pack     device bytes, 16-byte aligned, desc->weight_pack_bytes of
 *                  them (>= moe_tiled_pack_bytes(desc), else MOE_ERR_WORKSPACE)
 *   tiled_offsets  device int64 [E x 2]: written with the tiled pack's offsets
 *   status         device int32 [1] or NULL: MOE_STATUS_BAD_OFFSET is or-ed
 *                  in when a source offset is misaligned or runs past
 *                  weight_pack_bytes (that matrix is written as zeros)
 * The tiled pack and its offsets are what moe_prefill_layer, moe_gate_up and
 * moe_down take as weight_pack and expert_offsets. */
int moe_tile_weights(const MoeLayerDesc *desc, const uint8_t *weight_pack,
                     int64_t weight_pack_bytes, const int64_t *expert_offsets,
                     uint8_t *tiled_pack, int64_t *tiled_offsets, int32_t *status,
                     moe_stream_t stream);

/* The whole layer: route -> q8 -> gate/up with swiglu_quant fused -> down ->
 * combine (the gu region of the workspace is not written).
 *   x              device fp32 [T x d], row-major
 *   topk_ids       device int32 [T x k], expert of each (token, rank)
 *   topk_w         device fp32 [T x k], combine weight of each (token, rank)
 *   weight_pack    device bytes [weight_pack_bytes], 16-byte aligned: the
 *                  tiled pack written by moe_tile_weights
 *   expert_offsets device int64 [E x 2]: byte offsets in weight_pack of expert
 *                  e's gate/up matrix [2*n_ff x d] and down matrix [d x n_ff]
 *                  (the tiled offsets of moe_tile_weights); each must be a
 *                  multiple of 16 ("a per-layer offset table, + the down
 *                  offset", Strata #3752 commit "moe_ws kernels")
 *   out            device fp32 [T x d]
 *   workspace      device, 256-byte aligned, >= moe_prefill_workspace_bytes
 * Returns MOE_OK once everything is enqueued on `stream`. */
int moe_prefill_layer(const MoeLayerDesc *desc, const float *x,
                      const int32_t *topk_ids, const float *topk_w,
                      const uint8_t *weight_pack, const int64_t *expert_offsets,
                      float *out, void *workspace, size_t workspace_bytes,
                      moe_stream_t stream);

/* The same layer with x, topk_ids, topk_w and out in HOST memory (pinned
 * memory makes the copies asynchronous; pageable memory works but the copies
 * then synchronise).  The weights, offsets and workspace stay on the device.
 * The host inputs are copied into `io`, a caller-owned device staging buffer
 * of moe_host_io_bytes(desc) bytes (256-byte aligned); out is copied back
 * from it.  The call returns after enqueueing: the caller synchronises
 * `stream` before reading out or reusing the host inputs.
 * The transfers overlap compute where the order allows: x is copied on a
 * per-device copy stream that waits only until the previous call on the same
 * `io` has quantised its x (so a call enqueued while the previous one
 * computes brings its x in meanwhile), and out leaves in token chunks on a
 * second copy stream right behind the combine; `stream` waits for the last
 * chunk (unless desc->flags has MOE_FLAG_HOST_OUT_DEFERRED).  Calls whose
 * work overlaps on the same `io` (other streams, other threads) race, as on
 * one workspace.  Under stream capture all copies run on `stream` in order.
 *
 * moe_host_out_join makes `stream` wait for every out copy that host-buffer
 * calls on the current device have enqueued so far (MOE_OK and nothing
 * enqueued when there is none, or when `stream` is being captured: there
 * the copies run on the stream in order); with MOE_FLAG_HOST_OUT_DEFERRED
 * the caller enqueues it, then synchronises `stream`, before reading any
 * h_out. */
size_t moe_host_io_bytes(const MoeLayerDesc *desc);
int moe_prefill_layer_host(const MoeLayerDesc *desc, const float *h_x,
                           const int32_t *h_topk_ids, const float *h_topk_w,
                           const uint8_t *weight_pack,
                           const int64_t *expert_offsets, float *h_out,
                           void *io, size_t io_bytes, void *workspace,
                           size_t workspace_bytes, moe_stream_t stream);
int moe_host_out_join(moe_stream_t stream);

/* Stage entry points (tests and profiling).  Each runs one step of the
 * layer, reading and writing the workspace regions of MoeWorkspaceView, in
 * the order route, quant_q8, gate_up, swiglu_quant, down, combine (a stage
 * run on a workspace that moe_route has not filled reads garbage routing data;
 * it bounds-checks it, skips what is out of range and sets
 * MOE_STATUS_BAD_ROUTING, never reading or writing outside the buffers).  A later
 * stage may be re-run on workspace contents written by the caller (for
 * example the down product alone on a reference Hq). */
int moe_route(const MoeLayerDesc *desc, const int32_t *topk_ids,
              void *workspace, size_t workspace_bytes, moe_stream_t stream);
int moe_quant_q8(const MoeLayerDesc *desc, const float *x, void *workspace,
                 size_t workspace_bytes, moe_stream_t stream);
int moe_gate_up(const MoeLayerDesc *desc, const uint8_t *weight_pack,
                const int64_t *expert_offsets, void *workspace,
                size_t workspace_bytes, moe_stream_t stream);
/* gate/up with swiglu_quant fused into its epilogue: writes hq and dh (as
 * moe_gate_up followed by moe_swiglu_quant would, bit for bit) and leaves gu
 * unwritten.  This is the step moe_prefill_layer runs. */
int moe_gate_up_swiglu(const MoeLayerDesc *desc, const uint8_t *weight_pack,
                       const int64_t *expert_offsets, void *workspace,
                       size_t workspace_bytes, moe_stream_t stream);
int moe_swiglu_quant(const MoeLayerDesc *desc, void *workspace,
                     size_t workspace_bytes, moe_stream_t stream);
int moe_down(const MoeLayerDesc *desc, const uint8_t *weight_pack,
             const int64_t *expert_offsets, void *workspace,
             size_t workspace_bytes, moe_stream_t stream);
/* The down product with the combine fused into its epilogue (the step
 * moe_prefill_layer runs under MOE_FLAG_FUSED_COMBINE; here regardless of
 * the flag): writes dm and out [T x d] (device fp32, 16-byte aligned) from
 * topk_w (device fp32 [T x k]), the routing of moe_route and the workspace's
 * hq and dh. */
int moe_down_combine(const MoeLayerDesc *desc, const uint8_t *weight_pack,
                     const int64_t *expert_offsets, const float *topk_w, float *out,
                     void *workspace, size_t workspace_bytes, moe_stream_t stream);
int moe_combine(const MoeLayerDesc *desc, const float *topk_w, float *out,
                void *workspace, size_t workspace_bytes, moe_stream_t stream);

/* Synchronise `stream`, copy the device status word of the workspace to
 * *status, and clear it on the device.  Returns MOE_OK, or
 * MOE_ERR_DEVICE_STATUS when any bit was set. */
int moe_read_status(const MoeLayerDesc *desc, void *workspace,
                    size_t workspace_bytes, int32_t *status,
                    moe_stream_t stream);

/* Routing (the same outputs as moe_route) for callers that cannot allocate
 * device memory -- code that may only use the buffers handed to it, or that
 * runs where allocation is not allowed.  The pages have no counterpart: this
 * entry point is an addition of this library.
 *   topk_ids  device int32 [T x k] (desc: T, E, k; other fields unused)
 *   counts    device int32 [E]     rows per expert
 *   offsets   device int32 [E+1]   exclusive prefix sum of counts
 *   row_src   device int32 [T*k]   routed row -> flat entry t*k+r (the first
 *                                  offsets[E] entries are written)
 *   dst_of    device int32 [T*k]   flat entry -> routed row, -1 where the
 *                                  expert id is outside [0, E)
 * Its scratch is a fixed 1 MiB array in the library's device memory (held by
 * every GPU that loads the library until the process exits) instead of a
 * workspace: (c + ceil(c/8))*E + 4*floor(T*k/128) + 9*E + 71 int32, with
 * c = ceil(T*k/1024), must fit in 262144 (T*k = 163840 with E = 512 needs
 * about 102,000), or
 * MOE_ERR_SCRATCH is returned with nothing enqueued.  Every call looks the
 * array's device address up (cudaGetSymbolAddress) with the current device
 * current; the first call on a device also loads the library's device code
 * there, so make it before any stream capture.  No status word reaches the
 * caller on this path: an expert id outside [0, E) shows only as dst_of = -1
 * for that entry (and offsets[E] < T*k).  All calls share the array: calls
 * whose work overlaps on the GPU (other streams, other threads) race.
 * Nothing is allocated or freed. */
int moe_route_noalloc(const MoeLayerDesc *desc, const int32_t *topk_ids,
                      int32_t *counts, int32_t *offsets, int32_t *row_src,
                      int32_t *dst_of, moe_stream_t stream);

/* Self-test of the failure path of the bounded pipeline waits (tests only).
 * Enqueues one warp that waits on an mbarrier nothing ever completes,
 * through the wait routine the product kernels use: sleep = 1 takes the
 * timed wait of the producer and decode roles (gives up after 20 ms of
 * global time), sleep = 0 the polling wait of the epilogue and MMA roles
 * (gives up after its fixed count of polls, about 1.4 s on a GB300).  On
 * giving up it or-s MOE_STATUS_PIPE_TIMEOUT into *status (device int32,
 * 4-byte aligned) and exits; nothing faults or traps and the context stays
 * usable.  Returns MOE_OK once enqueued, MOE_ERR_NULL / MOE_ERR_ALIGN /
 * MOE_ERR_SHAPE (sleep not 0 or 1) / MOE_ERR_DEVICE before enqueueing. */
int moe_selftest_wait_timeout(int32_t *status, int sleep, moe_stream_t stream);

/* MOE_OK when the current CUDA device is an sm_103 part, else MOE_ERR_DEVICE. */
int moe_check_device(void);

/* Human-readable text of a MOE_* code (static storage). */
const char *moe_status_string(int code);

/* Kernels this library has launched in this process (all threads). */
uint64_t moe_kernel_launches(void);

#ifdef __cplusplus
}
#endif
#endif /* MOE_PREFILL_H */
