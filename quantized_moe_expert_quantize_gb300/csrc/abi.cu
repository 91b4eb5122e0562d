// C ABI of libmoeprefill.so: argument validation, workspace layout and the
// order of the stages.  See include/moe_prefill.h for the contract.
#include <cuda.h>

#include <atomic>
#include <cstring>
#include <mutex>

#include "common.cuh"

namespace moe {

static std::atomic<uint64_t> g_launches{0};
void count_launch(int n) { g_launches.fetch_add((uint64_t)n, std::memory_order_relaxed); }

// Per-device values looked up once are cached in relaxed atomics: two
// threads may both look one up, and both store the same value.
int device_sm_count() {
  static std::atomic<int> cache[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 1;
  if (dev >= 0 && dev < 64) {
    const int c = cache[dev].load(std::memory_order_relaxed);
    if (c > 0) return c;
  }
  int n = 1;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1)
    return 1;
  if (dev >= 0 && dev < 64) cache[dev].store(n, std::memory_order_relaxed);
  return n;
}

// The two driver calls are looked up through the runtime (as the tensor-map
// encoder is), so that loading the library needs no libcuda on a host
// without a GPU.
uint64_t current_context_id() {
  using GetCurrent = CUresult (*)(CUcontext*);
  using GetId = CUresult (*)(CUcontext, unsigned long long*);
  static GetCurrent get_current = nullptr;
  static GetId get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<GetCurrent>(p);
    p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<GetId>(p);
  });
  CUcontext c = nullptr;
  unsigned long long id = 0;
  if (!get_current || !get_id || get_current(&c) != CUDA_SUCCESS || !c ||
      get_id(c, &id) != CUDA_SUCCESS)
    return 0;
  return (uint64_t)id;
}

namespace {

constexpr size_t kAlign = 256;
inline size_t align_up(size_t v) { return (v + kAlign - 1) / kAlign * kAlign; }

struct Layout {
  size_t status, counts, offsets, order, tiles, row_src, dst_of, hist, xq, dx, gu, hq, dh, dm, cnt;
  size_t total;
};

inline int64_t rows_max(const MoeLayerDesc& d) { return (int64_t)d.T * d.k; }

Layout layout(const MoeLayerDesc& d) {
  Layout L{};
  size_t p = 0;
  auto take = [&](size_t bytes) {
    const size_t o = p;
    p = align_up(p + bytes);
    return o;
  };
  const int64_t R = rows_max(d);
  const int nchunks = route_chunks(R);
  L.status = take(kAlign);
  L.counts = take(sizeof(int32_t) * d.E);
  L.offsets = take(sizeof(int32_t) * (d.E + 1));
  L.order = take(sizeof(int32_t) * d.E);
  L.tiles = take(sizeof(int4) * (size_t)max_tiles(R, d.E));
  L.row_src = take(sizeof(int32_t) * R);
  L.dst_of = take(sizeof(int32_t) * R);
  L.hist = take(sizeof(int32_t) * (size_t)route_hist_rows(R) * d.E);
  L.xq = take(sizeof(uint16_t) * (size_t)R * d.d);
  L.dx = take(sizeof(float) * (size_t)R * scale_stride(d.d));
  L.hq = take(sizeof(uint16_t) * (size_t)R * d.n_ff);
  L.dh = take(sizeof(float) * (size_t)R * scale_stride(d.n_ff));
  // gu lives from the gate/up product to swiglu_quant (the whole layer never
  // writes it), dm from the down product to the combine: one region for both
  L.dm = take(sizeof(float) * (size_t)R * std::max(d.d, 2 * d.n_ff));
  L.gu = L.dm;
  L.cnt = take(sizeof(int32_t) * (size_t)d.T * (d.d / 32));  // fused combine's counters
  L.total = p;
  return L;
}

int validate_desc(const MoeLayerDesc* d) {
  if (!d) return MOE_ERR_NULL;
  if (d->T < 0 || d->d < 128 || d->d > 8192 || d->d % 128 != 0 || d->n_ff < 64 ||
      d->n_ff > 4096 || d->n_ff % 64 != 0 || d->E < 1 || d->E > 1024 || d->k < 1 ||
      d->k > d->E)
    return MOE_ERR_SHAPE;
  if ((int64_t)d->T * d->k >= ((int64_t)1 << 24)) return MOE_ERR_SHAPE;
  auto fmt_ok = [](int f) { return f == MOE_FMT_W2 || f == MOE_FMT_W4NL || f == MOE_FMT_Q8_0; };
  if (!fmt_ok(d->gu_fmt) || !fmt_ok(d->down_fmt) ||
      (d->gu_layout != MOE_GU_SPLIT && d->gu_layout != MOE_GU_INTERLEAVED) ||
      (d->flags & ~(uint32_t)(MOE_FLAG_FUSED_COMBINE | MOE_FLAG_HOST_OUT_DEFERRED)) != 0 ||
      d->reserved != 0)
    return MOE_ERR_FORMAT;
  if (d->weight_pack_bytes < 0) return MOE_ERR_SHAPE;
  if (!tc_supported(*d)) return MOE_ERR_SHAPE;
  return MOE_OK;
}

inline bool aligned(const void* p, size_t a) { return ((uintptr_t)p % a) == 0; }

int check_device() {
  int dev = 0, major = 0, minor = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_DEVICE;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
    return MOE_ERR_DEVICE;
  return (major == 10 && minor == 3) ? MOE_OK : MOE_ERR_DEVICE;
}

struct Ctx {
  MoeLayerDesc d;
  Layout L;
  uint8_t* ws;
  MoeWorkspaceView v;
};

int open_ctx(const MoeLayerDesc* desc, void* workspace, size_t bytes, Ctx& c) {
  int rc = validate_desc(desc);
  if (rc) return rc;
  if (!workspace) return MOE_ERR_NULL;
  if (!aligned(workspace, kAlign)) return MOE_ERR_ALIGN;
  c.d = *desc;
  c.L = layout(c.d);
  if (bytes < c.L.total) return MOE_ERR_WORKSPACE;
  c.ws = static_cast<uint8_t*>(workspace);
  auto at = [&](size_t off) { return (void*)(c.ws + off); };
  c.v.status = (int32_t*)at(c.L.status);
  c.v.counts = (int32_t*)at(c.L.counts);
  c.v.offsets = (int32_t*)at(c.L.offsets);
  c.v.order = (int32_t*)at(c.L.order);
  c.v.row_src = (int32_t*)at(c.L.row_src);
  c.v.dst_of = (int32_t*)at(c.L.dst_of);
  c.v.xq = (uint16_t*)at(c.L.xq);
  c.v.dx = (float*)at(c.L.dx);
  c.v.gu = (float*)at(c.L.gu);
  c.v.hq = (uint16_t*)at(c.L.hq);
  c.v.dh = (float*)at(c.L.dh);
  c.v.dm = (float*)at(c.L.dm);
  return MOE_OK;
}

inline int launch_rc(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_LAUNCH; }

// A second stream per device for the small-row launch, so that it runs
// beside the tcgen05 launch (the two read the same inputs and write disjoint
// rows) and fills the multiprocessors the tcgen05 tiles leave idle.  It
// forks from the caller's stream and joins back before the call returns, so
// to the caller the stage is ordered on its own stream as before (also under
// stream capture, where the fork and join become graph edges).  One stream
// and two events per device and context, created on the first call that is
// not being captured and kept until the process exits (a context replaced by
// cudaDeviceReset gets new ones); calls enqueue under a lock, as the events
// are shared.  Without them the two launches share the caller's stream.
struct SideStream {
  cudaStream_t s = nullptr;
  cudaEvent_t fork = nullptr, join = nullptr;
  // moe_prefill_layer_host's copy streams and their events (see there)
  cudaStream_t h2d = nullptr, d2h = nullptr;
  cudaEvent_t x_in = nullptr, x_free = nullptr, comb = nullptr, out_done = nullptr,
              entry = nullptr;
  const void* last_io = nullptr;  // staging buffer x_free was last recorded for
  bool out_pending = false;       // out_done has been recorded
  uint64_t ctx = 0;    // context the handles belong to
  bool tried = false;  // creation was attempted in that context
};
std::mutex g_side_mu;
SideStream g_side[64];

SideStream* side_stream(cudaStream_t st) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  SideStream& sd = g_side[dev];
  const uint64_t ctx = current_context_id();
  if (ctx == 0) return nullptr;
  if (sd.ctx != ctx) sd = SideStream{};  // handles of a destroyed context are dead
  if (!sd.s && !sd.tried) {
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(st, &cs) != cudaSuccess || cs != cudaStreamCaptureStatusNone)
      return nullptr;
    sd.tried = true;
    sd.ctx = ctx;
    if (cudaStreamCreateWithFlags(&sd.s, cudaStreamNonBlocking) != cudaSuccess ||
        cudaEventCreateWithFlags(&sd.fork, cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&sd.join, cudaEventDisableTiming) != cudaSuccess ||
        cudaStreamCreateWithFlags(&sd.h2d, cudaStreamNonBlocking) != cudaSuccess ||
        cudaStreamCreateWithFlags(&sd.d2h, cudaStreamNonBlocking) != cudaSuccess ||
        cudaEventCreateWithFlags(&sd.x_in, cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&sd.x_free, cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&sd.comb, cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&sd.out_done, cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&sd.entry, cudaEventDisableTiming) != cudaSuccess) {
      cudaGetLastError();
      sd.s = nullptr;
      return nullptr;
    }
  }
  return sd.s ? &sd : nullptr;
}

// The status word starts every layer (and every moe_route) at zero.
int run_route(Ctx& c, const int32_t* ids, cudaStream_t st) {
  return launch_rc(launch_route(ids, rows_max(c.d), c.d.E, (int32_t*)(c.ws + c.L.hist),
                                c.v.counts, c.v.offsets, c.v.order, c.v.row_src, c.v.dst_of,
                                (int4*)(c.ws + c.L.tiles), c.v.status + 1, c.v.status, true, st));
}

int run_quant(Ctx& c, const float* x, cudaStream_t st) {
  return launch_rc(launch_quant_q8(x, c.d.T, c.d.d, c.d.k, c.v.dst_of, rows_max(c.d),
                                  (__half*)c.v.xq, c.v.dx, st));
}

GemmArgs gemm_args(Ctx& c, int which, const uint8_t* pack, const int64_t* eoff,
                   bool fuse_swiglu = false, const float* comb_w = nullptr,
                   float* comb_out = nullptr) {
  GemmArgs a{};
  a.pack = pack;
  a.eoff = eoff;
  a.which = which;
  a.fmt = which == 0 ? c.d.gu_fmt : c.d.down_fmt;
  a.pack_bytes = c.d.weight_pack_bytes;
  a.tiles = (const int4*)(c.ws + c.L.tiles);
  a.ntiles = c.v.status + 1;
  a.sched = c.v.status + 4 + 2 * which;  // zeroed by routing (ntiles[3..6])
  a.E = c.d.E;
  a.status = c.v.status;
  a.rows_max = rows_max(c.d);
  a.gu_layout = c.d.gu_layout;
  if (which == 0) {
    a.act = (const __half*)c.v.xq;
    a.act_d = c.v.dx;
    a.K = c.d.d;
    a.N_out = 2 * c.d.n_ff;
    a.out = c.v.gu;
    if (fuse_swiglu) {
      a.hq = (__half*)c.v.hq;
      a.dh = c.v.dh;
    }
  } else {
    a.act = (const __half*)c.v.hq;
    a.act_d = c.v.dh;
    a.K = c.d.n_ff;
    a.N_out = c.d.d;
    a.out = c.v.dm;
    if (comb_out) {
      a.comb.out = comb_out;
      a.comb.topk_w = comb_w;
      a.comb.dst_of = c.v.dst_of;
      a.comb.row_src = c.v.row_src;
      a.comb.cnt = (int32_t*)(c.ws + c.L.cnt);
      a.comb.k = c.d.k;
    }
  }
  return a;
}

int run_gemm(Ctx& c, int which, const uint8_t* pack, const int64_t* eoff, cudaStream_t st,
             bool fuse_swiglu = false, const float* comb_w = nullptr, float* comb_out = nullptr) {
  const GemmArgs a = gemm_args(c, which, pack, eoff, fuse_swiglu, comb_w, comb_out);
  // 128-row tiles on the tcgen05 kernel, short remainders on the small-row
  // tier (both read the tile list's split point on the device), the latter
  // on the side stream when there is one
  std::lock_guard<std::mutex> lock(g_side_mu);
  SideStream* sd = side_stream(st);
  if (sd && (cudaEventRecord(sd->fork, st) != cudaSuccess ||
             cudaStreamWaitEvent(sd->s, sd->fork, 0) != cudaSuccess))
    return MOE_ERR_LAUNCH;
  const cudaError_t e = launch_gemm_tc(a, st);
  const cudaError_t e2 = e == cudaSuccess ? launch_gemm_small(a, sd ? sd->s : st) : e;
  // always join, so that a failed launch leaves no open fork (nor an unjoined
  // stream in a capture)
  if (sd && (cudaEventRecord(sd->join, sd->s) != cudaSuccess ||
             cudaStreamWaitEvent(st, sd->join, 0) != cudaSuccess))
    return MOE_ERR_LAUNCH;
  return launch_rc(e2);
}

// Both product stages of the layer (gate/up with swiglu_quant fused, then
// down), with one fork and one join: the tcgen05 launches run one after the
// other on the caller's stream and the small-row launches on the side
// stream.  A small-row tile's down product reads only the Hq rows that its
// own gate/up launch wrote (every routed row is in one tile, and both stages
// split the tile list at the same point), so neither chain waits for the
// other before the join.
int run_products(Ctx& c, const uint8_t* pack, const int64_t* eoff, cudaStream_t st,
                 const float* comb_w = nullptr, float* comb_out = nullptr) {
  const GemmArgs g = gemm_args(c, 0, pack, eoff, true);
  const GemmArgs d = gemm_args(c, 1, pack, eoff, false, comb_w, comb_out);
  std::lock_guard<std::mutex> lock(g_side_mu);
  SideStream* sd = side_stream(st);
  if (sd && (cudaEventRecord(sd->fork, st) != cudaSuccess ||
             cudaStreamWaitEvent(sd->s, sd->fork, 0) != cudaSuccess))
    return MOE_ERR_LAUNCH;
  cudaStream_t ss = sd ? sd->s : st;
  cudaError_t e = launch_gemm_tc(g, st);
  if (e == cudaSuccess) e = launch_gemm_small(g, ss);
  if (e == cudaSuccess) e = launch_gemm_tc(d, st);
  if (e == cudaSuccess) e = launch_gemm_small(d, ss);
  if (sd && (cudaEventRecord(sd->join, sd->s) != cudaSuccess ||
             cudaStreamWaitEvent(st, sd->join, 0) != cudaSuccess))
    return MOE_ERR_LAUNCH;
  return launch_rc(e);
}

int run_swiglu(Ctx& c, cudaStream_t st) {
  return launch_rc(launch_swiglu_quant(c.v.gu, c.v.offsets + c.d.E, rows_max(c.d), c.d.n_ff,
                                       c.d.gu_layout, (__half*)c.v.hq, c.v.dh, st));
}

int run_combine(Ctx& c, const float* w, float* out, cudaStream_t st) {
  return launch_rc(
      launch_combine(w, c.v.dst_of, c.v.dm, 0, c.d.T, c.d.k, c.d.d, rows_max(c.d), out, st));
}

// The down product with the combine fused into its epilogue: the arrival
// counters first (on the caller's stream, before the products fork).
int run_down_combine(Ctx& c, const uint8_t* pack, const int64_t* eoff, const float* w,
                     float* out, cudaStream_t st) {
  int rc = launch_rc(launch_combine_init(c.v.dst_of, c.d.T, c.d.k, c.d.d / 32,
                                         (int32_t*)(c.ws + c.L.cnt), st));
  if (rc) return rc;
  return run_gemm(c, 1, pack, eoff, st, false, w, out);
}

// The layer after quant_q8: both products, then the combine (or, with
// MOE_FLAG_FUSED_COMBINE, the combine inside the down epilogues, its arrival
// counters set up first).
int run_layer_tail(Ctx& c, const uint8_t* pack, const int64_t* eoff, const float* w, float* out,
                   cudaStream_t st) {
  int rc;
  if (c.d.flags & MOE_FLAG_FUSED_COMBINE) {
    if ((rc = launch_rc(launch_combine_init(c.v.dst_of, c.d.T, c.d.k, c.d.d / 32,
                                            (int32_t*)(c.ws + c.L.cnt), st))))
      return rc;
    return run_products(c, pack, eoff, st, w, out);
  }
  if ((rc = run_products(c, pack, eoff, st))) return rc;
  return run_combine(c, w, out, st);
}

int check_weights(const MoeLayerDesc* d, const uint8_t* pack, const int64_t* eoff) {
  if (!pack || !eoff) return MOE_ERR_NULL;
  if (!aligned(pack, 16) || !aligned(eoff, 8)) return MOE_ERR_ALIGN;
  (void)d;
  return MOE_OK;
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" {

size_t moe_prefill_workspace_bytes(const MoeLayerDesc* desc) {
  if (validate_desc(desc)) return 0;
  return layout(*desc).total;
}

int moe_workspace_view(const MoeLayerDesc* desc, void* workspace, size_t bytes,
                       MoeWorkspaceView* view) {
  if (!view) return MOE_ERR_NULL;
  Ctx c;
  const int rc = open_ctx(desc, workspace, bytes, c);
  if (rc) return rc;
  *view = c.v;
  return MOE_OK;
}

int moe_check_device(void) { return check_device(); }

int64_t moe_tiled_pack_bytes(const MoeLayerDesc* desc) {
  if (validate_desc(desc)) return 0;
  return tiled_pack_bytes(*desc);
}

int moe_tile_weights(const MoeLayerDesc* desc, const uint8_t* weight_pack,
                     int64_t weight_pack_bytes, const int64_t* expert_offsets,
                     uint8_t* tiled_pack, int64_t* tiled_offsets, int32_t* status,
                     moe_stream_t stream) {
  int rc = validate_desc(desc);
  if (rc) return rc;
  if (!weight_pack || !expert_offsets || !tiled_pack || !tiled_offsets) return MOE_ERR_NULL;
  if (weight_pack_bytes < 0) return MOE_ERR_SHAPE;
  if (desc->weight_pack_bytes < tiled_pack_bytes(*desc)) return MOE_ERR_WORKSPACE;
  if (!aligned(weight_pack, 16) || !aligned(tiled_pack, 16) || !aligned(expert_offsets, 8) ||
      !aligned(tiled_offsets, 8) || !aligned(status, 4))
    return MOE_ERR_ALIGN;
  if ((rc = check_device())) return rc;
  return launch_rc(launch_tile_weights(*desc, weight_pack, weight_pack_bytes, expert_offsets,
                                       tiled_pack, tiled_offsets, status, (cudaStream_t)stream));
}

int moe_route(const MoeLayerDesc* desc, const int32_t* topk_ids, void* ws, size_t bytes,
              moe_stream_t stream) {
  Ctx c;
  int rc = open_ctx(desc, ws, bytes, c);
  if (rc) return rc;
  if (!topk_ids && rows_max(c.d) > 0) return MOE_ERR_NULL;
  if ((rc = check_device())) return rc;
  return run_route(c, topk_ids, (cudaStream_t)stream);
}

int moe_quant_q8(const MoeLayerDesc* desc, const float* x, void* ws, size_t bytes,
                 moe_stream_t stream) {
  Ctx c;
  int rc = open_ctx(desc, ws, bytes, c);
  if (rc) return rc;
  if (!x && c.d.T > 0) return MOE_ERR_NULL;
  if (!aligned(x, 16)) return MOE_ERR_ALIGN;
  if ((rc = check_device())) return rc;
  return run_quant(c, x, (cudaStream_t)stream);
}

int moe_gate_up(const MoeLayerDesc* desc, const uint8_t* pack, const int64_t* eoff, void* ws,
                size_t bytes, moe_stream_t stream) {
  Ctx c;
  int rc = open_ctx(desc, ws, bytes, c);
  if (rc) return rc;
  if ((rc = check_weights(desc, pack, eoff))) return rc;
  if ((rc = check_device())) return rc;
  return run_gemm(c, 0, pack, eoff, (cudaStream_t)stream);
}

int moe_gate_up_swiglu(const MoeLayerDesc* desc, const uint8_t* pack, const int64_t* eoff,
                       void* ws, size_t bytes, moe_stream_t stream) {
  Ctx c;
  int rc = open_ctx(desc, ws, bytes, c);
  if (rc) return rc;
  if ((rc = check_weights(desc, pack, eoff))) return rc;
  if ((rc = check_device())) return rc;
  return run_gemm(c, 0, pack, eoff, (cudaStream_t)stream, true);
}

int moe_swiglu_quant(const MoeLayerDesc* desc, void* ws, size_t bytes, moe_stream_t stream) {
  Ctx c;
  int rc = open_ctx(desc, ws, bytes, c);
  if (rc) return rc;
  if ((rc = check_device())) return rc;
  return run_swiglu(c, (cudaStream_t)stream);
}

int moe_down(const MoeLayerDesc* desc, const uint8_t* pack, const int64_t* eoff, void* ws,
             size_t bytes, moe_stream_t stream) {
  Ctx c;
  int rc = open_ctx(desc, ws, bytes, c);
  if (rc) return rc;
  if ((rc = check_weights(desc, pack, eoff))) return rc;
  if ((rc = check_device())) return rc;
  return run_gemm(c, 1, pack, eoff, (cudaStream_t)stream);
}

int moe_down_combine(const MoeLayerDesc* desc, const uint8_t* pack, const int64_t* eoff,
                     const float* topk_w, float* out, void* ws, size_t bytes,
                     moe_stream_t stream) {
  Ctx c;
  int rc = open_ctx(desc, ws, bytes, c);
  if (rc) return rc;
  if ((rc = check_weights(desc, pack, eoff))) return rc;
  if ((!topk_w || !out) && c.d.T > 0) return MOE_ERR_NULL;
  if (!aligned(out, 16)) return MOE_ERR_ALIGN;
  if ((rc = check_device())) return rc;
  return run_down_combine(c, pack, eoff, topk_w, out, (cudaStream_t)stream);
}

int moe_combine(const MoeLayerDesc* desc, const float* topk_w, float* out, void* ws, size_t bytes,
                moe_stream_t stream) {
  Ctx c;
  int rc = open_ctx(desc, ws, bytes, c);
  if (rc) return rc;
  if ((!topk_w || !out) && c.d.T > 0) return MOE_ERR_NULL;
  if (!aligned(out, 16)) return MOE_ERR_ALIGN;
  if ((rc = check_device())) return rc;
  return run_combine(c, topk_w, out, (cudaStream_t)stream);
}

int moe_prefill_layer(const MoeLayerDesc* desc, const float* x, const int32_t* topk_ids,
                      const float* topk_w, const uint8_t* weight_pack,
                      const int64_t* expert_offsets, float* out, void* ws, size_t bytes,
                      moe_stream_t stream) {
  Ctx c;
  int rc = open_ctx(desc, ws, bytes, c);
  if (rc) return rc;
  if (c.d.T > 0 && (!x || !topk_ids || !topk_w || !out)) return MOE_ERR_NULL;
  if (!aligned(x, 16) || !aligned(out, 16) || !aligned(topk_ids, 4) || !aligned(topk_w, 4))
    return MOE_ERR_ALIGN;
  if ((rc = check_weights(desc, weight_pack, expert_offsets))) return rc;
  if ((rc = check_device())) return rc;
  cudaStream_t st = (cudaStream_t)stream;
  if ((rc = run_route(c, topk_ids, st))) return rc;
  if ((rc = run_quant(c, x, st))) return rc;
  return run_layer_tail(c, weight_pack, expert_offsets, topk_w, out, st);
}

size_t moe_host_io_bytes(const MoeLayerDesc* desc) {
  if (validate_desc(desc)) return 0;
  const size_t T = (size_t)desc->T;
  return align_up(sizeof(float) * T * desc->d) + align_up(sizeof(int32_t) * T * desc->k) +
         align_up(sizeof(float) * T * desc->k) + align_up(sizeof(float) * T * desc->d);
}

// The host-buffer layer overlaps its transfers with compute where the call's
// order allows (x is 168 MB in and out 168 MB back at 16,384 tokens; the
// link moves about 200 GB/s, about 0.85 ms each way):
//  - x is copied on a copy stream of its own, which waits only until the
//    previous call's q8 step has read the staging buffer: a call enqueued
//    while the previous one computes brings its x in behind those products
//    (when the previous call used another staging buffer, the copy waits
//    for everything enqueued on `stream` before this call instead);
//  - the routing ids and weights (small) are copied on the caller's stream;
//  - the combine runs in token chunks, and each chunk's rows of out go back
//    on a second copy stream as soon as they are written; the caller's
//    stream then waits for the last chunk, so out is complete once `stream`
//    is -- or, with MOE_FLAG_HOST_OUT_DEFERRED, it does not, and the copy
//    runs on under the next call's products (out is then complete after
//    moe_host_out_join).  The first combine chunk waits for the previous
//    call's last out copy, so the staging buffer is not overwritten while it
//    is still being read.
// Under stream capture, or without the copy streams, every copy runs on the
// caller's stream in order.
constexpr int kOutChunks = 8;

int moe_prefill_layer_host(const MoeLayerDesc* desc, const float* h_x, const int32_t* h_ids,
                           const float* h_w, const uint8_t* weight_pack,
                           const int64_t* expert_offsets, float* h_out, void* io,
                           size_t io_bytes, void* ws, size_t bytes, moe_stream_t stream) {
  Ctx c;
  int rc = open_ctx(desc, ws, bytes, c);
  if (rc) return rc;
  if (c.d.T > 0 && (!h_x || !h_ids || !h_w || !h_out)) return MOE_ERR_NULL;
  if (!io) return MOE_ERR_NULL;
  if (!aligned(io, kAlign)) return MOE_ERR_ALIGN;
  if (io_bytes < moe_host_io_bytes(desc)) return MOE_ERR_WORKSPACE;
  if ((rc = check_weights(desc, weight_pack, expert_offsets))) return rc;
  if ((rc = check_device())) return rc;
  const size_t T = (size_t)c.d.T;
  const size_t bx = sizeof(float) * T * c.d.d, bi = sizeof(int32_t) * T * c.d.k,
               bw = sizeof(float) * T * c.d.k;
  uint8_t* p = static_cast<uint8_t*>(io);
  float* d_x = (float*)p;
  int32_t* d_ids = (int32_t*)(p + align_up(bx));
  float* d_w = (float*)(p + align_up(bx) + align_up(bi));
  float* d_out = (float*)(p + align_up(bx) + align_up(bi) + align_up(bw));
  cudaStream_t st = (cudaStream_t)stream;
  if (T == 0) {
    if ((rc = run_route(c, d_ids, st))) return rc;
    return MOE_OK;
  }
  // under stream capture every copy runs on `stream` in order: the copy
  // streams' events from earlier calls lie outside the capture
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(st, &cs) != cudaSuccess) return MOE_ERR_LAUNCH;
  std::unique_lock<std::mutex> lock(g_side_mu);
  SideStream* sd = cs == cudaStreamCaptureStatusNone ? side_stream(st) : nullptr;
  const bool overlap = sd != nullptr;
  auto ok = [](cudaError_t e) { return e == cudaSuccess; };
  if (overlap) {
    cudaEvent_t guard = sd->x_free;
    if (sd->last_io != io) {
      guard = sd->entry;
      if (!ok(cudaEventRecord(guard, st))) return MOE_ERR_LAUNCH;
    }
    if (!ok(cudaStreamWaitEvent(sd->h2d, guard, 0)) ||
        !ok(cudaMemcpyAsync(d_x, h_x, bx, cudaMemcpyHostToDevice, sd->h2d)) ||
        !ok(cudaEventRecord(sd->x_in, sd->h2d)))
      return MOE_ERR_LAUNCH;
  } else if (!ok(cudaMemcpyAsync(d_x, h_x, bx, cudaMemcpyHostToDevice, st))) {
    return MOE_ERR_LAUNCH;
  }
  if (!ok(cudaMemcpyAsync(d_ids, h_ids, bi, cudaMemcpyHostToDevice, st)) ||
      !ok(cudaMemcpyAsync(d_w, h_w, bw, cudaMemcpyHostToDevice, st)))
    return MOE_ERR_LAUNCH;
  lock.unlock();
  if ((rc = run_route(c, d_ids, st))) return rc;
  if (overlap && !ok(cudaStreamWaitEvent(st, sd->x_in, 0))) return MOE_ERR_LAUNCH;
  if ((rc = run_quant(c, d_x, st))) return rc;
  if (overlap) {
    lock.lock();
    const bool rec = ok(cudaEventRecord(sd->x_free, st));
    sd->last_io = io;
    lock.unlock();
    if (!rec) return MOE_ERR_LAUNCH;
  }
  if (!overlap || (c.d.flags & MOE_FLAG_FUSED_COMBINE)) {
    if ((rc = run_layer_tail(c, weight_pack, expert_offsets, d_w, d_out, st))) return rc;
    if (!ok(cudaMemcpyAsync(h_out, d_out, bx, cudaMemcpyDeviceToHost, st))) return MOE_ERR_LAUNCH;
    return MOE_OK;
  }
  if ((rc = run_products(c, weight_pack, expert_offsets, st))) return rc;
  lock.lock();
  if (!ok(cudaStreamWaitEvent(st, sd->out_done, 0))) return MOE_ERR_LAUNCH;
  const size_t row_bytes = sizeof(float) * c.d.d;
  for (int ch = 0; ch < kOutChunks; ch++) {
    const int64_t t0 = (int64_t)(T * ch / kOutChunks), t1 = (int64_t)(T * (ch + 1) / kOutChunks);
    if (t1 == t0) continue;
    if (!ok(launch_combine(d_w, c.v.dst_of, c.v.dm, t0, t1 - t0, c.d.k, c.d.d, rows_max(c.d),
                           d_out, st)) ||
        !ok(cudaEventRecord(sd->comb, st)) || !ok(cudaStreamWaitEvent(sd->d2h, sd->comb, 0)) ||
        !ok(cudaMemcpyAsync(reinterpret_cast<uint8_t*>(h_out) + t0 * row_bytes,
                            reinterpret_cast<uint8_t*>(d_out) + t0 * row_bytes,
                            (t1 - t0) * row_bytes, cudaMemcpyDeviceToHost, sd->d2h)))
      return MOE_ERR_LAUNCH;
  }
  if (!ok(cudaEventRecord(sd->out_done, sd->d2h))) return MOE_ERR_LAUNCH;
  sd->out_pending = true;
  if (!(c.d.flags & MOE_FLAG_HOST_OUT_DEFERRED) && !ok(cudaStreamWaitEvent(st, sd->out_done, 0)))
    return MOE_ERR_LAUNCH;
  return MOE_OK;
}

int moe_host_out_join(moe_stream_t stream) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return MOE_ERR_DEVICE;
  // a stream being captured copies out in order itself (no copy streams), and
  // may not wait on an event recorded outside the capture
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing((cudaStream_t)stream, &cs) != cudaSuccess) return MOE_ERR_LAUNCH;
  if (cs != cudaStreamCaptureStatusNone) return MOE_OK;
  std::lock_guard<std::mutex> lock(g_side_mu);
  const SideStream& sd = g_side[dev];
  if (sd.ctx != current_context_id() || !sd.out_pending) return MOE_OK;
  return cudaStreamWaitEvent((cudaStream_t)stream, sd.out_done, 0) == cudaSuccess ? MOE_OK
                                                                                    : MOE_ERR_LAUNCH;
}

int moe_read_status(const MoeLayerDesc* desc, void* ws, size_t bytes, int32_t* status,
                    moe_stream_t stream) {
  Ctx c;
  int rc = open_ctx(desc, ws, bytes, c);
  if (rc) return rc;
  if (!status) return MOE_ERR_NULL;
  if ((rc = check_device())) return rc;
  cudaStream_t st = (cudaStream_t)stream;
  int32_t v = 0;
  if (cudaMemcpyAsync(&v, c.v.status, sizeof(v), cudaMemcpyDeviceToHost, st) != cudaSuccess ||
      cudaMemsetAsync(c.v.status, 0, sizeof(int32_t), st) != cudaSuccess ||
      cudaStreamSynchronize(st) != cudaSuccess)
    return MOE_ERR_LAUNCH;
  *status = v;
  return v ? MOE_ERR_DEVICE_STATUS : MOE_OK;
}

const char* moe_status_string(int code) {
  switch (code) {
    case MOE_OK: return "ok";
    case MOE_ERR_NULL: return "a required pointer is NULL";
    case MOE_ERR_SHAPE: return "unsupported shape";
    case MOE_ERR_FORMAT: return "unknown weight format, layout or flags";
    case MOE_ERR_ALIGN: return "misaligned pointer";
    case MOE_ERR_WORKSPACE: return "workspace too small";
    case MOE_ERR_DEVICE: return "no sm_103 device is current";
    case MOE_ERR_LAUNCH: return "a CUDA call failed while enqueueing";
    case MOE_ERR_DEVICE_STATUS: return "device-side status bits were set";
    case MOE_ERR_SCRATCH: return "too large for the fixed scratch of moe_route_noalloc";
    default: return "unknown status code";
  }
}

uint64_t moe_kernel_launches(void) { return g_launches.load(std::memory_order_relaxed); }

}  // extern "C"
