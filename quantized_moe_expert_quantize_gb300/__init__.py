"""Quantized MoE prefill experts on GB300 (sm_103a).

A thin ctypes binding over ``libmoeprefill.so`` (C ABI in
``include/moe_prefill.h``).  Every function marshals torch tensors into the
C call of the same name; every step of the layer runs in the library's CUDA
kernels.  There is no CPU fallback: if the library is missing or the current
device is not an sm_103 part, calls raise.
"""
from __future__ import annotations

import ctypes
import os

import torch

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libmoeprefill.so")

MOE_FMT_W2 = 1
MOE_FMT_W4NL = 2
MOE_FMT_Q8_0 = 3
MOE_GU_SPLIT = 0
MOE_GU_INTERLEAVED = 1
MOE_FLAG_FUSED_COMBINE = 1
MOE_FLAG_HOST_OUT_DEFERRED = 2

MOE_OK = 0
MOE_ERR_NULL = -1
MOE_ERR_SHAPE = -2
MOE_ERR_FORMAT = -3
MOE_ERR_ALIGN = -4
MOE_ERR_WORKSPACE = -5
MOE_ERR_DEVICE = -6
MOE_ERR_LAUNCH = -7
MOE_ERR_DEVICE_STATUS = -8
MOE_ERR_SCRATCH = -9

MOE_STATUS_BAD_EXPERT_ID = 1
MOE_STATUS_BAD_OFFSET = 2
MOE_STATUS_PIPE_TIMEOUT = 4
MOE_STATUS_BAD_ROUTING = 8

# every symbol include/moe_prefill.h declares
EXPORTS = (
    "moe_prefill_workspace_bytes", "moe_workspace_view", "moe_prefill_layer",
    "moe_host_io_bytes", "moe_prefill_layer_host", "moe_host_out_join", "moe_route", "moe_quant_q8",
    "moe_gate_up", "moe_swiglu_quant", "moe_down", "moe_down_combine", "moe_combine",
    "moe_read_status",
    "moe_check_device", "moe_status_string", "moe_kernel_launches", "moe_route_noalloc",
    "moe_tiled_pack_bytes", "moe_tile_weights", "moe_gate_up_swiglu",
    "moe_selftest_wait_timeout",
)


class MoeError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {status_string(code)} ({code})")


class MoeLayerDesc(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int32), ("d", ctypes.c_int32), ("n_ff", ctypes.c_int32),
                ("E", ctypes.c_int32), ("k", ctypes.c_int32), ("gu_fmt", ctypes.c_int32),
                ("down_fmt", ctypes.c_int32), ("gu_layout", ctypes.c_int32),
                ("flags", ctypes.c_uint32), ("reserved", ctypes.c_int32),
                ("weight_pack_bytes", ctypes.c_int64)]


class MoeWorkspaceView(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in
                ("counts", "offsets", "order", "row_src", "dst_of", "xq", "dx", "gu",
                 "hq", "dh", "dm", "status")]


_lib = None


def lib(build_if_missing: bool = False) -> ctypes.CDLL:
    """The loaded library; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            if build_if_missing:
                from . import build as _b
                _b.build()
            else:
                raise RuntimeError(
                    f"{LIB_PATH} is missing: build it with "
                    "`python -m quantized_moe_expert_quantize_gb300.build`")
        L = ctypes.CDLL(LIB_PATH)
        vp, sz, i32 = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int
        dp = ctypes.POINTER(MoeLayerDesc)
        L.moe_prefill_workspace_bytes.argtypes = [dp]
        L.moe_prefill_workspace_bytes.restype = sz
        L.moe_workspace_view.argtypes = [dp, vp, sz, ctypes.POINTER(MoeWorkspaceView)]
        L.moe_workspace_view.restype = i32
        L.moe_prefill_layer.argtypes = [dp, vp, vp, vp, vp, vp, vp, vp, sz, vp]
        L.moe_prefill_layer.restype = i32
        L.moe_host_io_bytes.argtypes = [dp]
        L.moe_host_io_bytes.restype = sz
        L.moe_prefill_layer_host.argtypes = [dp, vp, vp, vp, vp, vp, vp, vp, sz, vp, sz, vp]
        L.moe_prefill_layer_host.restype = i32
        L.moe_host_out_join.argtypes = [vp]
        L.moe_host_out_join.restype = i32
        L.moe_route.argtypes = [dp, vp, vp, sz, vp]
        L.moe_route.restype = i32
        L.moe_quant_q8.argtypes = [dp, vp, vp, sz, vp]
        L.moe_quant_q8.restype = i32
        L.moe_gate_up.argtypes = [dp, vp, vp, vp, sz, vp]
        L.moe_gate_up.restype = i32
        L.moe_gate_up_swiglu.argtypes = [dp, vp, vp, vp, sz, vp]
        L.moe_gate_up_swiglu.restype = i32
        L.moe_swiglu_quant.argtypes = [dp, vp, sz, vp]
        L.moe_swiglu_quant.restype = i32
        L.moe_down.argtypes = [dp, vp, vp, vp, sz, vp]
        L.moe_down.restype = i32
        L.moe_down_combine.argtypes = [dp, vp, vp, vp, vp, vp, sz, vp]
        L.moe_down_combine.restype = i32
        L.moe_combine.argtypes = [dp, vp, vp, vp, sz, vp]
        L.moe_combine.restype = i32
        L.moe_route_noalloc.argtypes = [dp, vp, vp, vp, vp, vp, vp]
        L.moe_route_noalloc.restype = i32
        L.moe_read_status.argtypes = [dp, vp, sz, ctypes.POINTER(ctypes.c_int32), vp]
        L.moe_read_status.restype = i32
        L.moe_check_device.argtypes = []
        L.moe_check_device.restype = i32
        L.moe_status_string.argtypes = [i32]
        L.moe_status_string.restype = ctypes.c_char_p
        L.moe_tiled_pack_bytes.argtypes = [dp]
        L.moe_tiled_pack_bytes.restype = ctypes.c_int64
        L.moe_tile_weights.argtypes = [dp, vp, ctypes.c_int64, vp, vp, vp, vp, vp]
        L.moe_tile_weights.restype = i32
        L.moe_selftest_wait_timeout.argtypes = [vp, i32, vp]
        L.moe_selftest_wait_timeout.restype = i32
        L.moe_kernel_launches.argtypes = []
        L.moe_kernel_launches.restype = ctypes.c_uint64
        _lib = L
    return _lib


def status_string(code: int) -> str:
    return lib().moe_status_string(code).decode()


def _check(rc: int, where: str):
    if rc != MOE_OK:
        raise MoeError(rc, where)


def make_desc(T, d, n_ff, E, k, gu_fmt=MOE_FMT_W2, down_fmt=MOE_FMT_W2,
              weight_pack_bytes=0, gu_layout=MOE_GU_SPLIT, flags=0) -> MoeLayerDesc:
    return MoeLayerDesc(T, d, n_ff, E, k, gu_fmt, down_fmt, int(gu_layout), int(flags), 0,
                        int(weight_pack_bytes))


def _ptr(t: torch.Tensor | None, dtype=None, device=True):
    if t is None:
        return None
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"expected {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError("tensors must be contiguous")
    if device and not t.is_cuda:
        raise ValueError("expected a CUDA tensor")
    if not device and t.is_cuda:
        raise ValueError("expected a host tensor")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def workspace_bytes(desc: MoeLayerDesc) -> int:
    n = lib().moe_prefill_workspace_bytes(ctypes.byref(desc))
    if n == 0:
        raise MoeError(MOE_ERR_SHAPE, "moe_prefill_workspace_bytes")
    return int(n)


def alloc_workspace(desc: MoeLayerDesc, device=None) -> torch.Tensor:
    """Device workspace of the right size (torch's allocator aligns to 512 B)."""
    return torch.empty(workspace_bytes(desc), dtype=torch.uint8, device=device or "cuda")


def host_io_bytes(desc: MoeLayerDesc) -> int:
    return int(lib().moe_host_io_bytes(ctypes.byref(desc)))


def workspace_view(desc: MoeLayerDesc, ws: torch.Tensor) -> dict:
    """Torch views of the workspace regions (shapes as in the header)."""
    v = MoeWorkspaceView()
    _check(lib().moe_workspace_view(ctypes.byref(desc), _ptr(ws, torch.uint8), ws.numel(),
                                    ctypes.byref(v)), "moe_workspace_view")
    base = ws.data_ptr()
    T, d, n_ff, E, k = desc.T, desc.d, desc.n_ff, desc.E, desc.k
    R = T * k
    ssd, ssf = ((d // 32) + 3) // 4 * 4, ((n_ff // 32) + 3) // 4 * 4  # padded scale rows
    spec = dict(counts=((E,), torch.int32), offsets=((E + 1,), torch.int32),
                order=((E,), torch.int32), row_src=((R,), torch.int32),
                dst_of=((R,), torch.int32), xq=((R, d), torch.float16),
                dx=((R, ssd), torch.float32), gu=((R, 2 * n_ff), torch.float32),
                hq=((R, n_ff), torch.float16), dh=((R, ssf), torch.float32),
                dm=((R, d), torch.float32), status=((1,), torch.int32))
    out = {}
    for name, (shape, dt) in spec.items():
        off = getattr(v, name) - base
        n = 1
        for s in shape:
            n *= s
        nbytes = n * torch.tensor([], dtype=dt).element_size()
        out[name] = ws[off:off + nbytes].view(dt).view(*shape)
    return out


def tiled_pack_bytes(desc: MoeLayerDesc) -> int:
    n = lib().moe_tiled_pack_bytes(ctypes.byref(desc))
    if n <= 0:
        raise MoeError(MOE_ERR_SHAPE, "moe_tiled_pack_bytes")
    return int(n)


def moe_tile_weights(desc, weight_pack, expert_offsets, tiled_pack, tiled_offsets, status=None,
                     stream=None):
    """Row-major weight pack -> the device-tiled pack the layer reads."""
    _check(lib().moe_tile_weights(
        ctypes.byref(desc), _ptr(weight_pack, torch.uint8), weight_pack.numel(),
        _ptr(expert_offsets, torch.int64), _ptr(tiled_pack, torch.uint8),
        _ptr(tiled_offsets, torch.int64), _ptr(status, torch.int32), _stream(stream)),
        "moe_tile_weights")


def tile_weights(T, d, n_ff, E, k, gu_fmt, down_fmt, weight_pack, expert_offsets, stream=None,
                 gu_layout=MOE_GU_SPLIT):
    """Tile a device-resident row-major pack; returns (desc, tiled pack,
    tiled offsets), desc.weight_pack_bytes being the tiled pack's size."""
    desc = make_desc(T, d, n_ff, E, k, gu_fmt, down_fmt, 0, gu_layout)
    desc.weight_pack_bytes = tiled_pack_bytes(desc)
    dev = weight_pack.device
    tiled = torch.empty(desc.weight_pack_bytes, dtype=torch.uint8, device=dev)
    toffs = torch.empty((E, 2), dtype=torch.int64, device=dev)
    moe_tile_weights(desc, weight_pack, expert_offsets, tiled, toffs, None, stream)
    return desc, tiled, toffs


def moe_prefill_layer(desc, x, topk_ids, topk_w, weight_pack, expert_offsets, out, workspace,
                      stream=None):
    _check(lib().moe_prefill_layer(
        ctypes.byref(desc), _ptr(x, torch.float32), _ptr(topk_ids, torch.int32),
        _ptr(topk_w, torch.float32), _ptr(weight_pack, torch.uint8),
        _ptr(expert_offsets, torch.int64), _ptr(out, torch.float32),
        _ptr(workspace, torch.uint8), workspace.numel(), _stream(stream)), "moe_prefill_layer")


def moe_prefill_layer_host(desc, h_x, h_topk_ids, h_topk_w, weight_pack, expert_offsets, h_out,
                           io, workspace, stream=None):
    _check(lib().moe_prefill_layer_host(
        ctypes.byref(desc), _ptr(h_x, torch.float32, device=False),
        _ptr(h_topk_ids, torch.int32, device=False), _ptr(h_topk_w, torch.float32, device=False),
        _ptr(weight_pack, torch.uint8), _ptr(expert_offsets, torch.int64),
        _ptr(h_out, torch.float32, device=False), _ptr(io, torch.uint8), io.numel(),
        _ptr(workspace, torch.uint8), workspace.numel(), _stream(stream)),
        "moe_prefill_layer_host")


def moe_host_out_join(stream=None):
    _check(lib().moe_host_out_join(_stream(stream)), "moe_host_out_join")


def moe_route(desc, topk_ids, workspace, stream=None):
    _check(lib().moe_route(ctypes.byref(desc), _ptr(topk_ids, torch.int32),
                           _ptr(workspace, torch.uint8), workspace.numel(), _stream(stream)),
           "moe_route")


def moe_route_noalloc(desc, topk_ids, counts, offsets, row_src, dst_of, stream=None):
    """Routing into caller buffers with no workspace and no allocation (the
    library's fixed device scratch is used instead; see the C header)."""
    _check(lib().moe_route_noalloc(ctypes.byref(desc), _ptr(topk_ids, torch.int32),
                                   _ptr(counts, torch.int32), _ptr(offsets, torch.int32),
                                   _ptr(row_src, torch.int32), _ptr(dst_of, torch.int32),
                                   _stream(stream)), "moe_route_noalloc")


def moe_quant_q8(desc, x, workspace, stream=None):
    _check(lib().moe_quant_q8(ctypes.byref(desc), _ptr(x, torch.float32),
                              _ptr(workspace, torch.uint8), workspace.numel(), _stream(stream)),
           "moe_quant_q8")


def moe_gate_up(desc, weight_pack, expert_offsets, workspace, stream=None):
    _check(lib().moe_gate_up(ctypes.byref(desc), _ptr(weight_pack, torch.uint8),
                             _ptr(expert_offsets, torch.int64), _ptr(workspace, torch.uint8),
                             workspace.numel(), _stream(stream)), "moe_gate_up")


def moe_gate_up_swiglu(desc, weight_pack, expert_offsets, workspace, stream=None):
    _check(lib().moe_gate_up_swiglu(ctypes.byref(desc), _ptr(weight_pack, torch.uint8),
                                    _ptr(expert_offsets, torch.int64),
                                    _ptr(workspace, torch.uint8), workspace.numel(),
                                    _stream(stream)), "moe_gate_up_swiglu")


def moe_swiglu_quant(desc, workspace, stream=None):
    _check(lib().moe_swiglu_quant(ctypes.byref(desc), _ptr(workspace, torch.uint8),
                                  workspace.numel(), _stream(stream)), "moe_swiglu_quant")


def moe_down(desc, weight_pack, expert_offsets, workspace, stream=None):
    _check(lib().moe_down(ctypes.byref(desc), _ptr(weight_pack, torch.uint8),
                          _ptr(expert_offsets, torch.int64), _ptr(workspace, torch.uint8),
                          workspace.numel(), _stream(stream)), "moe_down")


def moe_down_combine(desc, weight_pack, expert_offsets, topk_w, out, workspace, stream=None):
    _check(lib().moe_down_combine(ctypes.byref(desc), _ptr(weight_pack, torch.uint8),
                                  _ptr(expert_offsets, torch.int64), _ptr(topk_w, torch.float32),
                                  _ptr(out, torch.float32), _ptr(workspace, torch.uint8),
                                  workspace.numel(), _stream(stream)), "moe_down_combine")


def moe_combine(desc, topk_w, out, workspace, stream=None):
    _check(lib().moe_combine(ctypes.byref(desc), _ptr(topk_w, torch.float32),
                             _ptr(out, torch.float32), _ptr(workspace, torch.uint8),
                             workspace.numel(), _stream(stream)), "moe_combine")


def moe_read_status(desc, workspace, stream=None) -> int:
    st = ctypes.c_int32(0)
    rc = lib().moe_read_status(ctypes.byref(desc), _ptr(workspace, torch.uint8),
                               workspace.numel(), ctypes.byref(st), _stream(stream))
    if rc not in (MOE_OK, MOE_ERR_DEVICE_STATUS):
        raise MoeError(rc, "moe_read_status")
    return int(st.value)


def moe_selftest_wait_timeout(status, sleep: int, stream=None):
    """Enqueue the bounded-wait self-test: a wait nothing completes must
    give up and or MOE_STATUS_PIPE_TIMEOUT into ``status`` (device int32)."""
    _check(lib().moe_selftest_wait_timeout(_ptr(status, torch.int32), int(sleep),
                                           _stream(stream)), "moe_selftest_wait_timeout")


def moe_check_device() -> int:
    return int(lib().moe_check_device())


def moe_kernel_launches() -> int:
    return int(lib().moe_kernel_launches())


class Layer:
    """Device-resident weights of one layer (tiled once, from the row-major
    pack) plus its workspace, for repeated calls at a fixed token count."""

    def __init__(self, T, d, n_ff, E, k, gu_fmt, down_fmt, weight_pack: torch.Tensor,
                 expert_offsets: torch.Tensor, device="cuda", gu_layout=MOE_GU_SPLIT):
        self.desc, self.weight_pack, self.expert_offsets = tile_weights(
            T, d, n_ff, E, k, gu_fmt, down_fmt, weight_pack, expert_offsets,
            gu_layout=gu_layout)
        self.workspace = alloc_workspace(self.desc, device)

    def __call__(self, x, topk_ids, topk_w, out=None, stream=None):
        if out is None:
            out = torch.empty_like(x)
        moe_prefill_layer(self.desc, x, topk_ids, topk_w, self.weight_pack,
                          self.expert_offsets, out, self.workspace, stream)
        return out

    def status(self, stream=None) -> int:
        return moe_read_status(self.desc, self.workspace, stream)
