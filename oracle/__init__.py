"""CPU oracle of the quantized MoE prefill layer -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` may import this package.  The
library under ``quantized_moe_expert_quantize_gb300`` never does.

The arithmetic lives in ``moe_oracle.c`` (plain C, fp32 with explicit
roundings); this module only marshals numpy arrays into it.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

from . import build as _build

W2 = 1
W4NL = 2

_LIB = None


def lib():
    global _LIB
    if _LIB is None:
        path = _build.build()
        L = ctypes.CDLL(path)
        i64, i32, vp = ctypes.c_int64, ctypes.c_int, ctypes.c_void_p
        L.orc_route.argtypes = [i64, i32, i32, vp, vp, vp, vp, vp]
        L.orc_route.restype = i64
        L.orc_quant_q8.argtypes = [i64, i32, vp, vp, vp]
        L.orc_quant_q8.restype = None
        L.orc_expert_rows.argtypes = [i32, i32, i32, vp, i64, vp, vp, vp]
        L.orc_expert_rows.restype = None
        L.orc_block_sums.argtypes = [i32, i32, vp, vp, vp]
        L.orc_block_sums.restype = None
        L.orc_swiglu_quant.argtypes = [i64, i32, i32, vp, vp, vp]
        L.orc_swiglu_quant.restype = None
        L.orc_combine.argtypes = [i64, i32, i32, vp, vp, vp, vp]
        L.orc_combine.restype = None
        L.orc_row_bytes.argtypes = [i32, i32]
        L.orc_row_bytes.restype = i64
        L.orc_w_value.argtypes = [i32, vp, i32]
        L.orc_w_value.restype = ctypes.c_double
        L.orc_layer.argtypes = [i64, i32, i32, i32, i32, i32, i32, i32] + [vp] * 16 + [i32]
        L.orc_layer.restype = i64
        _LIB = L
    return _LIB


def use_library(path: str | None):
    """Point the wrappers at another build of the oracle (the mutant tests
    load deliberately broken copies); ``None`` restores the normal build."""
    global _LIB
    _LIB = None
    if path is not None:
        real = _build.build
        try:
            _build.build = lambda force=False: path
            lib()
        finally:
            _build.build = real


def _p(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def route(topk_ids: np.ndarray, E: int):
    """Stable bucketing of the flat (token, rank) rows by expert.

    Returns counts[E], offsets[E+1], row_src[R], dst_of[T*k], bad-id count.
    """
    ids = _c(topk_ids, np.int32)
    T, k = ids.shape
    n = T * k
    counts = np.zeros(E, np.int32)
    offsets = np.zeros(E + 1, np.int32)
    row_src = np.zeros(max(n, 1), np.int32)
    dst_of = np.zeros(max(n, 1), np.int32)
    bad = lib().orc_route(T, k, E, _p(ids), _p(counts), _p(offsets), _p(row_src), _p(dst_of))
    R = int(offsets[E])
    return counts, offsets, row_src[:R].copy(), dst_of[:n].copy(), int(bad)


def quant_q8(x: np.ndarray):
    """q8 of each 32-value block of each row: (int8 q [rows, K], fp32 d [rows, K/32])."""
    x = _c(x, np.float32)
    rows, K = x.shape
    q = np.zeros((rows, K), np.int8)
    d = np.zeros((rows, K // 32), np.float32)
    lib().orc_quant_q8(rows, K, _p(x), _p(q), _p(d))
    return q, d


def row_bytes(fmt: int, K: int) -> int:
    return int(lib().orc_row_bytes(fmt, K))


def expert_rows(fmt: int, K: int, n_out: int, wmat: np.ndarray,
                q: np.ndarray, dq: np.ndarray) -> np.ndarray:
    """Activation rows (q, dq) against one expert's weight matrix bytes."""
    wmat = _c(wmat, np.uint8)
    q = _c(q, np.int8).reshape(-1, K)
    dq = _c(dq, np.float32).reshape(-1, K // 32)
    assert wmat.size >= n_out * row_bytes(fmt, K)
    out = np.zeros((q.shape[0], n_out), np.float32)
    lib().orc_expert_rows(fmt, K, n_out, _p(wmat), q.shape[0], _p(q), _p(dq), _p(out))
    return out


def block_sums(fmt: int, K: int, wrow: np.ndarray, q: np.ndarray) -> np.ndarray:
    wrow = _c(wrow, np.uint8)
    q = _c(q, np.int8)
    out = np.zeros(K // 32, np.int32)
    lib().orc_block_sums(fmt, K, _p(wrow), _p(q), _p(out))
    return out


def w_value(fmt: int, wrow: np.ndarray, j: int) -> float:
    wrow = _c(wrow, np.uint8)
    return float(lib().orc_w_value(fmt, _p(wrow), j))


def swiglu_quant(gu: np.ndarray, n_ff: int, layout: int = 0):
    """H = silu(gate)*up of GU rows, then q8.  layout 0: gate j at column j,
    up j at n_ff + j ("split"); 1: gate j at 2j, up j at 2j + 1."""
    gu = _c(gu, np.float32).reshape(-1, 2 * n_ff)
    rows = gu.shape[0]
    hq = np.zeros((rows, n_ff), np.int8)
    dh = np.zeros((rows, n_ff // 32), np.float32)
    lib().orc_swiglu_quant(rows, n_ff, int(layout), _p(gu), _p(hq), _p(dh))
    return hq, dh


def combine(topk_w: np.ndarray, dst_of: np.ndarray, dm: np.ndarray, d: int):
    w = _c(topk_w, np.float32)
    T, k = w.shape
    dst = _c(dst_of, np.int32).reshape(-1)
    dm = _c(dm, np.float32).reshape(-1, d)
    out = np.zeros((T, d), np.float32)
    lib().orc_combine(T, k, d, _p(w), _p(dst), _p(dm), _p(out))
    return out


def default_threads() -> int:
    return max(1, os.cpu_count() or 1)


def layer(L, threads: int | None = None) -> dict:
    """The whole layer on synthetic inputs ``L`` (a ``synth.Layer``).

    Returns every intermediate: counts, offsets, row_src, dst_of, xq, dx,
    gu, hq, dh, dm, out, bad.
    """
    s = L.shape
    T, d, n_ff, E, k = s.T, s.d, s.n_ff, s.E, s.k
    threads = threads or default_threads()
    x = _c(L.x, np.float32)
    ids = _c(L.topk_ids, np.int32)
    w = _c(L.topk_w, np.float32)
    pack = _c(L.weight_pack, np.uint8)
    eoff = _c(L.expert_offsets, np.int64)
    n = T * k
    # valid rows = entries with an in-range id
    R = int(np.count_nonzero((ids >= 0) & (ids < E)))
    o = dict(
        counts=np.zeros(E, np.int32), offsets=np.zeros(E + 1, np.int32),
        row_src=np.zeros(max(R, 1), np.int32), dst_of=np.zeros(max(n, 1), np.int32),
        xq=np.zeros((max(T, 1), d), np.int8), dx=np.zeros((max(T, 1), d // 32), np.float32),
        gu=np.zeros((max(R, 1), 2 * n_ff), np.float32),
        hq=np.zeros((max(R, 1), n_ff), np.int8), dh=np.zeros((max(R, 1), n_ff // 32), np.float32),
        dm=np.zeros((max(R, 1), d), np.float32), out=np.zeros((max(T, 1), d), np.float32))
    bad = lib().orc_layer(T, d, n_ff, E, k, s.gu_fmt, s.down_fmt, getattr(s, "gu_layout", 0),
                          _p(x), _p(ids), _p(w),
                          _p(pack), _p(eoff), _p(o["counts"]), _p(o["offsets"]),
                          _p(o["row_src"]), _p(o["dst_of"]), _p(o["xq"]), _p(o["dx"]),
                          _p(o["gu"]), _p(o["hq"]), _p(o["dh"]), _p(o["dm"]), _p(o["out"]),
                          threads)
    for key, rows in (("row_src", R), ("gu", R), ("hq", R), ("dh", R), ("dm", R),
                      ("dst_of", n), ("xq", T), ("dx", T), ("out", T)):
        o[key] = o[key][:rows]
    o["bad"] = int(bad)
    o["threads"] = threads
    return o
