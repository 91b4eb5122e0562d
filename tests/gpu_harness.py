"""Helpers for the GPU parity tests: upload a synthetic layer, run the library
through its C ABI (Python binding), and compare with the CPU oracle.

Tolerances (the layer spec's parity bar):
  routing permutation, q8 of x          bit-exact
  GU, Dm                                rel RMS <= 1e-5 vs the oracle
  Hq                                    <= 1e-4 of values differ, each by +-1
  dh (the scales of Hq)                 each within 1e-4 relative
  out                                   rel RMS <= 1e-4
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import synth

TOL_GU = 1e-5
TOL_DM = 1e-5
TOL_HQ_FRAC = 1e-4
TOL_OUT = 1e-4
# A scale d = amax/127 of Hq follows the block's largest |H|, which carries
# GU's ulp-level differences (the folded W2 epilogue, host and device expf)
# through silu; a relative error e of d moves every h/d by at most 127e, so
# at 1e-4 a q can only flip where h/d is within 0.013 of a half-integer --
# the flips the Hq bound already counts.
TOL_DH_REL = 1e-4


def require_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import quantized_moe_expert_quantize_gb300 as M
    from quantized_moe_expert_quantize_gb300 import build as B
    B.build()
    assert M.moe_check_device() == M.MOE_OK, "current device is not an sm_103 part"
    return M


# The library stores q8 values pair-interleaved in each 16-value group:
# stored position 2i holds value i, 2i+1 holds value i+8.
_UNPAIR = np.array([2 * (o % 8) + o // 8 for o in range(16)])
_PAIR = np.array([(p >> 1) + 8 * (p & 1) for p in range(16)])


def unpair16(a: np.ndarray) -> np.ndarray:
    """Stored (pair-interleaved) order -> natural order along the last axis."""
    sh = a.shape
    return a.reshape(*sh[:-1], sh[-1] // 16, 16)[..., _UNPAIR].reshape(sh)


def pair16(a: np.ndarray) -> np.ndarray:
    """Natural order -> stored (pair-interleaved) order along the last axis."""
    sh = a.shape
    return a.reshape(*sh[:-1], sh[-1] // 16, 16)[..., _PAIR].reshape(sh)


def rel_rms(a, b) -> float:
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    den = np.sqrt((b ** 2).mean()) if b.size else 0.0
    if den == 0.0:
        return 0.0 if np.all(a == b) else float("inf")
    return float(np.sqrt(((a - b) ** 2).mean()) / den)


class DeviceLayer:
    """A synth.Layer resident on the GPU plus a workspace and views."""

    def __init__(self, M, L: synth.Layer):
        self.M = M
        self.L = L
        s = L.shape
        dev = "cuda"
        self.x = torch.from_numpy(L.x).to(dev)
        self.ids = torch.from_numpy(L.topk_ids).to(dev)
        self.w = torch.from_numpy(L.topk_w).to(dev)
        # row-major pack as drawn, then the tiled pack the layer reads
        self.raw_pack = torch.from_numpy(L.weight_pack).to(dev)
        self.raw_eoff = torch.from_numpy(L.expert_offsets).to(dev)
        self.desc = M.make_desc(s.T, s.d, s.n_ff, s.E, s.k, s.gu_fmt, s.down_fmt, 0, s.gu_layout)
        self.desc.weight_pack_bytes = M.tiled_pack_bytes(self.desc)
        self.pack = torch.full((self.desc.weight_pack_bytes,), 0xA5, dtype=torch.uint8, device=dev)
        self.eoff = torch.full((s.E, 2), -1, dtype=torch.int64, device=dev)
        self.tile_status = torch.zeros(1, dtype=torch.int32, device=dev)
        M.moe_tile_weights(self.desc, self.raw_pack, self.raw_eoff, self.pack, self.eoff,
                           self.tile_status)
        self.out = torch.full((max(s.T, 1), s.d), float("nan"), device=dev)[: s.T]
        self.ws = M.alloc_workspace(self.desc)
        self.ws.fill_(0xFF)  # poison: nothing may rely on zeroed workspace
        self.v = M.workspace_view(self.desc, self.ws)
        self.gu_copy = None  # gu as the stage sequence left it (dm overwrites it)

    def run_layer(self):
        """The whole layer (gate/up with swiglu_quant fused: gu is not written)."""
        self.M.moe_prefill_layer(self.desc, self.x, self.ids, self.w, self.pack, self.eoff,
                                 self.out, self.ws)
        torch.cuda.synchronize()
        self.has_gu = False
        self.gu_copy = None

    def run_stages(self):
        M = self.M
        M.moe_route(self.desc, self.ids, self.ws)
        M.moe_quant_q8(self.desc, self.x, self.ws)
        M.moe_gate_up(self.desc, self.pack, self.eoff, self.ws)
        M.moe_swiglu_quant(self.desc, self.ws)
        # gu shares its bytes with dm, which the down product overwrites
        self.gu_copy = self.v["gu"].clone()
        M.moe_down(self.desc, self.pack, self.eoff, self.ws)
        M.moe_combine(self.desc, self.w, self.out, self.ws)
        torch.cuda.synchronize()
        self.has_gu = True

    def status(self) -> int:
        return self.M.moe_read_status(self.desc, self.ws)

    def get(self, name, rows=None) -> np.ndarray:
        """A workspace region as numpy, in natural order: q8 values
        un-interleaved, scale rows without their padding."""
        t = self.gu_copy if name == "gu" and self.gu_copy is not None else self.v[name]
        if name == "dx":
            t = t[:, : self.L.shape.d // 32]
        if name == "dh":
            t = t[:, : self.L.shape.n_ff // 32]
        if rows is not None:
            t = t[:rows]
        a = t.contiguous().cpu().numpy()
        if name in ("xq", "hq"):
            a = unpair16(a)
        return a


def check_route(dl: DeviceLayer, o: dict):
    s = dl.L.shape
    R = int(o["offsets"][-1])
    assert np.array_equal(dl.get("counts"), o["counts"])
    assert np.array_equal(dl.get("offsets"), o["offsets"])
    assert np.array_equal(dl.get("row_src", R), o["row_src"])
    assert np.array_equal(dl.get("dst_of", s.T * s.k), o["dst_of"])
    order = dl.get("order")
    # largest first, ties by id: the unique order
    want = np.lexsort((np.arange(s.E), -o["counts"]))
    assert np.array_equal(order, want)


def check_q8_x(dl: DeviceLayer, o: dict):
    """q8 of x, scattered to routed rows: row r holds token row_src[r] // k.
    Compared bit for bit on the device (the full-size layers are large)."""
    k = dl.L.shape.k
    row_src = torch.from_numpy(np.ascontiguousarray(o["row_src"])).long().cuda()
    R = row_src.numel()
    tok = row_src // k
    want_q = torch.from_numpy(np.ascontiguousarray(o["xq"])).cuda()[tok].to(torch.float16)
    got_q = dl.v["xq"][:R]
    perm = torch.from_numpy(_UNPAIR).cuda()
    got_q = got_q.view(R, -1, 16)[:, :, perm].reshape(R, -1)
    assert torch.equal(got_q, want_q), "q8 values of x differ from the oracle"
    want_d = torch.from_numpy(np.ascontiguousarray(o["dx"])).cuda()[tok]
    got_d = dl.v["dx"][:R, : dl.L.shape.d // 32]
    assert torch.equal(got_d, want_d), "q8 scales of x differ from the oracle"


def hq_compare(hq_gpu: np.ndarray, hq_ref: np.ndarray):
    """Fraction of differing q8 values and the largest difference."""
    a = hq_gpu.astype(np.int32)
    b = hq_ref.astype(np.int32)
    diff = np.abs(a - b)
    n = int(np.count_nonzero(diff))
    return n / max(diff.size, 1), int(diff.max()) if diff.size else 0, n


def check_full(dl: DeviceLayer, o: dict, report: dict | None = None):
    """Every stage of a full run against a full oracle run."""
    check_route(dl, o)
    check_q8_x(dl, o)
    R = int(o["offsets"][-1])
    r_gu, gu = None, None
    if dl.has_gu:
        gu = dl.get("gu", R)
        r_gu = rel_rms(gu, o["gu"])
        assert r_gu <= TOL_GU, r_gu
    hq = dl.get("hq", R)
    frac, mx, n = hq_compare(hq, o["hq"])
    assert frac <= TOL_HQ_FRAC and mx <= 1, (frac, mx, n)
    dh = dl.get("dh", R)
    ddh = np.abs(dh.astype(np.float64) - o["dh"])
    assert np.all(ddh <= TOL_DH_REL * np.abs(o["dh"])), float(np.max(ddh))
    dm = dl.get("dm", R)
    r_dm = rel_rms(dm, dm_reference(dl.L, o, hq, dh))
    assert r_dm <= TOL_DM, r_dm
    r_out = rel_rms(dl.out.cpu().numpy(), o["out"])
    assert r_out <= TOL_OUT, r_out
    if report is not None:
        report.update(gu_rel_rms=r_gu,
                      gu_exact=None if gu is None else bool(np.array_equal(gu, o["gu"])),
                      hq_diff=n, dh_exact=bool(np.array_equal(dh, o["dh"])), dm_rel_rms=r_dm,
                      out_rel_rms=r_out)
    return dict(gu=r_gu, hq=n, dm=r_dm, out=r_out)


def dm_reference(L: synth.Layer, o: dict, hq_gpu: np.ndarray, dh_gpu: np.ndarray,
                 rows: np.ndarray | None = None) -> np.ndarray:
    """The oracle's Dm on the GPU's own Hq: the bound on Dm (rel RMS 1e-5)
    is the down product's, given its input, while the Hq values that may
    flip by 1 where H's rounding falls the other way are bounded on their
    own.  Rows whose Hq equals the oracle's take the oracle's Dm (their
    scales can differ only in the last bits); the few rows holding a flip
    are recomputed by the oracle from the GPU's Hq and scales.  ``rows``
    lists the rows with a flip when the caller already knows them."""
    s = L.shape
    R = int(o["offsets"][-1])
    if rows is None:
        rows = np.nonzero((hq_gpu[:R].astype(np.int32) != o["hq"].astype(np.int32)).any(axis=1))[0]
    ref = o["dm"].copy() if len(rows) else o["dm"]
    for r in rows:
        e = int(L.topk_ids.reshape(-1)[o["row_src"][r]])
        ref[r] = oracle.expert_rows(s.down_fmt, s.n_ff, s.d,
                                    L.weight_pack[L.expert_offsets[e, 1]:],
                                    hq_gpu[r][None].astype(np.int8), dh_gpu[r][None])[0]
    return ref

