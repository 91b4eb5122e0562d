"""GPU parity: the CUDA path through the C ABI against the CPU oracle."""
from __future__ import annotations

import dataclasses

import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_harness import (DeviceLayer, TOL_DH_REL, TOL_DM, TOL_GU, TOL_HQ_FRAC, TOL_OUT, check_full,
                         check_q8_x, check_route, pair16, rel_rms, require_gpu)
from oracle_pins import np_decode_matrix

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def M():
    return require_gpu()


# ------------------------------------------------------------ small layers
SMALL = {
    "cfg0_tiny": lambda: synth.config_layer(0),
    # several tiles per expert with ragged tails, both down formats
    "mid_w2_w2": lambda: synth.make_layer(synth.LayerShape(300, 512, 192, 16, 4, synth.W2, synth.W2),
                                          seed=7, routing="topk", bias=True, outliers=True),
    "mid_w2_w4nl": lambda: synth.make_layer(synth.LayerShape(257, 384, 128, 12, 3, synth.W2, synth.W4NL),
                                            seed=8, routing="topk", bias=True, outliers=True),
    "mid_w4nl_w4nl": lambda: synth.make_layer(synth.LayerShape(130, 256, 64, 5, 2, synth.W4NL, synth.W4NL),
                                              seed=9, routing="topk", bias=False, outliers=True),
    "flat_w2_w4nl": lambda: synth.make_layer(synth.LayerShape(128, 256, 128, 16, 4, synth.W2, synth.W4NL),
                                             seed=10, routing="flat", outliers=True),
    # interleaved gate/up rows (gate j at row 2j, up j at 2j+1)
    "mid_w2_w2_inter": lambda: synth.make_layer(
        synth.LayerShape(300, 512, 192, 16, 4, synth.W2, synth.W2, synth.GU_INTERLEAVED),
        seed=7, routing="topk", bias=True, outliers=True),
    "mid_w4nl_w2_inter": lambda: synth.make_layer(
        synth.LayerShape(257, 384, 128, 12, 3, synth.W4NL, synth.W2, synth.GU_INTERLEAVED),
        seed=8, routing="topk", bias=True, outliers=True),
    # Q8_0 down (and gate/up) matrices
    "mid_w2_q8": lambda: synth.make_layer(
        synth.LayerShape(300, 512, 192, 16, 4, synth.W2, synth.Q8_0),
        seed=14, routing="topk", bias=True, outliers=True),
    "mid_q8_q8_inter": lambda: synth.make_layer(
        synth.LayerShape(257, 384, 128, 12, 3, synth.Q8_0, synth.Q8_0, synth.GU_INTERLEAVED),
        seed=15, routing="topk", bias=True, outliers=True),
    "flat_w4nl_q8": lambda: synth.make_layer(
        synth.LayerShape(128, 256, 128, 16, 4, synth.W4NL, synth.Q8_0),
        seed=16, routing="flat", outliers=True),
}


@pytest.mark.parametrize("name", list(SMALL))
@pytest.mark.parametrize("mode", ["layer", "stages"])
def test_small_layer_full_parity(M, name, mode):
    L = SMALL[name]()
    o = oracle.layer(L)
    dl = DeviceLayer(M, L)
    dl.run_layer() if mode == "layer" else dl.run_stages()
    assert dl.status() == 0
    check_full(dl, o)


def test_layer_replays_from_a_cuda_graph(M):
    """The layer enqueues only stream-ordered work (its small-row launches
    fork to a side stream and join back), so a CUDA graph captures it; the
    replay gives the eager call's bits, also for new inputs."""
    L = SMALL["mid_w2_w2"]()
    dl = DeviceLayer(M, L)
    dl.run_layer()  # eager first: sets the kernels up and makes the side stream
    ref = dl.out.clone()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        M.moe_prefill_layer(dl.desc, dl.x, dl.ids, dl.w, dl.pack, dl.eoff, dl.out, dl.ws)
    dl.out.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert dl.status() == 0
    assert torch.equal(dl.out, ref)
    # new activations through the same graph, against an eager call
    dl.x.mul_(-0.5)
    g.replay()
    torch.cuda.synchronize()
    got = dl.out.clone()
    dl.run_layer()
    assert torch.equal(got, dl.out)
    assert not torch.equal(got, ref)


def test_interleaved_gate_up_equals_split(M):
    """The same layer with its gate/up rows interleaved instead of split
    gives the same Hq, Dm and out bits on the GPU, and GU permuted."""
    Ls = SMALL["mid_w2_w2"]()
    Li = SMALL["mid_w2_w2_inter"]()
    a, b = DeviceLayer(M, Ls), DeviceLayer(M, Li)
    for mode in ("layer", "stages"):
        for dl in (a, b):
            dl.run_layer() if mode == "layer" else dl.run_stages()
            assert dl.status() == 0
        R = int(a.get("offsets")[-1])
        for key in ("hq", "dh", "dm"):
            assert np.array_equal(a.get(key, R), b.get(key, R)), (mode, key)
        assert torch.equal(a.out, b.out), mode
    n_ff = Ls.shape.n_ff
    perm = np.stack([np.arange(n_ff), n_ff + np.arange(n_ff)], axis=1).reshape(-1)
    assert np.array_equal(b.get("gu", R), a.get("gu", R)[:, perm])


@pytest.mark.parametrize("name", ["mid_w2_w2", "mid_w2_w4nl", "mid_w4nl_w4nl", "flat_w2_w4nl",
                                  "mid_w2_w2_inter", "mid_q8_q8_inter"])
def test_fused_swiglu_equals_stages(M, name):
    """The layer's gate/up epilogue with swiglu_quant fused writes the same Hq
    and dh bits as the gate/up stage followed by the swiglu_quant stage."""
    L = SMALL[name]()
    dl = DeviceLayer(M, L)
    dl.run_layer()
    R = int(dl.get("offsets")[-1])
    hq_f, dh_f = dl.get("hq", R), dl.get("dh", R)
    M.moe_gate_up(dl.desc, dl.pack, dl.eoff, dl.ws)
    M.moe_swiglu_quant(dl.desc, dl.ws)
    torch.cuda.synchronize()
    assert np.array_equal(dl.get("hq", R), hq_f)
    assert np.array_equal(dl.get("dh", R), dh_f)


@pytest.mark.parametrize("name", ["cfg0_tiny", "mid_w2_w2", "mid_w2_w4nl", "mid_w2_q8",
                                  "flat_w4nl_q8"])
def test_fused_combine_equals_unfused(M, name):
    """The combine fused into the down epilogue (MOE_FLAG_FUSED_COMBINE)
    gives the unfused layer's out bit for bit: the last of a token's rows
    to finish a 32-column group sums the k rows in rank order, one fma per
    rank, as the combine step does; the stage entry point moe_down_combine
    does the same after the earlier stages."""
    L = SMALL[name]()
    s = L.shape
    a = DeviceLayer(M, L)
    a.run_layer()
    assert a.status() == 0
    ref = a.out.clone()
    b = DeviceLayer(M, L)
    b.desc.flags = M.MOE_FLAG_FUSED_COMBINE
    b.run_layer()
    assert b.status() == 0
    assert torch.equal(b.out, ref)
    R = int(a.get("offsets")[-1])
    assert np.array_equal(b.get("dm", R), a.get("dm", R))
    # the stage entry point, on a fresh output, twice in a row (the arrival
    # counters are set again by every call)
    for _ in range(2):
        b.out.fill_(float("nan"))
        M.moe_down_combine(b.desc, b.pack, b.eoff, b.w, b.out, b.ws)
        torch.cuda.synchronize()
        assert torch.equal(b.out, ref)


def test_fused_combine_with_dropped_rows(M):
    """A token whose rank has an out-of-range expert id has one routed row
    fewer; its groups complete at k - 1 arrivals and out still matches the
    unfused layer bit for bit."""
    shape = synth.LayerShape(40, 256, 64, 8, 2)
    L = synth.make_layer(shape, seed=5, routing="topk")
    L.topk_ids[4, 1] = 8
    L.topk_ids[11, 0] = -3
    a = DeviceLayer(M, L)
    a.run_layer()
    b = DeviceLayer(M, L)
    b.desc.flags = M.MOE_FLAG_FUSED_COMBINE
    b.run_layer()
    assert b.status() & M.MOE_STATUS_BAD_EXPERT_ID
    assert torch.equal(b.out, a.out)


def test_config4_full_parity(M):
    """T=128 full layer (the weight-bandwidth-bound configuration), every
    output against the full oracle."""
    L = synth.config_layer(4)
    o = oracle.layer(L)
    dl = DeviceLayer(M, L)
    dl.run_layer()
    assert dl.status() == 0
    check_full(dl, o)


def test_down_alone_on_oracle_hq(M):
    """The down product alone, fed the oracle's Hq (the pages' parity test
    also ran the down alone on reference H)."""
    L = SMALL["mid_w2_w4nl"]()
    o = oracle.layer(L)
    dl = DeviceLayer(M, L)
    dl.run_layer()
    R = int(o["offsets"][-1])
    dl.v["hq"][:R].copy_(torch.from_numpy(pair16(o["hq"]).astype(np.float16)))
    dl.v["dh"][:R, : L.shape.n_ff // 32].copy_(torch.from_numpy(o["dh"]))
    M.moe_down(dl.desc, dl.pack, dl.eoff, dl.ws)
    torch.cuda.synchronize()
    assert rel_rms(dl.get("dm", R), o["dm"]) <= TOL_DM


# --------------------------------------------------------- full-size layers
def _dev(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def _rel_rms_dev(got: torch.Tensor, want: torch.Tensor) -> float:
    """rel RMS in float64 on the device (the full-size arrays are large)."""
    g, w = got.double(), want.double()
    den = torch.sqrt((w * w).mean())
    num = torch.sqrt(((g - w) ** 2).mean())
    if float(den) == 0.0:
        return 0.0 if float(num) == 0.0 else float("inf")
    return float(num / den)


def _report(name: str, values: dict) -> None:
    """Measured maxima of a parity test: printed, and written as JSON under
    $MOE_PARITY_REPORT_DIR when that is set."""
    import json
    import os
    print(name, values)
    d = os.environ.get("MOE_PARITY_REPORT_DIR")
    if d:
        os.makedirs(d, exist_ok=True)
        with open(os.path.join(d, f"{name}.json"), "w") as f:
            json.dump(values, f, indent=1)


@pytest.mark.parametrize("cfg", [1, 3, 2])
def test_full_size_config_full(M, cfg):
    """Configurations 1-3 at full size against the whole oracle layer: the
    routing and the q8 of x bit for bit, and for EVERY routed row its GU
    (gate/up stage), Hq (at most 1e-4 of the values differ, each by 1), dh
    (each scale within TOL_DH_REL) and Dm (against the oracle's down
    product of the same Hq: the rows holding one of the allowed Hq flips are
    recomputed from the GPU's Hq), and out for every token against the
    oracle's layer, at the layer spec's bounds."""
    L = synth.config_layer(cfg)
    s = L.shape
    o = oracle.layer(L)
    assert o["bad"] == 0
    dl = DeviceLayer(M, L)
    dl.run_layer()
    assert dl.status() == 0
    check_route(dl, o)
    check_q8_x(dl, o)
    R = int(o["offsets"][-1])
    assert R == s.T * s.k
    # Hq of every routed row (stored pair-interleaved on the device)
    perm = torch.from_numpy(np.array([2 * (j % 8) + j // 8 for j in range(16)])).cuda()
    hq_g = dl.v["hq"][:R].view(R, -1, 16)[:, :, perm].reshape(R, -1).to(torch.int32)
    hq_o = _dev(o["hq"]).to(torch.int32)
    dq = (hq_g - hq_o).abs()
    n_hq = int((dq != 0).sum())
    assert int(dq.max()) <= 1 and n_hq <= TOL_HQ_FRAC * dq.numel(), (n_hq, int(dq.max()))
    # dh of every block
    dh_g = dl.v["dh"][:R, : s.n_ff // 32].double()
    dh_o = _dev(o["dh"]).double()
    ddh = (dh_g - dh_o).abs()
    n_dh = int((ddh != 0).sum())
    dh_rel = float((ddh / dh_o.abs().clamp_min(1e-30)).max())
    assert bool((ddh <= TOL_DH_REL * dh_o.abs()).all()), dh_rel
    # Dm of every routed row against the oracle's down product on the same
    # Hq (rows with an allowed Hq flip recomputed from the GPU's Hq), and
    # out of every token against the oracle's layer
    flip_rows = torch.nonzero((dq != 0).any(dim=1)).flatten().cpu().numpy()
    hq_flip = hq_g[torch.from_numpy(flip_rows).cuda()].cpu().numpy() if len(flip_rows) else None
    dh_flip = dh_g[torch.from_numpy(flip_rows).cuda()].float().cpu().numpy() if len(flip_rows) else None
    dm_ref = _dev(o["dm"])
    for i, r in enumerate(flip_rows):
        e = int(L.topk_ids.reshape(-1)[o["row_src"][r]])
        dm_ref[int(r)] = _dev(oracle.expert_rows(s.down_fmt, s.n_ff, s.d,
                                                 L.weight_pack[L.expert_offsets[e, 1]:],
                                                 hq_flip[i][None].astype(np.int8),
                                                 dh_flip[i][None])[0])
    r_dm = _rel_rms_dev(dl.v["dm"][:R], dm_ref)
    assert r_dm <= TOL_DM, r_dm
    r_dm_layer = _rel_rms_dev(dl.v["dm"][:R], _dev(o["dm"]))
    r_out = _rel_rms_dev(dl.out, _dev(o["out"]))
    assert r_out <= TOL_OUT, r_out
    assert bool(torch.isfinite(dl.out).all())
    # GU of every routed row from the gate/up stage (the layer fuses it away)
    M.moe_gate_up(dl.desc, dl.pack, dl.eoff, dl.ws)
    torch.cuda.synchronize()
    gu_o = _dev(o["gu"])
    r_gu = _rel_rms_dev(dl.v["gu"][:R], gu_o)
    assert r_gu <= TOL_GU, r_gu
    gu_max = float(((dl.v["gu"][:R].double() - gu_o.double()).abs().max() /
                    gu_o.double().abs().max()))
    _report(f"parity_full_cfg{cfg}",
            dict(rows=R, tokens=s.T, gu_rel_rms=r_gu, gu_max_abs_over_max=gu_max,
                 hq_values_differing=n_hq, hq_fraction=n_hq / dq.numel(),
                 dh_blocks_differing=n_dh, dh_fraction=n_dh / ddh.numel(),
                 dh_max_rel=dh_rel,
                 hq_rows_with_flip=len(flip_rows), dm_rel_rms=r_dm,
                 dm_rel_rms_vs_oracle_layer=r_dm_layer, out_rel_rms=r_out))


# -------------------------------------------- the epilogues at real scales
EPI_COUNTS = [129, 31, 160, 5, 300, 1]  # tiles on both product kernels


def _fold_bound(fmt, wmat, nrows, K, q, dq):
    """Per-output bound on |GPU - oracle| for the W2 epilogue, whose scale is
    folded into the operand: the GPU computes acc = fma(d_x, d_w*isum, acc)
    with d_w*isum exact, the oracle acc = fma(fl(d_w*d_x), isum, acc).  Per
    block the two terms differ by at most u*|t_b| (u = 2^-24, t_b = d_w*d_x*
    isum_b exactly) and each side rounds once more by at most u*|acc_b|, with
    |acc_b| <= (1+u)^b * sum |t|; so over nb blocks |GPU - oracle| <=
    (2*nb + 1) * u * sum_b |t_b| (times 1.01 for the (1+u)^b factors).
    Returns that bound [rows of q, nrows], from a float64 evaluation of the
    block sums (exact: every block sum is an integer below 2^24)."""
    ints, scales = np_decode_matrix(fmt, wmat, nrows, K)
    nb = K // 32
    S = np.zeros((q.shape[0], nrows))
    qf = q.astype(np.float64)
    for b in range(nb):
        sl = slice(32 * b, 32 * b + 32)
        isum = qf[:, sl] @ ints[:, sl].T.astype(np.float64)   # [rows, nrows]
        S += np.abs(isum * (dq[:, b:b + 1].astype(np.float64) *
                            scales[None, :, 32 * b].astype(np.float64)))
    return (2 * nb + 1) * 2.0 ** -24 * 1.01 * S


def _check_product(fmt, got, want, wmats, K, nrows, groups, q, dq, what):
    """got/want [R, nrows]; bit-exact when the GPU keeps the oracle's
    epilogue order (W4NL, Q8_0), else within _fold_bound per element (W2)."""
    if fmt != synth.W2:
        assert np.array_equal(got, want), (what, float(np.max(np.abs(got - want))))
        return 0.0
    worst = 0.0
    for e, rows in groups:
        if len(rows) == 0:
            continue
        bound = _fold_bound(fmt, wmats[e], nrows, K, q[rows], dq[rows])
        diff = np.abs(got[rows].astype(np.float64) - want[rows].astype(np.float64))
        assert np.all(diff <= bound), (what, e, float(np.max(diff - bound)))
        worst = max(worst, float(np.max(diff / np.maximum(bound, 1e-300))))
    return worst


@pytest.mark.parametrize("fmts", [(synth.W2, synth.W2), (synth.W4NL, synth.Q8_0),
                                  (synth.Q8_0, synth.W4NL)])
def test_epilogues_at_real_scales(M, fmts):
    """The per-32-block K-ordered epilogue at the seeded (non-unit) scales,
    on both product kernels (row counts give full, partial and small-row
    tiles):
      - GU: bit for bit where the GPU keeps the oracle's order fma(fl(d_w*
        d_x), isum, acc) (W4NL, Q8_0 gate/up); for W2, whose weight scale is
        folded into the tensor-core operand, every output within the
        derived per-element bound of _fold_bound;
      - Dm of the oracle's own Hq: the same two rules for the down format;
      - out of the oracle's own Dm: bit for bit (one fma per rank, in rank
        order, on both sides)."""
    counts = EPI_COUNTS
    ids = np.random.default_rng(21).permutation(
        np.concatenate([np.full(c, e, np.int64) for e, c in enumerate(counts)]))
    shape = synth.LayerShape(len(ids), 512, 128, len(counts), 1, *fmts)
    L = _layer_with_ids(shape, ids, seed=22)
    s = L.shape
    o = oracle.layer(L)
    dl = DeviceLayer(M, L)
    dl.run_stages()
    assert dl.status() == 0
    check_route(dl, o)
    check_q8_x(dl, o)
    R = int(o["offsets"][-1])
    tok = o["row_src"] // s.k
    groups = [(e, np.arange(o["offsets"][e], o["offsets"][e + 1])) for e in range(s.E)]
    gu_w = [L.weight_pack[L.expert_offsets[e, 0]:] for e in range(s.E)]
    dn_w = [L.weight_pack[L.expert_offsets[e, 1]:] for e in range(s.E)]
    w_gu = _check_product(s.gu_fmt, dl.get("gu", R), o["gu"], gu_w, s.d, 2 * s.n_ff, groups,
                          o["xq"][tok], o["dx"][tok], "gu")
    # the down product alone on the oracle's Hq and scales
    dl.v["hq"][:R].copy_(torch.from_numpy(pair16(o["hq"]).astype(np.float16)))
    dl.v["dh"][:R, : s.n_ff // 32].copy_(torch.from_numpy(o["dh"]))
    M.moe_down(dl.desc, dl.pack, dl.eoff, dl.ws)
    torch.cuda.synchronize()
    w_dm = _check_product(s.down_fmt, dl.get("dm", R), o["dm"], dn_w, s.n_ff, s.d, groups,
                          o["hq"], o["dh"], "dm")
    # the combine alone on the oracle's Dm
    dl.v["dm"][:R].copy_(torch.from_numpy(o["dm"]))
    M.moe_combine(dl.desc, dl.w, dl.out, dl.ws)
    torch.cuda.synchronize()
    assert np.array_equal(dl.out.cpu().numpy(), o["out"])
    _report(f"epilogue_bound_{synth.FMT_NAMES[s.gu_fmt]}_{synth.FMT_NAMES[s.down_fmt]}",
            dict(gu_worst_fraction_of_bound=w_gu, dm_worst_fraction_of_bound=w_dm))


# ------------------------------------------------------------- edge cases
def _layer_with_ids(shape, ids, seed=3, x_override=None):
    L = synth.make_layer(shape, seed=seed, routing="topk",
                         topk_ids=np.asarray(ids, np.int32).reshape(shape.T, shape.k))
    if x_override is not None:
        L.x = np.ascontiguousarray(x_override, np.float32)
    return L


@pytest.mark.parametrize("T,E", [(1638, 512), (1639, 512), (40000, 512), (1000, 1024),
                                 (3000, 1024)])
def test_route_both_paths_bit_exact(M, T, E):
    """Routing runs in one CTA up to 2^14 flat entries and in three kernels
    beyond; both give the oracle's counts, bounds, stable permutation and
    largest-first order bit for bit (T*k = 16,380 / 16,390 / 400,000, and
    10,000 / 30,000 over the largest expert count, 1024)."""
    k = 10
    rng = np.random.default_rng(T)
    ids_np, _ = synth.draw_topk_routing(rng, T, E, k, True)
    ids_np[7, 3] = E + 5  # one bad id: dropped and flagged
    desc = M.make_desc(T, 256, 64, E, k)
    ws = M.alloc_workspace(desc)
    M.moe_route(desc, torch.from_numpy(ids_np).cuda(), ws)
    torch.cuda.synchronize()
    v = M.workspace_view(desc, ws)
    counts, offsets, row_src, dst_of, bad = oracle.route(ids_np, E)
    R = int(offsets[-1])
    assert bad == 1
    assert np.array_equal(v["counts"].cpu().numpy(), counts)
    assert np.array_equal(v["offsets"].cpu().numpy(), offsets)
    assert np.array_equal(v["row_src"][:R].cpu().numpy(), row_src)
    assert np.array_equal(v["dst_of"][: T * k].cpu().numpy(), dst_of)
    want = np.lexsort((np.arange(E), -counts))
    assert np.array_equal(v["order"].cpu().numpy(), want)
    assert M.moe_read_status(desc, ws) & M.MOE_STATUS_BAD_EXPERT_ID


def test_empty_layer(M):
    shape = synth.LayerShape(0, 256, 64, 8, 2)
    L = synth.make_layer(shape, seed=1)
    dl = DeviceLayer(M, L)
    dl.run_layer()
    assert dl.status() == 0
    assert np.array_equal(dl.get("counts"), np.zeros(8, np.int32))


def test_single_token_top1(M):
    shape = synth.LayerShape(1, 256, 64, 4, 1)
    L = synth.make_layer(shape, seed=2, routing="topk")
    o = oracle.layer(L)
    dl = DeviceLayer(M, L)
    dl.run_layer()
    check_full(dl, o)


def test_expert_row_counts_0_1_65(M):
    """Experts with 0, 1, 64, 65 and 129 rows (tile boundaries and tails)."""
    k, E = 1, 6
    ids = [1] * 1 + [2] * 64 + [3] * 65 + [5] * 129  # experts 0 and 4 empty
    rng = np.random.default_rng(0)
    ids = rng.permutation(np.array(ids))
    shape = synth.LayerShape(len(ids), 256, 128, E, k, synth.W2, synth.W4NL)
    L = _layer_with_ids(shape, ids)
    o = oracle.layer(L)
    dl = DeviceLayer(M, L)
    dl.run_layer()
    check_full(dl, o)
    assert dl.get("counts").tolist() == [0, 1, 64, 65, 0, 129]


SPLIT_COUNTS = [0, 1, 2, 3, 4, 5, 7, 8, 9, 16, 17, 24, 25, 31, 32, 33, 64, 128, 129, 132, 160,
                161, 300]


@pytest.mark.parametrize("fmts", [(synth.W2, synth.W2), (synth.W2, synth.W2, synth.GU_INTERLEAVED),
                                  (synth.W4NL, synth.Q8_0)])
def test_tile_split_row_counts(M, fmts):
    """Row counts around every tile rule: W2 tiles of 1 to 4 rows (the dp4a
    path, alone and as the remainder of a full tile: 129, 132), small-row
    tiles of 1 to 4 n8 fragments (5..32 rows), the 32/33-row cutoff, a full
    128-row tile alone, with a 32-row small remainder (160), with a 33-row
    tcgen05 remainder (161), and 2 full tiles + 44 (300); in the layer, in
    stages (GU in both gate/up layouts) and with the combine fused."""
    k, E = 1, len(SPLIT_COUNTS)
    ids = np.concatenate([np.full(c, e, np.int64) for e, c in enumerate(SPLIT_COUNTS)])
    ids = np.random.default_rng(1).permutation(ids)
    shape = synth.LayerShape(len(ids), 256, 128, E, k, *fmts)
    L = _layer_with_ids(shape, ids)
    o = oracle.layer(L)
    for mode in ("layer", "stages"):
        dl = DeviceLayer(M, L)
        dl.run_layer() if mode == "layer" else dl.run_stages()
        assert dl.status() == 0
        assert dl.get("counts").tolist() == SPLIT_COUNTS
        check_full(dl, o)
    # the combine fused into the down epilogue, on both product kernels
    ref = dl.out.clone()
    dl.desc.flags = M.MOE_FLAG_FUSED_COMBINE
    dl.run_layer()
    assert dl.status() == 0
    assert torch.equal(dl.out, ref)


def _two_expert_ids(T: int) -> np.ndarray:
    """k = 2 over 3 experts: every token routes to expert 0 and to expert 1
    (tokens < T - 3) or 2 (the last 3), ranks in a seeded order.  Counts
    [T, T - 3, 3]: for T = 132, a full 128-row tile plus a 4-row remainder,
    a full tile plus a 1-row remainder, and a 3-row small tile."""
    rng = np.random.default_rng(11)
    ids = np.zeros((T, 2), np.int64)
    ids[:, 1] = 1
    ids[T - 3:, 1] = 2
    swap = rng.random(T) < 0.5
    ids[swap] = ids[swap][:, ::-1]
    return ids.reshape(-1)


EXTREME = {
    # the largest d (gate/up K = 8192, 256 blocks in the epilogue; down
    # output 8192 rows = 32 weight tiles) with the smallest n_ff
    "d8192_nff64_w2_w2": (synth.LayerShape(132, 8192, 64, 3, 2, synth.W2, synth.W2), "two"),
    # the largest n_ff (down K = 4096, gate/up output 8192 rows) with the
    # smallest d (gate/up K = 128: two W2 or four W4NL blocks a row)
    "d128_nff4096_w4nl_q8": (synth.LayerShape(132, 128, 4096, 3, 2, synth.W4NL, synth.Q8_0), "two"),
    "d128_nff4096_w2_w2_inter": (synth.LayerShape(132, 128, 4096, 3, 2, synth.W2, synth.W2,
                                                  synth.GU_INTERLEAVED), "two"),
    # the largest E, most experts with 0-3 rows
    "E1024_w2_w4nl": (synth.LayerShape(300, 128, 64, 1024, 4, synth.W2, synth.W4NL), "topk"),
}


@pytest.mark.parametrize("name", list(EXTREME))
def test_extreme_shapes(M, name):
    """The ends of the supported shape range (d 128 and 8192, n_ff 64 and
    4096, E 1024), every stage against the oracle, as one layer call and as
    stages."""
    shape, routing = EXTREME[name]
    if routing == "two":
        L = _layer_with_ids(shape, _two_expert_ids(shape.T))
    else:
        L = synth.make_layer(shape, seed=12, routing="topk", bias=True, outliers=True)
    o = oracle.layer(L)
    for mode in ("layer", "stages"):
        dl = DeviceLayer(M, L)
        dl.run_layer() if mode == "layer" else dl.run_stages()
        assert dl.status() == 0
        check_full(dl, o)


def test_zero_and_huge_rows(M):
    """A zero token (every block d = 0, q = 0) and a token with one huge
    value (its block quantizes the rest to 0)."""
    shape = synth.LayerShape(40, 256, 64, 8, 2)
    L = synth.make_layer(shape, seed=4, routing="topk")
    L.x[3] = 0.0
    L.x[7, 10] = 3.0e6
    L.x[9, :32] = 0.0
    o = oracle.layer(L)
    dl = DeviceLayer(M, L)
    dl.run_layer()
    check_full(dl, o)
    xq, dx = dl.get("xq"), dl.get("dx")
    r3 = o["dst_of"][3 * 2:(3 + 1) * 2]   # routed rows of token 3
    r7 = o["dst_of"][7 * 2:(7 + 1) * 2]
    assert np.all(xq[r3] == 0) and np.all(dx[r3] == 0)
    assert np.all(xq[r7, 10] == 127) and all(np.count_nonzero(xq[r, :32]) == 1 for r in r7)


def test_bad_expert_id_is_dropped_and_flagged(M):
    shape = synth.LayerShape(20, 256, 64, 8, 2)
    L = synth.make_layer(shape, seed=5, routing="topk")
    L.topk_ids[4, 1] = 8      # out of range
    L.topk_ids[11, 0] = -3    # out of range
    o = oracle.layer(L)
    assert o["bad"] == 2
    dl = DeviceLayer(M, L)
    dl.run_layer()
    st = dl.status()
    assert st & M.MOE_STATUS_BAD_EXPERT_ID
    check_full(dl, o)


def test_bad_expert_offset_is_skipped_and_flagged(M):
    """A row-major offset that is misaligned or runs past the pack is flagged
    by the tiling step (that matrix becomes zeros); a tiled offset that is
    misaligned or runs past the tiled pack is flagged by the layer, and that
    expert is skipped."""
    shape = synth.LayerShape(16, 256, 64, 4, 1)
    L = synth.make_layer(shape, seed=6, routing="topk")
    L.expert_offsets = L.expert_offsets.copy()
    L.expert_offsets[0, 1] = L.weight_pack.size - 8   # runs past the pack
    dl = DeviceLayer(M, L)
    torch.cuda.synchronize()
    assert int(dl.tile_status.item()) & M.MOE_STATUS_BAD_OFFSET
    dl.run_layer()
    assert dl.status() == 0
    dl.eoff[1:, 0] += 2                                 # misaligned
    dl.eoff[2, 1] = dl.desc.weight_pack_bytes - 16      # runs past the tiled pack
    dl.run_layer()
    assert dl.status() & M.MOE_STATUS_BAD_OFFSET


def _tile_reference(pack, eoff, fmt_gu, fmt_dn, d, n_ff, E, gu_layout=synth.GU_SPLIT):
    """The tiled layout of the C header, written out with numpy."""
    out = []
    for e in range(E):
        for which, (fmt, N, K) in enumerate(((fmt_gu, 2 * n_ff, d), (fmt_dn, d, n_ff))):
            bpr = K // synth.BLOCK_VALUES[fmt]
            bb = synth.BLOCK_BYTES_OF[fmt]
            cb = 2 if fmt == synth.Q8_0 else 4         # blocks per chunk
            m = pack[eoff[e, which]:eoff[e, which] + N * bpr * bb].reshape(N, bpr, bb)
            if which == 0 and gu_layout == synth.GU_INTERLEAVED:
                gate, up = m[0::2], m[1::2]
            else:
                gate, up = m[:n_ff], m[n_ff:]
            for t in range(0, N, 256):
                nw = min(256, N - t)
                if which == 0:   # gate rows t/2 .., then the matching up rows
                    g0 = t // 2
                    rows = np.concatenate([gate[g0:g0 + nw // 2], up[g0:g0 + nw // 2]])
                else:
                    rows = m[t:t + nw]
                for c in range(0, bpr, cb):
                    blk = rows[:, c:c + cb]                    # [nw, nbc, bb]
                    out.append(blk[:, :, 2:].transpose(1, 0, 2).reshape(-1))
                    out.append(blk[:, :, :2].transpose(1, 0, 2).reshape(-1))
    return np.concatenate(out)


@pytest.mark.parametrize("shape", [synth.LayerShape(8, 384, 192, 3, 2, synth.W2, synth.W4NL),
                                   synth.LayerShape(8, 640, 320, 2, 1, synth.W4NL, synth.W2),
                                   synth.LayerShape(8, 384, 192, 3, 2, synth.W2, synth.W2,
                                                    synth.GU_INTERLEAVED),
                                   synth.LayerShape(8, 640, 320, 2, 1, synth.Q8_0, synth.Q8_0)])
def test_tiled_pack_layout(M, shape):
    """moe_tile_weights writes exactly the documented byte permutation, with
    ragged last tiles (N_out % 256 == 128) and ragged last chunks."""
    L = synth.make_layer(shape, seed=12, routing="topk")
    dl = DeviceLayer(M, L)
    torch.cuda.synchronize()
    assert int(dl.tile_status.item()) == 0
    ref = _tile_reference(L.weight_pack, L.expert_offsets, shape.gu_fmt, shape.down_fmt,
                          shape.d, shape.n_ff, shape.E, shape.gu_layout)
    got = dl.pack.cpu().numpy()
    assert got.size == ref.size
    assert np.array_equal(got, ref)
    gu = 2 * shape.n_ff * synth.row_bytes(shape.gu_fmt, shape.d)
    dn = shape.d * synth.row_bytes(shape.down_fmt, shape.n_ff)
    want = np.array([[e * (gu + dn), e * (gu + dn) + gu] for e in range(shape.E)])
    assert np.array_equal(dl.eoff.cpu().numpy(), want)


def test_host_buffers_entry_point(M):
    """moe_prefill_layer_host (host x/ids/w/out) equals the device entry."""
    L = SMALL["mid_w2_w2"]()
    dl = DeviceLayer(M, L)
    dl.run_layer()
    ref = dl.out.cpu().numpy()
    hx = torch.from_numpy(L.x).pin_memory()
    hi = torch.from_numpy(L.topk_ids).pin_memory()
    hw = torch.from_numpy(L.topk_w).pin_memory()
    ho = torch.empty((L.shape.T, L.shape.d), dtype=torch.float32).pin_memory()
    io = torch.empty(M.host_io_bytes(dl.desc), dtype=torch.uint8, device="cuda")
    M.moe_prefill_layer_host(dl.desc, hx, hi, hw, dl.pack, dl.eoff, ho, io, dl.ws)
    torch.cuda.synchronize()
    assert np.array_equal(ho.numpy(), ref)
    # two calls enqueued back to back on one staging buffer: the second
    # call's x (copied on the copy stream) must wait for the first call's q8
    # step
    ho2 = torch.empty_like(ho)
    hx2 = hx.clone()
    hx2.mul_(-1.0)
    M.moe_prefill_layer_host(dl.desc, hx2, hi, hw, dl.pack, dl.eoff, ho2, io, dl.ws)
    M.moe_prefill_layer_host(dl.desc, hx, hi, hw, dl.pack, dl.eoff, ho, io, dl.ws)
    torch.cuda.synchronize()
    assert np.array_equal(ho.numpy(), ref)
    dl.x.copy_(hx2.cuda())
    dl.run_layer()
    assert np.array_equal(ho2.numpy(), dl.out.cpu().numpy())


def test_host_buffers_deferred_out(M):
    """With MOE_FLAG_HOST_OUT_DEFERRED, three host-buffer calls enqueued back
    to back on one staging buffer (each call's out copy left running under
    the next call's products, the next combine waiting for it) give, after
    moe_host_out_join and a synchronise, each call's device-entry result."""
    L = SMALL["mid_w2_w2"]()
    dl = DeviceLayer(M, L)
    hi = torch.from_numpy(L.topk_ids).pin_memory()
    hw = torch.from_numpy(L.topk_w).pin_memory()
    xs = [torch.from_numpy(L.x).pin_memory()]
    xs.append(xs[0].clone().mul_(-1.0))
    xs.append(xs[0].clone().mul_(0.5))
    refs = []
    for hx in xs:
        dl.x.copy_(hx.cuda())
        dl.run_layer()
        refs.append(dl.out.cpu().numpy().copy())
    desc = type(dl.desc).from_buffer_copy(dl.desc)
    desc.flags = M.MOE_FLAG_HOST_OUT_DEFERRED
    io = torch.empty(M.host_io_bytes(desc), dtype=torch.uint8, device="cuda")
    outs = [torch.full((L.shape.T, L.shape.d), float("nan")).pin_memory() for _ in xs]
    for hx, ho in zip(xs, outs):
        M.moe_prefill_layer_host(desc, hx, hi, hw, dl.pack, dl.eoff, ho, io, dl.ws)
    M.moe_host_out_join()
    torch.cuda.synchronize()
    for ho, ref in zip(outs, refs):
        assert np.array_equal(ho.numpy(), ref)
    # nothing pending: the join enqueues a wait on a completed copy
    M.moe_host_out_join()
    torch.cuda.synchronize()


def test_host_buffers_captured_in_a_graph(M):
    """The host-buffer layer captured in a CUDA graph after an ordinary call
    (its copy streams exist by then), with MOE_FLAG_HOST_OUT_DEFERRED and the
    join: under capture every copy runs on the capturing stream in order,
    and each replay gives the device entry's out bit for bit."""
    L = SMALL["mid_w2_w2"]()
    dl = DeviceLayer(M, L)
    dl.run_layer()
    ref = dl.out.cpu().numpy()
    hx = torch.from_numpy(L.x).pin_memory()
    hi = torch.from_numpy(L.topk_ids).pin_memory()
    hw = torch.from_numpy(L.topk_w).pin_memory()
    ho = torch.empty((L.shape.T, L.shape.d), dtype=torch.float32).pin_memory()
    io = torch.empty(M.host_io_bytes(dl.desc), dtype=torch.uint8, device="cuda")
    desc = type(dl.desc).from_buffer_copy(dl.desc)
    desc.flags = M.MOE_FLAG_HOST_OUT_DEFERRED
    M.moe_prefill_layer_host(desc, hx, hi, hw, dl.pack, dl.eoff, ho, io, dl.ws)
    M.moe_host_out_join()
    torch.cuda.synchronize()
    assert np.array_equal(ho.numpy(), ref)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        M.moe_prefill_layer_host(desc, hx, hi, hw, dl.pack, dl.eoff, ho, io, dl.ws)
        M.moe_host_out_join()
    for _ in range(2):
        ho.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert np.array_equal(ho.numpy(), ref)


def test_host_buffers_fewer_tokens_than_chunks(M):
    """The host-buffer layer at T = 5 (some token chunks of its combine and
    out copy are empty) equals the device entry."""
    s = synth.LayerShape(5, 256, 64, 8, 2, synth.W2, synth.W2)
    L = synth.make_layer(s, seed=21)
    dl = DeviceLayer(M, L)
    dl.run_layer()
    ref = dl.out.cpu().numpy()
    hx = torch.from_numpy(L.x).pin_memory()
    hi = torch.from_numpy(L.topk_ids).pin_memory()
    hw = torch.from_numpy(L.topk_w).pin_memory()
    ho = torch.empty((s.T, s.d), dtype=torch.float32).pin_memory()
    io = torch.empty(M.host_io_bytes(dl.desc), dtype=torch.uint8, device="cuda")
    M.moe_prefill_layer_host(dl.desc, hx, hi, hw, dl.pack, dl.eoff, ho, io, dl.ws)
    torch.cuda.synchronize()
    assert np.array_equal(ho.numpy(), ref)


def test_repeat_is_deterministic(M):
    L = SMALL["mid_w2_w2"]()
    dl = DeviceLayer(M, L)
    dl.run_layer()
    a = dl.out.cpu().numpy().copy()
    dl.run_layer()
    assert np.array_equal(dl.out.cpu().numpy(), a)


def test_launch_counter_counts(M):
    L = SMALL["cfg0_tiny"]()
    dl = DeviceLayer(M, L)
    n0 = M.moe_kernel_launches()
    dl.run_layer()
    assert M.moe_kernel_launches() - n0 >= 6


def test_smoke_entry_point(M):
    """__graft_entry__.smoke(): the tiny layer through the C ABI against the
    oracle (tiled weights, routed-row q8, Hq and out tolerances)."""
    import __graft_entry__
    __graft_entry__.smoke()


def test_layer_class_equals_device_entry(M):
    """The binding's Layer (weights tiled when it is built, workspace kept)
    gives the device entry point's output bit for bit."""
    L = SMALL["mid_w4nl_w2_inter"]()
    s = L.shape
    dl = DeviceLayer(M, L)
    dl.run_layer()
    layer = M.Layer(s.T, s.d, s.n_ff, s.E, s.k, s.gu_fmt, s.down_fmt,
                    torch.from_numpy(L.weight_pack).cuda(),
                    torch.from_numpy(L.expert_offsets).cuda(), gu_layout=s.gu_layout)
    out = layer(dl.x, dl.ids, dl.w)
    torch.cuda.synchronize()
    assert torch.equal(out, dl.out)
    assert layer.status() == 0


def _unit_scales_and_extremes(L: synth.Layer, n_extreme: int, rng) -> None:
    """Every weight block scale set to fp16 1.0, the first ``n_extreme`` rows
    of every gate/up matrix set to the format's most negative code (W2 c = 0,
    value -2; W4NL index 0, value -127; Q8_0 -127), and x to integers in
    [-127, 127] whose every 32-value block holds a +-127 (so d_x = 1)."""
    s = L.shape
    for e in range(s.E):
        for m, (fmt, rows, K) in enumerate(((s.gu_fmt, 2 * s.n_ff, s.d),
                                            (s.down_fmt, s.d, s.n_ff))):
            bb = synth.BLOCK_BYTES_OF[fmt]
            nb = K // synth.BLOCK_VALUES[fmt]
            o = int(L.expert_offsets[e, m])
            mat = L.weight_pack[o:o + rows * nb * bb].reshape(rows, nb, bb)
            mat[:, :, 0] = 0x00
            mat[:, :, 1] = 0x3C
            if m == 0:
                mat[:n_extreme, :, 2:] = 0x81 if fmt == synth.Q8_0 else 0x00
    x = rng.integers(-127, 128, size=(s.T, s.d)).astype(np.float32)
    x[:, ::32] = np.where(rng.random((s.T, s.d // 32)) < 0.5, -127.0, 127.0)
    x[:10] = -127.0
    L.x = x


@pytest.mark.parametrize("fmts", [(synth.W2, synth.W2), (synth.W4NL, synth.Q8_0),
                                  (synth.Q8_0, synth.W4NL)])
def test_block_sums_exact_at_extremes(M, fmts):
    """The block sums are exact on both tensor-core paths: with every scale
    1.0 (d_w = d_x = 1) GU is the K-ordered fp32 sum of the integer block
    sums on both sides, so it must equal the oracle bit for bit, including
    blocks at the integer extremes (|isum| = 8,128 for W2 and 516,128 for
    W4NL and Q8_0).  Row counts put tiles on both product kernels."""
    counts = [129, 31, 160, 5]
    ids = np.random.default_rng(5).permutation(
        np.concatenate([np.full(c, e, np.int64) for e, c in enumerate(counts)]))
    shape = synth.LayerShape(len(ids), 512, 128, len(counts), 1, *fmts)
    L = _layer_with_ids(shape, ids)
    _unit_scales_and_extremes(L, 16, np.random.default_rng(6))
    o = oracle.layer(L)
    dl = DeviceLayer(M, L)
    dl.run_stages()
    assert dl.status() == 0
    check_route(dl, o)
    check_q8_x(dl, o)
    R = int(o["offsets"][-1])
    gu = dl.get("gu", R)
    assert np.array_equal(gu, o["gu"]), float(np.max(np.abs(gu - o["gu"])))
