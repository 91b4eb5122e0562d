#!/usr/bin/env python
"""Benchmark of the quantized MoE prefill layer on GB300.

One step = one whole layer (route -> q8 -> gate/up -> swiglu_quant -> down ->
combine) over one batch of synthetic input: by default the 16,384-token
layer (d = 2560, n_ff = 640, 512 experts, top-10, W2 gate/up and down,
skewed lognormal routing, seed 1002).  Prints ONE JSON line on rank 0.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--config C]
  python bench.py --impl reference ...   # the CPU oracle, timed on host cores

Multi-GPU runs (torchrun, one process per GPU) are independent replicas:
every rank runs the same layer with no data exchange ("scaling": "weak");
value = all ranks' tokens / the slowest rank's time.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = "MoE-layer prefill tokens/s and effective int8 TOPS at 16K tokens, top-10"
UNIT = "tokens/s"
# peaks: MEASURED_PEAKS.json when present, else these fallbacks
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
FALLBACK_BF16_TFLOPS_SUSTAINED = 1700.0
FP32_LANES_PER_SM = 128
# sm_103a's int8 tensor peak: mma.sync.m16n8k32.s8 as measured on a
# GB300 (tcgen05 kind::i8 does not exist there); MEASURED_PEAKS.json has no
# int8 figure
INT8_MMA_PEAK_TOPS = 150.0
# DRAM bytes (read + write) of one gate/up stage -- the tcgen05 launch plus
# the small-row launch -- at the 16,384-token layer, from a one-pass ncu
# capture (dram__bytes_read.sum + dram__bytes_write.sum); reported while the
# product kernels' code hashes as it did at that capture, else null
TRAFFIC_GATE_UP = {2: 1.5908e9}
TRAFFIC_SOURCES_SHA = "33afc4917d73b401"
TRAFFIC_SOURCES = ("gemm_tc.cu", "gemm_small.cu", "route.cu", "sm100_ptx.cuh", "common.cuh")
ALGO_BYTES_GATE_UP = {2: 1.586e9}
OTHER_CONFIGS = (1, 3, 4)


def sources_sha() -> str:
    """sha256 (first 16 hex digits) of the product kernels' code: the files of
    TRAFFIC_SOURCES with // comments, trailing blanks and empty lines taken
    out, so that only a change of code invalidates a capture."""
    import hashlib
    import re
    csrc = os.path.join(ROOT, "quantized_moe_expert_quantize_gb300", "csrc")
    h = hashlib.sha256()
    for f in TRAFFIC_SOURCES:
        with open(os.path.join(csrc, f)) as fh:
            lines = [re.sub(r"//.*$", "", ln).rstrip() for ln in fh.read().split("\n")]
        h.update(("\n".join(ln for ln in lines if ln.strip()) + "\n").encode())
    return h.hexdigest()[:16]


def measured_traffic(config: int):
    """(bytes, source) of the recorded capture, or (None, why not)."""
    sha = sources_sha()
    if sha != TRAFFIC_SOURCES_SHA:
        return None, (f"no capture of the current kernels (code hash {sha}; the last "
                      f"capture was of {TRAFFIC_SOURCES_SHA})")
    if config not in TRAFFIC_GATE_UP:
        return None, f"no capture of configuration {config}"
    return TRAFFIC_GATE_UP[config], (f"ncu dram__bytes_read.sum + dram__bytes_write.sum, one "
                                     f"pass, kernel code hash {TRAFFIC_SOURCES_SHA}")


def ops_per_row(s: synth.LayerShape) -> int:
    """Effective int8 ops of one routed row: 2 per multiply-add."""
    return 2 * (2 * s.n_ff * s.d + s.d * s.n_ff)


def layer_bytes(L) -> dict:
    """Algorithmic HBM bytes of one layer step: the weights of the experts the
    routing touches, x, the routing, out, and the staged intermediates (q8 of
    x and H with their scales, Dm), each written once and read once."""
    s = L.shape
    R = s.T * s.k
    touched = np.unique(L.topk_ids.reshape(-1))
    touched = touched[(touched >= 0) & (touched < s.E)]
    g = synth.row_bytes(s.gu_fmt, s.d) * 2 * s.n_ff
    dn = synth.row_bytes(s.down_fmt, s.n_ff) * s.d
    sd, sf = ((s.d // 32 + 3) & ~3), ((s.n_ff // 32 + 3) & ~3)
    parts = {
        "weights": len(touched) * (g + dn),
        "x": s.T * s.d * 4,
        "routing": s.T * s.k * 8,
        "out": s.T * s.d * 4,
        "xq+dx": 2 * R * (s.d * 2 + sd * 4),
        "hq+dh": 2 * R * (s.n_ff * 2 + sf * 4),
        "dm": 2 * R * s.d * 4,
    }
    parts["total"] = sum(parts.values())
    return parts


L2_BYTES = 129e6  # GB300 L2


def l2_note(parts: dict) -> str:
    """How the timed steps stand to the L2 (no flush between steps): the bytes
    one step touches, each buffer counted once."""
    once = parts["total"] - (parts["xq+dx"] + parts["hq+dh"] + parts["dm"]) / 2
    if once > 2 * L2_BYTES:
        return (f"no flush: every step touches {once / 1e9:.2f} GB (expert weights "
                f"{parts['weights'] / 1e9:.2f} GB) through a 129 MB L2")
    return (f"no flush: a step touches only {once / 1e6:.1f} MB, which the 129 MB L2 can "
            f"hold: L2-warm timing")


def config_layer(args) -> synth.Layer:
    """The seeded layer of --config, with --down-fmt / --gu-layout applied."""
    fmt = {"w2": synth.W2, "w4nl": synth.W4NL, "q8_0": synth.Q8_0}
    lay = {"split": synth.GU_SPLIT, "interleaved": synth.GU_INTERLEAVED}
    return synth.config_layer(args.config,
                              down_fmt=fmt[args.down_fmt] if args.down_fmt else None,
                              gu_layout=lay[args.gu_layout] if args.gu_layout else None)


def graph_leg(M, layer_call, out, ref_out, steps: int, world: int, T: int) -> dict:
    """Time `steps` replays of one CUDA-graph capture of `layer_call` (the
    single-call layer, enqueued on the capture stream); the output must keep
    the eager call's bits."""
    import torch
    try:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            layer_call()
        for _ in range(2):
            g.replay()
        torch.cuda.synchronize()
        cur = torch.cuda.current_stream()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(cur)
        for _ in range(steps):
            g.replay()
        e1.record(cur)
        torch.cuda.synchronize()
        if not torch.equal(out, ref_out):
            return {"error": "graph replay disagrees with the eager layer"}
        ms = reduce_max(e0.elapsed_time(e1), world)
        return {"ms_per_step": ms / steps, "value": world * T * steps / (ms / 1e3),
                "unit": UNIT, "steps": steps}
    except Exception as exc:  # reported, not fatal: the main line stands on its own
        return {"error": f"{type(exc).__name__}: {exc}"[:200]}


def layer_call_leg(M, dl, ref_out, steps: int, world: int, stream, T: int) -> dict:
    """`steps` calls of the single-call layer (moe_prefill_layer) back to back
    on one stream, CUDA events around them only.  It runs the same kernels as
    the stage sequence that `value` times, but forks the small-row launches
    once for both products (a small-row tile's down product needs only its
    own gate/up rows) where the stage entry points fork and join per stage,
    and it has no events between the steps."""
    import torch
    try:
        for _ in range(2):
            dl.layer(stream)
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(steps):
            dl.layer(stream)
        e1.record(stream)
        torch.cuda.synchronize()
        if not torch.equal(dl.out, ref_out):
            return {"error": "the single-call layer disagrees with the stage sequence"}
        ms = reduce_max(e0.elapsed_time(e1), world)
        return {"ms_per_step": ms / steps, "value": world * T * steps / (ms / 1e3),
                "unit": UNIT, "steps": steps}
    except Exception as exc:  # reported, not fatal
        return {"error": f"{type(exc).__name__}: {exc}"[:200]}


def fused_combine_leg(M, dl, ref_out, steps: int, world: int, stream) -> dict:
    """ms per layer step of the single-call layer, unfused and with the
    combine fused into the down epilogue, timed back to back."""
    import copy
    import torch
    try:
        fd = copy.copy(dl.desc)
        fd.flags = M.MOE_FLAG_FUSED_COMBINE
        out = torch.empty_like(dl.out)

        def run(desc, n):
            for _ in range(n):
                M.moe_prefill_layer(desc, dl.x, dl.ids, dl.w, dl.pack, dl.eoff, out, dl.ws, stream)

        res = {}
        for name, desc in (("unfused", dl.desc), ("fused", fd)):
            run(desc, 2)
            torch.cuda.synchronize()
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            run(desc, steps)
            e1.record(stream)
            torch.cuda.synchronize()
            res[name + "_ms_per_step"] = reduce_max(e0.elapsed_time(e1), world) / steps
            if not torch.equal(out, ref_out):
                return {"error": f"{name} layer disagrees with the stage sequence"}
        return res
    except Exception as exc:  # reported, not fatal
        return {"error": f"{type(exc).__name__}: {exc}"[:200]}


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            j = json.load(f)
        return dict(hbm=float(j.get("hbm_gbs", FALLBACK_HBM_GBS)),
                    bf16=float(j.get("bf16_tflops", FALLBACK_BF16_TFLOPS)),
                    bf16_sustained=float(j.get("bf16_tflops_sustained",
                                               j.get("bf16_tflops", FALLBACK_BF16_TFLOPS))),
                    source="measured")
    return dict(hbm=FALLBACK_HBM_GBS, bf16=FALLBACK_BF16_TFLOPS,
                bf16_sustained=FALLBACK_BF16_TFLOPS_SUSTAINED, source="fallback")


def tensor_peak(peaks: dict, clk: dict | None):
    """The bf16 denominator for a product stage timed inside the layer's
    steps: the burst figure when the clock record of the timed region shows
    the SM clock at its maximum with no power-cap or thermal reason (the
    burst figure's conditions), else the sustained one."""
    clk = clk or {}
    sm, smax, reasons = clk.get("sm_mhz"), clk.get("sm_max_mhz"), clk.get("reasons") or []
    burst = (sm is not None and smax and sm >= 0.97 * smax and
             not any(r in reasons for r in ("sw_power_cap", "hw_slowdown", "hw_thermal_slowdown",
                                             "sw_thermal_slowdown")))
    if burst:
        return peaks["bf16"], (f"{peaks['source']} bf16 dense, burst: the timed region ran at "
                               f"{sm:.0f} of {smax:.0f} MHz with no throttle reason")
    return peaks["bf16_sustained"], (f"{peaks['source']} bf16 dense, sustained: the clock record "
                                     f"of the timed region ({sm} of {smax} MHz, reasons "
                                     f"{reasons}) is not the burst figure's")


# ------------------------------------------------------------------ clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    REASONS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self):
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(prefix="clocks", suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.1)
        self.proc.terminate()
        self.proc.wait()
        sm, smax, reasons = [], [], set()
        with open(self.path) as f:
            for line in f:
                p = [x.strip() for x in line.split(",")]
                if len(p) < 9:
                    continue
                try:
                    sm.append(float(p[1]))
                    smax.append(float(p[2]))
                except ValueError:
                    continue
                for name, val in zip(self.REASONS, p[5:9]):
                    if val.lower().startswith("active"):
                        reasons.add(name)
        os.unlink(self.path)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# -------------------------------------------------------------- distributed
def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("gloo")  # host-side timing reductions only
    return world, rank, local


def reduce_max(value: float, world: int) -> float:
    """Largest value over ranks (gloo, host tensors); identity for 1 rank."""
    if world == 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ------------------------------------------------------------ CPU oracle
def time_oracle(L: synth.Layer, tokens: int, t0: int = 0):
    import oracle
    S = synth.token_slice(L, t0, t0 + tokens)
    threads = oracle.default_threads()
    t = time.perf_counter()
    oracle.layer(S, threads=threads)
    return time.perf_counter() - t, threads


def cpu_baseline(L: synth.Layer, tokens: int) -> dict:
    dt, threads = time_oracle(L, tokens)
    return {"value": tokens / dt, "unit": UNIT, "cores": threads, "kind": "oracle",
            "sample": f"first {tokens} tokens ({tokens * L.shape.k} routed rows) of the "
                      f"{L.shape.T}-token layer, one pass, {dt:.1f} s"}


def run_reference(args):
    world, rank, _ = dist_setup(args)
    if rank != 0:
        return 0
    L = config_layer(args)
    s = L.shape
    tok = args.ref_tokens
    for w in range(args.warmup):
        time_oracle(L, tok, (w * tok) % max(s.T - tok, 1))
    times = []
    threads = 1
    for i in range(args.steps):
        dt, threads = time_oracle(L, tok, ((args.warmup + i) * tok) % max(s.T - tok, 1))
        times.append(dt)
    total = sum(times)
    value = tok * args.steps / total
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * total / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32 (int32 block sums)", "data": "synthetic",
        "config": {"workload": L.name, "T": s.T, "d": s.d, "n_ff": s.n_ff, "E": s.E, "k": s.k,
                   "step": f"{tok} tokens of the layer per step (bounded sample)"},
        "effective_int8_tops": value * s.k * ops_per_row(s) / 1e12,
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle",
                         "sample": f"{tok} tokens ({tok * s.k} routed rows) per step"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------------ GPU arm
class DeviceLayer:
    """One seeded layer resident on the GPU: inputs, the tiled weight pack
    (tiled once at load time, outside every timed region), out, workspace."""

    def __init__(self, M, L: synth.Layer, dev: str):
        import torch
        s = L.shape
        self.L, self.M = L, M
        self.x = torch.from_numpy(L.x).to(dev)
        self.ids = torch.from_numpy(L.topk_ids).to(dev)
        self.w = torch.from_numpy(L.topk_w).to(dev)
        raw = torch.from_numpy(L.weight_pack).to(dev)
        roff = torch.from_numpy(L.expert_offsets).to(dev)
        self.desc, self.pack, self.eoff = M.tile_weights(s.T, s.d, s.n_ff, s.E, s.k, s.gu_fmt,
                                                         s.down_fmt, raw, roff,
                                                         gu_layout=s.gu_layout)
        torch.cuda.synchronize()
        del raw, roff
        self.out = torch.empty((s.T, s.d), dtype=torch.float32, device=dev)
        self.ws = M.alloc_workspace(self.desc, dev)

    def layer(self, stream=None):
        self.M.moe_prefill_layer(self.desc, self.x, self.ids, self.w, self.pack, self.eoff,
                                 self.out, self.ws, stream)

    def stage_calls(self, stream):
        """moe_prefill_layer's own launch sequence, one stage entry point each."""
        M, d = self.M, self.desc
        return [("route", lambda: M.moe_route(d, self.ids, self.ws, stream)),
                ("quant_q8", lambda: M.moe_quant_q8(d, self.x, self.ws, stream)),
                ("gate_up_swiglu",
                 lambda: M.moe_gate_up_swiglu(d, self.pack, self.eoff, self.ws, stream)),
                ("down", lambda: M.moe_down(d, self.pack, self.eoff, self.ws, stream)),
                ("combine", lambda: M.moe_combine(d, self.w, self.out, self.ws, stream))]


def time_stages(calls, steps: int, stream) -> dict:
    """`steps` layers as their stage sequence on one stream, with CUDA events
    between the stages: the whole span and each stage's duration, measured
    live inside the timed region."""
    import torch
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(len(calls) + 1)]
          for _ in range(steps)]
    for i in range(steps):
        ev[i][0].record(stream)
        for j, (_, c) in enumerate(calls):
            c()
            ev[i][j + 1].record(stream)
    torch.cuda.synchronize()
    per = {name: [ev[i][j].elapsed_time(ev[i][j + 1]) for i in range(steps)]
           for j, (name, _) in enumerate(calls)}
    return {"ms": ev[0][0].elapsed_time(ev[-1][-1]),
            "median": {k: statistics.median(v) for k, v in per.items()},
            "mean": {k: statistics.fmean(v) for k, v in per.items()}}


def product_rooflines(s: synth.LayerShape, mean_ms: dict, peak: float) -> dict:
    """Tensor-pipe fractions of the two product stages (2 flop per
    multiply-add of the gate/up and down products, all routed rows)."""
    R = s.T * s.k
    out = {}
    for stage, flops in (("gate_up_swiglu", 2.0 * R * (2 * s.n_ff) * s.d),
                         ("down", 2.0 * R * s.d * s.n_ff)):
        ms = mean_ms[stage]
        ach = flops / (ms * 1e-3) / 1e12 if ms > 0 else 0.0
        out[stage] = {"launch_ms": ms, "achieved_tflops": ach, "frac": ach / peak}
    return out


def other_config_line(M, cfg: int, steps: int, warmup: int, dev: str, stream,
                      peaks: dict, peak: float) -> dict:
    """Configuration `cfg` timed in this process: the layer as its stage
    sequence (as the main line), its binding roofline and the effective int8
    rate."""
    import torch
    L = synth.config_layer(cfg)
    s = L.shape
    dl = DeviceLayer(M, L, dev)
    calls = dl.stage_calls(stream)
    for _ in range(warmup):
        dl.layer(stream)
    torch.cuda.synchronize()
    if M.moe_read_status(dl.desc, dl.ws) != 0:
        return {"workload": L.name, "error": "device status bits set"}
    t = time_stages(calls, steps, stream)
    ms = t["ms"] / steps
    # the single-call layer, launched and replayed from one CUDA graph (no
    # launch gaps)
    dl.layer()
    torch.cuda.synchronize()
    ref_out = dl.out.clone()
    layer_call = layer_call_leg(M, dl, ref_out, steps, 1, stream, s.T)
    graph = graph_leg(M, lambda: dl.layer(), dl.out, ref_out, steps, 1, s.T)
    hbm = layer_bytes(L)
    hbm_gbs = hbm["total"] / (ms * 1e-3) / 1e9
    prod = product_rooflines(s, t["mean"], peak)
    line = {"workload": L.name, "T": s.T, "steps": steps, "ms_per_step": ms,
            "value": s.T / (ms * 1e-3), "unit": UNIT,
            "effective_int8_tops": s.T / (ms * 1e-3) * s.k * ops_per_row(s) / 1e12,
            "stage_ms": t["median"],
            "roofline_tensor": {"kernel": "gate_up_swiglu", "peak": peak,
                                "unit": "TFLOP/s", **prod["gate_up_swiglu"]},
            "roofline_tensor_down": {"kernel": "down", "peak": peak, "unit": "TFLOP/s",
                                     **prod["down"]},
            "roofline_hbm": {"kernel": "layer", "achieved": hbm_gbs, "peak": peaks["hbm"],
                             "unit": "GB/s", "frac": hbm_gbs / peaks["hbm"],
                             "algorithmic_bytes": hbm["total"],
                             "weights_bytes": hbm["weights"]},
            "l2": l2_note(hbm), "layer_call": layer_call, "graph": graph}
    line["binding"] = ("hbm" if line["roofline_hbm"]["frac"] >
                       line["roofline_tensor"]["frac"] else "tensor")
    del dl
    torch.cuda.empty_cache()
    return line


def run_ours(args):
    import torch
    world, rank, local = dist_setup(args)
    torch.cuda.set_device(local)
    import quantized_moe_expert_quantize_gb300 as M
    from quantized_moe_expert_quantize_gb300 import build as B
    if rank == 0 or not os.path.exists(M.LIB_PATH):
        B.build()
    barrier(world)
    if M.moe_check_device() != M.MOE_OK:
        raise SystemExit("current device is not an sm_103 GPU")

    L = config_layer(args)
    s = L.shape
    dev = f"cuda:{local}"
    stream = torch.cuda.current_stream()
    dl = DeviceLayer(M, L, dev)
    desc, x, ids, w, pack, eoff, out, ws = (dl.desc, dl.x, dl.ids, dl.w, dl.pack, dl.eoff,
                                            dl.out, dl.ws)
    sm_count = torch.cuda.get_device_properties(dev).multi_processor_count

    for _ in range(args.warmup):
        dl.layer(stream)
    torch.cuda.synchronize()
    if M.moe_read_status(desc, ws) != 0:
        raise SystemExit("device status bits set")

    # ---- timed region: exactly K layers.  Each layer is the library's own
    # launch sequence (moe_prefill_layer's steps, one stage entry point each,
    # same stream), with CUDA events between the steps, so every kernel's
    # duration is measured live inside the timed region.
    calls = dl.stage_calls(stream)
    clocks = ClockSampler()
    if rank == 0:
        clocks.start()
    barrier(world)
    torch.cuda.synchronize()
    n0 = M.moe_kernel_launches()
    t = time_stages(calls, args.steps, stream)
    launches = M.moe_kernel_launches() - n0
    barrier(world)
    clk = clocks.stop() if rank == 0 else None
    ms = reduce_max(t["ms"], world)
    ms_per_step = ms / args.steps
    value = world * s.T * args.steps / (ms / 1e3)
    stage_ms = t["median"]
    # the single-call entry point computes the same layer, bit for bit
    ref_out = out.clone()
    dl.layer(stream)
    torch.cuda.synchronize()
    if not torch.equal(out, ref_out):
        raise SystemExit("moe_prefill_layer disagrees with its own stage sequence")

    # ---- A/B of the combine fused into the down epilogue: the single-call
    # layer with and without MOE_FLAG_FUSED_COMBINE, back to back (the
    # fused layer must give the same bits)
    fused = fused_combine_leg(M, dl, ref_out, args.steps, world, stream)

    # ---- the single-call layer launched back to back (one fork for both
    # products, no events between steps)
    layer_call = layer_call_leg(M, dl, ref_out, args.steps, world, stream, s.T)

    # ---- the single-call layer captured once in a CUDA graph and replayed:
    # the same kernels without the host's launch gaps (reported beside
    # `value`, which times the launch sequence itself)
    graph = graph_leg(M, lambda: M.moe_prefill_layer(desc, x, ids, w, pack, eoff, out, ws),
                      out, ref_out, args.steps, world, s.T)

    # ---- end to end through the host-buffer entry point
    hx = torch.from_numpy(L.x).pin_memory()
    hi = torch.from_numpy(L.topk_ids).pin_memory()
    hw = torch.from_numpy(L.topk_w).pin_memory()
    ho = torch.empty((s.T, s.d), dtype=torch.float32).pin_memory()
    io = torch.empty(M.host_io_bytes(desc), dtype=torch.uint8, device=dev)

    # desc_deferred: each call's out copy back is left running under the next
    # call's products (MOE_FLAG_HOST_OUT_DEFERRED); the timed region ends
    # after moe_host_out_join, so it holds every step's copies either way
    desc_deferred = type(desc).from_buffer_copy(desc)
    desc_deferred.flags |= M.MOE_FLAG_HOST_OUT_DEFERRED

    def e2e_run(d):
        for _ in range(2):
            M.moe_prefill_layer_host(d, hx, hi, hw, pack, eoff, ho, io, ws, stream)
        M.moe_host_out_join(stream)
        torch.cuda.synchronize()
        barrier(world)
        f0 = torch.cuda.Event(enable_timing=True)
        f1 = torch.cuda.Event(enable_timing=True)
        f0.record(stream)
        for _ in range(e2e_steps):
            M.moe_prefill_layer_host(d, hx, hi, hw, pack, eoff, ho, io, ws, stream)
        M.moe_host_out_join(stream)
        f1.record(stream)
        torch.cuda.synchronize()
        return world * s.T * e2e_steps / (reduce_max(f0.elapsed_time(f1), world) / 1e3)

    e2e_steps = max(10, args.steps)
    e2e_sync_value = e2e_run(desc)
    if not np.allclose(ho.numpy(), out.cpu().numpy(), rtol=0, atol=0):
        raise SystemExit("host-buffer entry point disagrees with the device entry point")
    ho.fill_(float("nan"))
    e2e_value = e2e_run(desc_deferred)
    if not np.allclose(ho.numpy(), out.cpu().numpy(), rtol=0, atol=0):
        raise SystemExit("host-buffer entry point disagrees with the device entry point")
    h2d = int(L.x.nbytes + L.topk_ids.nbytes + L.topk_w.nbytes)
    del hx, hi, hw, ho, io

    if rank != 0:
        return 0

    peaks = load_peaks()
    peak, peak_source = tensor_peak(peaks, clk)
    prod = product_rooflines(s, t["mean"], peak)
    gu = prod["gate_up_swiglu"]
    R = s.T * s.k
    gu_flops = 2.0 * R * (2 * s.n_ff) * s.d
    pairs = R * (2 * s.n_ff) * (s.d // 32)
    sm_mhz = (clk or {}).get("sm_mhz") or (clk or {}).get("sm_max_mhz") or 2070.0
    alu_peak = sm_count * FP32_LANES_PER_SM * sm_mhz * 1e6 / 1e12  # T lane-ops/s
    alu_achieved = pairs / (gu["launch_ms"] * 1e-3) / 1e12
    eff_tops = value * s.k * ops_per_row(s) / 1e12
    # the recorded traffic and algorithmic bytes are for the configuration as listed
    variant = args.down_fmt is not None or args.gu_layout is not None
    traffic, traffic_source = ((None, "a format or layout variant of the configuration")
                               if variant else measured_traffic(args.config))
    hbm = layer_bytes(L)
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "int8 values in f16 MMA operands, f32 accumulate and epilogue",
        "data": "synthetic",
        "config": {"workload": L.name, "T": s.T, "d": s.d, "n_ff": s.n_ff, "E": s.E, "k": s.k,
                   "gu_fmt": synth.FMT_NAMES[s.gu_fmt], "down_fmt": synth.FMT_NAMES[s.down_fmt],
                   "gu_layout": "interleaved" if s.gu_layout == synth.GU_INTERLEAVED else "split",
                   "seed": 1000 + args.config, "parallelism": f"replicas x{world}",
                   "l2": l2_note(hbm)},
        "effective_int8_tops": eff_tops,
        "stage_ms": stage_ms,
        "roofline": {"bound": "tensor",
                     "kernel": "gate_up_swiglu (tcgen05 launch + small-row launch)",
                     "achieved": gu["achieved_tflops"], "peak": peak, "unit": "TFLOP/s",
                     "frac": gu["frac"], "traffic": traffic, "traffic_source": traffic_source,
                     "peak_source": peak_source + "; fp16 operands run at the bf16 rate",
                     "algorithmic": f"2*R*2*n_ff*d = {gu_flops:.4g} flop per stage; "
                                    f"{ALGO_BYTES_GATE_UP.get(args.config, float('nan')):.4g} "
                                    "algorithmic bytes per stage",
                     "launch_ms": gu["launch_ms"]},
        "roofline_down": {"bound": "tensor", "kernel": "down (tcgen05 + small-row launch)",
                          "achieved": prod["down"]["achieved_tflops"], "peak": peak,
                          "unit": "TFLOP/s", "frac": prod["down"]["frac"],
                          "launch_ms": prod["down"]["launch_ms"]},
        "roofline_alu": {"bound": "alu", "kernel": "gate_up_swiglu", "achieved": alu_achieved,
                         "peak": alu_peak, "unit": "T fp32 fma/s",
                         "frac": alu_achieved / alu_peak,
                         "algorithmic": "one fma per (output, 32-value block); "
                                        f"{sm_count} SMs x {FP32_LANES_PER_SM} fp32 lanes x "
                                        f"{sm_mhz:.0f} MHz"},
        "roofline_hbm": {"bound": "hbm", "kernel": "layer (all launches of a step)",
                         "achieved": hbm["total"] / (ms_per_step * 1e-3) / 1e9,
                         "peak": peaks["hbm"], "unit": "GB/s",
                         "frac": hbm["total"] / (ms_per_step * 1e-3) / 1e9 / peaks["hbm"],
                         "algorithmic_bytes": hbm,
                         "note": "binds at small T (the weight stream); at large T the "
                                 "products' tensor and epilogue rooflines bind"},
        "roofline_int8": {"bound": "tensor (int8)", "kernel": "layer",
                          "achieved": eff_tops, "peak": INT8_MMA_PEAK_TOPS, "unit": "TOPS",
                          "frac": eff_tops / INT8_MMA_PEAK_TOPS,
                          "note": "the layer's effective int8 rate against the sm_103a int8 "
                                  "tensor peak (mma.sync s8, measured); the products run as "
                                  "exact fp16 integers instead"},
        "layer_call": layer_call,
        "graph": graph,
        "fused_combine": fused,
        "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": int(s.T * s.d * 4), "steps": e2e_steps,
                "api": "moe_prefill_layer_host with MOE_FLAG_HOST_OUT_DEFERRED, "
                       "moe_host_out_join at the end of the timed region",
                "sync_out": {"value": e2e_sync_value, "unit": UNIT,
                             "note": "the same calls without the flag: each call's "
                                     "stream waits for its out copy"}},
        "gpu_launches": int(launches),
        "clocks": clk,
    }
    if world == 1 and not args.no_other_configs and not variant:
        # the other benched layers of the spec, timed in this process (their
        # own lines, not part of `value`); the main layer's buffers go first
        del dl, x, ids, w, pack, eoff, out, ws, ref_out
        torch.cuda.empty_cache()
        line["other_configs"] = {
            str(c): other_config_line(M, c, max(20, args.steps), args.warmup, dev, stream,
                                      peaks, peak)
            for c in OTHER_CONFIGS if c != args.config}
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(L, args.cpu_tokens)
    print(json.dumps(line), flush=True)
    return 0


def main():
    return main_args(sys.argv[1:])


def main_args(argv):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--config", type=int, default=2)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--cpu-tokens", type=int, default=2048)
    ap.add_argument("--ref-tokens", type=int, default=16)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-other-configs", action="store_true",
                    help="skip the other configurations' lines")
    ap.add_argument("--down-fmt", choices=["w2", "w4nl", "q8_0"], default=None,
                    help="the configuration with its down matrices in another format")
    ap.add_argument("--gu-layout", choices=["split", "interleaved"], default=None,
                    help="the configuration with its gate/up rows in another layout")
    args = ap.parse_args(argv)
    args.warmup = max(3, args.warmup)  # at least 3 untimed warm-up steps
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
