"""Seeded synthetic inputs for one quantized MoE prefill layer.

This module is shared by the CUDA path's tests/bench and by the CPU oracle.
It holds no arithmetic of the method itself (no quantisation, no products,
no SwiGLU, no combine): it only draws random numbers and lays them out in the
byte format the library reads.

Workloads follow the pages' shapes: one layer of 512 experts, top-10 routing,
hidden size 2560 and expert width 640 (the "Strata #3752" page, commit
"moe_ws kernels": gate/up [1280 x 2560], down [2560 x 640]); routings are
skewed lognormal or flat (same page, "Addendum": lognormal and flat-32
routings of the down bench).  The pages used real GGUF experts and real
prompts; seeded synthetic layers with those shapes stand in for them.

Weight formats (byte layout is this library's own choice; the pages name
the formats but never lay out their bytes):

* W2   -- 64 values per block, 18 bytes: fp16 scale ``d`` (little endian) in
  bytes 0-1, then 16 bytes of 2-bit codes.  Code ``j`` (0..63) sits in byte
  ``2 + j // 4`` at bit ``2 * (j % 4)``.  Value = d * (code - 2).
* W4NL -- 32 values per block, 18 bytes: fp16 ``d`` in bytes 0-1, then 16
  bytes of 4-bit indices.  Index ``j`` (0..31) sits in byte ``2 + j // 2``,
  low nibble for even ``j``.  Value = d * NL4_TABLE[index].
* Q8_0 -- 32 values per block, 34 bytes: fp16 ``d`` in bytes 0-1, then the 32
  int8 codes ``q_j`` in bytes 2..33.  Value = d * q_j.  (The pages name the
  type without laying it out; this is the common layout of that name.)
  Drawn codes lie in [-127, 127].

A weight matrix [rows x K] is row-major: each row is its K/64 (W2) or K/32
(W4NL) blocks back to back.  An expert's gate/up matrix holds the gate rows
0..n_ff-1 then the up rows n_ff..2*n_ff-1 ("split" layout), or gate row j
at row 2j and up row j at row 2j+1 ("interleaved").  An interleaved layer
draws the same blocks as the split layer of the same seed, with the gate/up
rows permuted.  The weight pack
is every expert's gate/up matrix then its down matrix, each start 16-byte
aligned; ``expert_offsets[e] = (gate/up byte offset, down byte offset)``.
"""
from __future__ import annotations

import dataclasses
import numpy as np

W2 = 1
W4NL = 2
Q8_0 = 3
GU_SPLIT = 0
GU_INTERLEAVED = 1

# 4-bit non-linear table of the W4NL format (the layer spec's mixed-format
# configuration lists these 16 integers).
NL4_TABLE = np.array([-127, -104, -83, -65, -49, -35, -22, -10,
                      1, 13, 25, 38, 53, 69, 89, 113], dtype=np.int8)

BLOCK_BYTES = 18                       # W2 and W4NL
BLOCK_BYTES_OF = {W2: 18, W4NL: 18, Q8_0: 34}
BLOCK_VALUES = {W2: 64, W4NL: 32, Q8_0: 32}


@dataclasses.dataclass(frozen=True)
class LayerShape:
    T: int
    d: int
    n_ff: int
    E: int
    k: int
    gu_fmt: int = W2
    down_fmt: int = W2
    gu_layout: int = GU_SPLIT


def row_bytes(fmt: int, K: int) -> int:
    """Bytes of one weight row of K values in format ``fmt``."""
    return (K // BLOCK_VALUES[fmt]) * BLOCK_BYTES_OF[fmt]


def _align16(n: int) -> int:
    return (n + 15) // 16 * 16


# The five seeded layers.  Seeds are 1000 + index; draws happen in the order
# x, routing, weights.
CONFIGS = {
    0: dict(name="tiny_T64_d256_nff64_E8_top2_w2w2",
            shape=LayerShape(64, 256, 64, 8, 2, W2, W2),
            routing="topk", bias=False, outliers=False),
    1: dict(name="moe_T2048_d2560_nff640_E512_top10_w2w2_lognormal",
            shape=LayerShape(2048, 2560, 640, 512, 10, W2, W2),
            routing="topk", bias=True, outliers=True),
    2: dict(name="moe_T16384_d2560_nff640_E512_top10_w2w2_lognormal",
            shape=LayerShape(16384, 2560, 640, 512, 10, W2, W2),
            routing="topk", bias=True, outliers=True),
    3: dict(name="moe_T8192_d2560_nff640_E512_top10_w2gu_w4nldown_flat",
            shape=LayerShape(8192, 2560, 640, 512, 10, W2, W4NL),
            routing="flat", bias=False, outliers=True),
    4: dict(name="moe_T128_d2560_nff640_E512_top10_w2w2_lognormal",
            shape=LayerShape(128, 2560, 640, 512, 10, W2, W2),
            routing="topk", bias=True, outliers=True),
}


@dataclasses.dataclass
class Layer:
    shape: LayerShape
    x: np.ndarray            # fp32 [T, d]
    topk_ids: np.ndarray     # int32 [T, k]
    topk_w: np.ndarray       # fp32 [T, k]
    weight_pack: np.ndarray  # uint8 [bytes]
    expert_offsets: np.ndarray  # int64 [E, 2]
    name: str = ""


def draw_x(rng: np.random.Generator, T: int, d: int, outliers: bool) -> np.ndarray:
    """x ~ N(0,1) fp32; with outliers, round(0.001*T*d) distinct entries x20."""
    x = rng.standard_normal((T, d), dtype=np.float32)
    if outliers and T * d > 0:
        n_out = int(round(0.001 * T * d))
        pos = rng.choice(T * d, size=n_out, replace=False)
        flat = x.reshape(-1)
        flat[pos] = flat[pos] * np.float32(20.0)
    return x


def draw_topk_routing(rng: np.random.Generator, T: int, E: int, k: int, bias: bool):
    """Top-k of N(0,1) logits (+ a per-expert log(lognormal(0,1)) bias).

    Ties take the lower expert id first; weights are a softmax over the k
    selected logits in float64, rounded to fp32.
    """
    logits = rng.standard_normal((T, E))
    if bias:
        b = np.log(rng.lognormal(0.0, 1.0, E))
        logits = logits + b[None, :]
    order = np.argsort(-logits, axis=1, kind="stable")[:, :k]
    sel = np.take_along_axis(logits, order, axis=1)
    m = sel.max(axis=1, keepdims=True) if T > 0 else sel
    ex = np.exp(sel - m)
    w = ex / ex.sum(axis=1, keepdims=True)
    return order.astype(np.int32), w.astype(np.float32)


def draw_flat_routing(rng: np.random.Generator, T: int, E: int, k: int):
    """Balanced assignment: e(t, r) = pi[(tau[t]*k + r) mod E], weights 1/k.

    With T*k a multiple of E every expert gets exactly T*k/E rows, and the k
    experts of a token are distinct as long as k <= E.
    """
    pi = rng.permutation(E)
    tau = rng.permutation(T)
    r = np.arange(k)
    ids = pi[(tau[:, None] * k + r[None, :]) % E]
    w = np.full((T, k), np.float32(1.0) / np.float32(k), dtype=np.float32)
    return ids.astype(np.int32), w


def draw_blocks(rng: np.random.Generator, n_blocks: int, fmt: int = W2) -> np.ndarray:
    """n_blocks random blocks of format ``fmt``: fp16 d = 0.02*U(0.5,1.5),
    random codes.  Uniform code bytes give uniform 2-bit codes and uniform
    4-bit indices (W2 and W4NL share the 18-byte draw); Q8_0 codes are
    uniform in [-127, 127].
    """
    d = (0.02 * rng.uniform(0.5, 1.5, n_blocks)).astype(np.float16)
    blocks = np.empty((n_blocks, BLOCK_BYTES_OF[fmt]), dtype=np.uint8)
    blocks[:, 0:2] = d.view(np.uint8).reshape(n_blocks, 2)
    if fmt == Q8_0:
        q = rng.integers(-127, 128, size=(n_blocks, 32)).astype(np.int8)
        blocks[:, 2:] = q.view(np.uint8)
    else:
        blocks[:, 2:] = rng.integers(0, 256, size=(n_blocks, 16), dtype=np.uint8)
    return blocks


def pack_layout(shape: LayerShape):
    """Byte offsets of every expert's (gate/up, down) matrix and the total."""
    gu_bytes = 2 * shape.n_ff * row_bytes(shape.gu_fmt, shape.d)
    dn_bytes = shape.d * row_bytes(shape.down_fmt, shape.n_ff)
    offs = np.zeros((shape.E, 2), dtype=np.int64)
    pos = 0
    for e in range(shape.E):
        offs[e, 0] = pos
        pos = _align16(pos + gu_bytes)
        offs[e, 1] = pos
        pos = _align16(pos + dn_bytes)
    return offs, pos, gu_bytes, dn_bytes


def draw_weights(rng: np.random.Generator, shape: LayerShape):
    offs, total, gu_bytes, dn_bytes = pack_layout(shape)
    pack = np.zeros(total, dtype=np.uint8)
    n_gu = gu_bytes // BLOCK_BYTES_OF[shape.gu_fmt]
    n_dn = dn_bytes // BLOCK_BYTES_OF[shape.down_fmt]
    rb = row_bytes(shape.gu_fmt, shape.d)
    for e in range(shape.E):
        gu = draw_blocks(rng, n_gu, shape.gu_fmt).reshape(2 * shape.n_ff, rb)
        if shape.gu_layout == GU_INTERLEAVED:
            gu = np.stack([gu[:shape.n_ff], gu[shape.n_ff:]], axis=1).reshape(2 * shape.n_ff, rb)
        pack[offs[e, 0]:offs[e, 0] + gu_bytes] = gu.reshape(-1)
        pack[offs[e, 1]:offs[e, 1] + dn_bytes] = draw_blocks(rng, n_dn, shape.down_fmt).reshape(-1)
    return pack, offs


def make_layer(shape: LayerShape, seed: int, routing: str = "topk",
               bias: bool = False, outliers: bool = False,
               topk_ids: np.ndarray | None = None,
               topk_w: np.ndarray | None = None, name: str = "") -> Layer:
    """Draw one layer.  ``topk_ids``/``topk_w`` override the routing draw."""
    rng = np.random.default_rng(seed)
    x = draw_x(rng, shape.T, shape.d, outliers)
    if routing == "topk":
        ids, w = draw_topk_routing(rng, shape.T, shape.E, shape.k, bias)
    elif routing == "flat":
        ids, w = draw_flat_routing(rng, shape.T, shape.E, shape.k)
    else:
        raise ValueError(routing)
    if topk_ids is not None:
        ids = np.ascontiguousarray(topk_ids, dtype=np.int32)
    if topk_w is not None:
        w = np.ascontiguousarray(topk_w, dtype=np.float32)
    pack, offs = draw_weights(rng, shape)
    return Layer(shape, x, ids, w, pack, offs, name)


FMT_NAMES = {W2: "W2", W4NL: "W4NL", Q8_0: "Q8_0"}


def config_layer(index: int, down_fmt: int | None = None,
                 gu_layout: int | None = None) -> Layer:
    """Seeded layer of configuration ``index`` (seed 1000 + index), optionally
    with another down format or gate/up row layout (named in ``name``)."""
    c = CONFIGS[index]
    shape, name = c["shape"], c["name"]
    if down_fmt is not None and down_fmt != shape.down_fmt:
        shape = dataclasses.replace(shape, down_fmt=down_fmt)
        name += "_down" + FMT_NAMES[down_fmt].lower()
    if gu_layout is not None and gu_layout != shape.gu_layout:
        shape = dataclasses.replace(shape, gu_layout=gu_layout)
        name += "_gu_interleaved" if gu_layout == GU_INTERLEAVED else "_gu_split"
    return make_layer(shape, 1000 + index, c["routing"], c["bias"], c["outliers"], name=name)


def token_slice(layer: Layer, t0: int, t1: int) -> Layer:
    """Tokens t0..t1-1 of a layer, same weights (a bounded sample)."""
    shape = dataclasses.replace(layer.shape, T=t1 - t0)
    return Layer(shape, np.ascontiguousarray(layer.x[t0:t1]),
                 np.ascontiguousarray(layer.topk_ids[t0:t1]),
                 np.ascontiguousarray(layer.topk_w[t0:t1]),
                 layer.weight_pack, layer.expert_offsets, layer.name)
