"""The routing entry point for callers that cannot allocate device memory.

moe_route_noalloc keeps its scratch in a fixed array inside the library
instead of a caller workspace, for code that may only touch the buffers it
is given.  Its outputs must equal those of moe_route (which uses a
workspace) bit for bit -- routing is integer work -- on two calls in a row,
the second on a different routing, since every call reuses the same array.
This file is collected near the end (before only the wait self-test), so
that a run stopping at the first failure has already run the parity tests.
"""
import numpy as np
import pytest
import torch

import synth
from gpu_harness import require_gpu

pytestmark = pytest.mark.gpu


def _route_both(M, L):
    s = L.shape
    desc = M.make_desc(s.T, s.d, s.n_ff, s.E, s.k, s.gu_fmt, s.down_fmt, L.weight_pack.size)
    ids = torch.from_numpy(L.topk_ids).cuda()
    ws = M.alloc_workspace(desc)
    ws.fill_(0xFF)
    M.moe_route(desc, ids, ws)
    v = M.workspace_view(desc, ws)
    n = s.T * s.k
    counts = torch.full((s.E,), -7, dtype=torch.int32, device="cuda")
    offsets = torch.full((s.E + 1,), -7, dtype=torch.int32, device="cuda")
    row_src = torch.full((max(n, 1),), -7, dtype=torch.int32, device="cuda")
    dst_of = torch.full((max(n, 1),), -7, dtype=torch.int32, device="cuda")
    M.moe_route_noalloc(desc, ids, counts, offsets, row_src, dst_of)
    torch.cuda.synchronize()
    R = int(v["offsets"][-1])
    assert torch.equal(counts, v["counts"])
    assert torch.equal(offsets, v["offsets"])
    assert torch.equal(row_src[:R], v["row_src"][:R])
    assert torch.equal(dst_of[:n], v["dst_of"][:n])
    return counts.cpu().numpy()


def test_noalloc_route_matches_workspace_route_twice():
    M = require_gpu()
    first = synth.config_layer(1)                  # 2,048 tokens, 512 experts, top-10
    second = synth.make_layer(synth.LayerShape(300, 256, 64, 16, 4), seed=11,
                              routing="topk", bias=True)
    second.topk_ids[5, 2] = 16                     # one out-of-range id: dropped, -1
    c1 = _route_both(M, first)
    c2 = _route_both(M, second)
    assert c1.sum() == 2048 * 10
    assert c2.sum() == 300 * 4 - 1
