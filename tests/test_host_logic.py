"""Host-side logic with no GPU: the work-list capacity the workspace and the
routing scratch are sized for, the bench's algorithmic byte count, and the
code hash that keys the recorded DRAM traffic."""
import os
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import synth  # noqa: E402



def _constant(name: str) -> int:
    """A tiling constant as the library's shared header defines it."""
    import re
    src = open(os.path.join(ROOT, "quantized_moe_expert_quantize_gb300", "csrc", "common.cuh")).read()
    m = re.search(r"constexpr int %s = (\d+);" % name, src)
    assert m, name
    return int(m.group(1))


TILE_ROWS = _constant("kTileRows")
SMALL_TILE_ROWS = _constant("kSmallTileRows")
SMALL_SPLIT = _constant("kSmallSplit")


def count_tiles(counts):
    """The split rule of the routing step, restated: full 128-row tiles, then
    the remainder as one more tcgen05 tile, or as 32-row small-row tiles when
    it is at most SMALL_SPLIT rows."""
    big = small = 0
    for c in counts:
        full, rem = divmod(int(c), TILE_ROWS)
        big += full
        if 0 < rem <= SMALL_SPLIT:
            small += -(-rem // SMALL_TILE_ROWS)
        elif rem:
            big += 1
    return big, small


def capacity(rows, E):
    """The work list's capacity: floor(rows/128) + E*(1 + split/32) + 1 tiles
    (the bound behind the workspace size and the routing scratch bound of the
    header, 4*floor(T*k/128) + 9*E + 71 int32 with the histogram)."""
    return rows // TILE_ROWS + E * (1 + SMALL_SPLIT // SMALL_TILE_ROWS) + 1


@pytest.mark.parametrize("seed", range(6))
def test_tile_count_within_capacity(seed):
    rng = np.random.default_rng(seed)
    E = int(rng.integers(1, 1025))
    rows = int(rng.integers(0, 200_000))
    # adversarial mixes: every expert just past a tile boundary, or just
    # under the small-row cutoff, or random
    kind = seed % 3
    if kind == 0:
        counts = np.full(E, 129)
    elif kind == 1:
        counts = np.full(E, SMALL_SPLIT)
    else:
        counts = rng.multinomial(rows, rng.dirichlet(np.ones(E) * 0.3))
    big, small = count_tiles(counts)
    assert big + small <= capacity(int(counts.sum()), E)


def test_split_rule_examples():
    # rows: (tcgen05 tiles, small-row tiles)
    cases = {0: (0, 0), 1: (0, 1), 32: (0, 1), 33: (1, 0), 128: (1, 0), 160: (1, 1),
             161: (2, 0), 300: (3, 0), 256 + 31: (2, 1)}
    for rows, want in cases.items():
        assert count_tiles([rows]) == want, rows


def test_layer_bytes_counts_touched_experts():
    import bench
    s = synth.LayerShape(8, 256, 64, 6, 2, synth.W2, synth.Q8_0)
    ids = np.array([[0, 1]] * 4 + [[1, 3]] * 4, np.int32)
    L = synth.make_layer(s, seed=1, topk_ids=ids)
    b = bench.layer_bytes(L)
    g = synth.row_bytes(synth.W2, 256) * 128
    dn = synth.row_bytes(synth.Q8_0, 64) * 256
    assert b["weights"] == 3 * (g + dn)                 # experts 0, 1, 3
    R = 16
    assert b["dm"] == 2 * R * 256 * 4
    assert b["total"] == sum(v for k, v in b.items() if k != "total")


def test_sources_sha_ignores_comments(tmp_path, monkeypatch):
    import bench
    csrc = tmp_path / "quantized_moe_expert_quantize_gb300" / "csrc"
    csrc.mkdir(parents=True)
    for f in bench.TRAFFIC_SOURCES:
        (csrc / f).write_text("int a;  // one\n\nint b;\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    h0 = bench.sources_sha()
    (csrc / bench.TRAFFIC_SOURCES[0]).write_text("// header\nint a;   // other\nint b;\n\n")
    assert bench.sources_sha() == h0
    (csrc / bench.TRAFFIC_SOURCES[0]).write_text("int a;\nint c;\n")
    assert bench.sources_sha() != h0


def test_l2_note_follows_the_step_footprint():
    """The bench's L2 statement: a layer step that touches more than twice the
    L2 streams through it; a tiny one says it is timed L2-warm."""
    import bench
    big = bench.l2_note(bench.layer_bytes(synth.config_layer(4)))
    assert big.startswith("no flush: every step touches") and "GB" in big
    small = bench.l2_note(bench.layer_bytes(synth.config_layer(0)))
    assert "L2-warm" in small


def test_oracle_layer_does_not_depend_on_its_thread_count():
    """The oracle splits routed rows over threads; each row's arithmetic is
    fixed, so every output is the same bits for 1, 3 and 8 threads."""
    import oracle
    L = synth.make_layer(synth.LayerShape(40, 256, 64, 6, 3, synth.W4NL, synth.W2), seed=31,
                         routing="topk", bias=True, outliers=True)
    runs = [oracle.layer(L, threads=t) for t in (1, 3, 8)]
    for o in runs[1:]:
        for key, v in runs[0].items():
            if key != "threads":
                assert np.array_equal(np.asarray(v), np.asarray(o[key])), key
