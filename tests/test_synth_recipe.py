"""The seeded inputs follow their stated recipe (no GPU): the shapes and
routings of the five configurations, the outlier count, flat routing's exact
balance, top-k's distinct experts and softmax weights, the scale and code
ranges of the weight blocks, and the interleaved layout as a row
permutation of the split one."""
import numpy as np
import pytest

import synth


def test_configuration_table():
    want = {0: (64, 256, 64, 8, 2, synth.W2, synth.W2, "topk", False, False),
            1: (2048, 2560, 640, 512, 10, synth.W2, synth.W2, "topk", True, True),
            2: (16384, 2560, 640, 512, 10, synth.W2, synth.W2, "topk", True, True),
            3: (8192, 2560, 640, 512, 10, synth.W2, synth.W4NL, "flat", False, True),
            4: (128, 2560, 640, 512, 10, synth.W2, synth.W2, "topk", True, True)}
    for i, w in want.items():
        c = synth.CONFIGS[i]
        s = c["shape"]
        assert (s.T, s.d, s.n_ff, s.E, s.k, s.gu_fmt, s.down_fmt) == w[:7], i
        assert (c["routing"], c["bias"], c["outliers"]) == w[7:], i
        assert s.gu_layout == synth.GU_SPLIT


@pytest.mark.parametrize("T,d", [(64, 256), (300, 512), (7, 2560)])
def test_outliers_are_round_0p001_Td_entries_times_20(T, d):
    base = synth.draw_x(np.random.default_rng(9), T, d, outliers=False)
    x = synth.draw_x(np.random.default_rng(9), T, d, outliers=True)
    changed = x != base
    assert int(changed.sum()) == int(round(0.001 * T * d))
    assert np.array_equal(x[changed], base[changed] * np.float32(20.0))
    assert x.dtype == np.float32


def test_flat_routing_is_exactly_balanced():
    T, E, k = 8192, 512, 10
    ids, w = synth.draw_flat_routing(np.random.default_rng(3), T, E, k)
    assert np.array_equal(np.bincount(ids.reshape(-1), minlength=E), np.full(E, T * k // E))
    assert all(len(set(row)) == k for row in ids)
    assert np.all(w == np.float32(1.0) / np.float32(k))


@pytest.mark.parametrize("bias", [False, True])
def test_topk_routing(bias):
    T, E, k = 500, 64, 6
    ids, w = synth.draw_topk_routing(np.random.default_rng(4), T, E, k, bias)
    assert ids.dtype == np.int32 and w.dtype == np.float32
    assert all(len(set(row)) == k for row in ids)
    assert np.all((ids >= 0) & (ids < E))
    assert np.allclose(w.astype(np.float64).sum(axis=1), 1.0, atol=1e-6)
    # ranks in descending weight order (the softmax keeps the logit order)
    assert np.all(np.diff(w, axis=1) <= 0)


def test_skewed_routing_is_skewed():
    """The per-expert bias makes the row counts uneven: the largest expert
    of configuration 2's routing has several times the mean."""
    s = synth.CONFIGS[2]["shape"]
    ids, _ = synth.draw_topk_routing(np.random.default_rng(0), 4096, s.E, s.k, True)
    c = np.bincount(ids.reshape(-1), minlength=s.E)
    assert c.max() > 3 * c.mean()


@pytest.mark.parametrize("fmt", [synth.W2, synth.W4NL, synth.Q8_0])
def test_weight_blocks(fmt):
    n = 4000
    b = synth.draw_blocks(np.random.default_rng(5), n, fmt)
    assert b.shape == (n, synth.BLOCK_BYTES_OF[fmt])
    d = b[:, 0:2].copy().view(np.float16)[:, 0].astype(np.float64)
    assert np.all((d >= 0.0099) & (d <= 0.0301))
    if fmt == synth.Q8_0:
        q = b[:, 2:].view(np.int8)
        assert q.min() == -127 and q.max() == 127      # never -128
    else:
        assert b[:, 2:].min() == 0 and b[:, 2:].max() == 255


def test_interleaved_layer_permutes_the_split_rows():
    s = synth.LayerShape(4, 256, 64, 3, 2, synth.W2, synth.W2)
    a = synth.make_layer(s, seed=21)
    b = synth.make_layer(synth.LayerShape(4, 256, 64, 3, 2, synth.W2, synth.W2,
                                          synth.GU_INTERLEAVED), seed=21)
    assert np.array_equal(a.x, b.x) and np.array_equal(a.topk_ids, b.topk_ids)
    rb = synth.row_bytes(s.gu_fmt, s.d)
    for e in range(s.E):
        o = int(a.expert_offsets[e, 0])
        ga = a.weight_pack[o:o + 2 * s.n_ff * rb].reshape(2 * s.n_ff, rb)
        gb = b.weight_pack[o:o + 2 * s.n_ff * rb].reshape(2 * s.n_ff, rb)
        assert np.array_equal(gb[0::2], ga[:s.n_ff]) and np.array_equal(gb[1::2], ga[s.n_ff:])


def test_offsets_are_16_byte_aligned_and_disjoint():
    s = synth.LayerShape(4, 384, 192, 5, 2, synth.W4NL, synth.Q8_0)
    offs, total, gu, dn = synth.pack_layout(s)
    assert np.all(offs % 16 == 0)
    flat = sorted((int(o), int(o) + size) for o, size in
                  [(offs[e, 0], gu) for e in range(s.E)] + [(offs[e, 1], dn) for e in range(s.E)])
    assert all(a1 <= b0 for (_, a1), (b0, _) in zip(flat, flat[1:]))
    assert flat[-1][1] <= total
