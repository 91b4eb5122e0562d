"""Plant plausible mistakes in copies of the oracle and check that the pins
catch every one (no GPU).  A mutant that passes every pin would mean the
pins cannot tell that mistake from the method."""
import os
import subprocess
import tempfile

import pytest

import oracle
import oracle.build as ob
import oracle_pins as P

# (name, exact source text, replacement)
MUTANTS = [
    ("w2_code_offset", "return c - 2;", "return c - 1;"),
    ("w2_bit_order", "(2 * (jj % 4))", "(2 * (3 - jj % 4))"),
    ("w4nl_nibble_order", "(4 * (jj % 2))", "(4 * (1 - jj % 2))"),
    ("q8_0_unsigned_codes", "return (int)(int8_t)blk[2 + jj];", "return (int)blk[2 + jj];"),
    ("q8_0_block_bytes", "return fmt == ORC_Q8_0 ? 34 : 18;", "return fmt == ORC_Q8_0 ? 33 : 18;"),
    ("half_exponent_bias", "ex - 25", "ex - 24"),
    ("dropped_last_block", "for (int b = 0; b < nb; b++) {\n      int32_t isum",
     "for (int b = 0; b < nb - 1; b++) {\n      int32_t isum"),
    ("act_scale_index", "float s = ws[b] * dq[b];", "float s = ws[b] * dq[0];"),
    ("weight_scale_block0", "ws[b] = orc_w_scale(fmt, wrow, 32 * b);",
     "ws[b] = orc_w_scale(fmt, wrow, 0);"),
    ("acc_reset", "acc = fmaf(s, (float)isum, acc);", "acc = fmaf(s, (float)isum, 0.0f);"),
    ("q8_divisor", "float db = amax / 127.0f;", "float db = amax / 128.0f;"),
    ("q8_round_away", "rintf(xb[i] / db)", "roundf(xb[i] / db)"),
    ("q8_amax_first_only", "if (a > amax) amax = a;", "if (i == 0) amax = a;"),
    ("silu_swapped_gu", "hbuf[j] = (g / (1.0f + expf(-g))) * u;",
     "hbuf[j] = (u / (1.0f + expf(-u))) * g;"),
    ("silu_sign", "expf(-g)", "expf(g)"),
    ("up_half_index", "float u = gu[n_ff + j];", "float u = gu[j];"),
    ("route_unstable", "int32_t pos = fill[e]++;",
     "int32_t pos = offsets[e + 1] - 1 - (fill[e]++ - offsets[e]);"),
    ("combine_reverse", "for (int r = 0; r < k; r++) {\n        int32_t pos = dst_of[t * k + r];",
     "for (int r = k - 1; r >= 0; r--) {\n        int32_t pos = dst_of[t * k + r];"),
    ("combine_weight_index", "fmaf(w[t * k + r]", "fmaf(w[t * k]"),
    ("interleaved_swapped", "g = gu[2 * j];\n      u = gu[2 * j + 1];",
     "g = gu[2 * j + 1];\n      u = gu[2 * j];"),
    ("scale_big_endian", "blk[0] | (blk[1] << 8)", "blk[1] | (blk[0] << 8)"),
    ("half_subnormal_exponent", "ldexpf((float)man, -24)", "ldexpf((float)man, -25)"),
    ("nl4_table_entry", "1,    13,   25,  38,  53,  69,  89,  113}",
     "1,    13,   25,  38,  53,  69,  89,  112}"),
    ("layer_token_of_row", "int64_t t = src / j->k;", "int64_t t = src % j->k;"),
    ("layer_down_offset", "j->eoff[2 * e + 1]", "j->eoff[2 * e]"),
    ("layer_expert_of_row", "int e = j->ids[src];", "int e = j->ids[r];"),
    ("w2_scale_per_32", "const uint8_t *blk = row + (int64_t)(j / bv) * orc_block_bytes(fmt);\n  return orc_half",
     "const uint8_t *blk = row + (int64_t)(j / 32) * orc_block_bytes(fmt);\n  return orc_half"),
    ("q8_scale_fp16", "    d[b] = db;", "    d[b] = (float)(_Float16)db;"),
    ("q8_signed_amax", "float a = fabsf(xb[i]);", "float a = xb[i];"),
    ("product_q_unsigned", "isum += wi[32 * b + i] * (int32_t)q[32 * b + i];",
     "isum += wi[32 * b + i] * (int32_t)(uint8_t)q[32 * b + i];"),
    ("route_bad_id_to_row_0", "      dst_of[i] = -1;", "      dst_of[i] = 0;"),
    ("swiglu_scale_row", "dh + r * (n_ff / 32), h);", "dh + r * (n_ff / 32 - 1), h);"),
    # rounding-level mistakes: each against a hand example where it changes a bit
    ("q8_reciprocal", "rintf(xb[i] / db)", "rintf(xb[i] * (1.0f / db))"),
    ("epilogue_unfused", "acc = fmaf(s, (float)isum, acc);", "acc = acc + s * (float)isum;"),
    ("combine_unfused", "acc = fmaf(w[t * k + r], dm[(int64_t)pos * d + j], acc);",
     "acc = acc + w[t * k + r] * dm[(int64_t)pos * d + j];"),
]


def _build_mutant(tmp, name, old, new):
    src = open(ob.SRC).read()
    assert src.count(old) >= 1, f"mutation anchor for {name} not found"
    src = src.replace(old, new)
    cpath = os.path.join(tmp, f"{name}.c")
    with open(cpath, "w") as f:
        f.write(src)
    so = os.path.join(tmp, f"lib{name}.so")
    subprocess.run(["gcc", *ob.CFLAGS, cpath, "-o", so, "-lm"], check=True,
                   capture_output=True)
    return so


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(name, old, new):
    with tempfile.TemporaryDirectory() as tmp:
        so = _build_mutant(tmp, name, old, new)
        caught = []
        try:
            oracle.use_library(so)
            for check in P.ALL_PINS:
                try:
                    check()
                except AssertionError:
                    caught.append(check.__name__)
        finally:
            oracle.use_library(None)
        assert caught, f"mutant {name} passed every pin"
