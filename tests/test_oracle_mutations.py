"""Mutation checks: plant one known mistake in a copy of the oracle source, build
it on the CPU, and confirm that the pins fail on it. A pin that passes a broken
oracle pins nothing.
"""
import tempfile
from pathlib import Path

import numpy as np
import pytest

import oracle
from tests import exact as ex
from tests import test_oracle_formats as fmt
from tests import test_oracle_gemv as gem

SRC = oracle.SRC.read_text()


def build_mutant(old: str, new: str) -> oracle.Oracle:
    assert SRC.count(old) == 1, f"mutation anchor not found exactly once: {old!r}"
    td = Path(tempfile.mkdtemp(prefix="orc_mut_"))
    return oracle.Oracle(oracle.compile_source(SRC.replace(old, new), td / "libmut.so"))


def fails(check, *args) -> bool:
    try:
        check(*args)
    except AssertionError:
        return True
    return False


Q4K_PINS = [
    (fmt.test_q4k_scale_min_roundtrip,),
    (fmt.test_q4k_high_bits_only_matter_for_last_four,),
    (fmt.test_q4k_handbuilt_block_closed_form,),
    (fmt.test_q4k_subblock_pairing,),
    (fmt.test_q4k_equals_exactly_rounded_formula, "workload"),
]

MUTANTS_Q4K = {
    "top bits from bits 5-6": ("*bit = 6 + (b - 4);", "*bit = 5 + (b - 4);"),
    "top bits from the byte of field j": ("*byte = 4 * k + (j - 4);", "*byte = 4 * k + j;"),
    "min low bits from low nibble": ("*bit = 4 * k + b;", "*bit = b;"),
    "low bits of fields 4-7 from byte j+3": ("*byte = j + 4;", "*byte = j + 3;"),
    "fields read as 7 bits": ("for (int b = 0; b < 6; ++b) {", "for (int b = 0; b < 7; ++b) {"),
    "nibble halves swapped": ("(i < 32) ? (qs[32 * c + i] & 15) : (qs[32 * c + i - 32] >> 4)",
                              "(i < 32) ? (qs[32 * c + i] >> 4) : (qs[32 * c + i - 32] & 15)"),
    "low nibbles paired with odd sub-block": ("int s = 2 * c + (i >= 32);",
                                              "int s = 2 * c + (i < 32);"),
    "dmin and d swapped": ("float d = rd_fp16(blk), dmin = rd_fp16(blk + 2);",
                           "float dmin = rd_fp16(blk), d = rd_fp16(blk + 2);"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS_Q4K))
def test_q4k_pins_catch_mutant(name):
    m = build_mutant(*MUTANTS_Q4K[name])
    assert any(fails(p[0], m, *p[1:]) for p in Q4K_PINS), f"no Q4_K pin caught: {name}"


Q6K_PINS = [
    (fmt.test_q6k_struct_offsets_and_16_grouping,),
    (fmt.test_q6k_quant_range_and_offset,),
    (fmt.test_q6k_scale_signs,),
    (fmt.test_q6k_equals_exactly_rounded_formula, "workload"),
]

MUTANTS_Q6K = {
    "one scale per 32 weights": ("(float)scales[e / 16];", "(float)scales[(e / 32) * 2];"),
    "no -32 offset": ("int q = (low | (high << 4)) - 32;", "int q = (low | (high << 4));"),
    "unsigned scales": ("const int8_t *scales = (const int8_t *)(blk + 192);",
                        "const uint8_t *scales = (const uint8_t *)(blk + 192);"),
    "high bits shifted by k": ("(qh[32 * h + l] >> (2 * k)) & 3", "(qh[32 * h + l] >> k) & 3"),
    "d read from the front": ("float d = rd_fp16(blk + 208);", "float d = rd_fp16(blk);"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS_Q6K))
def test_q6k_pins_catch_mutant(name):
    m = build_mutant(*MUTANTS_Q6K[name])
    assert any(fails(p[0], m, *p[1:]) for p in Q6K_PINS), f"no Q6_K pin caught: {name}"


def test_q6k_scale32_bug_has_the_reported_signature(orc):
    """The Q6_K bug story: with one scale applied to 32 weights, weights 0-15 of
    each 32 are right and 16-31 are wrong, strictly alternating in groups of 16,
    and wrong/right equals scale[0]/scale[1] in the first group."""
    m = build_mutant(*MUTANTS_Q6K["one scale per 32 weights"])
    rng = np.random.default_rng(7)
    scales = [int(v) for v in rng.choice([v for v in range(-128, 128) if v != 0], 16)]
    q6 = [int(v) for v in rng.integers(0, 64, 256)]
    q6 = [v if v != 32 else 33 for v in q6]  # no zero quants: ratios defined everywhere
    blk = np.frombuffer(ex.q6k_block(0x3C00, scales, q6), np.uint8)
    good = orc.dequant(oracle.Q6_K, blk, 256)
    bad = m.dequant(oracle.Q6_K, blk, 256)
    for e in range(256):
        m32, r = divmod(e, 32)
        if r < 16:
            assert bad[e] == good[e]
        else:
            assert bad[e] / good[e] == pytest.approx(scales[2 * m32] / scales[2 * m32 + 1])
    assert bad[16] / good[16] == pytest.approx(scales[0] / scales[1])
    # and the 16-grouping pin catches it
    assert fails(fmt.test_q6k_struct_offsets_and_16_grouping, m)


MUTANTS_PETIT = {
    "q8_0 scale read as fp16": ("memcpy(&d, blk, 4);", "d = rd_fp16(blk);"),
    "q8_0 unsigned quants": ("const int8_t *q = (const int8_t *)(blk + 4);",
                             "const uint8_t *q = (const uint8_t *)(blk + 4);"),
    "q4_0 nibbles interleaved": ("int q = (i < 16) ? (qs[i] & 15) : (qs[i - 16] >> 4);",
                                 "int q = (i % 2 == 0) ? (qs[i / 2] & 15) : (qs[i / 2] >> 4);"),
    "q4_0 no -8 offset": ("out[i] = (float)(q - 8) * d;", "out[i] = (float)q * d;"),
}

PETIT_PINS = [
    (fmt.test_q8_0_handbuilt,), (fmt.test_q8_0_extremes,),
    (fmt.test_q4_0_handbuilt_nibble_order,), (fmt.test_q4_0_equals_exactly_rounded_formula,),
]


@pytest.mark.parametrize("name", sorted(MUTANTS_PETIT))
def test_petit_pins_catch_mutant(name):
    m = build_mutant(*MUTANTS_PETIT[name])
    assert any(fails(p[0], m, *p[1:]) for p in PETIT_PINS), f"no pin caught: {name}"


MUTANTS_GEMV = {
    "x indexed by row": ("double p = (double)row_buf[c] * (double)xb[c];",
                         "double p = (double)row_buf[c] * (double)xb[r % cols];"),
    "fp32 accumulation": ("acc += p;", "acc = (float)(acc + p);"),
    "S without abs": ("sabs += fabs(p);", "sabs += p;"),
    "y laid out [rows][batch]": ("y[(int64_t)b * rows + r] = acc;", "y[r * batch + b] = acc;"),
}

GEMV_PINS = [
    (gem.test_gemv_unit_vectors_pick_columns, oracle.Q4_K),
    (gem.test_gemv_exact_rational_sum, oracle.Q6_K),
    (gem.test_gemv_abs_sum,), (gem.test_gemv_batch_layout,),
]


@pytest.mark.parametrize("name", sorted(MUTANTS_GEMV))
def test_gemv_pins_catch_mutant(name):
    m = build_mutant(*MUTANTS_GEMV[name])
    assert any(fails(p[0], m, *p[1:]) for p in GEMV_PINS), f"no GEMV pin caught: {name}"
