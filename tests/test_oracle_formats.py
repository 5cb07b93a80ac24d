"""Pins for the oracle's block decoders (no GPU).

Each test holds the oracle to something the pages or the mathematics fix: the
IEEE binary16 definition (checked against numpy), hand-built blocks with values
known in closed form, the Q4_K 12-byte field layout, the Q6_K one-scale-per-16
rule, and the exactly rounded value of each format's formula.
"""
from fractions import Fraction

import numpy as np
import pytest

import oracle
from quant_dequant_gemv_gb300 import synth
from tests import exact as ex

Q4_0, Q8_0, Q4_K, Q6_K = oracle.Q4_0, oracle.Q8_0, oracle.Q4_K, oracle.Q6_K


def assert_exact(got: np.ndarray, want: list[Fraction]):
    w = np.array([ex.round_f32(v) for v in want], dtype=np.float32)
    bad = np.nonzero(got != w)[0]
    assert bad.size == 0, f"{bad.size} mismatches, first at {bad[0]}: {got[bad[0]]!r} vs {w[bad[0]]!r}"


# ---------------------------------------------------------------- fp16 -------
def test_fp16_all_patterns_match_numpy(orc):
    h = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    got = orc.fp16_to_fp32(h)
    want = h.view(np.float16).astype(np.float32)
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan].view(np.uint32), want[~nan].view(np.uint32))


def test_fp16_definition_spot_values(orc):
    # 0x0001 is the smallest subnormal 2^-24; 0x3C00 = 1; 0x7BFF = 65504; 0xC000 = -2
    for h, v in [(0x0001, 2.0 ** -24), (0x03FF, 1023 * 2.0 ** -24), (0x0400, 2.0 ** -14),
                 (0x3C00, 1.0), (0x7BFF, 65504.0), (0xC000, -2.0), (0x8000, -0.0)]:
        got = orc.fp16_to_fp32(np.array([h]))[0]
        assert got == v and np.signbit(got) == np.signbit(v)


# ---------------------------------------------------------------- Q4_K -------
def test_q4k_field_table_is_a_bijection():
    # 16 fields x 6 bits use each of the 96 bits of the 12 bytes exactly once, so
    # uniform random bytes are uniform independent fields.
    seen = [pos for bits in ex.Q4K_TABLE.values() for pos in bits]
    assert len(seen) == 96 and len(set(seen)) == 96


def test_q4k_scale_min_roundtrip(orc):
    rng = np.random.default_rng(1)
    specials = [bytes([v] * 12) for v in (0x00, 0xFF, 0xC0, 0x3F, 0x0F, 0xF0)]
    randoms = [rng.integers(0, 256, 12, dtype=np.uint8).tobytes() for _ in range(3000)]
    for p in specials + randoms:
        got = [orc.q4k_scale_min(p, j) for j in range(8)]
        sc, mn = ex.q4k_unpack(p)
        assert got == list(zip(sc, mn))
        assert ex.q4k_pack([g[0] for g in got], [g[1] for g in got]) == p


def test_q4k_high_bits_only_matter_for_last_four(orc):
    # Sub-blocks 4..7 with fields in 48..63: their top bits live in bits 6-7 of
    # bytes 0..7, which sub-blocks 0..3 must ignore.
    sc = [5, 17, 33, 63, 48, 55, 60, 63]
    mn = [0, 1, 40, 2, 63, 50, 49, 62]
    p = ex.q4k_pack(sc, mn)
    assert all(b & 0xC0 for b in p[:8])  # every top-bit pair is in use
    assert [orc.q4k_scale_min(p, j) for j in range(8)] == list(zip(sc, mn))


def test_q4k_handbuilt_block_closed_form(orc):
    # d = 1, dmin = 1/2, q[e] = e mod 16: w[e] = sc[e//32]*(e%16) - mn[e//32]/2,
    # all exactly representable.
    sc = [1, 2, 3, 4, 49, 50, 51, 52]
    mn = [0, 1, 2, 3, 60, 61, 62, 63]
    q = [e % 16 for e in range(256)]
    blk = np.frombuffer(ex.q4k_block(0x3C00, 0x3800, sc, mn, q), dtype=np.uint8)
    got = orc.dequant(Q4_K, blk, 256)
    want = np.array([sc[e // 32] * (e % 16) - mn[e // 32] / 2 for e in range(256)], np.float32)
    assert np.array_equal(got, want)


def test_q4k_subblock_pairing(orc):
    # Only sub-block 1 gets a non-zero scale: exactly the high nibbles of chunk 0
    # (weights 32..63) must be non-zero.
    sc = [0, 7, 0, 0, 0, 0, 0, 0]
    blk = np.frombuffer(ex.q4k_block(0x3C00, 0, sc, [0] * 8, [9] * 256), dtype=np.uint8)
    got = orc.dequant(Q4_K, blk, 256)
    want = np.zeros(256, np.float32)
    want[32:64] = 63
    assert np.array_equal(got, want)


@pytest.mark.parametrize("source", ["workload", "any_finite_bytes"])
def test_q4k_equals_exactly_rounded_formula(orc, source):
    # d*sc*q has at most 11+6+4 = 21 significant bits and dmin*mn at most 17, so
    # the page's evaluation (d*sc)*q - dmin*mn rounds once: the result is the
    # correctly rounded real value of the formula.
    rng = np.random.default_rng(2)
    nb = 48
    if source == "workload":
        blocks = synth.gen_blocks(Q4_K, nb, rng).reshape(nb, 144)
    else:
        blocks = rng.integers(0, 256, (nb, 144), dtype=np.uint8)
        for b in blocks:  # keep d, dmin finite (exponent field != 31)
            b[1] &= 0xFB
            b[3] &= 0xFB
    got = orc.dequant(Q4_K, blocks.reshape(-1), nb * 256).reshape(nb, 256)
    for i in range(nb):
        assert_exact(got[i], ex.q4k_exact(blocks[i]))


def test_q4k_nonfinite_scale_propagates(orc):
    blk = bytearray(ex.q4k_block(0x7C00, 0x3C00, [1] * 8, [1] * 8, [e % 16 for e in range(256)]))
    got = orc.dequant(Q4_K, np.frombuffer(bytes(blk), np.uint8), 256)
    # inf * 1 * 0 = nan, inf * 1 * q = inf for q > 0
    assert np.all(np.isnan(got[::16])) and np.all(np.isinf(got[1::16]))


# ---------------------------------------------------------------- Q6_K -------
def test_q6k_struct_offsets_and_16_grouping(orc):
    # q6 = 33 everywhere (q = 1), scales[k] = k + 1, d = 1: w[e] = e//16 + 1.
    blk = ex.q6k_block(0x3C00, [k + 1 for k in range(16)], [33] * 256)
    got = orc.dequant(Q6_K, np.frombuffer(blk, np.uint8), 256)
    assert np.array_equal(got, np.array([e // 16 + 1 for e in range(256)], np.float32))
    # the same through raw bytes: ql nibbles all 1, qh fields all 2 (0b10101010)
    raw = bytes([0x11] * 128 + [0xAA] * 64 + list(range(1, 17))) + (0x3C00).to_bytes(2, "little")
    assert raw == blk


def test_q6k_quant_range_and_offset(orc):
    # q6 = 0 -> -32, q6 = 63 -> 31, d = 1/2, scale = -3
    q6 = [0 if e % 2 == 0 else 63 for e in range(256)]
    blk = ex.q6k_block(0x3800, [-3] * 16, q6)
    got = orc.dequant(Q6_K, np.frombuffer(blk, np.uint8), 256)
    want = np.array([(-3 * 0.5) * (-32 if e % 2 == 0 else 31) for e in range(256)], np.float32)
    assert np.array_equal(got, want)


def test_q6k_scale_signs(orc):
    # int8 scales: byte 0x80 is -128, 0x7F is 127
    blk = ex.q6k_block(0x3C00, [-128, 127] * 8, [33] * 256)
    got = orc.dequant(Q6_K, np.frombuffer(blk, np.uint8), 256)
    assert np.array_equal(got, np.array([(-128 if (e // 16) % 2 == 0 else 127)
                                         for e in range(256)], np.float32))


@pytest.mark.parametrize("source", ["workload", "any_finite_bytes"])
def test_q6k_equals_exactly_rounded_formula(orc, source):
    # d*sc is exact (11+8 bits), so (d*sc)*q rounds once.
    rng = np.random.default_rng(3)
    nb = 48
    if source == "workload":
        blocks = synth.gen_blocks(Q6_K, nb, rng).reshape(nb, 210)
    else:
        blocks = rng.integers(0, 256, (nb, 210), dtype=np.uint8)
        blocks[:, 209] &= 0xFB
    got = orc.dequant(Q6_K, blocks.reshape(-1), nb * 256).reshape(nb, 256)
    for i in range(nb):
        assert_exact(got[i], ex.q6k_exact(blocks[i]))


# ---------------------------------------------------------------- q8_0 / q4_0 --
def test_q8_0_handbuilt(orc):
    d = np.array([0.5], "<f4").view(np.uint8).tobytes()
    q = np.arange(-16, 16, dtype=np.int8).view(np.uint8).tobytes()
    got = orc.dequant(Q8_0, np.frombuffer(d + q, np.uint8), 32)
    assert np.array_equal(got, (np.arange(-16, 16) * 0.5).astype(np.float32))


def test_q8_0_extremes(orc):
    d = np.array([3.0], "<f4").view(np.uint8).tobytes()
    q = np.array([-128, -127, 127, 0] * 8, dtype=np.int8).view(np.uint8).tobytes()
    got = orc.dequant(Q8_0, np.frombuffer(d + q, np.uint8), 32)
    assert np.array_equal(got, np.array([-384, -381, 381, 0] * 8, np.float32))


def test_q8_0_equals_exactly_rounded_formula(orc):
    rng = np.random.default_rng(4)
    nb = 256
    blocks = synth.gen_blocks(Q8_0, nb, rng).reshape(nb, 36)
    got = orc.dequant(Q8_0, blocks.reshape(-1), nb * 32).reshape(nb, 32)
    for i in range(nb):
        assert_exact(got[i], ex.q8_0_exact(blocks[i]))


def test_q4_0_handbuilt_nibble_order(orc):
    # byte i = i | (15 - i) << 4, d = 1: weight i = i - 8, weight i + 16 = 7 - i
    qs = bytes([i | ((15 - i) << 4) for i in range(16)])
    got = orc.dequant(Q4_0, np.frombuffer((0x3C00).to_bytes(2, "little") + qs, np.uint8), 32)
    want = [i - 8 for i in range(16)] + [7 - i for i in range(16)]
    assert np.array_equal(got, np.array(want, np.float32))


def test_q4_0_equals_exactly_rounded_formula(orc):
    rng = np.random.default_rng(5)
    nb = 256
    blocks = synth.gen_blocks(Q4_0, nb, rng).reshape(nb, 18)
    got = orc.dequant(Q4_0, blocks.reshape(-1), nb * 32).reshape(nb, 32)
    for i in range(nb):
        assert_exact(got[i], ex.q4_0_exact(blocks[i]))


def test_dequant_rejects_partial_blocks(orc):
    with pytest.raises(ValueError):
        orc.dequant(Q4_K, np.zeros(144, np.uint8), 100)
