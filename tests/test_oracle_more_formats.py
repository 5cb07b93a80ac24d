"""Pins for the oracle's Q5_0, Q5_1, ggml q8_0 and Q2_K decoders (CPU only).

The pages name these formats ("S21 The Capstone: picoLM, in Python", section 2:
eight formats, Q2_K at 2.62 bits per weight, 84 bytes per 256) but print only
Q2_K's size; the layouts are the published ggml ones, a reading. The blocks here
are assembled in the test from that reading's description (which byte, which
bit), with values chosen so that every weight has a closed form, and planted
mutations of the oracle must fail them.
"""
import numpy as np
import pytest

import oracle
from quant_dequant_gemv_gb300 import synth
from tests.test_oracle_mutations import build_mutant, fails


def fp16(v) -> bytes:
    return np.array([v], dtype="<f2").tobytes()


def test_bits_per_weight_against_the_page():
    bpw = {t: 8 * oracle.BLOCK_BYTES[t] / oracle.BLOCK_WEIGHTS[t] for t in oracle.BLOCK_BYTES}
    assert round(bpw[oracle.Q2_K], 2) == 2.62 and oracle.BLOCK_BYTES[oracle.Q2_K] == 84  # the page's figures
    assert bpw[oracle.Q4_K] == 4.5 and round(bpw[oracle.Q6_K], 2) == 6.56
    assert (bpw[oracle.Q5_0], bpw[oracle.Q5_1], bpw[oracle.Q8_0G]) == (5.5, 6.0, 8.5)
    # the decoder reads exactly that many bytes
    for t in (oracle.Q5_0, oracle.Q5_1, oracle.Q8_0G, oracle.Q2_K):
        with pytest.raises(ValueError):
            oracle.dequant(t, np.zeros(oracle.BLOCK_BYTES[t] - 1, np.uint8), oracle.BLOCK_WEIGHTS[t])


# a permutation of 0..31: weights i and i + 16 differ in their low nibble and in
# their fifth bit, so a swapped nibble half or a misplaced bit changes a value
Q5 = np.array([9, 30, 4, 17, 25, 2, 13, 28, 7, 20, 31, 0, 18, 11, 26, 5,
               22, 3, 16, 27, 12, 29, 1, 14, 24, 8, 19, 6, 10, 23, 15, 21])


def q5_bytes(q) -> bytes:
    qs = bytes(int(q[i] & 15) | (int(q[i + 16] & 15) << 4) for i in range(16))
    qh = sum(int(q[i] >> 4) << i for i in range(32)).to_bytes(4, "little")
    return qh + qs


def check_q5_0(o):
    blk = np.frombuffer(fp16(0.5) + q5_bytes(Q5), np.uint8)
    np.testing.assert_array_equal(o.dequant(oracle.Q5_0, blk, 32), (Q5 - 16) * 0.5)


def check_q5_1(o):
    blk = np.frombuffer(fp16(0.25) + fp16(-2.0) + q5_bytes(Q5), np.uint8)
    np.testing.assert_array_equal(o.dequant(oracle.Q5_1, blk, 32), Q5 * 0.25 - 2.0)


def check_q8_0g(o):
    q = np.array([7 * i - 100 for i in range(32)], dtype=np.int8)
    blk = np.frombuffer(fp16(0.125) + q.tobytes(), np.uint8)
    np.testing.assert_array_equal(o.dequant(oracle.Q8_0G, blk, 32), q * 0.125)


def q2k_block():
    sc = np.array([(5 * i + 1) % 16 for i in range(16)])
    mn = np.array([(3 * i + 2) % 16 for i in range(16)])
    q = np.array([(e * e + e // 7) % 4 for e in range(256)])
    qs = np.zeros(64, dtype=np.uint8)
    want = np.empty(256)
    for e in range(256):
        n, j, l = e // 128, (e % 128) // 32, e % 32
        qs[32 * n + l] |= q[e] << (2 * j)
        i = 8 * n + 2 * j + l // 16
        want[e] = 0.5 * sc[i] * q[e] - 0.25 * mn[i]
    blk = bytes(int(s | (m << 4)) for s, m in zip(sc, mn)) + qs.tobytes() + fp16(0.5) + fp16(0.25)
    return np.frombuffer(blk, np.uint8), want


def check_q2k(o):
    blk, want = q2k_block()
    np.testing.assert_array_equal(o.dequant(oracle.Q2_K, blk, 256), want)


@pytest.mark.parametrize("check", [check_q5_0, check_q5_1, check_q8_0g, check_q2k])
def test_hand_built_blocks(check):
    check(oracle.get())


def test_gemv_matches_dequantised_dot_on_new_formats():
    rng = np.random.default_rng(4)
    for t in (synth.Q5_0, synth.Q5_1, synth.Q8_0G, synth.Q2_K):
        rows, cols = 5, 512
        W = synth.gen_matrix(t, rows, cols, 9)
        x = rng.standard_normal((2, cols)).astype(np.float32)
        y, S = oracle.gemv(t, W, rows, cols, x)
        w = oracle.dequant(t, W, rows * cols).astype(np.float64).reshape(rows, cols)
        np.testing.assert_allclose(y, x.astype(np.float64) @ w.T, rtol=1e-13, atol=1e-13)


MUTANTS = {
    "Q5 fifth bit of weight i+16 from bit i": (check_q5_0, "return nib | (int)(((qh >> i) & 1u) << 4);",
                                               "return nib | (int)(((qh >> (i & 15)) & 1u) << 4);"),
    "Q5 nibble halves swapped": (check_q5_1, "int nib = (i < 16) ? (qs[i] & 15) : (qs[i - 16] >> 4);",
                                 "int nib = (i < 16) ? (qs[i] >> 4) : (qs[i - 16] & 15);"),
    "Q5_0 offset 15": (check_q5_0, "(float)(q5_quant(blk + 2, blk + 6, i) - 16) * d",
                       "(float)(q5_quant(blk + 2, blk + 6, i) - 15) * d"),
    "Q5_1 subtracts m": (check_q5_1, "out[i] = a + m;", "out[i] = a - m;"),
    "Q5_1 m read as d": (check_q5_1, "float d = rd_fp16(blk), m = rd_fp16(blk + 2);",
                         "float d = rd_fp16(blk), m = rd_fp16(blk);"),
    "ggml q8_0 read with an fp32 scale": (check_q8_0g, "const int8_t *q = (const int8_t *)(blk + 2);",
                                          "const int8_t *q = (const int8_t *)(blk + 4);"),
    "Q2_K one scale per 32": (check_q2k, "int sm = scales[8 * n + 2 * j + l / 16];",
                              "int sm = scales[8 * n + 2 * j];"),
    "Q2_K shift j": (check_q2k, "int q = (qs[32 * n + l] >> (2 * j)) & 3;", "int q = (qs[32 * n + l] >> j) & 3;"),
    "Q2_K min from the low nibble": (check_q2k, "float b = dmin * (float)(sm >> 4);",
                                     "float b = dmin * (float)(sm & 15);"),
    "Q2_K d and dmin swapped": (check_q2k, "float d = rd_fp16(blk + 80), dmin = rd_fp16(blk + 82);",
                                "float d = rd_fp16(blk + 82), dmin = rd_fp16(blk + 80);"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_mutant(name):
    check, old, new = MUTANTS[name]
    assert fails(check, build_mutant(old, new)), f"pin passed a broken oracle: {name}"
