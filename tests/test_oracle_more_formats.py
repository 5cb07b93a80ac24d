"""Pins for the oracle's Q5_0, Q5_1, ggml q8_0, Q2_K, Q5_K and Q3_K decoders (CPU only).

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
from tests.exact import q4k_pack
from tests.test_oracle_mutations import build_mutant, fails


def fp16(v) -> bytes:
    return np.array([v], dtype="<f2").tobytes()


def test_bits_per_weight_against_the_page():
    bpw = {t: 8 * oracle.BLOCK_BYTES[t] / oracle.BLOCK_WEIGHTS[t] for t in oracle.BLOCK_BYTES}
    assert round(bpw[oracle.Q2_K], 2) == 2.62 and oracle.BLOCK_BYTES[oracle.Q2_K] == 84  # the page's figures
    assert bpw[oracle.Q4_K] == 4.5 and round(bpw[oracle.Q6_K], 2) == 6.56
    assert (bpw[oracle.Q5_0], bpw[oracle.Q5_1], bpw[oracle.Q8_0G]) == (5.5, 6.0, 8.5)
    assert (bpw[oracle.Q5_K], round(bpw[oracle.Q3_K], 4)) == (5.5, 3.4375)
    # the decoder reads exactly that many bytes
    for t in (oracle.Q5_0, oracle.Q5_1, oracle.Q8_0G, oracle.Q2_K, oracle.Q5_K, oracle.Q3_K):
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


def q5k_block():
    """fp16 d = 0.5, dmin = 0.25; 6-bit scales and mins in the Q4_K packing; weight
    e = 64c + 32h + l: low four bits in the low (h = 0) or high (h = 1) nibble of
    qs[32c + l], fifth bit at bit 2c + h of qh[l]; value 0.5 sc q - 0.25 mn."""
    sc = [(5 * s + 3) % 64 for s in range(8)]
    mn = [(7 * s + 1) % 64 for s in range(8)]
    q = [(13 * e + e // 9) % 32 for e in range(256)]
    qh, qs = [0] * 32, [0] * 128
    want = np.empty(256)
    for e in range(256):
        c, h, l = e // 64, (e % 64) // 32, e % 32
        qs[32 * c + l] |= (q[e] & 15) << (4 * h)
        qh[l] |= (q[e] >> 4) << (2 * c + h)
        want[e] = 0.5 * sc[2 * c + h] * q[e] - 0.25 * mn[2 * c + h]
    blk = fp16(0.5) + fp16(0.25) + q4k_pack(sc, mn) + bytes(qh) + bytes(qs)
    return np.frombuffer(blk, np.uint8), want


def check_q5k(o):
    blk, want = q5k_block()
    np.testing.assert_array_equal(o.dequant(oracle.Q5_K, blk, 256), want)


def q3k_block():
    """hmask[32], qs[64], 12 scale bytes, fp16 d = 0.5. Weight e = 128n + 32j + l:
    two bits at bit 2j of qs[32n + l], minus 4 unless bit 4n + j of hmask[l] is
    set; sub-block 8n + 2j + l // 16 of 16 weights; its 6-bit scale keeps the low
    nibble in byte s (s < 8) or the high nibble of byte s - 8, the top two bits
    at bit 2 (s // 4) of byte 8 + s % 4; value 0.5 (scale - 32) q."""
    sc6 = [(11 * s + 7) % 64 for s in range(16)]
    f = [0] * 12
    for s in range(16):
        f[s if s < 8 else s - 8] |= (sc6[s] & 15) << (0 if s < 8 else 4)
        f[8 + s % 4] |= (sc6[s] >> 4) << (2 * (s // 4))
    q = [((7 * e + e // 5) % 8) - 4 for e in range(256)]
    hmask, qs = [0] * 32, [0] * 64
    want = np.empty(256)
    for e in range(256):
        n, j, l = e // 128, (e % 128) // 32, e % 32
        hbit = 1 if q[e] >= 0 else 0
        qs[32 * n + l] |= (q[e] + (0 if hbit else 4)) << (2 * j)
        hmask[l] |= hbit << (4 * n + j)
        want[e] = 0.5 * (sc6[8 * n + 2 * j + l // 16] - 32) * q[e]
    blk = bytes(hmask) + bytes(qs) + bytes(f) + fp16(0.5)
    return np.frombuffer(blk, np.uint8), want


def check_q3k(o):
    blk, want = q3k_block()
    np.testing.assert_array_equal(o.dequant(oracle.Q3_K, blk, 256), want)


@pytest.mark.parametrize("check", [check_q5_0, check_q5_1, check_q8_0g, check_q2k, check_q5k, check_q3k])
def test_hand_built_blocks(check):
    check(oracle.get())


def test_gemv_matches_dequantised_dot_on_new_formats():
    rng = np.random.default_rng(4)
    for t in (synth.Q5_0, synth.Q5_1, synth.Q8_0G, synth.Q2_K, synth.Q5_K, synth.Q3_K):
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
    "Q5_K fifth bit at bit 2c for both halves": (check_q5k, "int q = nib | (((qh[l] >> sb) & 1) << 4);",
                                                 "int q = nib | (((qh[l] >> (2 * c)) & 1) << 4);"),
    "Q5_K nibble halves swapped": (check_q5k, "int nib = h ? (qs[32 * c + l] >> 4) : (qs[32 * c + l] & 15);",
                                   "int nib = h ? (qs[32 * c + l] & 15) : (qs[32 * c + l] >> 4);"),
    "Q5_K d and dmin swapped": (check_q5k, "const float dmin = rd_fp16(blk + 2), d = rd_fp16(blk);",
                                "const float dmin = rd_fp16(blk), d = rd_fp16(blk + 2);"),
    "Q5_K qh and qs regions swapped": (check_q5k, "const uint8_t *fields = blk + 4, *qh = blk + 16, *qs = blk + 48;",
                                       "const uint8_t *fields = blk + 4, *qh = blk + 144, *qs = blk + 16;"),
    "Q3_K hmask bit j of both halves": (check_q3k, "int q = ((hmask[l] >> (4 * n + j)) & 1) ? low2 : low2 - 4;",
                                        "int q = ((hmask[l] >> j) & 1) ? low2 : low2 - 4;"),
    "Q3_K hmask sense inverted": (check_q3k, "int q = ((hmask[l] >> (4 * n + j)) & 1) ? low2 : low2 - 4;",
                                  "int q = ((hmask[l] >> (4 * n + j)) & 1) ? low2 - 4 : low2;"),
    "Q3_K scale offset 31": (check_q3k, "return (low | (high << 4)) - 32;", "return (low | (high << 4)) - 31;"),
    "Q3_K top scale bits transposed": (check_q3k, "int high = (f[8 + s % 4] >> (2 * (s / 4))) & 3;",
                                       "int high = (f[8 + s / 4] >> (2 * (s % 4))) & 3;"),
    "Q3_K one scale per 32": (check_q3k, "float a = d * (float)q3k_scale(f, 8 * n + 2 * j + l / 16);",
                              "float a = d * (float)q3k_scale(f, 8 * n + 2 * j);"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_mutant(name):
    check, old, new = MUTANTS[name]
    assert fails(check, build_mutant(old, new)), f"pin passed a broken oracle: {name}"
