"""Pins for the quantiser oracle (oracle/quantize.py), CPU only.

The dequantiser that checks it is the C oracle's PETIT decoder, whose q8_0 /
q4_0 layouts are pinned on their own (hand-built blocks, tests/test_oracle_formats.py).
"""
import numpy as np

import oracle
from oracle import quantize as qz
from quant_dequant_gemv_gb300 import synth


def test_q8_0_round_trip_within_half_step():
    rng = np.random.default_rng(0)
    x = (rng.standard_normal(32 * 50) * rng.uniform(1e-3, 10, 32 * 50)).astype(np.float32)
    blocks = qz.quantize_q8_0(x)
    y = oracle.dequant(synth.Q8_0, blocks, x.size)
    d = blocks.reshape(-1, 36)[:, 0:4].copy().view("<f4").reshape(-1)
    assert np.all(np.abs(y - x).reshape(-1, 32) <= (d[:, None] / 2) * (1 + 1e-6))
    q = blocks.reshape(-1, 36)[:, 4:].view(np.int8)
    assert np.all(np.abs(q).max(axis=1) == 127)  # the largest |x| of each block lands on +-127


def test_q4_0_round_trip_within_half_step():
    rng = np.random.default_rng(1)
    x = rng.standard_normal(32 * 40).astype(np.float32)
    blocks = qz.quantize_q4_0(x)
    y = oracle.dequant(synth.Q4_0, blocks, x.size)
    d = blocks.reshape(-1, 18)[:, 0:2].copy().view("<f2").astype(np.float32).reshape(-1)
    # |x| <= 7 d up to the fp16 rounding of d, so every x is within half a step of a level
    err = np.abs(y - x).reshape(-1, 32)
    assert np.all(err <= d[:, None] * 0.5 + np.abs(x).reshape(-1, 32) * 2.0 ** -10)


def test_exact_multiples_and_extremes():
    d = np.float32(0.5)
    x = (np.arange(-127, 127, 254 / 32)[:32].round().astype(np.float32) * d)
    x[0] = -127 * d
    y = oracle.dequant(synth.Q8_0, qz.quantize_q8_0(x), 32)
    np.testing.assert_array_equal(y, x)
    x4 = np.array([k % 15 - 7 for k in range(32)], dtype=np.float32) * np.float32(0.25)
    x4[3] = 7 * 0.25
    y4 = oracle.dequant(synth.Q4_0, qz.quantize_q4_0(x4), 32)
    np.testing.assert_array_equal(y4, x4)


def test_halves_round_to_even_and_zero_block():
    # amax 127 -> d = 1; 2.5 -> 2, 3.5 -> 4, -2.5 -> -2
    x = np.zeros(32, dtype=np.float32)
    x[0], x[1], x[2], x[3] = 127, 2.5, 3.5, -2.5
    q = qz.quantize_q8_0(x).reshape(36)[4:].view(np.int8)
    assert list(q[:4]) == [127, 2, 4, -2]
    z = qz.quantize_q8_0(np.zeros(32, dtype=np.float32)).reshape(36)
    assert z[:4].view("<f4")[0] == 0 and not z[4:].any()
    z4 = qz.quantize_q4_0(np.zeros(32, dtype=np.float32)).reshape(18)
    assert z4[:2].view("<f2")[0] == 0 and np.all(z4[2:] == 0x88)


def test_q4_0_nibble_order_and_padding():
    # weight i in the low nibble of byte i, weight i + 16 in the high nibble
    x = np.zeros(20, dtype=np.float32)  # padded to 32 with zeros
    x[0], x[16] = 7.0, -7.0
    b = qz.quantize_q4_0(x).reshape(18)
    assert b[0:2].view("<f2")[0] == np.float16(1.0)
    assert b[2] == (15 | (1 << 4))
    assert np.all(b[3:] == 0x88)
