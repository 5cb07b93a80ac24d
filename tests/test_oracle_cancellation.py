"""The cancelling Q4_K blocks (tests/cancel_blocks.py) through the oracle.

The closed forms follow from w = d*sc*q - dmin*mn ("S21 The Capstone: picoLM, in
Python", section 2): with dmin = d and mn = sc*q_c, a quant at the centre q_c
gives w = 0 exactly (both products are exact in fp32), and q_c -+ 1 gives -+ d*sc.
These checks hold the builder to its description and the oracle to the format's
formula on exactly the inputs where a factored kernel is weakest.
"""
import numpy as np
import pytest

from tests.cancel_blocks import q4k_cancelling_blocks


def fields(b):
    from tests.exact import fp16_value, q4k_fields
    d16, dmin16, sc, mn, q = q4k_fields(b)
    return float(fp16_value(d16)), float(fp16_value(dmin16)), sc, mn, q


def test_exact_mode_every_weight_is_zero(orc):
    b = q4k_cancelling_blocks(300, np.random.default_rng(11), "exact")
    w = orc.dequant(3, b, 300 * 256)
    assert np.all(w == 0)


def test_pm1_mode_weights_are_minus_zero_plus_d_sc(orc):
    n = 200
    b = q4k_cancelling_blocks(n, np.random.default_rng(12), "pm1")
    w = orc.dequant(3, b, n * 256).reshape(n, 256)
    for i in range(0, n, 17):
        d, _, sc, _, _ = fields(b[144 * i:144 * (i + 1)])
        for j in range(8):
            ds = np.float32(d) * np.float32(sc[j])
            assert set(np.unique(w[i, 32 * j:32 * j + 32])) <= {-ds, np.float32(0.0), ds}


def test_near_mode_weights_are_small_rests(orc):
    n = 200
    b = q4k_cancelling_blocks(n, np.random.default_rng(13), "near")
    w = orc.dequant(3, b, n * 256).reshape(n, 256)
    for i in range(0, n, 13):
        d, dmin, sc, mn, q = fields(b[144 * i:144 * (i + 1)])
        for j in range(8):
            big = abs(d * sc[j] * q[32 * j])
            rest = w[i, 32 * j:32 * j + 32].astype(np.float64)
            # exactly the rounded rest -(dmin - d)*mn, at most 2^-9 of the cancelled terms
            assert np.all(rest == rest[0])
            assert abs(rest[0]) <= big * 2.0 ** -9 + 1e-30
            assert rest[0] == np.float32(np.float32(d) * np.float32(sc[j]) * np.float32(q[32 * j])
                                         - np.float32(dmin) * np.float32(mn[j]))


@pytest.mark.parametrize("mode", ["exact", "pm1", "near"])
def test_gemv_reference_is_zero_or_small(orc, mode):
    rows, cols = 4, 512
    b = q4k_cancelling_blocks(rows * cols // 256, np.random.default_rng(14), mode)
    x = np.random.default_rng(15).standard_normal((1, cols), dtype=np.float32)
    y, S = orc.gemv(3, b, rows, cols, x)
    if mode == "exact":
        assert np.all(y == 0) and np.all(S == 0)
    else:
        assert np.all(np.abs(y) <= S)
