"""Pins for the oracle's GEMV (no GPU).

y[b][r] = sum_c w[r][c] * x[b][c] in double, S[b][r] = sum_c |w[r][c] x[b][c]|,
W stored rows x cols (out x in), x as [batch][cols], y as [batch][rows]
("PETIT": weights stored out x in, one projection = one gemv).
"""
from fractions import Fraction

import numpy as np
import pytest

import oracle
from quant_dequant_gemv_gb300 import synth

TYPES = [oracle.Q4_0, oracle.Q8_0, oracle.Q4_K, oracle.Q6_K]


def small_case(qtype, rows, cols, batch, seed):
    W = synth.gen_matrix(qtype, rows, cols, seed)
    x = synth.gen_x(batch, cols, seed + 1000)
    return W, x


@pytest.mark.parametrize("qtype", TYPES)
def test_gemv_unit_vectors_pick_columns(orc, qtype):
    rows, cols = 5, 2 * oracle.BLOCK_WEIGHTS[qtype]
    W, _ = small_case(qtype, rows, cols, 1, 11)
    w = orc.dequant(qtype, W, rows * cols).reshape(rows, cols)
    js = [0, 17, cols // 2 + 3, cols - 1]
    x = np.zeros((len(js), cols), np.float32)
    for b, j in enumerate(js):
        x[b, j] = 1.0
    y, S = orc.gemv(qtype, W, rows, cols, x)
    for b, j in enumerate(js):
        assert np.array_equal(y[b], w[:, j].astype(np.float64))
        assert np.array_equal(S[b], np.abs(w[:, j]).astype(np.float64))


@pytest.mark.parametrize("qtype", TYPES)
def test_gemv_exact_rational_sum(orc, qtype):
    rows, cols = 3, oracle.BLOCK_WEIGHTS[qtype] * 2
    W, x = small_case(qtype, rows, cols, 1, 12)
    w = orc.dequant(qtype, W, rows * cols).reshape(rows, cols)
    y, S = orc.gemv(qtype, W, rows, cols, x)
    for r in range(rows):
        exact = sum(Fraction(float(w[r, c])) * Fraction(float(x[0, c])) for c in range(cols))
        assert abs(Fraction(y[0, r]) - exact) <= Fraction(1, 10 ** 13) * Fraction(S[0, r])


def test_gemv_abs_sum(orc):
    qtype, rows, cols = oracle.Q8_0, 4, 64
    W, _ = small_case(qtype, rows, cols, 1, 13)
    w = orc.dequant(qtype, W, rows * cols).reshape(rows, cols)
    x = np.where(np.arange(cols) % 2 == 0, 1.0, -1.0).astype(np.float32)[None, :]
    y, S = orc.gemv(qtype, W, rows, cols, x)
    want_S = np.abs(w.astype(np.float64)).sum(axis=1)
    assert np.allclose(S[0], want_S, rtol=1e-14, atol=0)
    assert np.all(S[0] >= np.abs(y[0]))


def test_gemv_batch_layout(orc):
    qtype, rows, cols, batch = oracle.Q4_0, 5, 96, 3
    W, x = small_case(qtype, rows, cols, batch, 14)
    y, S = orc.gemv(qtype, W, rows, cols, x)
    assert y.shape == (batch, rows)
    for b in range(batch):
        yb, Sb = orc.gemv(qtype, W, rows, cols, x[b:b + 1])
        assert np.array_equal(y[b], yb[0]) and np.array_equal(S[b], Sb[0])


@pytest.mark.parametrize("qtype", TYPES)
def test_gemv_matches_float64_matmul(orc, qtype):
    # dequantise-then-dot reduces to a plain float64 matrix product
    rows, cols, batch = 7, 3 * oracle.BLOCK_WEIGHTS[qtype], 2
    W, x = small_case(qtype, rows, cols, batch, 15)
    w = orc.dequant(qtype, W, rows * cols).reshape(rows, cols).astype(np.float64)
    y, S = orc.gemv(qtype, W, rows, cols, x)
    ref = x.astype(np.float64) @ w.T
    assert np.all(np.abs(y - ref) <= 1e-12 * S)


def test_gemv_row_range_sampling(orc):
    qtype, rows, cols = oracle.Q4_K, 9, 512
    W, x = small_case(qtype, rows, cols, 1, 16)
    y_all, _ = orc.gemv(qtype, W, rows, cols, x)
    y_part, _ = orc.gemv(qtype, W, rows, cols, x, 3, 6)
    assert np.array_equal(y_part[0, 3:6], y_all[0, 3:6])
    assert np.all(np.isnan(y_part[0, :3])) and np.all(np.isnan(y_part[0, 6:]))


def test_gemv_rejects_bad_shapes(orc):
    with pytest.raises(ValueError):
        orc.gemv(oracle.Q4_K, np.zeros(144, np.uint8), 1, 100, np.zeros((1, 100), np.float32))
