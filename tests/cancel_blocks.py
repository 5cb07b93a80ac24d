"""Q4_K blocks whose weights cancel, for the worst case of a factored dot product.

A Q4_K weight is w = d*sc*q - dmin*mn ("S21 The Capstone: picoLM, in Python",
section 2). A kernel that factors a sub-block as d*sc*sum(q x) - dmin*mn*sum(x)
subtracts two large, nearly equal sums when d*sc*q is close to dmin*mn for the
sub-block's quants. These blocks make that happen on purpose: each sub-block gets
a centre q_c with mn = sc*q_c (so that with dmin = d, dmin*mn = d*sc*q_c exactly)
and quants at or around q_c.

The fields are packed here from the layout description (six-bit scale and min
fields: sub-blocks 0-3 in the low six bits of bytes j and j+4, sub-blocks 4-7
split between the nibbles of byte j+4 and the top two bits of bytes j-4 / j;
chunk c of the nibble bytes holds sub-block 2c in its low nibbles and 2c+1 in its
high nibbles). Test input only: no decode arithmetic.
"""
from __future__ import annotations

import numpy as np

MODES = ("exact", "pm1", "near")


def _fp16_finite(rng, n, max_exp=29):
    """Random fp16 bit patterns with exponent field 1..max_exp and a random sign."""
    e = rng.integers(1, max_exp + 1, n).astype(np.uint16)
    f = rng.integers(0, 1024, n).astype(np.uint16)
    s = rng.integers(0, 2, n).astype(np.uint16)
    return (s << 15) | (e << 10) | f


def pack_scale_min(sc: np.ndarray, mn: np.ndarray) -> np.ndarray:
    """[n, 8] six-bit scales and mins -> [n, 12] packed bytes."""
    p = np.zeros((sc.shape[0], 12), dtype=np.uint16)
    for j in range(4):
        p[:, j] = (sc[:, j] & 63) | ((sc[:, j + 4] >> 4) << 6)
        p[:, j + 4] = (mn[:, j] & 63) | ((mn[:, j + 4] >> 4) << 6)
        p[:, j + 8] = (sc[:, j + 4] & 15) | ((mn[:, j + 4] & 15) << 4)
    return p.astype(np.uint8)


def q4k_cancelling_blocks(nblocks: int, rng: np.random.Generator, mode: str) -> np.ndarray:
    """`nblocks` Q4_K blocks as a flat uint8 array.

    mode "exact": dmin = d and every quant equals its sub-block's centre, so every
                  weight is exactly 0 (sum |w x| = 0).
    mode "pm1":   dmin = d and quants at centre - 1, centre, centre + 1 (clipped to
                  0..15): weights -d*sc, 0, +d*sc.
    mode "near":  every quant at the centre and dmin one fp16 step above d in
                  magnitude: every weight is the small rest -(dmin - d)*mn.
    """
    if mode not in MODES:
        raise ValueError(mode)
    d16 = _fp16_finite(rng, nblocks)
    dmin16 = d16 + 1 if mode == "near" else d16.copy()
    sc = rng.integers(1, 64, (nblocks, 8)).astype(np.uint16)
    qmax = np.minimum(15, 63 // sc)
    qc = (rng.random((nblocks, 8)) * (qmax + 1)).astype(np.uint16)
    mn = sc * qc
    q = np.repeat(qc, 32, axis=1).astype(np.int16)  # [n, 256], sub-block = e // 32
    if mode == "pm1":
        q = np.clip(q + rng.integers(-1, 2, q.shape), 0, 15)
    q = q.astype(np.uint8)
    qs = np.zeros((nblocks, 128), dtype=np.uint8)
    for c in range(4):
        qs[:, 32 * c:32 * c + 32] = q[:, 64 * c:64 * c + 32] | (q[:, 64 * c + 32:64 * c + 64] << 4)
    out = np.empty((nblocks, 144), dtype=np.uint8)
    out[:, 0:2] = d16.astype("<u2").view(np.uint8).reshape(-1, 2)
    out[:, 2:4] = dmin16.astype("<u2").view(np.uint8).reshape(-1, 2)
    out[:, 4:16] = pack_scale_min(sc, mn)
    out[:, 16:144] = qs
    return out.reshape(-1)
