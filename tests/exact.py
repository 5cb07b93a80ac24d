"""Test-side helpers that restate the block layouts as bit tables and evaluate the
formats' formulas in exact rational arithmetic.

They are written from the pages' layout descriptions independently of the
oracle's C code, so that the oracle can be pinned against them.
"""
from __future__ import annotations

from fractions import Fraction

import numpy as np


# -- binary16 / binary32 from their definitions --------------------------------
def fp16_value(h: int) -> Fraction | float:
    """Exact value of an IEEE binary16 pattern (inf/nan returned as floats)."""
    s, e, f = (h >> 15) & 1, (h >> 10) & 31, h & 1023
    if e == 31:
        return float("nan") if f else (float("-inf") if s else float("inf"))
    v = Fraction(f, 1 << 24) if e == 0 else Fraction(1024 + f) * Fraction(2) ** (e - 25)
    return -v if s else v


def round_f32(v: Fraction) -> np.float32:
    """Correctly rounded binary32 (round to nearest, ties to even)."""
    if v == 0:
        return np.float32(0.0)
    c = np.float32(float(v))
    if not np.isfinite(c):
        return c
    cands = [np.nextafter(c, np.float32(-np.inf)), c, np.nextafter(c, np.float32(np.inf))]
    best, best_err = None, None
    for k in cands:
        if not np.isfinite(k):
            continue
        err = abs(Fraction(float(k)) - v)
        if best is None or err < best_err or (
                err == best_err and (int(np.float32(k).view(np.uint32)) & 1) == 0):
            best, best_err = k, err
    return np.float32(best)


# -- Q4_K: the 12 packed bytes as a bit table -------------------------------------
# S21 section 2: eight 6-bit scales and eight 6-bit mins in 12 bytes. Sub-blocks
# 0-3 keep both fields in the low six bits of their own byte (scale in byte j, min
# in byte j+4). Sub-blocks 4-7 keep the low four bits in byte j+4 (scale in its
# low nibble, min in its high nibble) and the top two bits in bits 6-7 of byte j-4
# (scale) or byte j (min).
def q4k_bit_table() -> dict[tuple[str, int], list[tuple[int, int]]]:
    t = {}
    for j in range(8):
        if j < 4:
            t[("sc", j)] = [(j, b) for b in range(6)]
            t[("mn", j)] = [(j + 4, b) for b in range(6)]
        else:
            t[("sc", j)] = [(j + 4, b) for b in range(4)] + [(j - 4, 6), (j - 4, 7)]
            t[("mn", j)] = [(j + 4, 4 + b) for b in range(4)] + [(j, 6), (j, 7)]
    return t


Q4K_TABLE = q4k_bit_table()


def q4k_unpack(p12) -> tuple[list[int], list[int]]:
    p = [int(b) for b in p12]
    sc, mn = [], []
    for j in range(8):
        for kind, dst in (("sc", sc), ("mn", mn)):
            v = 0
            for i, (byte, bit) in enumerate(Q4K_TABLE[(kind, j)]):
                v |= ((p[byte] >> bit) & 1) << i
            dst.append(v)
    return sc, mn


def q4k_pack(sc, mn) -> bytes:
    p = [0] * 12
    for j in range(8):
        for kind, vals in (("sc", sc), ("mn", mn)):
            for i, (byte, bit) in enumerate(Q4K_TABLE[(kind, j)]):
                p[byte] |= ((vals[j] >> i) & 1) << bit
    return bytes(p)


def q4k_nibble(e: int) -> tuple[int, int]:
    """(byte index into the 128 nibble bytes, shift) of weight e; sub-block = e // 32."""
    c, i = divmod(e, 64)
    return 32 * c + (i % 32), (0 if i < 32 else 4)


def q4k_block(d16: int, dmin16: int, sc, mn, q) -> bytes:
    """Assemble a Q4_K block from fields; q = 256 nibbles in weight order."""
    qs = [0] * 128
    for e in range(256):
        b, sh = q4k_nibble(e)
        qs[b] |= (q[e] & 15) << sh
    return (d16.to_bytes(2, "little") + dmin16.to_bytes(2, "little") + q4k_pack(sc, mn)
            + bytes(qs))


def q4k_fields(blk) -> tuple:
    blk = bytes(blk)
    d16 = int.from_bytes(blk[0:2], "little")
    dmin16 = int.from_bytes(blk[2:4], "little")
    sc, mn = q4k_unpack(blk[4:16])
    qs = blk[16:144]
    q = []
    for e in range(256):
        b, sh = q4k_nibble(e)
        q.append((qs[b] >> sh) & 15)
    return d16, dmin16, sc, mn, q


def q4k_exact(blk) -> list[Fraction]:
    """Exact real values d*sc*q - dmin*mn for a block with finite d, dmin."""
    d16, dmin16, sc, mn, q = q4k_fields(blk)
    d, dmin = fp16_value(d16), fp16_value(dmin16)
    return [d * sc[e // 32] * q[e] - dmin * mn[e // 32] for e in range(256)]


# -- Q6_K: ql[128] qh[64] scales[16] d ------------------------------------------------
# Struct offsets from the block_q6_K struct; one int8 scale per 16 weights. The
# element -> (ql, qh) bit placement is the ggml layout (a reading; the pages do not
# print it): element e = 128h + 32k + l takes its low four bits from
# ql[64h + 32(k&1) + l] (low nibble for k < 2, high nibble for k >= 2) and its top
# two bits from bits 2k, 2k+1 of qh[32h + l].
def q6k_place(e: int) -> tuple[int, int, int, int]:
    h, r = divmod(e, 128)
    k, l = divmod(r, 32)
    return 64 * h + 32 * (k & 1) + l, (0 if k < 2 else 4), 32 * h + l, 2 * k


def q6k_block(d16: int, scales, q6) -> bytes:
    """Assemble a Q6_K block; q6 = 256 unsigned 6-bit values (q + 32)."""
    ql, qh = [0] * 128, [0] * 64
    for e in range(256):
        bl, sl, bh, sh = q6k_place(e)
        ql[bl] |= (q6[e] & 15) << sl
        qh[bh] |= ((q6[e] >> 4) & 3) << sh
    sc = bytes((s & 0xFF) for s in scales)
    return bytes(ql) + bytes(qh) + sc + d16.to_bytes(2, "little")


def q6k_fields(blk) -> tuple:
    blk = bytes(blk)
    q6 = []
    for e in range(256):
        bl, sl, bh, sh = q6k_place(e)
        q6.append(((blk[bl] >> sl) & 15) | (((blk[128 + bh] >> sh) & 3) << 4))
    scales = [int(np.int8(np.uint8(b))) for b in blk[192:208]]
    return int.from_bytes(blk[208:210], "little"), scales, q6


def q6k_exact(blk) -> list[Fraction]:
    d16, scales, q6 = q6k_fields(blk)
    d = fp16_value(d16)
    return [d * scales[e // 16] * (q6[e] - 32) for e in range(256)]


# -- PETIT q8_0 / q4_0 ------------------------------------------------------------------
def q8_0_exact(blk) -> list[Fraction]:
    blk = bytes(blk)
    d = Fraction(float(np.frombuffer(blk[0:4], dtype="<f4")[0]))
    return [d * int(np.int8(np.uint8(b))) for b in blk[4:36]]


def q4_0_exact(blk) -> list[Fraction]:
    blk = bytes(blk)
    d = fp16_value(int.from_bytes(blk[0:2], "little"))
    qs = blk[2:18]
    return [(((qs[i % 16] >> (0 if i < 16 else 4)) & 15) - 8) * d for i in range(32)]
