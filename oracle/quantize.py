"""CPU oracle for the quantiser (fp32 -> PETIT q8_0 / q4_0 blocks).

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg may import this module; the library never does.

Source: "PETIT -- a tiny, CPU-first, quantized LLM inference engine", What makes
it fast & small (q8_0: every 32 weights share one fp32 scale, stored as int8;
q4_0: the same block scheme with an fp16 scale and 4-bit nibbles, 18 bytes per
block) and How the pieces match (the exporter writes q8_0 blocks of an fp32
scale followed by 32 int8 values, zero-padded to a multiple of 32; q4_0 blocks of
an fp16 scale and 16 nibble bytes; the engine reads q4_0 as (q - 8) * d with
weights 0..15 in the low nibbles).

The scale rule is not on the pages. Reading (symmetric, round to nearest):
  q8_0: amax = max |x_i|; d = amax / 127; q_i = clamp(rint(x_i / d), -127, 127)
        (q = 0 when d = 0). Store d as fp32.
  q4_0: amax = max |x_i|; d = fp16(amax / 7); q_i = clamp(rint(x_i / d) + 8, 0, 15)
        with d the stored fp16 value (q = 8 when d = 0).
Every step is binary32 arithmetic (the division correctly rounded, rint halves to
even), because each quant is a discrete value that floating point decides: the
kernel takes the same decisions in the same precision.

Pins (tests/test_oracle_quantize.py): dequantising with the C oracle returns each
x within d/2; multiples of d come back exactly; the largest |x| lands on +-127 /
+-7; halves round to even; an all-zero block gives d = 0; padding to 32 is zeros.
"""
from __future__ import annotations

import numpy as np

QK = 32


def _blocks(x: np.ndarray) -> np.ndarray:
    x = np.asarray(x, dtype=np.float32).reshape(-1)
    pad = (-x.size) % QK  # the exporter zero-pads to a multiple of 32
    if pad:
        x = np.concatenate([x, np.zeros(pad, dtype=np.float32)])
    return x.reshape(-1, QK)


def quantize_q8_0(x: np.ndarray) -> np.ndarray:
    """fp32 values -> q8_0 blocks (fp32 d + 32 int8), as a flat uint8 array."""
    xb = _blocks(x)
    out = np.empty((xb.shape[0], 36), dtype=np.uint8)
    for b in range(xb.shape[0]):
        v = xb[b]
        amax = np.float32(np.max(np.abs(v)))
        d = np.float32(amax / np.float32(127.0))
        if d == 0:
            q = np.zeros(QK, dtype=np.int8)
        else:
            q = np.clip(np.rint(v / d), -127, 127).astype(np.int8)
        out[b, 0:4] = np.array([d], dtype="<f4").view(np.uint8)
        out[b, 4:36] = q.view(np.uint8)
    return out.reshape(-1)


def quantize_q4_0(x: np.ndarray) -> np.ndarray:
    """fp32 values -> q4_0 blocks (fp16 d + 16 nibble bytes), as a flat uint8 array."""
    xb = _blocks(x)
    out = np.empty((xb.shape[0], 18), dtype=np.uint8)
    for b in range(xb.shape[0]):
        v = xb[b]
        amax = np.float32(np.max(np.abs(v)))
        with np.errstate(over="ignore"):  # amax / 7 above 65504 has no finite fp16 scale: d = inf
            d16 = np.float16(np.float32(amax / np.float32(7.0)))
        d = np.float32(d16)
        if d == 0:
            q = np.full(QK, 8, dtype=np.uint8)
        else:
            q = np.clip(np.rint(v / d) + 8, 0, 15).astype(np.uint8)
        out[b, 0:2] = np.array([d16], dtype="<f2").view(np.uint8)
        out[b, 2:18] = q[:16] | (q[16:] << 4)
    return out.reshape(-1)
