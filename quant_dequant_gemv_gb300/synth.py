"""Seeded synthetic inputs: raw quantised blocks and fp32 activation vectors.

This module only lays random numbers out at the byte offsets of each block
format. It holds none of the decode or dot-product arithmetic, so both the CPU
oracle tests and the CUDA path can take their inputs from it.

Why uniform random bytes are the right draw:

* Q4_K ("S21 The Capstone: picoLM, in Python", section 2, the Q4_K super-block
  diagram and dequantize_q4_K): bytes 4..15 pack eight 6-bit scales and eight
  6-bit mins. Every one of the 96 bits belongs to exactly one field, so uniform
  random bytes give independent uniform fields in 0..63. The 128 nibble bytes
  give independent uniform nibbles in 0..15.
* Q6_K ("PicoLM Q6_K quantisation bug", the block_q6_K struct): ql[128] and
  qh[64] hold disjoint bits of each 6-bit quant, so random bytes give uniform
  quants in 0..63. scales[16] read as int8 are then uniform in -128..127.
* PETIT q4_0 ("PETIT", "How the pieces match"): fp16 scale + 16 nibble bytes.
* PETIT q8_0 (same section): fp32 scale + 32 int8, drawn in -127..127.

The scales d (and dmin) are drawn from U[1e-4, 1e-2] and rounded to fp16 by
numpy (round to nearest even); q8_0 keeps its scale in fp32.
"""
from __future__ import annotations

import hashlib
from dataclasses import dataclass

import numpy as np

# Type codes of the C ABI (include/qdq.h).
Q4_0 = 1
Q8_0 = 2  # PETIT q8_0: fp32 scale + 32 int8
Q4_K = 3
Q6_K = 4
# More GGUF block formats (ggml layouts): Q5_0 (22 B / 32), Q5_1 (24 B / 32),
# ggml's q8_0 with an fp16 scale (34 B / 32), Q2_K (84 B / 256), Q5_K (176 B /
# 256), Q3_K (110 B / 256).
Q5_0 = 5
Q5_1 = 6
Q8_0G = 7
Q2_K = 8
Q5_K = 9
Q3_K = 10

TYPE_NAMES = {Q4_0: "q4_0", Q8_0: "q8_0", Q4_K: "Q4_K", Q6_K: "Q6_K", Q5_0: "Q5_0", Q5_1: "Q5_1",
              Q8_0G: "q8_0 (ggml)", Q2_K: "Q2_K", Q5_K: "Q5_K", Q3_K: "Q3_K"}
BLOCK_BYTES = {Q4_0: 18, Q8_0: 36, Q4_K: 144, Q6_K: 210, Q5_0: 22, Q5_1: 24, Q8_0G: 34, Q2_K: 84, Q5_K: 176,
               Q3_K: 110}
BLOCK_WEIGHTS = {Q4_0: 32, Q8_0: 32, Q4_K: 256, Q6_K: 256, Q5_0: 32, Q5_1: 32, Q8_0G: 32, Q2_K: 256, Q5_K: 256,
                 Q3_K: 256}

SCALE_LO, SCALE_HI = 1e-4, 1e-2


def row_bytes(qtype: int, cols: int) -> int:
    return (cols // BLOCK_WEIGHTS[qtype]) * BLOCK_BYTES[qtype]


def _fp16_bytes(v: np.ndarray) -> np.ndarray:
    return v.astype("<f2").view(np.uint8).reshape(-1, 2)


def gen_blocks(qtype: int, nblocks: int, rng: np.random.Generator) -> np.ndarray:
    """Return `nblocks` random blocks of `qtype` as a flat uint8 array."""
    bb = BLOCK_BYTES[qtype]
    out = np.empty((nblocks, bb), dtype=np.uint8)
    if qtype in (Q4_K, Q5_K):  # fp16 d, dmin, then scale/min fields and quant bytes
        d = rng.uniform(SCALE_LO, SCALE_HI, nblocks)
        dmin = rng.uniform(SCALE_LO, SCALE_HI, nblocks)
        out[:, 0:2] = _fp16_bytes(d)
        out[:, 2:4] = _fp16_bytes(dmin)
        out[:, 4:bb] = rng.integers(0, 256, (nblocks, bb - 4), dtype=np.uint8)
    elif qtype == Q3_K:  # hmask, 2-bit quants, scale fields, then fp16 d
        out[:, 0:108] = rng.integers(0, 256, (nblocks, 108), dtype=np.uint8)
        out[:, 108:110] = _fp16_bytes(rng.uniform(SCALE_LO, SCALE_HI, nblocks))
    elif qtype == Q6_K:
        d = rng.uniform(SCALE_LO, SCALE_HI, nblocks)
        out[:, 0:208] = rng.integers(0, 256, (nblocks, 208), dtype=np.uint8)
        out[:, 208:210] = _fp16_bytes(d)
    elif qtype == Q8_0:
        d = rng.uniform(SCALE_LO, SCALE_HI, nblocks).astype("<f4")
        out[:, 0:4] = d.view(np.uint8).reshape(-1, 4)
        out[:, 4:36] = rng.integers(-127, 128, (nblocks, 32)).astype(np.int8).view(np.uint8)
    elif qtype in (Q4_0, Q5_0, Q8_0G):  # fp16 d, then quant bytes
        d = rng.uniform(SCALE_LO, SCALE_HI, nblocks)
        out[:, 0:2] = _fp16_bytes(d)
        out[:, 2:bb] = rng.integers(0, 256, (nblocks, bb - 2), dtype=np.uint8)
    elif qtype == Q5_1:  # fp16 d, fp16 m (a negative offset of the range), quant bytes
        d = rng.uniform(SCALE_LO, SCALE_HI, nblocks)
        out[:, 0:2] = _fp16_bytes(d)
        out[:, 2:4] = _fp16_bytes(-16 * d * rng.uniform(0.5, 1.5, nblocks))
        out[:, 4:24] = rng.integers(0, 256, (nblocks, 20), dtype=np.uint8)
    elif qtype == Q2_K:  # scale/min nibbles and 2-bit quants, then fp16 d, dmin
        out[:, 0:80] = rng.integers(0, 256, (nblocks, 80), dtype=np.uint8)
        out[:, 80:82] = _fp16_bytes(rng.uniform(SCALE_LO, SCALE_HI, nblocks))
        out[:, 82:84] = _fp16_bytes(rng.uniform(SCALE_LO, SCALE_HI, nblocks))
    else:
        raise ValueError(f"unknown block type {qtype}")
    return out.reshape(-1)


def gen_blocks_full_range(qtype: int, nblocks: int, rng: np.random.Generator) -> np.ndarray:
    """Uniform random bytes in every field of every block, except that the scales
    stay finite and bounded: an fp16 scale (Q4_K d and dmin, Q6_K d, q4_0 d) whose
    exponent field is all ones (inf/NaN) gets exponent 30 instead, and the fp32
    scale of q8_0 keeps an exponent field of at most 200 (|d| < 2^74), so that no
    dot product over a row overflows fp32. Everything else covers its full range:
    negative, subnormal and zero scales, 6-bit Q4_K scales and mins 0..63, int8
    Q6_K scales down to -128, q8_0 quants down to -128."""
    bb = BLOCK_BYTES[qtype]
    out = rng.integers(0, 256, (nblocks, bb), dtype=np.uint8)

    def clamp_fp16(col: int) -> None:
        h = out[:, col].astype(np.uint16) | (out[:, col + 1].astype(np.uint16) << 8)
        inf_nan = ((h >> 10) & 31) == 31
        h = np.where(inf_nan, h & ~np.uint16(0x0400), h)
        out[:, col] = (h & 0xFF).astype(np.uint8)
        out[:, col + 1] = (h >> 8).astype(np.uint8)

    if qtype in (Q4_K, Q5_K):
        clamp_fp16(0)
        clamp_fp16(2)
    elif qtype == Q3_K:
        clamp_fp16(108)
    elif qtype == Q6_K:
        clamp_fp16(208)
    elif qtype in (Q4_0, Q5_0, Q8_0G):
        clamp_fp16(0)
    elif qtype == Q5_1:
        clamp_fp16(0)
        clamp_fp16(2)
    elif qtype == Q2_K:
        clamp_fp16(80)
        clamp_fp16(82)
    elif qtype == Q8_0:
        w = out[:, 0:4].copy().view("<u4").reshape(-1)
        e = (w >> 23) & 0xFF
        w = np.where(e > 200, (w & ~np.uint32(0x7F800000)) | np.uint32(200 << 23), w)
        out[:, 0:4] = w.astype("<u4").view(np.uint8).reshape(-1, 4)
    else:
        raise ValueError(f"unknown block type {qtype}")
    return out.reshape(-1)


def gen_matrix(qtype: int, rows: int, cols: int, seed: int) -> np.ndarray:
    """A rows x cols weight matrix: row-major, each row a run of whole blocks."""
    if cols % BLOCK_WEIGHTS[qtype]:
        raise ValueError("cols must be a multiple of the block size")
    rng = np.random.default_rng(seed)
    return gen_blocks(qtype, rows * (cols // BLOCK_WEIGHTS[qtype]), rng)


def gen_x(batch: int, cols: int, seed: int) -> np.ndarray:
    """Activations x ~ N(0, 1), fp32, laid out [batch][cols]."""
    rng = np.random.default_rng(seed)
    return rng.standard_normal((batch, cols), dtype=np.float32)


def digest(a: np.ndarray) -> str:
    return hashlib.sha256(np.ascontiguousarray(a).view(np.uint8)).hexdigest()[:16]


# ---------------------------------------------------------------------------
# Workload shapes. Seeds: tensor t of a workload uses seed base + t, and its
# activation vector uses seed base + 1000 + t.
# ---------------------------------------------------------------------------
@dataclass(frozen=True)
class Gemv:
    name: str
    qtype: int
    rows: int
    cols: int

    @property
    def weight_bytes(self) -> int:
        return self.rows * row_bytes(self.qtype, self.cols)


# Single GEMVs.
Q4K_2048x2048 = Gemv("Q4_K 2048x2048", Q4_K, 2048, 2048)
Q6K_2048x5632 = Gemv("Q6_K 2048x5632 (ffn_down)", Q6_K, 2048, 5632)

# 1.1B Llama shape, Q4_K_M mix: hidden 2048, 32 q heads / 4 kv heads of 64,
# FFN 5632, vocab 32000, 22 layers.
LLAMA_1B = dict(n_layers=22, hidden=2048, n_heads=32, n_kv_heads=4, head_dim=64,
                ffn=5632, vocab=32000)


def llama_1b_layer(l: int) -> list[Gemv]:
    h, kv, f = 2048, 4 * 64, 5632
    return [
        Gemv(f"blk.{l}.attn_q", Q4_K, h, h),
        Gemv(f"blk.{l}.attn_k", Q4_K, kv, h),
        Gemv(f"blk.{l}.attn_v", Q6_K, kv, h),
        Gemv(f"blk.{l}.attn_output", Q4_K, h, h),
        Gemv(f"blk.{l}.ffn_gate", Q4_K, f, h),
        Gemv(f"blk.{l}.ffn_up", Q4_K, f, h),
        Gemv(f"blk.{l}.ffn_down", Q6_K, h, f),
    ]


def llama_1b_step(n_layers: int = 22) -> list[list[Gemv]]:
    """The GEMVs of one decode step, grouped into dependency levels.

    Within a level the GEMVs read the same input vector in a real forward pass
    ({q,k,v} read rmsnorm(x); {gate,up} read rmsnorm(h)); each level depends on
    the previous one. The output head is the last level.
    """
    levels: list[list[Gemv]] = []
    for l in range(n_layers):
        q, k, v, o, g, u, d = llama_1b_layer(l)
        levels += [[q, k, v], [o], [g, u], [d]]
    levels.append([Gemv("output", Q6_K, LLAMA_1B["vocab"], LLAMA_1B["hidden"])])
    return levels


def step_weight_bytes(levels: list[list[Gemv]]) -> int:
    return sum(g.weight_bytes for lv in levels for g in lv)


# ---------------------------------------------------------------------------
# A whole Llama-architecture model of random blocks, for the decode-step glue.
# Tensor types follow the Q4_K_M mix above; norm weights are fp32 ~ U[0.5, 1.5].
# ---------------------------------------------------------------------------
LAYER_TENSORS = ("q", "k", "v", "o", "gate", "up", "down")
LAYER_TYPES = {"q": Q4_K, "k": Q4_K, "v": Q6_K, "o": Q4_K, "gate": Q4_K, "up": Q4_K, "down": Q6_K}


def llama_shapes(dim: int, hidden: int, n_heads: int, n_kv_heads: int) -> dict:
    """(rows, cols) of each layer tensor: weights stored out x in."""
    kv = n_kv_heads * (dim // n_heads)
    return {"q": (dim, dim), "k": (kv, dim), "v": (kv, dim), "o": (dim, dim),
            "gate": (hidden, dim), "up": (hidden, dim), "down": (dim, hidden)}


def gen_llama_model(dim: int, hidden: int, n_layers: int, n_heads: int, n_kv_heads: int, vocab: int,
                    seed: int, embd_type: int = Q4_K, out_type: int = Q6_K, norm_scale: float = 1.0,
                    layer_types: dict | None = None) -> dict:
    """Raw blocks of every tensor and the fp32 norm vectors (times norm_scale), from one seed.

    With the workload's block draws a weight is of order 1, so q.k scores reach
    thousands and the softmax is one-hot; a norm_scale of about 0.02 keeps the
    scores of order 1 (every position then weighs in)."""
    rng = np.random.default_rng(seed)
    shapes = llama_shapes(dim, hidden, n_heads, n_kv_heads)
    m = {"token_embd": (embd_type, vocab, dim, gen_blocks(embd_type, vocab * dim // BLOCK_WEIGHTS[embd_type], rng)),
         "layers": []}
    for _ in range(n_layers):
        lw = {}
        for name in LAYER_TENSORS:
            r, c = shapes[name]
            t = (layer_types or LAYER_TYPES)[name]
            lw[name] = (t, r, c, gen_blocks(t, r * c // BLOCK_WEIGHTS[t], rng))
        lw["attn_norm"] = (norm_scale * rng.uniform(0.5, 1.5, dim)).astype(np.float32)
        lw["ffn_norm"] = (norm_scale * rng.uniform(0.5, 1.5, dim)).astype(np.float32)
        m["layers"].append(lw)
    m["output_norm"] = (norm_scale * rng.uniform(0.5, 1.5, dim)).astype(np.float32)
    m["output"] = (out_type, vocab, dim, gen_blocks(out_type, vocab * dim // BLOCK_WEIGHTS[out_type], rng))
    return m
