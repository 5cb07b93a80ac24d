"""CPU oracle for the decode-step glue around the GEMVs: one token through a
Llama-architecture model, in float64 NumPy.

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg may import this module; the library's compute path
never does, and nothing here imports the library. Weights are decoded by the C
oracle (``oracle.dequant``), so every weight is the pages' fp32 value; all other
arithmetic is float64, one operation at a time, in the order the cited passages
give it.

Sources (page title, section):
  [S21-4]  "S21 The Capstone: picoLM, in Python", section 4 "The forward pass"
           (model_forward(m, token, pos): embedding row, per layer rmsnorm, q/k/v
           projections, rope, fp16 key/value cache at `pos`, per-head attention
           with GQA (KV head g = h // kv_mul) and scores scaled by `inv`, output
           projection, SwiGLU, residuals; final rmsnorm and output matmul).
  [S21-3]  same page, section 3, "The RoPE layout is not the one you learned":
           llama.cpp / picoLM rotate pairs (x[2i], x[2i+1]); GPT-NeoX rotates
           (x[i], x[i + D/2]); the two differ by a permutation of the Q and K rows.
  [PETIT]  "PETIT -- a tiny, CPU-first, quantized LLM inference engine", What makes
           it fast & small (RoPE + RMSNorm + SwiGLU, Llama-style block) and How the
           pieces match (RoPE base 10000, applied per head).

Readings where the pages leave a step open (each is listed with its reason in
the design notes):
  * rmsnorm(x, w) = x / sqrt(mean(x^2) + eps) * w with eps = 1e-5 (the pages give
    rmsnorm's signature, not its body or eps).
  * RoPE angle of pair i at position p: p * base^(-2i / head_dim), base = 10000
    (PETIT gives the base; the frequency ladder is the standard one).
  * Attention scale inv = 1 / sqrt(head_dim) (the page names `inv` only).
  * SwiGLU: silu(gate) * up, silu(g) = g / (1 + exp(-g)).
  * The key and value of the current position are rounded to fp16 before the
    attention that uses them, as the cache is written before it is read.

Pin status: every function here is pinned by tests/test_oracle_decode_step.py
against closed forms, invariants and the pages' own checks (RoPE layouts that
differ by more than 0.1 yet agree after the row permutation; attention over
one key returning its value; GQA head mapping; the softmax scale).
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

from . import dequant as _dequant

EPS = 1e-5
ROPE_BASE = 10000.0


# ---------------------------------------------------------------- elementwise ops
def rmsnorm(x: np.ndarray, w: np.ndarray, eps: float = EPS) -> np.ndarray:
    """x / sqrt(mean(x^2) + eps) * w  [S21-4 rmsnorm(out, x, weight, dim); PETIT RMSNorm]."""
    x = np.asarray(x, dtype=np.float64)
    ms = np.sum(x * x) / x.size
    return x / np.sqrt(ms + eps) * np.asarray(w, dtype=np.float64)


def silu(g: np.ndarray) -> np.ndarray:
    g = np.asarray(g, dtype=np.float64)
    with np.errstate(over="ignore"):  # exp(-g) = inf below g = -709: g / inf is the limit, -0
        return g / (1.0 + np.exp(-g))


def swiglu(gate: np.ndarray, up: np.ndarray) -> np.ndarray:
    """silu(gate) * up, the FFN activation of the Llama block [S21-4; PETIT SwiGLU]."""
    return silu(gate) * np.asarray(up, dtype=np.float64)


# ------------------------------------------------------------------------- RoPE
def rope_angles(head_dim: int, pos: int, base: float = ROPE_BASE) -> tuple[np.ndarray, np.ndarray]:
    """cos and sin of pair i's angle pos * base^(-2i/head_dim), i < head_dim / 2."""
    i = np.arange(head_dim // 2, dtype=np.float64)
    theta = pos * base ** (-2.0 * i / head_dim)
    return np.cos(theta), np.sin(theta)


def rope_interleaved(v: np.ndarray, n_heads: int, head_dim: int, pos: int,
                     base: float = ROPE_BASE) -> np.ndarray:
    """Rotate pairs (v[2i], v[2i+1]) of every head by angle i [S21-3, llama.cpp layout]."""
    v = np.asarray(v, dtype=np.float64).reshape(n_heads, head_dim)
    c, s = rope_angles(head_dim, pos, base)
    out = np.empty_like(v)
    a, b = v[:, 0::2], v[:, 1::2]
    out[:, 0::2] = a * c - b * s
    out[:, 1::2] = a * s + b * c
    return out.reshape(-1)


def rope_neox(v: np.ndarray, n_heads: int, head_dim: int, pos: int,
              base: float = ROPE_BASE) -> np.ndarray:
    """Rotate pairs (v[i], v[i + D/2]) of every head by angle i [S21-3, GPT-NeoX layout]."""
    v = np.asarray(v, dtype=np.float64).reshape(n_heads, head_dim)
    h = head_dim // 2
    c, s = rope_angles(head_dim, pos, base)
    out = np.empty_like(v)
    out[:, :h] = v[:, :h] * c - v[:, h:] * s
    out[:, h:] = v[:, h:] * c + v[:, :h] * s
    return out.reshape(-1)


def neox_to_interleaved_perm(head_dim: int) -> np.ndarray:
    """Index map P with (P v)[2i] = v[i], (P v)[2i+1] = v[i + D/2] inside one head: the
    row permutation that turns a NeoX-ordered Q or K projection into the
    interleaved one [S21-3]."""
    h = head_dim // 2
    src = np.empty(head_dim, dtype=np.int64)
    src[0::2] = np.arange(h)
    src[1::2] = np.arange(h) + h
    return src


# -------------------------------------------------------------------- attention
def softmax(s: np.ndarray) -> np.ndarray:
    s = np.asarray(s, dtype=np.float64)
    e = np.exp(s - np.max(s))
    return e / np.sum(e)


def attention(q: np.ndarray, k_cache: np.ndarray, v_cache: np.ndarray, npos: int,
              n_heads: int, n_kv_heads: int, head_dim: int) -> np.ndarray:
    """Per query head h: p = softmax(K_g q_h * inv) over positions < npos, out_h = p V_g,
    with g = h // (n_heads / n_kv_heads) and inv = 1/sqrt(head_dim) [S21-4].
    k_cache, v_cache: [positions][n_kv_heads][head_dim]."""
    kv_mul = n_heads // n_kv_heads
    inv = 1.0 / np.sqrt(head_dim)
    q = np.asarray(q, dtype=np.float64).reshape(n_heads, head_dim)
    K = np.asarray(k_cache, dtype=np.float64)[:npos]
    V = np.asarray(v_cache, dtype=np.float64)[:npos]
    out = np.empty((n_heads, head_dim))
    for h in range(n_heads):
        g = h // kv_mul
        scores = (K[:, g, :] @ q[h]) * inv
        out[h] = softmax(scores) @ V[:, g, :]
    return out.reshape(-1)


# ------------------------------------------------------------------------ model
@dataclass
class LlamaConfig:
    dim: int
    hidden: int
    n_layers: int
    n_heads: int
    n_kv_heads: int
    vocab: int
    max_seq: int
    rope_base: float = ROPE_BASE
    eps: float = EPS

    @property
    def head_dim(self) -> int:
        return self.dim // self.n_heads

    @property
    def kv_dim(self) -> int:
        return self.n_kv_heads * self.head_dim


@dataclass
class QMatrix:
    """A quantised weight matrix: rows x cols, raw blocks (uint8), block type."""
    qtype: int
    rows: int
    cols: int
    blocks: np.ndarray

    def dense(self) -> np.ndarray:
        return _dequant(self.qtype, self.blocks, self.rows * self.cols).astype(np.float64).reshape(self.rows, self.cols)

    def row(self, r: int) -> np.ndarray:
        rb = self.blocks.size // self.rows
        return _dequant(self.qtype, self.blocks[r * rb:(r + 1) * rb], self.cols).astype(np.float64)


@dataclass
class LlamaWeights:
    cfg: LlamaConfig
    token_embd: QMatrix            # vocab x dim
    layers: list[dict]             # per layer: q k v o gate up down (QMatrix), attn_norm ffn_norm (fp32)
    output_norm: np.ndarray
    output: QMatrix                # vocab x dim
    _dense: dict = field(default_factory=dict, repr=False)

    def w(self, l: int, name: str) -> np.ndarray:
        key = (l, name)
        if key not in self._dense:
            self._dense[key] = self.layers[l][name].dense()
        return self._dense[key]

    def head(self) -> np.ndarray:
        if "output" not in self._dense:
            self._dense["output"] = self.output.dense()
        return self._dense["output"]


def fp16_round(v: np.ndarray) -> np.ndarray:
    return np.asarray(v, dtype=np.float64).astype(np.float16)


def forward(m: LlamaWeights, k_cache: np.ndarray, v_cache: np.ndarray, token: int, pos: int,
            trace: dict | None = None, rows: dict | None = None) -> np.ndarray:
    """Logits of one token at position `pos` [S21-4 model_forward / forward].

    k_cache, v_cache: float16 [n_layers][max_seq][kv_dim]; entries of positions
    < pos are read, and position pos is written (the key after RoPE). If `trace`
    is a dict, the unrounded key and value of each layer, the residual stream
    after the last layer and its norm go into it.

    Rounding a key or value to fp16 is a decision on a discrete value: a kernel
    that computes k in fp32 can land on the neighbouring fp16 value when k sits
    near a rounding boundary. `rows` ({"k": [layer][kv_dim], "v": ...} fp16)
    gives the row each layer stores at `pos` instead of fp16(k), fp16(v), so a
    comparison takes that decision once, on the kernel's side, after checking
    the kernel's rows against the unrounded values traced here."""
    c = m.cfg
    x = m.token_embd.row(token)
    for l in range(c.n_layers):
        xb = rmsnorm(x, m.layers[l]["attn_norm"], c.eps)
        q = m.w(l, "q") @ xb
        k = m.w(l, "k") @ xb
        v = m.w(l, "v") @ xb
        q = rope_interleaved(q, c.n_heads, c.head_dim, pos, c.rope_base)
        k = rope_interleaved(k, c.n_kv_heads, c.head_dim, pos, c.rope_base)
        if trace is not None:
            trace.setdefault("k", []).append(k)
            trace.setdefault("v", []).append(v)
        k_cache[l, pos] = fp16_round(k) if rows is None else rows["k"][l]  # the cache is fp16
        v_cache[l, pos] = fp16_round(v) if rows is None else rows["v"][l]
        att = attention(q, k_cache[l].reshape(c.max_seq, c.n_kv_heads, c.head_dim),
                        v_cache[l].reshape(c.max_seq, c.n_kv_heads, c.head_dim), pos + 1,
                        c.n_heads, c.n_kv_heads, c.head_dim)
        x = x + m.w(l, "o") @ att
        xb = rmsnorm(x, m.layers[l]["ffn_norm"], c.eps)
        hb = swiglu(m.w(l, "gate") @ xb, m.w(l, "up") @ xb)
        x = x + m.w(l, "down") @ hb
    if trace is not None:
        trace["h"] = x
    xn = rmsnorm(x, m.output_norm, c.eps)
    if trace is not None:
        trace["hn"] = xn
    return m.head() @ xn


def argmax_first(v: np.ndarray) -> int:
    """Index of the largest value; the smallest such index on ties."""
    v = np.asarray(v)
    return int(np.flatnonzero(v == v.max())[0])


def from_blocks(cfg: LlamaConfig, m: dict) -> LlamaWeights:
    """LlamaWeights from a dict of raw blocks: token_embd / output as (type, rows,
    cols, blocks); layers as dicts of such tuples plus attn_norm / ffn_norm."""
    def qm(t):
        return QMatrix(int(t[0]), int(t[1]), int(t[2]), np.ascontiguousarray(t[3], dtype=np.uint8))
    layers = []
    for lw in m["layers"]:
        d = {k: qm(v) for k, v in lw.items() if k not in ("attn_norm", "ffn_norm")}
        d["attn_norm"] = np.asarray(lw["attn_norm"], dtype=np.float64)
        d["ffn_norm"] = np.asarray(lw["ffn_norm"], dtype=np.float64)
        layers.append(d)
    return LlamaWeights(cfg, qm(m["token_embd"]), layers, np.asarray(m["output_norm"], dtype=np.float64),
                        qm(m["output"]))


def new_cache(cfg: LlamaConfig) -> tuple[np.ndarray, np.ndarray]:
    shape = (cfg.n_layers, cfg.max_seq, cfg.kv_dim)
    return np.zeros(shape, dtype=np.float16), np.zeros(shape, dtype=np.float16)
