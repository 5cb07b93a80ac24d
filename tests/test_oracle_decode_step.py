"""Pins for the decode-step oracle (oracle/decode_step.py), CPU only.

Each check is fixed by the pages or by mathematics, not by re-typing the
oracle's formulas:
* rmsnorm: closed forms on constant vectors, scale invariance, unit mean square.
* RoPE ("S21 The Capstone: picoLM, in Python", section 3): position 0 is the
  identity; rotations preserve pair norms and add up over positions; pair i of a
  4-wide head turns by p / 100 at base 10000; the interleaved and NeoX layouts
  differ by more than 0.1 on the same input, and agree once the input is
  permuted, as the page says (the conversion permutes Q and K rows).
* Attention (same page, section 4): one key returns its value; equal keys
  return the mean value; a score gap of ln 3 gives weights 3/4 and 1/4 only if
  the scale is 1/sqrt(head_dim); query head h reads KV head h // kv_mul.
* SwiGLU: silu(0) = 0, silu(1) = 1/(1 + 1/e), silu(g) -> g and -> 0 at the tails.
* The whole step: zero-weight layers leave the embedding row to the head; at
  position 0 the query weights cannot matter (one key); a NeoX-rope model with
  permuted Q/K rows reproduces the interleaved model's logits; the cache of an
  earlier position is never rewritten and a replay of the prefix is identical.
"""
import numpy as np
import pytest

import oracle
from oracle import decode_step as ds
from quant_dequant_gemv_gb300 import synth


# -------------------------------------------------------------------- rmsnorm
def test_rmsnorm_constant_vector():
    w = np.linspace(0.5, 2.0, 64)
    for c in (3.0, -0.25):
        np.testing.assert_allclose(ds.rmsnorm(np.full(64, c), w, eps=0.0), np.sign(c) * w, rtol=1e-15)
        np.testing.assert_allclose(ds.rmsnorm(np.full(64, c), w, eps=1e-5), c / np.sqrt(c * c + 1e-5) * w,
                                   rtol=1e-15)


def test_rmsnorm_scale_invariant_unit_mean_square():
    rng = np.random.default_rng(0)
    x = rng.standard_normal(256)
    w = np.ones(256)
    y = ds.rmsnorm(x, w, eps=0.0)
    assert abs(np.mean(y * y) - 1.0) < 1e-14
    np.testing.assert_allclose(ds.rmsnorm(37.5 * x, w, eps=0.0), y, rtol=1e-14)


# ----------------------------------------------------------------------- RoPE
@pytest.mark.parametrize("rope", [ds.rope_interleaved, ds.rope_neox])
def test_rope_identity_norms_and_additivity(rope):
    rng = np.random.default_rng(1)
    v = rng.standard_normal(4 * 64)
    np.testing.assert_array_equal(rope(v, 4, 64, 0), v)
    r = rope(v, 4, 64, 7)
    if rope is ds.rope_interleaved:
        n0, n1 = v[0::2] ** 2 + v[1::2] ** 2, r[0::2] ** 2 + r[1::2] ** 2
    else:
        a, b = v.reshape(4, 64), r.reshape(4, 64)
        n0, n1 = a[:, :32] ** 2 + a[:, 32:] ** 2, b[:, :32] ** 2 + b[:, 32:] ** 2
    np.testing.assert_allclose(n1, n0, rtol=1e-12)
    np.testing.assert_allclose(rope(rope(v, 4, 64, 3), 4, 64, 4), r, rtol=1e-9, atol=1e-12)


def test_rope_pair_frequency_closed_form():
    # head_dim 4, base 10000: pair 0 turns by p radians, pair 1 by p / 100
    p = 5
    e = np.zeros(4)
    e[2] = 1.0  # interleaved: pair 1 is (v[2], v[3])
    np.testing.assert_allclose(ds.rope_interleaved(e, 1, 4, p), [0, 0, np.cos(p / 100), np.sin(p / 100)],
                               atol=1e-15)
    e = np.zeros(4)
    e[1] = 1.0  # NeoX: pair 1 is (v[1], v[3])
    np.testing.assert_allclose(ds.rope_neox(e, 1, 4, p), [0, np.cos(p / 100), 0, np.sin(p / 100)], atol=1e-15)
    e = np.zeros(4)
    e[0] = 1.0  # pair 0: p radians
    np.testing.assert_allclose(ds.rope_interleaved(e, 1, 4, p), [np.cos(p), np.sin(p), 0, 0], atol=1e-15)


def test_rope_layouts_differ_then_agree_after_permutation():
    rng = np.random.default_rng(2)
    H, D, pos = 2, 64, 9
    v = rng.standard_normal(H * D)
    a, b = ds.rope_interleaved(v, H, D, pos), ds.rope_neox(v, H, D, pos)
    assert np.max(np.abs(a - b)) > 0.1  # the page's check: the layouts are not interchangeable
    P = np.concatenate([h * D + ds.neox_to_interleaved_perm(D) for h in range(H)])
    np.testing.assert_allclose(ds.rope_interleaved(v[P], H, D, pos), b[P], rtol=1e-13, atol=1e-13)


# ------------------------------------------------------------------ attention
def _kv(npos, nkv, D, rng):
    return rng.standard_normal((npos, nkv, D)), rng.standard_normal((npos, nkv, D))


def test_attention_one_key_returns_value_and_gqa_mapping():
    rng = np.random.default_rng(3)
    H, G, D = 8, 2, 16
    K, V = _kv(4, G, D, rng)
    q = rng.standard_normal(H * D)
    out = ds.attention(q, K, V, 1, H, G, D).reshape(H, D)
    for h in range(H):
        np.testing.assert_allclose(out[h], V[0, h // (H // G)], rtol=1e-15)
    assert not np.allclose(out[1], V[0, 1])  # head 1 reads KV head 0, not 1


def test_attention_equal_keys_mean_and_scale():
    rng = np.random.default_rng(4)
    D = 16
    K = np.zeros((3, 1, D))
    V = rng.standard_normal((3, 1, D))
    q = rng.standard_normal(D)
    np.testing.assert_allclose(ds.attention(q, K, V, 3, 1, 1, D), V[:, 0].mean(axis=0), rtol=1e-14)
    # scores q.k0 * inv - q.k1 * inv = ln 3  =>  p = (3/4, 1/4)
    q = np.zeros(D)
    q[0] = 2.0
    K = np.zeros((2, 1, D))
    K[0, 0, 0] = np.log(3.0) * np.sqrt(D) / 2.0
    out = ds.attention(q, K, V[:2], 2, 1, 1, D)
    np.testing.assert_allclose(out, 0.75 * V[0, 0] + 0.25 * V[1, 0], rtol=1e-13)


# --------------------------------------------------------------------- SwiGLU
def test_silu_closed_forms():
    assert ds.silu(np.array([0.0]))[0] == 0.0
    assert abs(ds.silu(np.array([1.0]))[0] - 1.0 / (1.0 + np.exp(-1.0))) < 1e-16
    assert abs(ds.silu(np.array([40.0]))[0] - 40.0) < 1e-12
    assert abs(ds.silu(np.array([-40.0]))[0]) < 1e-15
    np.testing.assert_allclose(ds.swiglu(np.array([1.0, 2.0]), np.array([3.0, -1.0])),
                               [3.0 / (1.0 + np.exp(-1.0)), -2.0 / (1.0 + np.exp(-2.0))], rtol=1e-15)


# ------------------------------------------------------------- the whole step
CFG = dict(dim=256, hidden=512, n_layers=2, n_heads=4, n_kv_heads=2, vocab=300)


def _model(seed=5, zero=()):
    m = synth.gen_llama_model(seed=seed, **CFG)
    for lw in m["layers"]:
        for name in zero:  # all-zero blocks decode to w = 0 in every format
            t, r, c, b = lw[name]
            lw[name] = (t, r, c, np.zeros_like(b))
    cfg = ds.LlamaConfig(max_seq=8, **CFG)
    return cfg, m


def test_step_zero_layers_leave_embedding_to_head():
    cfg, m = _model(zero=("o", "down"))
    w = ds.from_blocks(cfg, m)
    kc, vc = ds.new_cache(cfg)
    tok = 17
    logits = ds.forward(w, kc, vc, tok, 0)
    t, r, c, b = m["token_embd"]
    row = oracle.dequant(t, b[tok * (b.size // r):(tok + 1) * (b.size // r)], c).astype(np.float64)
    xn = row / np.sqrt(np.mean(row * row) + cfg.eps) * m["output_norm"]
    ot, orows, ocols, ob = m["output"]
    y, _ = oracle.gemv(ot, ob, orows, ocols, xn.astype(np.float32)[None, :])
    # the oracle GEMV takes fp32 x: compare at fp32 resolution of the normalised row
    np.testing.assert_allclose(logits, y[0], rtol=1e-6, atol=1e-6 * np.abs(y).max())


def test_step_position_zero_ignores_query_weights():
    cfg, m = _model()
    a = ds.forward(ds.from_blocks(cfg, m), *ds.new_cache(cfg), 3, 0)
    for lw in m["layers"]:
        t, r, c, b = lw["q"]
        lw["q"] = (t, r, c, np.zeros_like(b))
    b0 = ds.forward(ds.from_blocks(cfg, m), *ds.new_cache(cfg), 3, 0)
    np.testing.assert_allclose(a, b0, rtol=1e-12)


def test_step_neox_model_with_permuted_rows_matches_interleaved():
    cfg, m = _model()
    toks = [5, 9, 2]
    ref = ds.from_blocks(cfg, m)
    kc, vc = ds.new_cache(cfg)
    want = [ds.forward(ref, kc, vc, t, p) for p, t in enumerate(toks)]
    # rows of Q and K reordered so that NeoX pairs (i, i + D/2) hold what the
    # interleaved pairs (2i, 2i + 1) held
    D = cfg.head_dim
    inv = np.argsort(ds.neox_to_interleaved_perm(D))
    for lw in m["layers"]:
        for name in ("q", "k"):
            t, r, c, b = lw[name]
            rb = b.size // r
            perm = np.concatenate([h * D + inv for h in range(r // D)])
            lw[name] = (t, r, c, b.reshape(r, rb)[perm].reshape(-1))
    perm_model = ds.from_blocks(cfg, m)
    orig = ds.rope_interleaved
    try:
        ds.rope_interleaved = ds.rope_neox
        kc, vc = ds.new_cache(cfg)
        got = [ds.forward(perm_model, kc, vc, t, p) for p, t in enumerate(toks)]
    finally:
        ds.rope_interleaved = orig
    for g, w_ in zip(got, want):
        np.testing.assert_allclose(g, w_, rtol=1e-9, atol=1e-9 * np.abs(w_).max())
    # and the wrong layout on the unpermuted weights does change the logits
    try:
        ds.rope_interleaved = ds.rope_neox
        kc, vc = ds.new_cache(cfg)
        bad = [ds.forward(ref, kc, vc, t, p) for p, t in enumerate(toks)]
    finally:
        ds.rope_interleaved = orig
    # (random weights make the softmax nearly one-hot, so the change is small, but
    # it is far above the float64 rounding that the permuted model agrees within)
    assert np.max(np.abs(bad[-1] - want[-1])) > 1e-6 * np.abs(want[-1]).max()


def test_step_cache_immutable_and_prefix_replay():
    cfg, m = _model()
    w = ds.from_blocks(cfg, m)
    kc, vc = ds.new_cache(cfg)
    first = [ds.forward(w, kc, vc, t, p) for p, t in enumerate([4, 8])]
    k0 = kc[:, 0].copy()
    ds.forward(w, kc, vc, 6, 2)
    np.testing.assert_array_equal(kc[:, 0], k0)
    kc2, vc2 = ds.new_cache(cfg)
    again = [ds.forward(w, kc2, vc2, t, p) for p, t in enumerate([4, 8])]
    for a, b in zip(first, again):
        np.testing.assert_array_equal(a, b)


def test_argmax_first_on_ties():
    assert ds.argmax_first(np.array([1.0, 3.0, 3.0, 2.0])) == 1
