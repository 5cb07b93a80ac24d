"""The decode-step glue on the GPU against the oracle (oracle/decode_step.py).

* Plan options: a GEMV reading rmsnorm(x), silu(gate) * up or gate * up, writing
  y += W x or silu(W x), and the output head's fused argmax. The GEMV bound is the one every GEMV test
  uses, |y - y_ref| <= 1e-5 sum|w x'| + 1e-7, with x' the oracle's input in
  double precision (the prologue's own fp32 rounding is far inside it).
* qdq_rope_attention: the cache row it writes equals fp16 of the oracle's turned
  key (within one fp16 step: the fp32 and float64 keys can round to neighbouring
  fp16 values), and its output matches the oracle's attention over the GPU's own
  cache within 1e-5 of the largest |v|.
* The token step (qdq_llama): positions 0..4 of a two-layer model. Each fp16
  cache row the GPU writes lies within one fp16 step of the oracle's key or
  value (plus 1e-5 of the row's largest entry, for the fp32 GEMV before it);
  the oracle then takes those rows as its cache (rounding to fp16 decides a
  discrete value: both sides must take the decision once, the same way). Logits
  within 1e-4 of the head row's sum|w x| (two layers of GEMVs within 1e-5
  each, fp32 norms and attention), the argmax equal to that of the GPU's own
  logits.
"""
import numpy as np
import pytest

import oracle
from oracle import decode_step as ds
from quant_dequant_gemv_gb300 import synth

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def q():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from quant_dequant_gemv_gb300 import build, qdq
    build.build()
    torch.cuda.set_device(0)
    return qdq


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def assert_gemv_close(y, y_ref, S, what, extra=0.0):
    ok = np.abs(np.asarray(y, np.float64) - y_ref) <= 1e-5 * S + 1e-7 + extra
    if not ok.all():
        i = int(np.argwhere(~ok)[0][0])
        raise AssertionError(f"{what}: {int((~ok).sum())} out of tolerance; first {i}: {y[i]} vs {y_ref[i]}")


@pytest.mark.parametrize("qtype,rows,cols", [(synth.Q4_K, 300, 2048), (synth.Q6_K, 97, 5632), (synth.Q8_0, 64, 4096)])
def test_plan_rmsnorm_prologue(q, qtype, rows, cols):
    rng = np.random.default_rng(qtype * 7 + rows)
    W = synth.gen_matrix(qtype, rows, cols, 11)
    x = (rng.standard_normal(cols) * 3.0).astype(np.float32)
    w = rng.uniform(0.5, 1.5, cols).astype(np.float32)
    y = torch.full((1, rows), float("nan"), device="cuda")
    xd, wd = dev(x[None, :]), dev(w)
    plan = q.Plan([(qtype, dev(W), rows, cols, xd, y)], [0], 1,
                  opts=[{"x_op": q.X_RMSNORM, "norm_w": wd, "eps": 1e-5}])
    plan.run()
    assert q.get_device_status() == 0
    xn = ds.rmsnorm(x, w, 1e-5)
    y_ref, S = oracle.gemv(qtype, W, rows, cols, xn.astype(np.float32)[None, :])
    assert_gemv_close(y.cpu().numpy()[0], y_ref[0], S[0], "rmsnorm prologue")
    plan.close()


def test_plan_swiglu_prologue_and_residual_add(q):
    rng = np.random.default_rng(21)
    rows, cols = 2048, 5632
    W = synth.gen_matrix(synth.Q6_K, rows, cols, 12)
    g = (rng.standard_normal(cols) * 4).astype(np.float32)
    u = rng.standard_normal(cols).astype(np.float32)
    h0 = rng.standard_normal(rows).astype(np.float32) * 100
    y = dev(h0[None, :].copy())
    plan = q.Plan([(synth.Q6_K, dev(W), rows, cols, dev(g[None, :]), y)], [0], 1,
                  opts=[{"x_op": q.X_SWIGLU, "x2": dev(u[None, :]), "y_op": q.Y_ADD}])
    plan.run()
    assert q.get_device_status() == 0
    xs = ds.swiglu(g, u)
    y_ref, S = oracle.gemv(synth.Q6_K, W, rows, cols, xs.astype(np.float32)[None, :])
    # y = h0 + W x': the one extra fp32 addition rounds at |y| 2^-24
    got = y.cpu().numpy()[0]
    assert_gemv_close(got, y_ref[0] + h0, S[0], "swiglu + residual", extra=np.abs(got) * 2.0 ** -23)
    plan.close()


def test_plan_silu_store_then_product_stage(q):
    """gate stored through silu (Y_SILU) and up from rmsnorm(h); down reads
    gate * up (X_MUL) and adds into h: SwiGLU split between the two levels."""
    rng = np.random.default_rng(41)
    dim, hid = 2048, 5632
    Wg, Wu, Wd = (synth.gen_matrix(t, r, c, s) for t, r, c, s in
                  [(synth.Q4_K, hid, dim, 5), (synth.Q4_K, hid, dim, 6), (synth.Q6_K, dim, hid, 7)])
    h0 = rng.standard_normal(dim).astype(np.float32)
    nw = rng.uniform(0.5, 1.5, dim).astype(np.float32)
    h = dev(h0[None, :].copy())
    gbuf = torch.zeros(1, hid, device="cuda")
    ubuf = torch.zeros(1, hid, device="cuda")
    nwd = dev(nw)
    items = [(synth.Q4_K, dev(Wg), hid, dim, h, gbuf), (synth.Q4_K, dev(Wu), hid, dim, h, ubuf),
             (synth.Q6_K, dev(Wd), dim, hid, gbuf, h)]
    opts = [{"x_op": q.X_RMSNORM, "norm_w": nwd, "eps": 1e-5, "y_op": q.Y_SILU},
            {"x_op": q.X_RMSNORM, "norm_w": nwd, "eps": 1e-5},
            {"x_op": q.X_MUL, "x2": ubuf, "y_op": q.Y_ADD}]
    plan = q.Plan(items, [0, 0, 1], 1, opts=opts)
    plan.run()
    assert q.get_device_status() == 0
    g_gpu, u_gpu, h_gpu = gbuf.cpu().numpy()[0], ubuf.cpu().numpy()[0], h.cpu().numpy()[0]
    xn = ds.rmsnorm(h0, nw, 1e-5).astype(np.float32)[None, :]
    gr, gS = oracle.gemv(synth.Q4_K, Wg, hid, dim, xn)
    ur, uS = oracle.gemv(synth.Q4_K, Wu, hid, dim, xn)
    # silu has slope below 1.1: the GEMV bound carries over, plus the fp32 rounding
    # of silu itself (exp and the division, a few units of 2^-24)
    assert_gemv_close(g_gpu, ds.silu(gr[0]), 1.1 * gS[0], "silu(gate)", extra=np.abs(g_gpu) * 2.0 ** -20)
    assert_gemv_close(u_gpu, ur[0], uS[0], "up")
    # down reads the GPU's gate * up, each product rounded once to fp32
    xm = (g_gpu.astype(np.float64) * u_gpu).astype(np.float32)[None, :]
    dr, dS = oracle.gemv(synth.Q6_K, Wd, dim, hid, xm)
    assert_gemv_close(h_gpu, h0 + dr[0], dS[0], "down + residual", extra=np.abs(h_gpu) * 2.0 ** -23)
    plan.close()


def test_plan_chained_levels_with_options(q):
    """o (y += W att) -> gate/up from rmsnorm(h) -> down (swiglu, y += ...): one layer's plan."""
    rng = np.random.default_rng(31)
    dim, hid = 2048, 5632
    Wo, Wg, Wu, Wd = (synth.gen_matrix(t, r, c, s) for t, r, c, s in
                      [(synth.Q4_K, dim, dim, 1), (synth.Q4_K, hid, dim, 2), (synth.Q4_K, hid, dim, 3),
                       (synth.Q6_K, dim, hid, 4)])
    att = rng.standard_normal(dim).astype(np.float32)
    h0 = rng.standard_normal(dim).astype(np.float32)
    nw = rng.uniform(0.01, 0.03, dim).astype(np.float32)
    h = dev(h0[None, :].copy())
    gbuf = torch.zeros(1, hid, device="cuda")
    ubuf = torch.zeros(1, hid, device="cuda")
    items = [(synth.Q4_K, dev(Wo), dim, dim, dev(att[None, :]), h), (synth.Q4_K, dev(Wg), hid, dim, h, gbuf),
             (synth.Q4_K, dev(Wu), hid, dim, h, ubuf), (synth.Q6_K, dev(Wd), dim, hid, gbuf, h)]
    nwd = dev(nw)
    opts = [{"y_op": q.Y_ADD}, {"x_op": q.X_RMSNORM, "norm_w": nwd, "eps": 1e-5},
            {"x_op": q.X_RMSNORM, "norm_w": nwd, "eps": 1e-5}, {"x_op": q.X_SWIGLU, "x2": ubuf, "y_op": q.Y_ADD}]
    plan = q.Plan(items, [0, 1, 1, 2], 1, opts=opts)
    plan.run()
    assert q.get_device_status() == 0
    # check each level against the oracle fed with the GPU's input to that level
    h1 = h0 + oracle.gemv(synth.Q4_K, Wo, dim, dim, att[None, :])[0][0]
    g_gpu, u_gpu, h_gpu = gbuf.cpu().numpy()[0], ubuf.cpu().numpy()[0], h.cpu().numpy()[0]
    # gate/up read rmsnorm(h1): recompute from the oracle's h1 (rounded to fp32 as stored)
    xn = ds.rmsnorm(h1.astype(np.float32), nw).astype(np.float32)[None, :]
    gr, gS = oracle.gemv(synth.Q4_K, Wg, hid, dim, xn)
    ur, uS = oracle.gemv(synth.Q4_K, Wu, hid, dim, xn)
    # h1 itself carries the o GEMV's error into the norm: allow it on top
    assert_gemv_close(g_gpu, gr[0], gS[0] * 2, "gate")
    assert_gemv_close(u_gpu, ur[0], uS[0] * 2, "up")
    dr, dS = oracle.gemv(synth.Q6_K, Wd, dim, hid, ds.swiglu(g_gpu, u_gpu).astype(np.float32)[None, :])
    oS = oracle.gemv(synth.Q4_K, Wo, dim, dim, att[None, :])[1][0]
    assert_gemv_close(h_gpu, h1 + dr[0], dS[0] + oS, "down + residual", extra=np.abs(h_gpu) * 2.0 ** -22)
    plan.close()


def test_plan_argmax_head(q):
    rng = np.random.default_rng(41)
    rows, cols = 32000, 2048
    W = synth.gen_matrix(synth.Q6_K, rows, cols, 13)
    x = rng.standard_normal(cols).astype(np.float32)
    nw = rng.uniform(0.5, 1.5, cols).astype(np.float32)
    y = torch.zeros(1, rows, device="cuda")
    am = torch.full((1,), -1, dtype=torch.int64, device="cuda")
    plan = q.Plan([(synth.Q6_K, dev(W), rows, cols, dev(x[None, :]), y)], [0], 1,
                  opts=[{"x_op": q.X_RMSNORM, "norm_w": dev(nw), "eps": 1e-5, "argmax": am}])
    for _ in range(3):  # the slot is cleared for the next run
        am.fill_(-1)
        plan.run()
        assert q.get_device_status() == 0
        yg = y.cpu().numpy()[0]
        assert int(am.item()) == ds.argmax_first(yg)
    y_ref, S = oracle.gemv(synth.Q6_K, W, rows, cols, ds.rmsnorm(x, nw).astype(np.float32)[None, :])
    assert_gemv_close(yg, y_ref[0], S[0], "head")
    i_ref = ds.argmax_first(y_ref[0])
    top = np.sort(y_ref[0])[-2:]
    if top[1] - top[0] > 2e-5 * S[0].max():
        assert int(am.item()) == i_ref
    plan.close()


def test_plan_argmax_ties_take_smallest_index(q):
    rows, cols = 600, 256
    W = np.zeros(rows * (cols // 256) * 144, dtype=np.uint8)  # every weight 0: all logits 0
    x = np.ones((1, cols), dtype=np.float32)
    y = torch.zeros(1, rows, device="cuda")
    am = torch.full((1,), -1, dtype=torch.int64, device="cuda")
    plan = q.Plan([(synth.Q4_K, dev(W), rows, cols, dev(x), y)], [0], 1, opts=[{"argmax": am}])
    plan.run()
    assert q.get_device_status() == 0
    assert int(am.item()) == 0
    plan.close()


def test_plan_option_checks(q):
    W = dev(synth.gen_matrix(synth.Q4_K, 8, 256, 1))
    x = torch.zeros(1, 256, device="cuda")
    y = torch.zeros(1, 8, device="cuda")
    am = torch.zeros(1, dtype=torch.int64, device="cuda")
    bad = [
        [{"x_op": 7}],
        [{"x_op": q.X_RMSNORM, "norm_w": None}],
        [{"x_op": q.X_SWIGLU}],
        [{"argmax": am}, {"argmax": am}],  # two argmax GEMVs
        [{"y_op": 3}],
        [{"x_op": q.X_MUL, "x2": None}],
    ]
    for opts in bad:
        items = [(synth.Q4_K, W, 8, 256, x, y)] * len(opts)
        with pytest.raises(q.QdqError):
            q.Plan(items, [0] * len(opts), 1, opts=opts)
    # argmax outside the last level
    with pytest.raises(q.QdqError):
        q.Plan([(synth.Q4_K, W, 8, 256, x, y), (synth.Q4_K, W, 8, 256, x, y)], [0, 1], 1,
               opts=[{"argmax": am}, {}])
    # silu at the store and the staged product: batch 1 only; silu rows of at most 4096 columns
    W2 = dev(synth.gen_matrix(synth.Q4_K, 8, 4352, 2))
    xb = torch.zeros(2, 256, device="cuda")
    yb = torch.zeros(2, 8, device="cuda")
    xw = torch.zeros(1, 4352, device="cuda")
    for items, batch, opts in [([(synth.Q4_K, W, 8, 256, xb, yb)], 2, [{"y_op": q.Y_SILU}]),
                               ([(synth.Q4_K, W, 8, 256, xb, yb)], 2, [{"x_op": q.X_MUL, "x2": xb}]),
                               ([(synth.Q4_K, W2, 8, 4352, xw, y)], 1, [{"y_op": q.Y_SILU}])]:
        with pytest.raises(q.QdqError):
            q.Plan(items, [0], batch, opts=opts)
    # two GEMVs of a level read the same x with different options
    with pytest.raises(q.QdqError):
        q.Plan([(synth.Q4_K, W, 8, 256, x, y), (synth.Q4_K, W, 8, 256, x, torch.zeros(1, 8, device="cuda"))],
               [0, 0], 1, opts=[{"x_op": q.X_RMSNORM, "norm_w": x[0], "eps": 1e-5}, {}])


@pytest.mark.parametrize("H,G,D,pos", [(32, 4, 64, 0), (32, 4, 64, 37), (4, 2, 128, 100), (8, 8, 32, 5)])
def test_rope_attention(q, H, G, D, pos):
    rng = np.random.default_rng(H * 1000 + pos)
    max_seq = pos + 3
    qv = rng.standard_normal(H * D).astype(np.float32)
    kv = rng.standard_normal(G * D).astype(np.float32)
    vv = rng.standard_normal(G * D).astype(np.float32)
    kc = rng.standard_normal((max_seq, G * D)).astype(np.float16)
    vc = rng.standard_normal((max_seq, G * D)).astype(np.float16)
    kcd, vcd = dev(kc.view(np.uint16)), dev(vc.view(np.uint16))
    out = torch.full((H * D,), float("nan"), device="cuda")
    q.rope_attention(dev(qv), dev(kv), dev(vv), kcd, vcd, out, H, G, D, pos, max_seq)
    assert q.get_device_status() == 0
    kc_gpu = kcd.cpu().numpy().view(np.float16)
    vc_gpu = vcd.cpu().numpy().view(np.float16)
    # rows other than pos untouched; row pos = fp16 of the oracle's turned key / value
    np.testing.assert_array_equal(np.delete(kc_gpu, pos, 0), np.delete(kc, pos, 0))
    k_ref = ds.rope_interleaved(kv, G, D, pos)
    ulp = np.abs(np.spacing(k_ref.astype(np.float16)).astype(np.float64))
    assert np.all(np.abs(kc_gpu[pos].astype(np.float64) - k_ref) <= ulp)
    np.testing.assert_array_equal(vc_gpu[pos], vv.astype(np.float16))
    q_ref = ds.rope_interleaved(qv, H, D, pos)
    o_ref = ds.attention(q_ref, kc_gpu.reshape(max_seq, G, D), vc_gpu.reshape(max_seq, G, D), pos + 1, H, G, D)
    o = out.cpu().numpy()
    assert np.max(np.abs(o - o_ref)) <= 1e-5 * np.abs(vc_gpu[:pos + 1]).max()


CFG = dict(dim=256, hidden=512, n_layers=2, n_heads=4, n_kv_heads=2, vocab=300)


def _gpu_model(q, m, max_seq):
    t = lambda a: dev(a)
    layers = []
    for lw in m["layers"]:
        d = {name: (lw[name][0], t(lw[name][3])) for name in synth.LAYER_TENSORS}
        d["attn_norm"] = t(lw["attn_norm"])
        d["ffn_norm"] = t(lw["ffn_norm"])
        layers.append(d)
    e, o = m["token_embd"], m["output"]
    return q.Llama(max_seq=max_seq, embd=(e[0], t(e[3])), layers=layers, output_norm=t(m["output_norm"]),
                   output=(o[0], t(o[3])), **CFG)


PETIT_TYPES = {"q": synth.Q8_0, "k": synth.Q4_0, "v": synth.Q8_0, "o": synth.Q4_0, "gate": synth.Q8_0,
               "up": synth.Q4_0, "down": synth.Q8_0}


@pytest.mark.parametrize("norm_scale,petit", [(0.02, False), (1.0, False), (0.02, True)])
def test_token_step(q, norm_scale, petit):
    max_seq = 8
    kw = dict(layer_types=PETIT_TYPES, embd_type=synth.Q8_0, out_type=synth.Q4_0) if petit else {}
    m = synth.gen_llama_model(seed=77, norm_scale=norm_scale, **kw, **CFG)
    model = _gpu_model(q, m, max_seq)
    assert model.launches == 2  # the embedding row's decode, then one plan launch
    cfg = ds.LlamaConfig(max_seq=max_seq, **CFG)
    w = ds.from_blocks(cfg, m)
    kc, vc = ds.new_cache(cfg)
    for pos, tok in enumerate([5, 17, 3, 299, 0]):
        model.forward(tok, pos)
        assert q.get_device_status() == 0
        kg = model.k_cache.cpu().numpy()
        vg = model.v_cache.cpu().numpy()
        kc[:, :pos], vc[:, :pos] = kg[:, :pos], vg[:, :pos]  # the GPU's earlier rows
        tr = {}
        # the oracle stores the GPU's fp16 rows of this position (the rounding
        # decision taken once), after they are checked against its own k and v
        ref = ds.forward(w, kc, vc, tok, pos, trace=tr, rows={"k": kg[:, pos], "v": vg[:, pos]})
        for l in range(CFG["n_layers"]):
            for got, want in ((kg[l, pos], tr["k"][l]), (vg[l, pos], tr["v"][l])):
                step = np.abs(np.spacing(want.astype(np.float16)).astype(np.float64))
                assert np.all(np.abs(got.astype(np.float64) - want) <= step + 1e-5 * np.abs(want).max()), (pos, l)
        logits = model.logits.cpu().numpy()
        ot, orows, ocols, ob = m["output"]
        _, S = oracle.gemv(ot, ob, orows, ocols, tr["hn"].astype(np.float32)[None, :])
        err = np.abs(logits.astype(np.float64) - ref)
        assert np.all(err <= 1e-4 * S[0] + 1e-6), (pos, float(err.max()), float(S[0].max()))
        assert int(model.argmax.item()) == ds.argmax_first(logits)
    model.close()


def _check_positions(q, cfg1, max_seq, check, seed):
    """Decode positions 0 .. max_seq - 1 of a model of shape cfg1 and compare the
    logits with the oracle's at the positions in `check`."""
    m = synth.gen_llama_model(seed=seed, norm_scale=0.02, **cfg1)
    t = lambda a: dev(a)
    layers = [{**{k: (lw[k][0], t(lw[k][3])) for k in synth.LAYER_TENSORS},
               "attn_norm": t(lw["attn_norm"]), "ffn_norm": t(lw["ffn_norm"])} for lw in m["layers"]]
    model = q.Llama(max_seq=max_seq, embd=(m["token_embd"][0], t(m["token_embd"][3])), layers=layers,
                    output_norm=t(m["output_norm"]), output=(m["output"][0], t(m["output"][3])), **cfg1)
    w = ds.from_blocks(ds.LlamaConfig(max_seq=max_seq, **cfg1), m)
    kc, vc = ds.new_cache(w.cfg)
    for pos in range(max_seq):
        tok = (pos * 37 + 11) % cfg1["vocab"]
        model.forward(tok, pos)
        if pos not in check:
            continue
        assert q.get_device_status() == 0
        kg, vg = model.k_cache.cpu().numpy(), model.v_cache.cpu().numpy()
        kc[:, :pos], vc[:, :pos] = kg[:, :pos], vg[:, :pos]
        tr = {}
        ref = ds.forward(w, kc, vc, tok, pos, trace=tr, rows={"k": kg[:, pos], "v": vg[:, pos]})
        ot, orows, ocols, ob = m["output"]
        _, S = oracle.gemv(ot, ob, orows, ocols, tr["hn"].astype(np.float32)[None, :])
        err = np.abs(model.logits.cpu().numpy().astype(np.float64) - ref)
        assert np.all(err <= 1e-4 * S[0] + 1e-6), (pos, float(err.max()))
    model.close()


def test_token_step_long_context(q):
    """Positions up to 519 of a one-layer model with 64-dimensional heads: the
    attention level's chunks of eight positions spread over the fifteen consumer
    warps (a new round every 120 positions, each warp's next chunk loaded ahead),
    and the warps' states merged. Checked at the chunk and round boundaries."""
    cfg1 = dict(dim=256, hidden=512, n_layers=1, n_heads=4, n_kv_heads=2, vocab=300)
    _check_positions(q, cfg1, 520, {0, 7, 8, 9, 31, 32, 33, 119, 120, 121, 239, 240, 250, 479, 480, 481, 519}, 78)


@pytest.mark.parametrize("n_heads,n_kv_heads", [(8, 2), (2, 1), (8, 8)])
def test_token_step_head_dims(q, n_heads, n_kv_heads):
    """Heads of 32 dimensions (the eight-position chunks with one 16-byte key load
    per lane) and of 128 (the per-32-position loop), grouped and ungrouped, over
    several rounds of chunks."""
    cfg1 = dict(dim=256, hidden=512, n_layers=1, n_heads=n_heads, n_kv_heads=n_kv_heads, vocab=300)
    _check_positions(q, cfg1, 136, {0, 7, 8, 31, 32, 64, 119, 120, 135}, 79 + n_heads)


@pytest.mark.parametrize("batch", [3, 8])
def test_plan_options_batched(q, batch):
    """rmsnorm (per batch column), SwiGLU and the residual add in the 4- and
    8-column instantiations of the streaming kernel."""
    rng = np.random.default_rng(50 + batch)
    dim, hid = 2048, 5632
    Wg = synth.gen_matrix(synth.Q4_K, hid, dim, 21)
    Wd = synth.gen_matrix(synth.Q6_K, dim, hid, 22)
    h0 = (rng.standard_normal((batch, dim)) * rng.uniform(0.5, 3, (batch, 1))).astype(np.float32)
    nw = rng.uniform(0.01, 0.03, dim).astype(np.float32)
    u = rng.standard_normal((batch, hid)).astype(np.float32)
    h = dev(h0.copy())
    g = torch.zeros(batch, hid, device="cuda")
    ud = dev(u)
    plan = q.Plan([(synth.Q4_K, dev(Wg), hid, dim, h, g), (synth.Q6_K, dev(Wd), dim, hid, g, h)], [0, 1], batch,
                  opts=[{"x_op": q.X_RMSNORM, "norm_w": dev(nw), "eps": 1e-5},
                        {"x_op": q.X_SWIGLU, "x2": ud, "y_op": q.Y_ADD}])
    plan.run()
    assert q.get_device_status() == 0
    g_gpu, h_gpu = g.cpu().numpy(), h.cpu().numpy()
    xn = np.stack([ds.rmsnorm(h0[b], nw) for b in range(batch)]).astype(np.float32)
    gr, gS = oracle.gemv(synth.Q4_K, Wg, hid, dim, xn)
    for b in range(batch):
        assert_gemv_close(g_gpu[b], gr[b], gS[b], f"rmsnorm gate, column {b}")
    xs = np.stack([ds.swiglu(g_gpu[b], u[b]) for b in range(batch)]).astype(np.float32)
    dr, dS = oracle.gemv(synth.Q6_K, Wd, dim, hid, xs)
    for b in range(batch):
        assert_gemv_close(h_gpu[b], h0[b] + dr[b], dS[b], f"swiglu down + residual, column {b}",
                          extra=np.abs(h_gpu[b]) * 2.0 ** -23)
    plan.close()
