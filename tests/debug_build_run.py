"""Parity cases run against the library built with -DQDQ_DEBUG (device-side index
and alignment checks that record QDQ_ERR_BOUNDS instead of trapping).

Run as a separate process by tests/test_gpu_debug_build.py, with QDQ_BUILD_DIR
and QDQ_EXTRA_NVCC_FLAGS set, so that the debug library is the one loaded. Every
case must match the oracle within the GEMV bound and leave the device status at
0 (no check fired). Exits non-zero on the first failure.
"""
import sys

import numpy as np
import torch

import oracle
from oracle import decode_step as ds
from quant_dequant_gemv_gb300 import build, qdq, synth


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def status_ok(what):
    rc = qdq.get_device_status()
    if rc != 0:
        raise SystemExit(f"{what}: device status {rc} ({qdq.status_string(rc)})")


def gemv_case(qtype, rows, cols, batch, seed):
    W = synth.gen_matrix(qtype, rows, cols, seed)
    x = synth.gen_x(batch, cols, seed + 1)
    y = torch.full((batch, rows), float("nan"), device="cuda")
    qdq.gemv(qtype, dev(W), rows, cols, dev(x), y, batch)
    status_ok(f"gemv {synth.TYPE_NAMES[qtype]} {rows}x{cols} b{batch}")
    y_ref, S = oracle.gemv(qtype, W, rows, cols, x)
    if not np.all(np.abs(y.cpu().numpy().astype(np.float64) - y_ref) <= 1e-5 * S + 1e-7):
        raise SystemExit(f"gemv {synth.TYPE_NAMES[qtype]} {rows}x{cols} b{batch}: out of tolerance")


def main():
    path = build.build()
    assert "QDQ_DEBUG" in " ".join(build.NVCC_FLAGS), "not a debug build"
    torch.cuda.set_device(0)
    print("library", path)
    # streaming kernel at batch 1, 2, 8 (whole-row and chunked tiles, ragged rows),
    # the tensor-core kernel at 16 and 40, the warp-per-row kernel of a further format
    for qtype, rows, cols, batch in [(synth.Q4_K, 300, 2048, 1), (synth.Q6_K, 97, 5632, 1),
                                     (synth.Q8_0, 64, 14336, 1), (synth.Q4_0, 33, 4096, 2),
                                     (synth.Q4_K, 1000, 2048, 8), (synth.Q4_K, 640, 2048, 16),
                                     (synth.Q6_K, 384, 2048, 40), (synth.Q3_K, 37, 5632, 3)]:
        gemv_case(qtype, rows, cols, batch, 11 * rows + batch)
    # standalone dequantisation
    for qtype in (synth.Q4_K, synth.Q6_K, synth.Q5_K):
        n = 4099 * synth.BLOCK_WEIGHTS[qtype]
        B = synth.gen_matrix(qtype, 1, n, 5)
        out = torch.empty(n, device="cuda")
        qdq.dequant(qtype, dev(B), n, out)
        status_ok(f"dequant {synth.TYPE_NAMES[qtype]}")
        if not np.array_equal(out.cpu().numpy().view(np.uint32), oracle.dequant(qtype, B, n).view(np.uint32)):
            raise SystemExit(f"dequant {synth.TYPE_NAMES[qtype]}: not bit-exact")
    # a chained multi-level plan: two layers of the 1.1B step shapes
    levels = synth.llama_1b_step(2)
    items, lv, ref = [], [], []
    for li, level in enumerate(levels):
        x = synth.gen_x(1, level[0].cols, 700 + li)
        xd = dev(x)
        for gi, g in enumerate(level):
            W = synth.gen_matrix(g.qtype, g.rows, g.cols, 40 * li + gi)
            y = torch.full((1, g.rows), float("nan"), device="cuda")
            items.append((g.qtype, dev(W), g.rows, g.cols, xd, y))
            lv.append(li)
            ref.append((g.qtype, W, g.rows, g.cols, x, y))
    plan = qdq.Plan(items, lv, 1)
    plan.run()
    status_ok("plan")
    for qtype, W, rows, cols, x, y in ref:  # the first and last 48 rows of every GEMV
        got = y.cpu().numpy().astype(np.float64)
        for r0 in (0, max(rows - 48, 0)):
            r1 = min(r0 + 48, rows)
            y_ref, S = oracle.gemv(qtype, W, rows, cols, x, r0, r1)  # full-width arrays, rows r0..r1 filled
            if not np.all(np.abs(got[:, r0:r1] - y_ref[:, r0:r1]) <= 1e-5 * S[:, r0:r1] + 1e-7):
                raise SystemExit(f"plan: {synth.TYPE_NAMES[qtype]} {rows}x{cols} rows {r0}..{r1} out of tolerance")
    plan.close()
    # the token step of a one-layer model over 40 positions (attention levels)
    cfg = dict(dim=256, hidden=512, n_layers=1, n_heads=4, n_kv_heads=2, vocab=300)
    m = synth.gen_llama_model(seed=5, norm_scale=0.02, **cfg)
    layers = [{**{k: (lw[k][0], dev(lw[k][3])) for k in synth.LAYER_TENSORS},
               "attn_norm": dev(lw["attn_norm"]), "ffn_norm": dev(lw["ffn_norm"])} for lw in m["layers"]]
    model = qdq.Llama(max_seq=40, embd=(m["token_embd"][0], dev(m["token_embd"][3])), layers=layers,
                      output_norm=dev(m["output_norm"]), output=(m["output"][0], dev(m["output"][3])), **cfg)
    w = ds.from_blocks(ds.LlamaConfig(max_seq=40, **cfg), m)
    kc, vc = ds.new_cache(w.cfg)
    for pos in range(40):
        tok = (pos * 37 + 11) % cfg["vocab"]
        model.forward(tok, pos)
        status_ok(f"token step at {pos}")
        if pos in (0, 9, 39):
            kg, vg = model.k_cache.cpu().numpy(), model.v_cache.cpu().numpy()
            kc[:, :pos], vc[:, :pos] = kg[:, :pos], vg[:, :pos]
            tr = {}
            logits_ref = ds.forward(w, kc, vc, tok, pos, trace=tr, rows={"k": kg[:, pos], "v": vg[:, pos]})
            ot, orows, ocols, ob = m["output"]
            _, S = oracle.gemv(ot, ob, orows, ocols, tr["hn"].astype(np.float32)[None, :])
            err = np.abs(model.logits.cpu().numpy().astype(np.float64) - logits_ref)
            if not np.all(err <= 1e-4 * S[0] + 1e-6):
                raise SystemExit(f"token step at {pos}: out of tolerance")
    model.close()
    print("debug build: every case within the bound, no check fired")


if __name__ == "__main__":
    sys.exit(main())
