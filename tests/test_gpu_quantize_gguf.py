"""The quantiser kernel against the oracle (bit-exact: every quant and scale is
a discrete value both sides decide in binary32), and a model loaded from a
mapped synthetic GGUF file run through the one-token forward pass."""
import mmap

import numpy as np
import pytest

import oracle
from oracle import decode_step as ds
from oracle import quantize as qz
from quant_dequant_gemv_gb300 import synth
from tests import gguf_file as gf

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


def _inputs(n, kind, rng):
    if kind == "normal":
        return rng.standard_normal(n).astype(np.float32)
    if kind == "scaled":  # blocks whose magnitudes span many binades
        return (rng.standard_normal(n) * 10.0 ** rng.uniform(-30, 30, n)).astype(np.float32)
    if kind == "halves":  # x / d lands on .5 often: round half to even decides
        v = (rng.integers(-254, 255, n) / 2.0).astype(np.float32)
        v[::32] = 127.0
        return v
    v = rng.standard_normal(n).astype(np.float32)
    v[: n // 2] = 0.0  # zero blocks and a zero-padded tail
    return v


@pytest.mark.parametrize("qtype", [synth.Q8_0, synth.Q4_0])
@pytest.mark.parametrize("kind", ["normal", "scaled", "halves", "zeros"])
@pytest.mark.parametrize("n", [32, 1000, 32 * 4099, 1 << 20])
def test_quantize_bit_exact(q, qtype, kind, n):
    rng = np.random.default_rng(n + qtype)
    x = _inputs(n, kind, rng)
    bb = synth.BLOCK_BYTES[qtype]
    nb = (n + 31) // 32
    out = torch.full((nb * bb,), 0xAB, dtype=torch.uint8, device="cuda")
    q.quantize(qtype, torch.from_numpy(x).cuda(), n, out)
    assert q.get_device_status() == 0
    want = qz.quantize_q8_0(x) if qtype == synth.Q8_0 else qz.quantize_q4_0(x)
    got = out.cpu().numpy()
    if not np.array_equal(got, want):
        i = int(np.flatnonzero(got != want)[0])
        raise AssertionError(f"byte {i} (block {i // bb}): {got[i]} vs {want[i]}")


def test_llama_from_mapped_gguf(q, tmp_path):
    cfg = dict(dim=256, hidden=512, n_layers=2, n_heads=4, n_kv_heads=2, vocab=300)
    m = synth.gen_llama_model(seed=9, norm_scale=0.02, **cfg)
    path = tmp_path / "tiny.gguf"
    path.write_bytes(gf.llama_file(m, cfg))
    with open(path, "rb") as fh, mmap.mmap(fh.fileno(), 0, access=mmap.ACCESS_READ) as mm:
        tensors, _, _ = q.gguf_parse(mm)
        by = {t["name"]: t for t in tensors}

        def meta(key):
            t, off = q.gguf_find_kv(mm, key)
            return gf.read_value(mm, t, off)

        dim, nl = meta("llama.embedding_length"), meta("llama.block_count")
        load = lambda name: torch.from_numpy(gf.tensor_array(mm, by[name]).copy()).cuda()
        wt = lambda name: (by[name]["qdq_type"], load(name))
        f32 = lambda name: torch.from_numpy(gf.tensor_array(mm, by[name], np.float32).copy()).cuda()
        names = {"q": "attn_q", "k": "attn_k", "v": "attn_v", "o": "attn_output", "gate": "ffn_gate",
                 "up": "ffn_up", "down": "ffn_down"}
        layers = []
        for l in range(nl):
            d = {k: wt(f"blk.{l}.{v}.weight") for k, v in names.items()}
            d["attn_norm"], d["ffn_norm"] = f32(f"blk.{l}.attn_norm.weight"), f32(f"blk.{l}.ffn_norm.weight")
            layers.append(d)
        model = q.Llama(dim=dim, hidden=meta("llama.feed_forward_length"), n_layers=nl,
                        n_heads=meta("llama.attention.head_count"), n_kv_heads=meta("llama.attention.head_count_kv"),
                        vocab=by["token_embd.weight"]["dims"][1], max_seq=4, embd=wt("token_embd.weight"),
                        layers=layers, output_norm=f32("output_norm.weight"), output=wt("output.weight"),
                        rope_base=meta("llama.rope.freq_base"), norm_eps=meta("llama.attention.layer_norm_rms_epsilon"))
    w = ds.from_blocks(ds.LlamaConfig(max_seq=4, **cfg), m)
    kc, vc = ds.new_cache(w.cfg)
    for pos, tok in enumerate([7, 123]):
        model.forward(tok, pos)
        assert q.get_device_status() == 0
        kg, vg = model.k_cache.cpu().numpy(), model.v_cache.cpu().numpy()
        kc[:, :pos], vc[:, :pos] = kg[:, :pos], vg[:, :pos]
        tr = {}
        ref = ds.forward(w, kc, vc, tok, pos, trace=tr, rows={"k": kg[:, pos], "v": vg[:, pos]})
        ot, orows, ocols, ob = m["output"]
        _, S = oracle.gemv(ot, ob, orows, ocols, tr["hn"].astype(np.float32)[None, :])
        err = np.abs(model.logits.cpu().numpy().astype(np.float64) - ref)
        assert np.all(err <= 1e-4 * S[0] + 1e-6)
    model.close()
