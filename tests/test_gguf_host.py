"""The GGUF reader (qdq_gguf_parse / qdq_gguf_find_kv): host-only code, so these
run without a GPU. The layout pins come from the page ("S21 The Capstone:
picoLM, in Python", section 1: header, metadata, tensor index of (name, shape,
type, offset), padding to general.alignment, blob) and a file whose bytes are
written out by hand below."""
import struct

import numpy as np
import pytest

from quant_dequant_gemv_gb300 import synth
from tests import gguf_file as gf


@pytest.fixture(scope="module")
def q():
    from quant_dequant_gemv_gb300 import build, qdq
    build.build()
    qdq.lib()
    return qdq


def test_hand_built_file_offsets(q):
    # header: magic, version 3, one tensor, one metadata entry (alignment 64)
    b = struct.pack("<IIQQ", 0x46554747, 3, 1, 1)
    b += struct.pack("<Q", 17) + b"general.alignment" + struct.pack("<II", 4, 64)
    # tensor "w": 2 dims (256, 3), type 12 (Q4_K), offset 0 in the blob
    b += struct.pack("<Q", 1) + b"w" + struct.pack("<IQQIQ", 2, 256, 3, 12, 0)
    assert len(b) == 24 + 8 + 17 + 8 + 8 + 1 + 4 + 16 + 4 + 8  # 98 bytes of header
    blob_at = 128  # the next multiple of 64
    data = bytes(range(256)) * 2 + bytes(432 - 512 % 432)  # 3 rows of 144 bytes, any content
    f = b + bytes(blob_at - len(b)) + data[:432]
    tensors, data_off, align = q.gguf_parse(f)
    assert (data_off, align) == (128, 64)
    assert tensors == [{"name": "w", "dims": [256, 3], "ggml_type": 12, "qdq_type": synth.Q4_K,
                        "offset": 128, "bytes": 432}]


def test_writer_file_and_metadata(q):
    cfg = dict(dim=256, hidden=512, n_layers=2, n_heads=4, n_kv_heads=2, vocab=50)
    m = synth.gen_llama_model(seed=3, **cfg)
    f = gf.llama_file(m, cfg)
    tensors, data_off, align = q.gguf_parse(f)
    assert align == 32 and data_off % 32 == 0
    assert len(tensors) == 2 + cfg["n_layers"] * 9 + 1
    by = {t["name"]: t for t in tensors}
    wq = by["blk.1.attn_q.weight"]
    assert wq["dims"] == [256, 256] and wq["qdq_type"] == synth.Q4_K and wq["bytes"] == 256 * 144
    np.testing.assert_array_equal(gf.tensor_array(f, wq), m["layers"][1]["q"][3])
    assert by["blk.0.attn_v.weight"]["qdq_type"] == synth.Q6_K
    assert by["output_norm.weight"]["ggml_type"] == gf.GGML_F32 and by["output_norm.weight"]["qdq_type"] == 0
    np.testing.assert_array_equal(gf.tensor_array(f, by["output_norm.weight"], np.float32), m["output_norm"])
    for t in tensors:
        assert t["offset"] % align == 0 and t["offset"] + t["bytes"] <= len(f)
    # metadata after a string array and a float array is still found
    t, off = q.gguf_find_kv(f, "llama.attention.head_count_kv")
    assert (t, gf.read_value(f, t, off)) == (gf.U32, 2)
    t, off = q.gguf_find_kv(f, "general.architecture")
    assert gf.read_value(f, t, off) == "llama"
    with pytest.raises(q.QdqError) as e:
        q.gguf_find_kv(f, "llama.no_such_key")
    assert e.value.rc == -10


def test_malformed_files_are_rejected(q):
    f = gf.build([("a", gf.ARRAY, (gf.STRING, ["x", "yy"]))],
                 [("t", [32, 2], gf.GGML_Q4_0, bytes(36))])
    tensors, _, _ = q.gguf_parse(f)
    assert tensors[0]["qdq_type"] == synth.Q4_0 and tensors[0]["bytes"] == 36
    end = tensors[0]["offset"]
    for cut in range(0, end):  # every truncation of the header and index
        with pytest.raises(q.QdqError) as e:
            q.gguf_parse(f[:cut])
        assert e.value.rc == -9
    with pytest.raises(q.QdqError):
        q.gguf_parse(b"GGUX" + f[4:])  # magic
    with pytest.raises(q.QdqError):
        q.gguf_parse(f[:4] + struct.pack("<I", 9) + f[8:])  # version
    bad = gf.build([], [("t", [30, 2], gf.GGML_Q4_0, bytes(36))])  # a row that is not whole blocks
    with pytest.raises(q.QdqError):
        q.gguf_parse(bad)
    with pytest.raises(q.QdqError) as e:
        q.gguf_parse(f, max_tensors=0)
    assert e.value.rc == -8


def test_further_formats_map_to_their_decoders(q):
    f = gf.build([], [("a", [32, 1], 6, bytes(22)), ("b", [32, 1], 7, bytes(24)), ("c", [32, 1], 8, bytes(34)),
                      ("d", [256, 1], 10, bytes(84)), ("e", [256, 1], 13, bytes(176)),
                      ("g", [256, 1], 11, bytes(110)), ("h", [32, 1], 3, bytes(20))])
    t, _, _ = q.gguf_parse(f)
    assert [x["qdq_type"] for x in t] == [synth.Q5_0, synth.Q5_1, synth.Q8_0G, synth.Q2_K, synth.Q5_K, synth.Q3_K, 0]
    assert [x["bytes"] for x in t] == [22, 24, 34, 84, 176, 110, 20]
