"""Writes synthetic GGUF files for the reader's tests (test input only).

Layout ("S21 The Capstone: picoLM, in Python", section 1: header, metadata,
tensor index of (name, shape, type, offset), padding to general.alignment, one
blob), with the published GGUF encodings: little-endian u32 magic "GGUF" and
version, u64 tensor and metadata counts; strings as a u64 length and the bytes;
a metadata entry as key, u32 value type, value (arrays: u32 element type, u64
count, elements); a tensor entry as name, u32 dimension count, u64 dims
(innermost first), u32 type, u64 offset from the start of the blob.
"""
from __future__ import annotations

import struct

import numpy as np

U8, I8, U16, I16, U32, I32, F32, BOOL, STRING, ARRAY, U64, I64, F64 = range(13)
_FMT = {U8: "<B", I8: "<b", U16: "<H", I16: "<h", U32: "<I", I32: "<i", F32: "<f", BOOL: "<?", U64: "<Q",
        I64: "<q", F64: "<d"}
GGML_F32, GGML_Q4_0, GGML_Q8_0, GGML_Q4_K, GGML_Q6_K = 0, 2, 8, 12, 14


def _str(s: str) -> bytes:
    b = s.encode()
    return struct.pack("<Q", len(b)) + b


def _value(t: int, v) -> bytes:
    if t == STRING:
        return _str(v)
    if t == ARRAY:
        et, items = v
        return struct.pack("<IQ", et, len(items)) + b"".join(_value(et, x) for x in items)
    return struct.pack(_FMT[t], v)


def build(kvs: list[tuple], tensors: list[tuple], alignment: int | None = 32, version: int = 3) -> bytes:
    """kvs: (key, type, value); tensors: (name, dims, ggml_type, data bytes).
    general.alignment is written first when `alignment` is not None."""
    align = alignment or 32
    if alignment is not None:
        kvs = [("general.alignment", U32, alignment)] + list(kvs)
    head = struct.pack("<IIQQ", 0x46554747, version, len(tensors), len(kvs))
    head += b"".join(_str(k) + struct.pack("<I", t) + _value(t, v) for k, t, v in kvs)
    offs, off = [], 0
    for _, _, _, data in tensors:
        off = (off + align - 1) // align * align
        offs.append(off)
        off += len(data)
    for (name, dims, gt, _), o in zip(tensors, offs):
        head += _str(name) + struct.pack("<I", len(dims)) + b"".join(struct.pack("<Q", d) for d in dims)
        head += struct.pack("<IQ", gt, o)
    data_start = (len(head) + align - 1) // align * align
    blob = bytearray(data_start + off)
    blob[:len(head)] = head
    for (_, _, _, data), o in zip(tensors, offs):
        blob[data_start + o:data_start + o + len(data)] = data
    return bytes(blob)


def llama_file(m: dict, cfg: dict) -> bytes:
    """A GGUF holding a synthetic model from synth.gen_llama_model, llama.cpp tensor names."""
    from quant_dequant_gemv_gb300 import synth
    gg = {synth.Q4_K: GGML_Q4_K, synth.Q6_K: GGML_Q6_K, synth.Q4_0: GGML_Q4_0}
    names = {"q": "attn_q", "k": "attn_k", "v": "attn_v", "o": "attn_output", "gate": "ffn_gate",
             "up": "ffn_up", "down": "ffn_down"}
    T = []
    t, r, c, b = m["token_embd"]
    T.append(("token_embd.weight", [c, r], gg[t], b.tobytes()))
    for l, lw in enumerate(m["layers"]):
        T.append((f"blk.{l}.attn_norm.weight", [cfg["dim"]], GGML_F32, lw["attn_norm"].tobytes()))
        for key in synth.LAYER_TENSORS:
            t, r, c, b = lw[key]
            T.append((f"blk.{l}.{names[key]}.weight", [c, r], gg[t], b.tobytes()))
        T.append((f"blk.{l}.ffn_norm.weight", [cfg["dim"]], GGML_F32, lw["ffn_norm"].tobytes()))
    T.append(("output_norm.weight", [cfg["dim"]], GGML_F32, m["output_norm"].tobytes()))
    t, r, c, b = m["output"]
    T.append(("output.weight", [c, r], gg[t], b.tobytes()))
    kvs = [("general.architecture", STRING, "llama"),
           ("llama.embedding_length", U32, cfg["dim"]), ("llama.feed_forward_length", U32, cfg["hidden"]),
           ("llama.block_count", U32, cfg["n_layers"]), ("llama.attention.head_count", U32, cfg["n_heads"]),
           ("llama.attention.head_count_kv", U32, cfg["n_kv_heads"]),
           ("llama.attention.layer_norm_rms_epsilon", F32, 1e-5), ("llama.rope.freq_base", F32, 10000.0),
           ("tokenizer.ggml.tokens", ARRAY, (STRING, [f"<t{i}>" for i in range(cfg["vocab"])])),
           ("tokenizer.ggml.scores", ARRAY, (F32, [0.0] * cfg["vocab"]))]
    return build(kvs, T)


def read_value(buf: bytes, t: int, off: int):
    if t == STRING:
        n = struct.unpack_from("<Q", buf, off)[0]
        return buf[off + 8:off + 8 + n].decode()
    return struct.unpack_from(_FMT[t], buf, off)[0]


def tensor_array(buf, info: dict, dtype=np.uint8) -> np.ndarray:
    return np.frombuffer(buf, dtype=np.uint8, count=info["bytes"], offset=info["offset"]).view(dtype)
