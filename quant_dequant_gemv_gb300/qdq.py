"""ctypes binding of libqdq (the C ABI in include/qdq.h).

Argument marshalling only: every step of the computation runs in the library's
CUDA kernels. Buffers may be passed as torch tensors (their data_ptr() is used)
or as raw integer device addresses. `stream` defaults to torch's current CUDA
stream. Any non-zero status raises QdqError. If the library is not built or
cannot be loaded, every call raises: there is no fallback path.
"""
from __future__ import annotations

import ctypes
from typing import Sequence

from . import build as _build
from .synth import Q4_0, Q8_0, Q4_K, Q6_K  # noqa: F401

_lib = None

_P = ctypes.c_void_p
_I64 = ctypes.c_int64
_INT = ctypes.c_int


class QdqError(RuntimeError):
    def __init__(self, what: str, rc: int):
        self.rc = rc
        super().__init__(f"{what}: {status_string(rc)} ({rc})")


class GemvDesc(ctypes.Structure):
    _fields_ = [("type", ctypes.c_int32), ("reserved", ctypes.c_int32), ("W", _P), ("rows", _I64),
                ("cols", _I64), ("x", _P), ("y", _P)]


# qdq_gemv_opts: step glue fused into a plan's GEMV
X_PLAIN, X_RMSNORM, X_SWIGLU, X_MUL = 0, 1, 2, 3
Y_STORE, Y_ADD, Y_SILU = 0, 1, 2


class GemvOpts(ctypes.Structure):
    _fields_ = [("x_op", ctypes.c_int32), ("y_op", ctypes.c_int32), ("x2", _P), ("norm_w", _P),
                ("eps", ctypes.c_float), ("reserved", ctypes.c_int32), ("argmax", _P)]


class LlamaConfig(ctypes.Structure):
    _fields_ = [("dim", ctypes.c_int32), ("hidden", ctypes.c_int32), ("n_layers", ctypes.c_int32),
                ("n_heads", ctypes.c_int32), ("n_kv_heads", ctypes.c_int32), ("vocab", ctypes.c_int32),
                ("max_seq", ctypes.c_int32), ("reserved", ctypes.c_int32), ("rope_base", ctypes.c_float),
                ("norm_eps", ctypes.c_float)]


class LlamaLayer(ctypes.Structure):
    _fields_ = [("w", _P * 7), ("type", ctypes.c_int32 * 7), ("reserved", ctypes.c_int32),
                ("attn_norm", _P), ("ffn_norm", _P)]


class GgufTensor(ctypes.Structure):
    _fields_ = [("name", ctypes.c_char * 96), ("n_dims", ctypes.c_int32), ("ggml_type", ctypes.c_int32),
                ("qdq_type", ctypes.c_int32), ("reserved", ctypes.c_int32), ("dims", _I64 * 4),
                ("offset", _I64), ("bytes", _I64)]


def lib() -> ctypes.CDLL:
    """Load libqdq.so (built by __graft_entry__.build()). Raises if it is absent."""
    global _lib
    if _lib is None:
        path = _build.LIB
        if not path.exists():
            raise RuntimeError(f"{path} is not built; run __graft_entry__.build() (nvcc, sm_103a)")
        L = ctypes.CDLL(str(path))
        sig = {
            "qdq_block_bytes": (_INT, [_INT]),
            "qdq_block_weights": (_INT, [_INT]),
            "qdq_status_string": (ctypes.c_char_p, [_INT]),
            "qdq_device_sm_count": (_INT, []),
            "qdq_dequant": (_INT, [_INT, _P, _I64, _P]),
            "qdq_dequant_async": (_INT, [_INT, _P, _I64, _P, _P]),
            "qdq_gemv": (_INT, [_INT, _P, _I64, _I64, _P, _P, _INT, _P]),
            "qdq_gemv_group": (_INT, [ctypes.POINTER(GemvDesc), _INT, _INT, _P]),
            "qdq_plan_create": (_INT, [ctypes.POINTER(GemvDesc), ctypes.POINTER(_INT), _INT, _INT,
                                       ctypes.POINTER(_P)]),
            "qdq_plan_create_ex": (_INT, [ctypes.POINTER(GemvDesc), ctypes.POINTER(GemvOpts),
                                          ctypes.POINTER(_INT), _INT, _INT, ctypes.POINTER(_P)]),
            "qdq_plan_run": (_INT, [_P, _P]),
            "qdq_plan_run_io": (_INT, [_P, _P, _P, _P, ctypes.POINTER(_I64), ctypes.POINTER(_I64)]),
            "qdq_plan_reset": (_INT, [_P, _P]),
            "qdq_plan_destroy": (None, [_P]),
            "qdq_plan_launches": (_INT, [_P]),
            "qdq_get_device_status": (_INT, [_P]),
            "qdq_selftest_wait_timeout": (_INT, [_I64, _P]),
            "qdq_gemv_levels_noalloc": (_INT, [ctypes.POINTER(GemvDesc), ctypes.POINTER(_INT), _INT, _INT, _P]),
            "qdq_rope_attention": (_INT, [_P, _P, _P, _P, _P, _P, _INT, _INT, _INT, _INT, _INT, ctypes.c_float,
                                          _P]),
            "qdq_llama_create": (_INT, [ctypes.POINTER(LlamaConfig), _P, _INT, ctypes.POINTER(LlamaLayer), _P, _P,
                                        _INT, ctypes.POINTER(_P)]),
            "qdq_llama_forward": (_INT, [_P, _INT, _INT, _P]),
            "qdq_llama_buffers": (_INT, [_P, ctypes.POINTER(_P), ctypes.POINTER(_P), ctypes.POINTER(_P),
                                         ctypes.POINTER(_P), ctypes.POINTER(_P)]),
            "qdq_llama_launches": (_INT, [_P]),
            "qdq_llama_destroy": (None, [_P]),
            "qdq_quantize": (_INT, [_INT, _P, _I64, _P, _P]),
            "qdq_gguf_parse": (_INT, [_P, _I64, ctypes.POINTER(GgufTensor), _INT, ctypes.POINTER(_INT),
                                      ctypes.POINTER(_I64), ctypes.POINTER(ctypes.c_uint32)]),
            "qdq_gguf_find_kv": (_INT, [_P, _I64, ctypes.c_char_p, ctypes.POINTER(ctypes.c_uint32),
                                        ctypes.POINTER(_I64)]),
        }
        for name, (res, args) in sig.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _lib = L
    return _lib


# Every name the header declares (the C ABI's exported symbols).
EXPORTS = ["qdq_block_bytes", "qdq_block_weights", "qdq_status_string", "qdq_device_sm_count",
           "qdq_dequant", "qdq_dequant_async", "qdq_gemv", "qdq_gemv_group", "qdq_plan_create",
           "qdq_plan_create_ex",
           "qdq_plan_run", "qdq_plan_run_io", "qdq_plan_reset", "qdq_plan_destroy",
           "qdq_plan_launches", "qdq_get_device_status", "qdq_selftest_wait_timeout",
           "qdq_gemv_levels_noalloc", "qdq_rope_attention", "qdq_llama_create", "qdq_llama_forward",
           "qdq_llama_buffers", "qdq_llama_launches", "qdq_llama_destroy", "qdq_quantize", "qdq_gguf_parse",
           "qdq_gguf_find_kv"]


def _ptr(t) -> int:
    if t is None:
        return 0
    if isinstance(t, int):
        return t
    return int(t.data_ptr())


def _stream(stream) -> int:
    if stream is None:
        import torch
        return int(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, int):
        return stream
    return int(stream.cuda_stream)


def _check(rc: int, what: str) -> None:
    if rc != 0:
        raise QdqError(what, rc)


def status_string(rc: int) -> str:
    return lib().qdq_status_string(rc).decode()


def block_bytes(qtype: int) -> int:
    return lib().qdq_block_bytes(qtype)


def block_weights(qtype: int) -> int:
    return lib().qdq_block_weights(qtype)


def device_sm_count() -> int:
    n = lib().qdq_device_sm_count()
    if n < 0:
        raise QdqError("qdq_device_sm_count", n)
    return n


def dequant(qtype: int, blocks, n: int, out, stream=None) -> None:
    _check(lib().qdq_dequant_async(qtype, _ptr(blocks), n, _ptr(out), _stream(stream)), "qdq_dequant")


def gemv(qtype: int, W, rows: int, cols: int, x, y, batch: int = 1, stream=None) -> None:
    _check(lib().qdq_gemv(qtype, _ptr(W), rows, cols, _ptr(x), _ptr(y), batch, _stream(stream)), "qdq_gemv")


def _descs(items: Sequence[tuple]) -> ctypes.Array:
    arr = (GemvDesc * max(len(items), 1))()
    for i, (qtype, W, rows, cols, x, y) in enumerate(items):
        arr[i] = GemvDesc(qtype, 0, _ptr(W), rows, cols, _ptr(x), _ptr(y))
    return arr


def gemv_group(items: Sequence[tuple], batch: int = 1, stream=None) -> None:
    """items: (type, W, rows, cols, x, y) for each GEMV."""
    _check(lib().qdq_gemv_group(_descs(items), len(items), batch, _stream(stream)), "qdq_gemv_group")


class Plan:
    """A decode step's GEMVs in dependency levels, run as one persistent launch."""

    def __init__(self, items: Sequence[tuple], levels: Sequence[int], batch: int = 1,
                 opts: Sequence[dict | None] | None = None):
        """opts[i] (optional): dict with x_op, y_op, x2, norm_w, eps, argmax for items[i]."""
        self._keep = (items, opts)  # the caller's buffers must outlive the plan
        self.batch = batch
        lv = (_INT * len(levels))(*levels)
        h = _P()
        if opts is None:
            _check(lib().qdq_plan_create(_descs(items), lv, len(items), batch, ctypes.byref(h)), "qdq_plan_create")
        else:
            oa = (GemvOpts * max(len(items), 1))()
            for i, o in enumerate(opts):
                o = o or {}
                oa[i] = GemvOpts(o.get("x_op", X_PLAIN), o.get("y_op", Y_STORE), _ptr(o.get("x2")),
                                 _ptr(o.get("norm_w")), float(o.get("eps", 0.0)), 0, _ptr(o.get("argmax")))
            _check(lib().qdq_plan_create_ex(_descs(items), oa, lv, len(items), batch, ctypes.byref(h)),
                   "qdq_plan_create_ex")
        self._h = h

    def run(self, stream=None) -> None:
        _check(lib().qdq_plan_run(self._h, _stream(stream)), "qdq_plan_run")

    def run_io(self, x_host, y_host, stream=None) -> tuple[int, int]:
        hb, db = _I64(), _I64()
        _check(lib().qdq_plan_run_io(self._h, _ptr(x_host), _ptr(y_host), _stream(stream), ctypes.byref(hb),
                                     ctypes.byref(db)), "qdq_plan_run_io")
        return hb.value, db.value

    def reset(self, stream=None) -> None:
        _check(lib().qdq_plan_reset(self._h, _stream(stream)), "qdq_plan_reset")

    @property
    def launches(self) -> int:
        return lib().qdq_plan_launches(self._h)

    def close(self) -> None:
        if getattr(self, "_h", None) is not None and self._h.value:
            lib().qdq_plan_destroy(self._h)
            self._h = _P()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def gemv_levels_noalloc(items: Sequence[tuple], levels: Sequence[int], batch: int = 1, stream=None) -> None:
    """The plan computation in one call that allocates no device memory (its
    level counters live in a fixed 512-byte array inside the library)."""
    lv = (_INT * len(levels))(*levels)
    _check(lib().qdq_gemv_levels_noalloc(_descs(items), lv, len(items), batch, _stream(stream)),
           "qdq_gemv_levels_noalloc")


def get_device_status(stream=None) -> int:
    return lib().qdq_get_device_status(_stream(stream))


def selftest_wait_timeout(timeout_ns: int, stream=None) -> None:
    _check(lib().qdq_selftest_wait_timeout(timeout_ns, _stream(stream)), "qdq_selftest_wait_timeout")


def rope_attention(q, k, v, k_cache, v_cache, out, n_heads: int, n_kv_heads: int, head_dim: int, pos: int,
                   max_seq: int, rope_base: float = 10000.0, stream=None) -> None:
    """RoPE, fp16 cache append at `pos` and GQA attention of one position (qdq_rope_attention)."""
    _check(lib().qdq_rope_attention(_ptr(q), _ptr(k), _ptr(v), _ptr(k_cache), _ptr(v_cache), _ptr(out), n_heads,
                                    n_kv_heads, head_dim, pos, max_seq, rope_base, _stream(stream)),
           "qdq_rope_attention")


class _DeviceArray:
    """__cuda_array_interface__ over a library-owned device buffer (no copy)."""

    def __init__(self, ptr: int, shape: tuple, typestr: str):
        self.__cuda_array_interface__ = {"shape": shape, "typestr": typestr, "data": (ptr, False), "version": 2,
                                         "strides": None}


def device_view(ptr: int, shape: tuple, typestr: str):
    """A torch tensor viewing `ptr` (device memory the library owns)."""
    import torch
    return torch.as_tensor(_DeviceArray(ptr, shape, typestr), device="cuda")


class Llama:
    """One-token forward passes of a Llama-architecture model (qdq_llama_*).

    embd, output: (type, W) of the token embedding and output matrices;
    layers: per layer a dict of q k v o gate up down -> (type, W) and attn_norm,
    ffn_norm -> fp32 tensors; output_norm: fp32 tensor. The tensors must outlive
    the model."""

    def __init__(self, dim, hidden, n_layers, n_heads, n_kv_heads, vocab, max_seq, embd, layers, output_norm,
                 output, rope_base=10000.0, norm_eps=1e-5):
        self._keep = (embd, layers, output_norm, output)
        self.cfg = LlamaConfig(dim, hidden, n_layers, n_heads, n_kv_heads, vocab, max_seq, 0, rope_base, norm_eps)
        arr = (LlamaLayer * n_layers)()
        for i, lw in enumerate(layers):
            for j, name in enumerate(("q", "k", "v", "o", "gate", "up", "down")):
                t, W = lw[name]
                arr[i].w[j] = _ptr(W)
                arr[i].type[j] = t
            arr[i].attn_norm = _ptr(lw["attn_norm"])
            arr[i].ffn_norm = _ptr(lw["ffn_norm"])
        h = _P()
        _check(lib().qdq_llama_create(ctypes.byref(self.cfg), _ptr(embd[1]), embd[0], arr, _ptr(output_norm),
                                      _ptr(output[1]), output[0], ctypes.byref(h)), "qdq_llama_create")
        self._h = h
        ptrs = [_P() for _ in range(5)]
        _check(lib().qdq_llama_buffers(h, *[ctypes.byref(p) for p in ptrs]), "qdq_llama_buffers")
        kv = n_kv_heads * (dim // n_heads)
        self.logits = device_view(ptrs[0].value, (vocab,), "<f4")
        self.argmax = device_view(ptrs[1].value, (1,), "<i8")
        self.hidden = device_view(ptrs[2].value, (dim,), "<f4")
        self.k_cache = device_view(ptrs[3].value, (n_layers, max_seq, kv), "<f2")
        self.v_cache = device_view(ptrs[4].value, (n_layers, max_seq, kv), "<f2")

    def forward(self, token: int, pos: int, stream=None) -> None:
        _check(lib().qdq_llama_forward(self._h, token, pos, _stream(stream)), "qdq_llama_forward")

    @property
    def launches(self) -> int:
        return lib().qdq_llama_launches(self._h)

    def close(self) -> None:
        if getattr(self, "_h", None) is not None and self._h.value:
            lib().qdq_llama_destroy(self._h)
            self._h = _P()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def quantize(qtype: int, x, n: int, blocks, stream=None) -> None:
    """fp32 -> q8_0 / q4_0 blocks on the GPU (qdq_quantize)."""
    _check(lib().qdq_quantize(qtype, _ptr(x), n, _ptr(blocks), _stream(stream)), "qdq_quantize")


def gguf_parse(buf, max_tensors: int = 4096) -> tuple[list[dict], int, int]:
    """Tensor index of GGUF bytes in host memory (a bytes object, numpy array or
    mmap): ([{name, dims, ggml_type, qdq_type, offset, bytes}], data_offset, alignment)."""
    import numpy as np
    a = np.frombuffer(buf, dtype=np.uint8)
    arr = (GgufTensor * max(max_tensors, 1))()
    n, data, align = _INT(), _I64(), ctypes.c_uint32()
    _check(lib().qdq_gguf_parse(a.ctypes.data, a.size, arr, max_tensors, ctypes.byref(n), ctypes.byref(data),
                                ctypes.byref(align)), "qdq_gguf_parse")
    out = []
    for t in arr[:n.value]:
        out.append({"name": t.name.decode(), "dims": list(t.dims[:t.n_dims]), "ggml_type": t.ggml_type,
                    "qdq_type": t.qdq_type, "offset": t.offset, "bytes": t.bytes})
    return out, data.value, align.value


def gguf_find_kv(buf, key: str) -> tuple[int, int]:
    """(GGUF value type, byte offset of the value) of a metadata key."""
    import numpy as np
    a = np.frombuffer(buf, dtype=np.uint8)
    t, off = ctypes.c_uint32(), _I64()
    _check(lib().qdq_gguf_find_kv(a.ctypes.data, a.size, key.encode(), ctypes.byref(t), ctypes.byref(off)),
           "qdq_gguf_find_kv")
    return t.value, off.value
