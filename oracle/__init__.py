"""CPU oracle for the fused dequant-GEMV (ctypes wrapper around qdq_oracle.c).

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg may import this package. The library's compute path
(``quant_dequant_gemv_gb300``) never imports it, and it imports nothing from
there. It is compiled with gcc at first use (``-O2 -ffp-contract=off``) into
``oracle/_build``.

What each function computes, and which passage it follows, is stated in
``qdq_oracle.c``.
"""
from __future__ import annotations

import ctypes
import hashlib
import os
import subprocess
import tempfile
from pathlib import Path

import numpy as np

HERE = Path(__file__).resolve().parent
SRC = HERE / "qdq_oracle.c"
BUILD_DIR = HERE / "_build"
CFLAGS = ["-O2", "-ffp-contract=off", "-fno-fast-math", "-std=c11", "-shared", "-fPIC"]

Q4_0, Q8_0, Q4_K, Q6_K, Q5_0, Q5_1, Q8_0G, Q2_K, Q5_K, Q3_K = 1, 2, 3, 4, 5, 6, 7, 8, 9, 10
BLOCK_BYTES = {Q4_0: 18, Q8_0: 36, Q4_K: 144, Q6_K: 210, Q5_0: 22, Q5_1: 24, Q8_0G: 34, Q2_K: 84, Q5_K: 176,
               Q3_K: 110}
BLOCK_WEIGHTS = {Q4_0: 32, Q8_0: 32, Q4_K: 256, Q6_K: 256, Q5_0: 32, Q5_1: 32, Q8_0G: 32, Q2_K: 256, Q5_K: 256,
                 Q3_K: 256}

_P = ctypes.c_void_p
_I64 = ctypes.c_int64


def compile_source(source: str, out: Path) -> Path:
    """Compile oracle C source text into a shared library at `out`."""
    out.parent.mkdir(parents=True, exist_ok=True)
    with tempfile.TemporaryDirectory() as td:
        src = Path(td) / "oracle.c"
        src.write_text(source)
        tmp_out = Path(td) / out.name
        subprocess.run(["gcc", *CFLAGS, str(src), "-o", str(tmp_out), "-lm"], check=True)
        os.replace(tmp_out, out)
    return out


def build() -> Path:
    """Compile qdq_oracle.c (cached by content hash) and return the .so path."""
    text = SRC.read_text()
    tag = hashlib.sha256((text + " ".join(CFLAGS)).encode()).hexdigest()[:12]
    out = BUILD_DIR / f"liborc_{tag}.so"
    if not out.exists():
        compile_source(text, out)
    return out


class Oracle:
    """Bindings to one compiled oracle library (the real one, or a test mutant)."""

    def __init__(self, so_path: Path):
        lib = ctypes.CDLL(str(so_path))
        lib.orc_fp16_to_fp32.restype = ctypes.c_float
        lib.orc_fp16_to_fp32.argtypes = [ctypes.c_uint16]
        lib.orc_q4k_scale_min.restype = None
        lib.orc_q4k_scale_min.argtypes = [_P, ctypes.c_int, _P, _P]
        lib.orc_dequant.restype = ctypes.c_int
        lib.orc_dequant.argtypes = [ctypes.c_int, _P, _I64, _P]
        lib.orc_gemv_rows.restype = ctypes.c_int
        lib.orc_gemv_rows.argtypes = [ctypes.c_int, _P, _I64, _I64, _P, ctypes.c_int,
                                      _I64, _I64, _P, _P, _P]
        self.lib = lib

    def fp16_to_fp32(self, h: np.ndarray) -> np.ndarray:
        h = np.ascontiguousarray(h, dtype=np.uint16).reshape(-1)
        f = self.lib.orc_fp16_to_fp32
        return np.array([f(int(v)) for v in h], dtype=np.float32)

    def q4k_scale_min(self, packed12: bytes | np.ndarray, j: int) -> tuple[int, int]:
        p = np.ascontiguousarray(np.frombuffer(bytes(packed12), dtype=np.uint8))
        sc, mn = ctypes.c_int(), ctypes.c_int()
        self.lib.orc_q4k_scale_min(p.ctypes.data, j, ctypes.byref(sc), ctypes.byref(mn))
        return sc.value, mn.value

    def dequant(self, qtype: int, blocks: np.ndarray, n: int) -> np.ndarray:
        blocks = np.ascontiguousarray(blocks, dtype=np.uint8)
        if blocks.size < (n // BLOCK_WEIGHTS[qtype]) * BLOCK_BYTES[qtype]:
            raise ValueError("not enough block bytes")
        out = np.empty(n, dtype=np.float32)
        rc = self.lib.orc_dequant(qtype, blocks.ctypes.data, n, out.ctypes.data)
        if rc:
            raise ValueError(f"orc_dequant failed ({rc})")
        return out

    def gemv(self, qtype: int, W: np.ndarray, rows: int, cols: int, x: np.ndarray,
             r0: int = 0, r1: int | None = None) -> tuple[np.ndarray, np.ndarray]:
        """y, S as float64 [batch][rows]; only rows [r0, r1) are filled (rest NaN)."""
        W = np.ascontiguousarray(W, dtype=np.uint8)
        x = np.ascontiguousarray(x, dtype=np.float32)
        batch = x.shape[0] if x.ndim == 2 else 1
        if x.size != batch * cols:
            raise ValueError("x must be [batch][cols]")
        r1 = rows if r1 is None else r1
        y = np.full((batch, rows), np.nan)
        S = np.full((batch, rows), np.nan)
        buf = np.empty(max(cols, 1), dtype=np.float32)
        rc = self.lib.orc_gemv_rows(qtype, W.ctypes.data, rows, cols, x.ctypes.data, batch,
                                    r0, r1, y.ctypes.data, S.ctypes.data, buf.ctypes.data)
        if rc:
            raise ValueError(f"orc_gemv_rows failed ({rc})")
        return y, S


_default: Oracle | None = None


def get() -> Oracle:
    global _default
    if _default is None:
        _default = Oracle(build())
    return _default


def dequant(qtype: int, blocks: np.ndarray, n: int) -> np.ndarray:
    return get().dequant(qtype, blocks, n)


def gemv(qtype, W, rows, cols, x, r0=0, r1=None):
    return get().gemv(qtype, W, rows, cols, x, r0, r1)


def within_tolerance(y: np.ndarray, y_ref: np.ndarray, S: np.ndarray,
                     rel: float = 1e-5, abs_: float = 1e-7) -> np.ndarray:
    """The GEMV acceptance rule |y - y_ref| <= rel * S + abs_, elementwise."""
    return np.abs(np.asarray(y, np.float64) - y_ref) <= rel * S + abs_
