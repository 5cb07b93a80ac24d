"""The C ABI without a GPU: the library builds, loads, exports every symbol the
header declares, and its host-side argument checks answer before any device
work."""
import re
from pathlib import Path

import pytest

ROOT = Path(__file__).resolve().parents[1]


@pytest.fixture(scope="module")
def lib():
    from quant_dequant_gemv_gb300 import build, qdq
    build.build()
    return qdq.lib()


def header_functions():
    text = (ROOT / "include" / "qdq.h").read_text()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(qdq_[a-z0-9_]+)\s*\(", text)))


def test_every_declared_function_is_exported(lib):
    from quant_dequant_gemv_gb300 import qdq
    names = header_functions()
    assert len(names) >= 15
    for n in names:
        assert hasattr(lib, n), f"{n} declared in include/qdq.h but not exported"
    assert sorted(qdq.EXPORTS) == names


def test_block_geometry(lib):
    assert [lib.qdq_block_bytes(t) for t in (1, 2, 3, 4)] == [18, 36, 144, 210]
    assert [lib.qdq_block_weights(t) for t in (1, 2, 3, 4)] == [32, 32, 256, 256]
    # Q5_0, Q5_1, ggml q8_0, Q2_K (84 bytes per 256: the page's figure)
    assert [lib.qdq_block_bytes(t) for t in (5, 6, 7, 8)] == [22, 24, 34, 84]
    assert [lib.qdq_block_weights(t) for t in (5, 6, 7, 8)] == [32, 32, 32, 256]
    assert lib.qdq_block_bytes(0) == -1 and lib.qdq_block_weights(99) == -1


def test_status_strings(lib):
    from quant_dequant_gemv_gb300 import qdq
    for rc in range(0, -9, -1):
        assert qdq.status_string(rc) != "unknown status"
    assert qdq.status_string(-100) == "unknown status"


def test_argument_checks_precede_device_work(lib):
    # These return before the library touches a device, so they hold on any host.
    assert lib.qdq_gemv(99, 0, 4, 256, 0, 0, 1, 0) == -1           # type
    assert lib.qdq_gemv(3, 0, 4, 100, 0, 0, 1, 0) == -2            # cols % 256
    assert lib.qdq_gemv(3, 0, -1, 256, 0, 0, 1, 0) == -2           # rows < 0
    assert lib.qdq_gemv(3, 0, 4, 256, 0, 0, 0, 0) == -2            # batch < 1
    assert lib.qdq_gemv(3, 0, 0, 256, 0, 0, 1, 0) == 0             # rows == 0: no-op
    assert lib.qdq_dequant(4, 0, 100, 0) == -2                      # n % 256
    assert lib.qdq_dequant(99, 0, 256, 0) == -1
    assert lib.qdq_dequant(1, 0, 0, 0) == 0                         # n == 0: no-op
    assert lib.qdq_gemv_group(None, 9, 1, 0) == -8                  # more than 8 GEMVs
    assert lib.qdq_plan_create(None, None, 1, 1, None) == -4


def test_binding_has_no_fallback(monkeypatch, tmp_path):
    """Without the built library every call raises; nothing computes on the CPU."""
    from quant_dequant_gemv_gb300 import build, qdq
    monkeypatch.setattr(build, "LIB", tmp_path / "missing.so")
    monkeypatch.setattr(qdq, "_lib", None)
    with pytest.raises(RuntimeError):
        qdq.gemv(3, 0, 1, 256, 0, 0, 1, stream=0)


def test_group_and_plan_checks_precede_device_work(lib):
    # Batch limits and the level sequence of a plan are checked before any device
    # work, so these answers hold on any host.
    import ctypes
    assert lib.qdq_gemv_group(None, 0, 1, None) == 0                # no GEMVs: no-op
    assert lib.qdq_gemv_group(None, 3, 0, None) == -2               # batch < 1
    assert lib.qdq_gemv_group(None, 3, 9, None) == -8               # batch above 8
    assert lib.qdq_gemv_group(None, -1, 1, None) == -8

    def plan(levels, batch=1):
        lv = (ctypes.c_int * max(len(levels), 1))(*levels)
        out = ctypes.c_void_p(12345)
        rc = lib.qdq_plan_create(None, lv, len(levels), batch, ctypes.byref(out))
        assert out.value is None                                    # no plan on failure
        return rc

    assert plan([0, 1], batch=0) == -2
    assert plan([0, 1], batch=9) == -8
    assert plan([1, 1]) == -2                                       # must start at level 0
    assert plan([0, 2]) == -2                                       # levels go up one at a time
    assert plan([0, 1, 0]) == -2                                    # and never down
    assert plan(list(range(129))) == -8                             # more than 128 levels
    assert plan([0] * 193) == -8                                    # more than 192 GEMVs
    assert plan([]) == -8
