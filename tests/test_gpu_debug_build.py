"""The library built with -DQDQ_DEBUG: device-side index and alignment checks
(QDQ_CHECK) around the ring placement of weight tiles, the partial buffer's row
groups, the staged x window, the attention level's heads and the tensor-core
kernel's bulk and tensor copies, each recording QDQ_ERR_BOUNDS and skipping the
access instead of trapping. The parity cases of tests/debug_build_run.py run in a
separate process against that build (its own build directory), and must pass
with no check firing."""
import os
import subprocess
import sys
from pathlib import Path

import pytest

ROOT = Path(__file__).resolve().parents[1]
DEBUG_DIR = ROOT / "quant_dequant_gemv_gb300" / "_build" / "debug"


def _env():
    env = dict(os.environ)
    env["QDQ_BUILD_DIR"] = str(DEBUG_DIR)
    env["QDQ_EXTRA_NVCC_FLAGS"] = "-DQDQ_DEBUG"
    env["PYTHONPATH"] = str(ROOT) + os.pathsep + env.get("PYTHONPATH", "")
    return env


@pytest.mark.gpu
def test_debug_build_parity_without_a_check_firing():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    r = subprocess.run([sys.executable, str(ROOT / "tests" / "debug_build_run.py")], env=_env(), cwd=ROOT,
                       capture_output=True, text=True, timeout=1200)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-4000:]
    assert "no check fired" in r.stdout
