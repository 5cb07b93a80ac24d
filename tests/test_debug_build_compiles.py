"""The -DQDQ_DEBUG variants of the two persistent kernels' translation units
compile for sm_103a (a cross-compile: no GPU needed)."""
import shutil
import subprocess
import tempfile
from concurrent.futures import ThreadPoolExecutor
from pathlib import Path

import pytest

from quant_dequant_gemv_gb300 import build


@pytest.mark.skipif(shutil.which("nvcc") is None and not Path("/usr/local/cuda/bin/nvcc").exists(),
                    reason="no CUDA toolkit")
def test_debug_units_compile():
    out = Path(tempfile.mkdtemp(prefix="qdq_debug_"))
    flags = [x for x in build.NVCC_FLAGS] + ["-DQDQ_DEBUG"]

    def one(src):
        return subprocess.run([build.nvcc(), *build.ARCH, *flags, "-c", str(build.CSRC / src), "-o",
                               str(out / (src + ".o"))], capture_output=True, text=True)

    with ThreadPoolExecutor(2) as ex:
        results = list(ex.map(one, ["qdq_stream1.cu", "qdq_mma.cu"]))
    for r in results:
        assert r.returncode == 0, r.stderr[-3000:]
    shutil.rmtree(out, ignore_errors=True)
