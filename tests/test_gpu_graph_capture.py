"""A serving loop captures its calls in a CUDA graph. The very first library call of a
process may happen inside the capture, so each case runs in a fresh process: the
captured graph must replay with the same results as plain calls."""
import subprocess
import sys
import textwrap
from pathlib import Path

import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

ROOT = Path(__file__).resolve().parents[1]

SCRIPT = textwrap.dedent("""
    import sys, numpy as np, torch
    sys.path.insert(0, {root!r})
    from quant_dequant_gemv_gb300 import qdq, synth
    torch.cuda.set_device(0)
    case = {case!r}
    qtype, rows, cols, batch = synth.Q4_K, 640, 2048, case[1]
    W = torch.from_numpy(synth.gen_matrix(qtype, rows, cols, 7)).cuda()
    x = torch.from_numpy(synth.gen_x(batch, cols, 8)).cuda()
    y = torch.full((batch, rows), float("nan"), device="cuda")
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    if case[0] == "gemv":
        with torch.cuda.graph(g, stream=s):
            qdq.gemv(qtype, W, rows, cols, x, y, batch, torch.cuda.current_stream())
    else:
        plan = qdq.Plan([(qtype, W, rows, cols, x, y)], [0], batch)
        with torch.cuda.graph(g, stream=s):
            plan.run(torch.cuda.current_stream())
    g.replay(); torch.cuda.synchronize()
    got = y.cpu().numpy().copy()
    y.fill_(float("nan"))
    qdq.gemv(qtype, W, rows, cols, x, y, batch)
    torch.cuda.synchronize()
    ref = y.cpu().numpy()
    assert qdq.get_device_status() == 0
    assert np.array_equal(got, ref), "graph replay differs from a plain call"
    print("OK")
""")


@pytest.mark.parametrize("case", [("gemv", 1), ("gemv", 16), ("plan", 1)])
def test_first_call_inside_graph_capture(case):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from quant_dequant_gemv_gb300 import build
    build.build()
    r = subprocess.run([sys.executable, "-c", SCRIPT.format(root=str(ROOT), case=case)], capture_output=True,
                       text=True, timeout=300)
    assert r.returncode == 0 and "OK" in r.stdout, r.stdout[-2000:] + r.stderr[-2000:]
