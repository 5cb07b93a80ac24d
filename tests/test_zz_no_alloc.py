"""The allocation-free entry point against the oracle.

qdq_gemv_levels_noalloc serves callers that cannot call cudaMalloc (code handed
a fixed memory budget by a host framework, a serving loop that must not touch
the allocator, a process whose allocations all go through another component).
It runs the same multi-level GEMV as a plan, with its level counters in a fixed
array inside the library. This test calls it through the C ABI twice in a row
and checks each result against the CPU oracle, within the GEMV tolerance
|y - y_ref| <= 1e-5 * sum|w x| + 1e-7 used by the parity tests; it also checks
that the second call leaves the device's free memory unchanged. Batch 1 runs the
kernel's one-column instantiation, batch 3 its four-column one.
"""
import numpy as np
import pytest

import oracle
from quant_dequant_gemv_gb300 import synth

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


@pytest.mark.parametrize("batch", [1, 3])
def test_noalloc_matches_oracle_on_two_calls(q, orc, batch):
    levels = synth.llama_1b_step(2)[:-1] + [[synth.Gemv("output", synth.Q6_K, 512, 2048)]]
    items, lv, host = [], [], []
    for li, level in enumerate(levels):
        x = synth.gen_x(batch, level[0].cols, 500 + li)
        xd = torch.from_numpy(x).cuda()
        for gi, g in enumerate(level):
            W = synth.gen_matrix(g.qtype, g.rows, g.cols, 600 + 10 * li + gi)
            y = torch.full((batch, g.rows), float("nan"), device="cuda")
            items.append((g.qtype, torch.from_numpy(W).cuda(), g.rows, g.cols, xd, y))
            lv.append(li)
            host.append((g, W, x))
    ref = [orc.gemv(g.qtype, W, g.rows, g.cols, x) for g, W, x in host]

    for call in range(2):
        for it in items:
            it[5].fill_(float("nan"))
        torch.cuda.synchronize()
        free_before = torch.cuda.mem_get_info()[0]
        q.gemv_levels_noalloc(items, lv, batch)
        torch.cuda.synchronize()
        free_after = torch.cuda.mem_get_info()[0]
        assert q.get_device_status() == 0
        if call == 1:  # the first call on a device may still load the module's code
            assert free_after == free_before, f"free device memory changed by {free_before - free_after} bytes"
        for (g, _, _), (y_ref, S), it in zip(host, ref, items):
            y = it[5].cpu().numpy()
            ok = oracle.within_tolerance(y, y_ref, S)
            assert ok.all(), f"call {call}: {g.name}: {int((~ok).sum())} outputs out of tolerance"


def test_noalloc_rejects_too_many_levels(q):
    from quant_dequant_gemv_gb300.qdq import QdqError
    W = torch.zeros(144, dtype=torch.uint8, device="cuda")
    x = torch.zeros(256, device="cuda")
    ys = [torch.zeros(1, device="cuda") for _ in range(129)]
    items = [(synth.Q4_K, W, 1, 256, x, y) for y in ys]
    with pytest.raises(QdqError) as e:
        q.gemv_levels_noalloc(items, list(range(129)), 1)
    assert e.value.rc == -8
