"""The allocation-free entry point against the plan path.

qdq_gemv_levels_noalloc serves callers that cannot call cudaMalloc (code handed
a fixed memory budget by a host framework, a serving loop that must not touch
the allocator, a process whose allocations all go through another component).
It runs the same multi-level GEMV as a plan, with its level counters in a fixed
array inside the library. This test calls it through the C ABI twice in a row
and checks each result against the plan entry point's result, within the GEMV
tolerance |y - y_ref| <= 1e-5 * sum|w x| + 1e-7 used by the parity tests.
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


def test_noalloc_matches_plan_on_two_calls(q, orc):
    levels = synth.llama_1b_step(2)[:-1] + [[synth.Gemv("output", synth.Q6_K, 512, 2048)]]
    items_a, items_b, lv, host = [], [], [], []
    for li, level in enumerate(levels):
        x = synth.gen_x(1, level[0].cols, 500 + li)
        xd = torch.from_numpy(x).cuda()
        for gi, g in enumerate(level):
            W = synth.gen_matrix(g.qtype, g.rows, g.cols, 600 + 10 * li + gi)
            Wd = torch.from_numpy(W).cuda()
            ya = torch.full((1, g.rows), float("nan"), device="cuda")
            yb = torch.full((1, g.rows), float("nan"), device="cuda")
            items_a.append((g.qtype, Wd, g.rows, g.cols, xd, ya))
            items_b.append((g.qtype, Wd, g.rows, g.cols, xd, yb))
            lv.append(li)
            host.append((g, W, x))

    plan = q.Plan(items_a, lv, 1)
    plan.run()
    torch.cuda.synchronize()
    ref = [it[5].cpu().numpy().copy() for it in items_a]
    S = [orc.gemv(g.qtype, W, g.rows, g.cols, x)[1] for g, W, x in host]
    plan.close()

    for call in range(2):
        for it in items_b:
            it[5].fill_(float("nan"))
        q.gemv_levels_noalloc(items_b, lv, 1)
        torch.cuda.synchronize()
        assert q.get_device_status() == 0
        for (g, _, _), y_ref, s, it in zip(host, ref, S, items_b):
            y = it[5].cpu().numpy()
            ok = np.abs(y.astype(np.float64) - y_ref) <= 1e-5 * s + 1e-7
            assert ok.all(), f"call {call}: {g.name}: {int((~ok).sum())} outputs differ from the plan's"


def test_noalloc_rejects_too_many_levels(q):
    from quant_dequant_gemv_gb300.qdq import QdqError
    W = torch.zeros(144, dtype=torch.uint8, device="cuda")
    x = torch.zeros(256, device="cuda")
    ys = [torch.zeros(1, device="cuda") for _ in range(129)]
    items = [(synth.Q4_K, W, 1, 256, x, y) for y in ys]
    with pytest.raises(QdqError) as e:
        q.gemv_levels_noalloc(items, list(range(129)), 1)
    assert e.value.rc == -8
