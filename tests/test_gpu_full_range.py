"""GEMV parity outside the workload distribution, through the C ABI.

Two families of inputs, each at batch widths that reach every kernel: 1, 3, 4
and 8 run the streaming CUDA-core kernel (batch 3 pads to its four-column
instantiation), 16 and 64 the tensor-core kernel (q8_0 and q4_0 from batch 4).
Shapes reach whole-row tiles and, for wide rows, column chunks.

* Full-range blocks: uniform random bytes in every field, scales kept finite
  (synth.gen_blocks_full_range): negative, subnormal and large scales, Q6_K
  scales of -128, q8_0 quants of -128. The kernels' exponent-field integer
  conversion, nibbles left in place against pre-scaled x, and the factored
  per-group forms must all hold here, not only on the benchmark's narrow draws.
* Cancelling Q4_K blocks (tests/cancel_blocks.py): d*sc*q equal to or close to
  dmin*mn, where a factored sub-block sum subtracts two nearly equal terms; the
  kernels recentre each sub-block so that the bound still holds.

The bound is the one every GEMV test uses: |y - y_ref| <= 1e-5 * sum|w x| + 1e-7,
y_ref and sum|w x| from the oracle in double precision.
"""
import numpy as np
import pytest

import oracle
from quant_dequant_gemv_gb300 import synth
from tests.cancel_blocks import q4k_cancelling_blocks

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

REL, ABS = 1e-5, 1e-7
BATCHES = [1, 3, 4, 8, 16, 64]
SHAPES = {  # (rows, cols): whole-row tiles, then rows long enough for column chunks
    synth.Q4_K: [(97, 2048), (37, 20480)],
    synth.Q6_K: [(97, 2048), (37, 16896)],
    synth.Q8_0: [(97, 4096), (37, 32768)],
    synth.Q4_0: [(97, 4096), (37, 32800)],
}


@pytest.fixture(scope="module")
def q():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from quant_dequant_gemv_gb300 import build, qdq
    build.build()
    torch.cuda.set_device(0)
    return qdq


def run_gemv(q, qtype, W, rows, cols, x):
    batch = x.shape[0]
    y = torch.full((batch, rows), float("nan"), device="cuda")
    q.gemv(qtype, torch.from_numpy(W).cuda(), rows, cols, torch.from_numpy(x).cuda(), y, batch)
    torch.cuda.synchronize()
    assert q.get_device_status() == 0
    return y.cpu().numpy()


def assert_close(y, y_ref, S, what):
    ok = oracle.within_tolerance(y, y_ref, S, REL, ABS)
    if not ok.all():
        i = tuple(np.argwhere(~ok)[0])
        raise AssertionError(f"{what}: {int((~ok).sum())} of {ok.size} outputs out of tolerance; first {i}: "
                             f"y={y[i]!r} ref={y_ref[i]!r} S={S[i]!r}")


@pytest.mark.parametrize("qtype", [synth.Q4_K, synth.Q6_K, synth.Q8_0, synth.Q4_0])
@pytest.mark.parametrize("batch", BATCHES)
def test_gemv_full_range_blocks(q, orc, qtype, batch):
    for k, (rows, cols) in enumerate(SHAPES[qtype]):
        rng = np.random.default_rng(1000 * qtype + 10 * batch + k)
        W = synth.gen_blocks_full_range(qtype, rows * cols // synth.BLOCK_WEIGHTS[qtype], rng)
        x = rng.standard_normal((batch, cols), dtype=np.float32)
        y = run_gemv(q, qtype, W, rows, cols, x)
        y_ref, S = orc.gemv(qtype, W, rows, cols, x)
        assert_close(y, y_ref, S, f"{synth.TYPE_NAMES[qtype]} {rows}x{cols} batch {batch}")


@pytest.mark.parametrize("mode", ["exact", "pm1", "near"])
@pytest.mark.parametrize("batch", BATCHES)
def test_gemv_q4k_cancelling_blocks(q, orc, mode, batch):
    for k, (rows, cols) in enumerate([(64, 2048), (37, 20480)]):
        rng = np.random.default_rng(7 + 100 * batch + k)
        W = q4k_cancelling_blocks(rows * cols // 256, rng, mode)
        x = rng.standard_normal((batch, cols), dtype=np.float32)
        y = run_gemv(q, synth.Q4_K, W, rows, cols, x)
        y_ref, S = orc.gemv(synth.Q4_K, W, rows, cols, x)
        assert_close(y, y_ref, S, f"cancelling ({mode}) Q4_K {rows}x{cols} batch {batch}")


def test_plan_with_full_range_and_cancelling_levels(q, orc):
    """The decode-step launch (a multi-level plan, batch 1) on both input families."""
    n = 2048
    rng = np.random.default_rng(99)
    spec = [
        (0, synth.Q4_K, 300, lambda r: q4k_cancelling_blocks(300 * n // 256, r, "pm1")),
        (0, synth.Q6_K, 64, lambda r: synth.gen_blocks_full_range(synth.Q6_K, 64 * n // 256, r)),
        (1, synth.Q4_K, 200, lambda r: synth.gen_blocks_full_range(synth.Q4_K, 200 * n // 256, r)),
        (2, synth.Q4_K, 128, lambda r: q4k_cancelling_blocks(128 * n // 256, r, "near")),
    ]
    items, lv, host = [], [], []
    xs = [rng.standard_normal((1, n), dtype=np.float32) for _ in range(3)]
    xd = [torch.from_numpy(a).cuda() for a in xs]
    for level, t, rows, make in spec:
        W = make(rng)
        y = torch.full((1, rows), float("nan"), device="cuda")
        items.append((t, torch.from_numpy(W).cuda(), rows, n, xd[level], y))
        lv.append(level)
        host.append((t, W, rows, xs[level], y))
    plan = q.Plan(items, lv, 1)
    plan.run()
    torch.cuda.synchronize()
    assert q.get_device_status() == 0
    for t, W, rows, x, y in host:
        y_ref, S = orc.gemv(t, W, rows, n, x)
        assert_close(y.cpu().numpy(), y_ref, S, f"plan level {synth.TYPE_NAMES[t]} {rows}")
    plan.close()
