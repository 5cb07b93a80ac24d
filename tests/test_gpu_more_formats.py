"""Q5_0, Q5_1, ggml q8_0, Q2_K, Q5_K and Q3_K on the GPU against the oracle (ggml block
layouts, a reading: the pages name the formats and give Q2_K's size).

* Dequantisation bit for bit, on the workload draws and on full-range bytes.
* qdq_gemv within |y - y_ref| <= 1e-5 sum|w x| + 1e-7, at batch widths 1, 3, 8
  and 11 (two slices of the eight-column kernel), on both draws, including
  rows of a few blocks and long rows.
* Groups and plans refuse these types (QDQ_ERR_TYPE).
"""
import numpy as np
import pytest

import oracle
from quant_dequant_gemv_gb300 import synth

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")

TYPES = [synth.Q5_0, synth.Q5_1, synth.Q8_0G, synth.Q2_K, synth.Q5_K, synth.Q3_K]


@pytest.fixture(scope="module")
def q():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from quant_dequant_gemv_gb300 import build, qdq
    build.build()
    torch.cuda.set_device(0)
    return qdq


def blocks(qtype, nblocks, rng, full):
    return (synth.gen_blocks_full_range if full else synth.gen_blocks)(qtype, nblocks, rng)


@pytest.mark.parametrize("qtype", TYPES)
@pytest.mark.parametrize("full", [False, True])
def test_dequant_bit_exact(q, qtype, full):
    rng = np.random.default_rng(qtype * 3 + full)
    for nblocks in (1, 7, 4099):
        n = nblocks * synth.BLOCK_WEIGHTS[qtype]
        B = blocks(qtype, nblocks, rng, full)
        out = torch.full((n,), float("nan"), device="cuda")
        q.dequant(qtype, torch.from_numpy(B).cuda(), n, out)
        assert q.get_device_status() == 0
        np.testing.assert_array_equal(out.cpu().numpy().view(np.uint32),
                                      oracle.dequant(qtype, B, n).view(np.uint32))


@pytest.mark.parametrize("qtype", TYPES)
@pytest.mark.parametrize("batch", [1, 3, 8, 11])
@pytest.mark.parametrize("full", [False, True])
def test_gemv_parity(q, qtype, batch, full):
    rng = np.random.default_rng(100 * qtype + batch + 7 * full)
    for rows, cols in [(97, 256), (37, 5632), (300, 2048)]:
        W = blocks(qtype, rows * cols // synth.BLOCK_WEIGHTS[qtype], rng, full)
        x = rng.standard_normal((batch, cols)).astype(np.float32)
        y = torch.full((batch, rows), float("nan"), device="cuda")
        q.gemv(qtype, torch.from_numpy(W).cuda(), rows, cols, torch.from_numpy(x).cuda(), y, batch)
        assert q.get_device_status() == 0
        y_ref, S = oracle.gemv(qtype, W, rows, cols, x)
        ok = np.abs(y.cpu().numpy().astype(np.float64) - y_ref) <= 1e-5 * S + 1e-7
        assert ok.all(), f"{synth.TYPE_NAMES[qtype]} {rows}x{cols} batch {batch}: {int((~ok).sum())} out"


def test_groups_and_plans_refuse_the_further_formats(q):
    W = torch.zeros(8 * 22, dtype=torch.uint8, device="cuda")
    x = torch.zeros(1, 32, device="cuda")
    y = torch.zeros(1, 8, device="cuda")
    with pytest.raises(q.QdqError) as e:
        q.gemv_group([(synth.Q5_0, W, 8, 32, x, y)], 1)
    assert e.value.rc == -1
    with pytest.raises(q.QdqError):
        q.Plan([(synth.Q5_0, W, 8, 32, x, y)], [0], 1)
