"""GPU parity of the batched (tensor-core) GEMV path, batch >= 9, against the oracle.

The batched path multiplies each scale group's integer quants (exact in bf16,
recentred for Q4_K) by x split into bf16 hi + lo terms, accumulates the group
sums in fp32 in tensor memory and applies the group's scale (and, for Q4_K, its
min) in fp32; it must meet the same per-output bound as the streaming path,
|y - y_ref| <= 1e-5 * sum|w x| + 1e-7.
The cases cover every format, ragged row tiles, ragged K (q8_0/q4_0 widths
that are not a multiple of 256), split-K clusters of 1 to 8 CTAs, batches past
one 128-wide chunk, a matrix whose byte length is not a multiple of 16, and
run-to-run determinism.
"""
import numpy as np
import pytest

from quant_dequant_gemv_gb300 import synth

from .test_gpu_parity import assert_close, bits_equal, dev, q, run_gemv, sampled_rows, check_rows  # noqa: F401

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

TYPES = [synth.Q4_K, synth.Q6_K, synth.Q8_0, synth.Q4_0]


def worst_rel(y, y_ref, S):
    return float(np.max(np.abs(y.astype(np.float64) - y_ref) / np.maximum(S, 1e-30)))


@pytest.mark.parametrize("qtype", TYPES)
@pytest.mark.parametrize("batch", [4, 5, 9, 16, 33, 64])
def test_batched_all_formats_ragged(q, orc, qtype, batch):
    # batch 4: q8_0 on the tensor cores, the other formats on the streaming kernel
    rows = 300  # three row tiles, the last one 44 rows
    cols = 1024 if qtype in (synth.Q4_K, synth.Q6_K) else 416  # 416 = 256 + 160: a ragged last unit
    W = synth.gen_matrix(qtype, rows, cols, 80 + batch)
    x = synth.gen_x(batch, cols, 90 + batch)
    y = run_gemv(q, qtype, W, rows, cols, x)
    y_ref, S = orc.gemv(qtype, W, rows, cols, x)
    assert_close(y, y_ref, S, f"{synth.TYPE_NAMES[qtype]} batch {batch}")
    print(f"{synth.TYPE_NAMES[qtype]} b{batch}: worst |y-y_ref|/S = {worst_rel(y, y_ref, S):.3e}")


@pytest.mark.parametrize("units", [2, 5, 9])
def test_batched_split_k_cluster(q, orc, units):
    # one row tile, so the K range is split over min(8, units) CTAs of one cluster
    rows, cols, batch = 128, 256 * units, 24
    W = synth.gen_matrix(synth.Q4_K, rows, cols, 120 + units)
    x = synth.gen_x(batch, cols, 130 + units)
    y = run_gemv(q, synth.Q4_K, W, rows, cols, x)
    y_ref, S = orc.gemv(synth.Q4_K, W, rows, cols, x)
    assert_close(y, y_ref, S, f"split-K over {units} units")


def test_batched_many_row_tiles_no_split(q, orc):
    # more row tiles than SMs: one CTA per tile, no cluster
    rows, cols, batch = 152 * 128 + 3, 512, 16
    W = synth.gen_matrix(synth.Q6_K, rows, cols, 140)
    x = synth.gen_x(batch, cols, 141)
    y = run_gemv(q, synth.Q6_K, W, rows, cols, x)
    check_rows(orc, synth.Q6_K, W, rows, cols, x, y, sampled_rows(rows, 128), "19459x512 b16")


def test_batched_past_one_chunk(q, orc):
    rows, cols, batch = 200, 512, 130  # batch slices of 128 and 2
    W = synth.gen_matrix(synth.Q6_K, rows, cols, 150)
    x = synth.gen_x(batch, cols, 151)
    y = run_gemv(q, synth.Q6_K, W, rows, cols, x)
    y_ref, S = orc.gemv(synth.Q6_K, W, rows, cols, x)
    assert_close(y, y_ref, S, "batch 130")


@pytest.mark.parametrize("qtype,rows,cols", [(synth.Q6_K, 3, 256), (synth.Q4_0, 5, 32), (synth.Q8_0, 7, 96)])
def test_batched_matrix_length_not_multiple_of_16(q, orc, qtype, rows, cols):
    W = synth.gen_matrix(qtype, rows, cols, 160)
    assert W.nbytes % 16 != 0
    x = synth.gen_x(16, cols, 161)
    y = run_gemv(q, qtype, W, rows, cols, x)
    y_ref, S = orc.gemv(qtype, W, rows, cols, x)
    assert_close(y, y_ref, S, f"{synth.TYPE_NAMES[qtype]} {rows}x{cols}")


def test_batched_deterministic(q):
    rows, cols, batch = 2048, 5632, 16
    W = dev(synth.gen_matrix(synth.Q6_K, rows, cols, 170))
    x = dev(synth.gen_x(batch, cols, 171))
    ys = []
    for _ in range(3):
        y = torch.full((batch, rows), float("nan"), device="cuda")
        q.gemv(synth.Q6_K, W, rows, cols, x, y, batch)
        torch.cuda.synchronize()
        ys.append(y.cpu().numpy())
    assert q.get_device_status() == 0
    assert bits_equal(ys[0], ys[1]) and bits_equal(ys[0], ys[2])
