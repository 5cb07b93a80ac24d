"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle.

Dequantisation must match bit for bit (NaN compared as NaN). The GEMV must meet
|y - y_ref| <= 1e-5 * sum|w x| + 1e-7 elementwise, y_ref and sum|w x| from the
oracle in double precision.
"""
import numpy as np
import pytest

import oracle
from quant_dequant_gemv_gb300 import synth

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

TYPES = [synth.Q4_K, synth.Q6_K, synth.Q8_0, synth.Q4_0]
REL, ABS = 1e-5, 1e-7


@pytest.fixture(scope="module")
def q():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from quant_dequant_gemv_gb300 import build, qdq
    build.build()
    torch.cuda.set_device(0)
    return qdq


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def run_gemv(q, qtype, W, rows, cols, x):
    batch = x.shape[0]
    y = torch.full((batch, rows), float("nan"), device="cuda")
    q.gemv(qtype, dev(W), rows, cols, dev(x), y, batch)
    torch.cuda.synchronize()
    return y.cpu().numpy()


def assert_close(y, y_ref, S, what=""):
    ok = oracle.within_tolerance(y, y_ref, S, REL, ABS)
    if not ok.all():
        i = np.argwhere(~ok)[0]
        raise AssertionError(f"{what}: {int((~ok).sum())} outputs out of tolerance; first {tuple(i)}: "
                             f"y={y[tuple(i)]!r} ref={y_ref[tuple(i)]!r} S={S[tuple(i)]!r}")


def bits_equal(a, b):
    nan = np.isnan(a) & np.isnan(b)
    return np.all(nan | (a.view(np.uint32) == b.view(np.uint32)))


# ----------------------------------------------------------------- dequant ---
@pytest.mark.parametrize("qtype", TYPES)
@pytest.mark.parametrize("nblocks", [1, 7, 1000, 4099])
def test_dequant_bit_exact_workload(q, orc, qtype, nblocks):
    rng = np.random.default_rng(100 + nblocks)
    blocks = synth.gen_blocks(qtype, nblocks, rng)
    n = nblocks * synth.BLOCK_WEIGHTS[qtype]
    out = torch.empty(n, device="cuda")
    q.dequant(qtype, dev(blocks), n, out)
    torch.cuda.synchronize()
    assert bits_equal(out.cpu().numpy(), orc.dequant(qtype, blocks, n))


@pytest.mark.parametrize("qtype", TYPES)
def test_dequant_bit_exact_any_bytes(q, orc, qtype):
    # every byte pattern is a valid block: subnormal, infinite and NaN scales,
    # negative scales, signed zeros
    rng = np.random.default_rng(7)
    nblocks = 3000
    blocks = rng.integers(0, 256, nblocks * synth.BLOCK_BYTES[qtype], dtype=np.uint8)
    n = nblocks * synth.BLOCK_WEIGHTS[qtype]
    out = torch.empty(n, device="cuda")
    q.dequant(qtype, dev(blocks), n, out)
    torch.cuda.synchronize()
    got, want = out.cpu().numpy(), orc.dequant(qtype, blocks, n)
    assert bits_equal(got, want)
    assert np.array_equal(np.signbit(got[~np.isnan(got)]), np.signbit(want[~np.isnan(want)]))


# -------------------------------------------------------------------- gemv ---
SMALL_SHAPES = {
    synth.Q4_K: [(1, 256), (3, 512), (33, 2048), (97, 5632), (300, 1024)],
    synth.Q6_K: [(1, 256), (5, 768), (33, 2048), (41, 5632), (129, 1280)],
    synth.Q8_0: [(1, 32), (3, 96), (17, 4096), (65, 2080), (200, 544)],
    synth.Q4_0: [(1, 32), (3, 96), (17, 4096), (65, 2080), (201, 544)],
}


@pytest.mark.parametrize("qtype", TYPES)
def test_gemv_batch1_small_shapes(q, orc, qtype):
    for i, (rows, cols) in enumerate(SMALL_SHAPES[qtype]):
        W = synth.gen_matrix(qtype, rows, cols, 10 + i)
        x = synth.gen_x(1, cols, 20 + i)
        y = run_gemv(q, qtype, W, rows, cols, x)
        y_ref, S = orc.gemv(qtype, W, rows, cols, x)
        assert_close(y, y_ref, S, f"{synth.TYPE_NAMES[qtype]} {rows}x{cols}")


@pytest.mark.parametrize("qtype", TYPES)
@pytest.mark.parametrize("batch", [2, 3, 4, 5, 8])
def test_gemv_small_batches(q, orc, qtype, batch):
    rows, cols = (70, 2048) if qtype in (synth.Q4_K, synth.Q6_K) else (70, 4096)
    W = synth.gen_matrix(qtype, rows, cols, 30 + batch)
    x = synth.gen_x(batch, cols, 40 + batch)
    y = run_gemv(q, qtype, W, rows, cols, x)
    y_ref, S = orc.gemv(qtype, W, rows, cols, x)
    assert_close(y, y_ref, S, f"{synth.TYPE_NAMES[qtype]} batch {batch}")


@pytest.mark.parametrize("qtype", [synth.Q4_K, synth.Q6_K])
@pytest.mark.parametrize("batch", [9, 16, 64])
def test_gemv_large_batches(q, orc, qtype, batch):
    rows, cols = 200, 2048
    W = synth.gen_matrix(qtype, rows, cols, 50 + batch)
    x = synth.gen_x(batch, cols, 60 + batch)
    y = run_gemv(q, qtype, W, rows, cols, x)
    y_ref, S = orc.gemv(qtype, W, rows, cols, x)
    assert_close(y, y_ref, S, f"{synth.TYPE_NAMES[qtype]} batch {batch}")


@pytest.mark.parametrize("qtype,cols", [(synth.Q8_0, 32768), (synth.Q4_K, 20480), (synth.Q6_K, 16896),
                                        (synth.Q4_0, 32800)])
def test_gemv_wide_rows_column_chunks(q, orc, qtype, cols):
    # x no longer fits the shared-memory x buffer: the kernel splits columns
    rows = 37
    for batch in (1, 3):
        W = synth.gen_matrix(qtype, rows, cols, 70)
        x = synth.gen_x(batch, cols, 71)
        y = run_gemv(q, qtype, W, rows, cols, x)
        y_ref, S = orc.gemv(qtype, W, rows, cols, x)
        assert_close(y, y_ref, S, f"{synth.TYPE_NAMES[qtype]} cols {cols} batch {batch}")


@pytest.mark.parametrize("qtype,rows,cols", [(synth.Q8_0, 3648, 16384), (synth.Q4_0, 3000, 4096),
                                             (synth.Q8_0, 3000, 4096), (synth.Q4_0, 2000, 32800),
                                             (synth.Q6_K, 2000, 16896)])
def test_gemv_many_rows_per_cta(q, orc, qtype, rows, cols):
    # 13-24 rows per CTA: multi-pass tiles of padded whole rows (row length a
    # multiple of 128 bytes) and of column chunks (aligned and unaligned rows)
    for batch in (1, 3):
        W = synth.gen_matrix(qtype, rows, cols, 75)
        x = synth.gen_x(batch, cols, 76)
        y = run_gemv(q, qtype, W, rows, cols, x)
        y_ref, S = orc.gemv(qtype, W, rows, cols, x)
        assert_close(y, y_ref, S, f"{synth.TYPE_NAMES[qtype]} {rows}x{cols} batch {batch}")


def test_gemv_guard_bytes_and_determinism(q, orc):
    qtype, rows, cols = synth.Q6_K, 77, 5632
    W = synth.gen_matrix(qtype, rows, cols, 80)
    x = synth.gen_x(1, cols, 81)
    buf = torch.full((rows + 64,), 12345.0, device="cuda")
    y = buf[32:32 + rows]
    Wd, xd = dev(W), dev(x)
    q.gemv(qtype, Wd, rows, cols, xd, y, 1)
    first = y.clone()
    q.gemv(qtype, Wd, rows, cols, xd, y, 1)
    torch.cuda.synchronize()
    host = buf.cpu().numpy()
    assert np.all(host[:32] == 12345.0) and np.all(host[32 + rows:] == 12345.0)
    assert torch.equal(first, y)
    y_ref, S = orc.gemv(qtype, W, rows, cols, x)
    assert_close(y.cpu().numpy()[None, :], y_ref, S)


def test_gemv_zero_cols_writes_zeros(q):
    y = torch.full((2, 5), 3.0, device="cuda")
    x = torch.zeros(16, device="cuda")
    W = torch.zeros(16, dtype=torch.uint8, device="cuda")
    q.gemv(synth.Q4_K, W, 5, 0, x, y, 2)
    torch.cuda.synchronize()
    assert torch.count_nonzero(y) == 0


# ------------------------------------------------------- the listed workloads ---
def sampled_rows(rows, k=192):
    # first and last tiles plus evenly spread rows
    idx = set(range(min(32, rows))) | set(range(max(0, rows - 32), rows))
    idx |= set(np.linspace(0, rows - 1, k).astype(int).tolist())
    return sorted(idx)


def check_rows(orc, qtype, W, rows, cols, x, y, rowset, what):
    rb = synth.row_bytes(qtype, cols)
    for r in rowset:
        y_ref, S = orc.gemv(qtype, W[r * rb:(r + 1) * rb], 1, cols, x)
        assert_close(y[:, r:r + 1], y_ref, S, f"{what} row {r}")


def test_q4k_2048x2048_batch1_full(q, orc):
    g = synth.Q4K_2048x2048
    W = synth.gen_matrix(g.qtype, g.rows, g.cols, 0)
    x = synth.gen_x(1, g.cols, 1000)
    y = run_gemv(q, g.qtype, W, g.rows, g.cols, x)
    y_ref, S = orc.gemv(g.qtype, W, g.rows, g.cols, x)
    assert_close(y, y_ref, S, g.name)


def test_q6k_2048x5632_batch1_full(q, orc):
    g = synth.Q6K_2048x5632
    W = synth.gen_matrix(g.qtype, g.rows, g.cols, 0)
    x = synth.gen_x(1, g.cols, 1000)
    y = run_gemv(q, g.qtype, W, g.rows, g.cols, x)
    y_ref, S = orc.gemv(g.qtype, W, g.rows, g.cols, x)
    assert_close(y, y_ref, S, g.name)


@pytest.mark.parametrize("batch", [1, 4, 16, 64])
def test_ffn_shapes_batched(q, orc, batch):
    for qtype, rows, cols in [(synth.Q4_K, 5632, 2048), (synth.Q6_K, 2048, 5632)]:
        W = synth.gen_matrix(qtype, rows, cols, 3)
        x = synth.gen_x(batch, cols, 1003)
        y = run_gemv(q, qtype, W, rows, cols, x)
        check_rows(orc, qtype, W, rows, cols, x, y, sampled_rows(rows, 96), f"{rows}x{cols} b{batch}")


@pytest.mark.parametrize("qtype", [synth.Q8_0, synth.Q4_0])
@pytest.mark.parametrize("batch", [1, 8])
def test_petit_8b_ffn_shapes(q, orc, qtype, batch):
    for rows, cols in [(14336, 4096), (4096, 14336)]:
        W = synth.gen_matrix(qtype, rows, cols, 5)
        x = synth.gen_x(batch, cols, 1005)
        y = run_gemv(q, qtype, W, rows, cols, x)
        check_rows(orc, qtype, W, rows, cols, x, y, sampled_rows(rows, 64), f"{rows}x{cols} b{batch}")


# ------------------------------------------------------------ groups, plans ---
def test_group_qkv_mixed_formats(q, orc):
    cols = 2048
    x = synth.gen_x(1, cols, 90)
    xd = dev(x)
    specs = [(synth.Q4_K, 2048), (synth.Q4_K, 256), (synth.Q6_K, 256)]
    Ws = [synth.gen_matrix(t, r, cols, 91 + i) for i, (t, r) in enumerate(specs)]
    ys = [torch.empty(1, r, device="cuda") for _, r in specs]
    items = [(t, dev(W), r, cols, xd, y) for (t, r), W, y in zip(specs, Ws, ys)]
    q.gemv_group(items, 1)
    torch.cuda.synchronize()
    for (t, r), W, y in zip(specs, Ws, ys):
        y_ref, S = orc.gemv(t, W, r, cols, x)
        assert_close(y.cpu().numpy(), y_ref, S, f"group {synth.TYPE_NAMES[t]}")


def build_step(n_layers, seed=0):
    """Device buffers and plan items for n_layers of the 1.1B decode step."""
    levels = synth.llama_1b_step(n_layers)
    items, lv, host = [], [], []
    for li, level in enumerate(levels):
        x = synth.gen_x(1, level[0].cols, seed + 1000 + li)
        xd = dev(x)
        for gi, g in enumerate(level):
            W = synth.gen_matrix(g.qtype, g.rows, g.cols, seed + 10 * li + gi)
            y = torch.full((1, g.rows), float("nan"), device="cuda")
            items.append((g.qtype, dev(W), g.rows, g.cols, xd, y))
            lv.append(li)
            host.append((g, W, x))
    return items, lv, host


def test_plan_two_layers_repeated_runs(q, orc):
    items, lv, host = build_step(2)
    plan = q.Plan(items, lv, 1)
    outs = []
    for _ in range(3):
        for it in items:
            it[5].fill_(float("nan"))
        plan.run()
        torch.cuda.synchronize()
        outs.append([it[5].cpu().numpy().copy() for it in items])
    assert q.get_device_status() == 0
    for run in outs[1:]:  # deterministic across runs (the level counters reset themselves)
        for a, b in zip(outs[0], run):
            assert np.array_equal(a, b)
    for (g, W, x), y in zip(host, outs[0]):
        check_rows(orc, g.qtype, W, g.rows, g.cols, x, y, sampled_rows(g.rows, 48), g.name)
    plan.close()


def test_plan_run_io_host_buffers(q, orc):
    items, lv, host = build_step(1)
    plan = q.Plan(items, lv, 1)
    xs = []
    for g, W, x in host:
        if not any(x is seen for seen in xs):
            xs.append(x)
    x_host = torch.from_numpy(np.concatenate([a.reshape(-1) for a in xs])).pin_memory()
    y_host = torch.empty(sum(g.rows for g, _, _ in host), dtype=torch.float32).pin_memory()
    h2d, d2h = plan.run_io(x_host, y_host)
    torch.cuda.synchronize()
    assert h2d == x_host.numel() * 4 and d2h == y_host.numel() * 4
    off = 0
    for g, W, x in host:
        y = y_host[off:off + g.rows].numpy()[None, :]
        check_rows(orc, g.qtype, W, g.rows, g.cols, x, y, sampled_rows(g.rows, 16), g.name)
        off += g.rows
    plan.close()


@pytest.mark.parametrize("batch", [1, 3, 8])
def test_plan_chained_levels_read_previous_outputs(q, orc, batch):
    """A plan whose levels consume the previous level's outputs (x of level L+1 is a
    y of level L), in every format and with side outputs, run twice, at batch 1, 3
    (a padded batch width) and 8. Each level is checked against the oracle applied
    to the input it actually read from the GPU: a level that started before its
    input was complete would have read NaN or stale values (every y starts as NaN)."""
    n = 2048
    spec = [  # (level, name, format, rows, x from)
        (0, "A", synth.Q4_K, n, "x0"), (0, "B", synth.Q6_K, 512, "x0"),
        (1, "C", synth.Q6_K, n, "A"),
        (2, "D", synth.Q8_0, n, "C"), (2, "E", synth.Q4_0, 1024, "C"),
        (3, "F", synth.Q4_0, n, "D"),
    ]
    x0 = synth.gen_x(batch, n, 4242)
    bufs = {"x0": dev(x0)}
    items, lv, Ws = [], [], {}
    for li, name, t, rows, src in spec:
        Ws[name] = synth.gen_matrix(t, rows, n, 300 + len(items))
        bufs[name] = torch.full((batch, rows), float("nan"), device="cuda")
        items.append((t, dev(Ws[name]), rows, n, bufs[src], bufs[name]))
        lv.append(li)
    plan = q.Plan(items, lv, batch)
    for _ in range(2):
        for _, name, _, _, _ in spec:
            bufs[name].fill_(float("nan"))
        plan.run()
        torch.cuda.synchronize()
        assert q.get_device_status() == 0
        got = {k: v.cpu().numpy() for k, v in bufs.items()}
        for _, name, t, rows, src in spec:
            assert not np.isnan(got[name]).any(), name
            y_ref, S = orc.gemv(t, Ws[name], rows, n, got[src].astype(np.float32))
            assert y_ref.shape == (batch, rows)
            assert_close(got[name], y_ref, S, f"level output {name}")
    plan.close()


def test_full_decode_step_sampled(q, orc):
    """The 22-layer, 155-GEMV step in the launch configuration the benchmark
    times, checked on sampled rows of every GEMV."""
    items, lv, host = build_step(22)
    plan = q.Plan(items, lv, 1)
    plan.run()
    plan.run()
    torch.cuda.synchronize()
    assert q.get_device_status() == 0
    for (g, W, x), it in zip(host, items):
        y = it[5].cpu().numpy()
        assert not np.isnan(y).any(), g.name
        check_rows(orc, g.qtype, W, g.rows, g.cols, x, y, sampled_rows(g.rows, 8)[:24], g.name)
    plan.close()


# ------------------------------------------------------------------ errors ---
def test_errors_host_and_misaligned_pointers(q):
    from quant_dequant_gemv_gb300.qdq import QdqError
    W = torch.zeros(144 * 8, dtype=torch.uint8, device="cuda")
    x = torch.zeros(2048 + 4, device="cuda")
    y = torch.zeros(8, device="cuda")
    host_x = torch.zeros(2048)
    with pytest.raises(QdqError) as e:
        q.gemv(synth.Q4_K, W, 1, 2048, host_x, y, 1)
    assert e.value.rc == -4
    with pytest.raises(QdqError) as e:
        q.gemv(synth.Q4_K, W, 1, 2048, x[1:], y, 1)  # 4-byte offset
    assert e.value.rc == -3
    with pytest.raises(QdqError) as e:
        q.gemv(synth.Q4_K, W, 1, 2000, x, y, 1)
    assert e.value.rc == -2
    with pytest.raises(QdqError) as e:
        q.gemv(99, W, 1, 2048, x, y, 1)  # no such type
    assert e.value.rc == -1


def test_bounded_wait_times_out_and_context_survives(q, orc):
    q.selftest_wait_timeout(2_000_000)  # 2 ms on a flag nothing sets
    assert q.get_device_status() == -6
    assert q.get_device_status() == 0  # read-and-clear
    # the context is still usable
    W = synth.gen_matrix(synth.Q4_K, 8, 256, 1)
    x = synth.gen_x(1, 256, 2)
    y = run_gemv(q, synth.Q4_K, W, 8, 256, x)
    y_ref, S = orc.gemv(synth.Q4_K, W, 8, 256, x)
    assert_close(y, y_ref, S)
