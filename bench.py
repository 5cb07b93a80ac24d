"""Benchmark: the fused dequant-GEMV decode step on GB300.

Default workload: one batch-1 decode step of the 1.1B Llama shape (22 layers,
hidden 2048, 32/4 heads of 64, FFN 5632, vocab 32000; Q4_K for attn_q/k/o and
ffn_gate/up, Q6_K for attn_v, ffn_down and the output head), seeded random
blocks, a fresh N(0,1) input per dependency level. One step = one persistent
launch of the plan (155 GEMVs in 89 dependency levels). The 667 MB of weights
exceed the 129 MB L2 several times over, so no flush is needed between steps.

Prints one JSON line. `value` is HBM GB/s of algorithmic bytes (weights + x + y
per step) over the device-timed step; `tok_s` is steps per second.
  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload step|q4k|q6k|ffn_q4k|ffn_q6k|q8_0|q4_0|dequant_q4k|dequant_q6k|
                              dequant_q8_0|dequant_q4_0] [--batch B]
Under torchrun each rank runs an independent replica (the path has no data
exchange); rank 0 prints the aggregate.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time
from pathlib import Path

import numpy as np

ROOT = Path(__file__).resolve().parent
sys.path.insert(0, str(ROOT))

from quant_dequant_gemv_gb300 import synth  # noqa: E402

METRIC = "fused dequant-GEMV HBM GB/s (% of GB300 peak); 1.1B-shape decode-step tok/s"

WORKLOADS = {
    "step": "1.1B Llama-shape decode step, batch 1: 22 layers, Q4_K_M mix (Q4_K attn_q/k/o, ffn_gate/up; "
            "Q6_K attn_v, ffn_down, output 32000x2048), 155 GEMVs in 89 dependency levels, "
            "667,152,384 weight bytes",
    "q4k": "single Q4_K GEMV 2048x2048",
    "q6k": "single Q6_K GEMV 2048x5632",
    "ffn_q4k": "Q4_K GEMV 5632x2048 (ffn_gate/up shape)",
    "ffn_q6k": "Q6_K GEMV 2048x5632 (ffn_down shape)",
    "q8_0": "PETIT q8_0 GEMVs 14336x4096 and 4096x14336",
    "q4_0": "PETIT q4_0 GEMVs 14336x4096 and 4096x14336",
    "token": "1.1B Llama-shape token step, batch 1, greedy decode: embedding row, 22 layers of rmsnorm -> "
             "q/k/v -> RoPE + fp16 KV cache + GQA attention -> o + residual -> rmsnorm -> gate/up -> SwiGLU -> "
             "down + residual, final rmsnorm -> output head + argmax (Q4_K_M mix, 667,152,384 GEMV weight bytes)",
    "ffn_q5_0": "Q5_0 GEMV 5632x2048 (ffn_gate/up shape; ggml layout)",
    "ffn_q5_1": "Q5_1 GEMV 5632x2048 (ffn_gate/up shape; ggml layout)",
    "ffn_q8_0g": "ggml q8_0 (fp16 scale) GEMV 5632x2048 (ffn_gate/up shape)",
    "ffn_q2k": "Q2_K GEMV 5632x2048 (ffn_gate/up shape; ggml layout)",
    "ffn_q5k": "Q5_K GEMV 5632x2048 (ffn_gate/up shape; ggml layout)",
    "ffn_q3k": "Q3_K GEMV 5632x2048 (ffn_gate/up shape; ggml layout)",
    "dequant_q4k": "standalone dequantisation, Q4_K, 2^27 weights -> fp32",
    "dequant_q6k": "standalone dequantisation, Q6_K, 2^27 weights -> fp32",
    "dequant_q8_0": "standalone dequantisation, PETIT q8_0, 2^27 weights -> fp32",
    "dequant_q4_0": "standalone dequantisation, PETIT q4_0, 2^27 weights -> fp32",
    "dequant_q5_1": "standalone dequantisation, Q5_1 (ggml layout), 2^27 weights -> fp32",
    "dequant_q2k": "standalone dequantisation, Q2_K (ggml layout), 2^27 weights -> fp32",
    "dequant_q5k": "standalone dequantisation, Q5_K (ggml layout), 2^27 weights -> fp32",
    "dequant_q3k": "standalone dequantisation, Q3_K (ggml layout), 2^27 weights -> fp32",
}
MORE_GEMV = {"ffn_q5_0": synth.Q5_0, "ffn_q5_1": synth.Q5_1, "ffn_q8_0g": synth.Q8_0G, "ffn_q2k": synth.Q2_K,
             "ffn_q5k": synth.Q5_K, "ffn_q3k": synth.Q3_K}
DEQUANT_TYPES = {"dequant_q4k": synth.Q4_K, "dequant_q6k": synth.Q6_K, "dequant_q8_0": synth.Q8_0,
                 "dequant_q4_0": synth.Q4_0, "dequant_q5_1": synth.Q5_1, "dequant_q2k": synth.Q2_K,
                 "dequant_q5k": synth.Q5_K, "dequant_q3k": synth.Q3_K}
DEQUANT_N = 1 << 27  # weights per dequantisation step: in + out bytes are several times L2


def workload_levels(name: str, layers: int = 22) -> list[list[synth.Gemv]]:
    if name == "token":
        return synth.llama_1b_step(layers)
    if name in DEQUANT_TYPES:
        return []
    if name == "step":
        return synth.llama_1b_step(layers)
    if name == "q4k":
        return [[synth.Q4K_2048x2048]]
    if name == "q6k":
        return [[synth.Q6K_2048x5632]]
    if name == "ffn_q4k":
        return [[synth.Gemv("ffn_gate", synth.Q4_K, 5632, 2048)]]
    if name == "ffn_q6k":
        return [[synth.Gemv("ffn_down", synth.Q6_K, 2048, 5632)]]
    if name in MORE_GEMV:
        return [[synth.Gemv("ffn_gate", MORE_GEMV[name], 5632, 2048)]]
    if name in ("q8_0", "q4_0"):
        t = synth.Q8_0 if name == "q8_0" else synth.Q4_0
        return [[synth.Gemv("w_up", t, 14336, 4096)], [synth.Gemv("w_down", t, 4096, 14336)]]
    raise SystemExit(f"unknown workload {name}")


def dequant_bytes(qtype: int, n: int) -> int:
    """Standalone dequantisation: the blocks read once, n floats written once."""
    return n // synth.BLOCK_WEIGHTS[qtype] * synth.BLOCK_BYTES[qtype] + 4 * n


def algorithmic_bytes(levels, batch: int) -> int:
    """Weights once, each level's x once, every y once."""
    w = sum(g.weight_bytes for lv in levels for g in lv)
    x = sum(4 * batch * lv[0].cols for lv in levels)
    y = sum(4 * batch * g.rows for lv in levels for g in lv)
    return w + x + y


def load_peaks() -> dict:
    p = ROOT / "MEASURED_PEAKS.json"
    if p.exists():
        d = json.loads(p.read_text())
        return {"hbm_gbs": float(d["hbm_gbs"]), "source": "measured"}
    return {"hbm_gbs": 6800.0, "source": "fallback"}


def kernel_source_hash(exclude=()) -> str:
    """Hash of the kernel sources' code: line comments and blank lines are left
    out, so an edit to comments keeps recorded counters valid. `exclude` names
    source files the recorded kernel is not built from."""
    h = hashlib.sha256()
    for f in sorted((ROOT / "quant_dequant_gemv_gb300" / "csrc").glob("*")):
        if f.name in exclude:
            continue
        for line in f.read_text().splitlines():
            code = line.split("//", 1)[0].rstrip()
            if code:
                h.update(code.encode() + b"\n")
    return h.hexdigest()[:16]


def recorded_traffic(workload: str, batch: int):
    """DRAM bytes per launch from a committed ncu summary, if it was taken on the
    current sources of its kernel; else None."""
    p = ROOT / "profiles" / "dram_traffic.json"
    if not p.exists():
        return None
    d = json.loads(p.read_text())
    e = d.get(f"{workload}/b{batch}")
    if not e or e.get("source_hash") != kernel_source_hash(tuple(e.get("excluded_sources", ()))):
        return None
    return e.get("bytes_per_launch")


class ClockSampler:
    """nvidia-smi clock/throttle samples while the GPU is under load."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.file = None

    def start(self):
        try:
            self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=self.file, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self) -> dict | None:
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.file.flush()
        rows = []
        for line in Path(self.file.name).read_text().splitlines():
            f = [c.strip() for c in line.split(",")]
            if len(f) < 9:
                continue
            try:
                rows.append((float(f[1]), float(f[2]), f[5], f[6], f[7], f[8]))
            except ValueError:
                continue
        os.unlink(self.file.name)
        if not rows:
            return None
        reasons = set()
        for _, _, hw, hwt, swt, swp in rows:
            if hw == "Active":
                reasons.add("hw_slowdown")
            if hwt == "Active":
                reasons.add("hw_thermal_slowdown")
            if swt == "Active":
                reasons.add("sw_thermal_slowdown")
            if swp == "Active":
                reasons.add("sw_power_cap")
        return {"sm_mhz": statistics.median(r[0] for r in rows), "sm_max_mhz": max(r[1] for r in rows),
                "samples": len(rows), "reasons": sorted(reasons)}


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------
def build_inputs(levels, batch, device, seed=0):
    """Weights per GEMV; the activations live in two arenas (every level's x, then
    every y, back to back in plan order), as a serving engine lays them out, so the
    plan's host<->device transfers are one copy each way."""
    import torch
    items, lv = [], []
    xs_host = [synth.gen_x(batch, level[0].cols, seed + 1000 + li) for li, level in enumerate(levels)]
    x_all = torch.from_numpy(np.concatenate([a.reshape(-1) for a in xs_host])).to(device)
    y_all = torch.empty(sum(batch * g.rows for level in levels for g in level), dtype=torch.float32, device=device)
    xo = yo = 0
    for li, level in enumerate(levels):
        nx = batch * level[0].cols
        xd = x_all[xo:xo + nx].view(batch, level[0].cols)
        xo += nx
        for gi, g in enumerate(level):
            W = synth.gen_matrix(g.qtype, g.rows, g.cols, seed + 10 * li + gi)
            y = y_all[yo:yo + batch * g.rows].view(batch, g.rows)
            yo += batch * g.rows
            items.append((g.qtype, torch.from_numpy(W).to(device), g.rows, g.cols, xd, y))
            lv.append(li)
    return items, lv, xs_host


L2_BYTES = 129 * 2 ** 20   # GB300 L2
def mma_min_batch(qtype):  # single GEMVs from this batch on run on the tensor cores (library dispatch)
    if qtype in MORE_GEMV.values():
        return 1 << 30  # the further formats always run gemv_more_kernel
    return 4 if qtype in (synth.Q8_0, synth.Q4_0) else 5
GROUP = 8                  # single-GEMV workloads: steps per replayed CUDA graph


def gemv_launches(g, batch):
    """Kernel launches of one qdq_gemv call (mirrors the library's dispatch)."""
    if g.qtype in MORE_GEMV.values():
        return (batch + 7) // 8  # gemv_more_kernel per slice of at most 8 columns
    if batch < mma_min_batch(g.qtype):
        return 1
    per = 32 if g.qtype == synth.Q6_K else 64
    return (batch + per - 1) // per  # one tensor-core launch per batch slice


def run_dequant(args, device):
    """Standalone dequantisation: one qdq_dequant call per step on 2^27 weights
    (blocks and output exceed L2, so no flush is needed)."""
    import torch
    from quant_dequant_gemv_gb300 import build, qdq

    build.build()
    qtype = DEQUANT_TYPES[args.workload]
    n = DEQUANT_N
    blocks_host = synth.gen_blocks(qtype, n // synth.BLOCK_WEIGHTS[qtype], np.random.default_rng(0))
    blocks = torch.from_numpy(blocks_host).to(device)
    out = torch.empty(n, dtype=torch.float32, device=device)
    stream = torch.cuda.current_stream(device)
    for _ in range(args.warmup):
        qdq.dequant(qtype, blocks, n, out, stream)
    torch.cuda.synchronize(device)
    sampler = ClockSampler(device.index if device.index is not None else 0)
    sampler.start()
    t_load = time.perf_counter()
    while time.perf_counter() - t_load < 1.0:
        for _ in range(20):
            qdq.dequant(qtype, blocks, n, out, stream)
        torch.cuda.synchronize(device)
    K = args.steps
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    torch.cuda.synchronize(device)
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for e in evs:
        e[0].record(stream)
        qdq.dequant(qtype, blocks, n, out, stream)
        e[1].record(stream)
    t1.record(stream)
    torch.cuda.synchronize(device)
    clocks = sampler.stop()
    rc = qdq.get_device_status(stream)
    if rc != 0:
        raise SystemExit(f"device status after timing: {qdq.status_string(rc)}")
    # end to end: pinned host blocks in, fp32 weights out, every step
    b_pin = torch.from_numpy(blocks_host).pin_memory()
    o_pin = torch.empty(n, dtype=torch.float32).pin_memory()
    E = 3
    te = time.perf_counter()
    for _ in range(E):
        blocks.copy_(b_pin, non_blocking=True)
        qdq.dequant(qtype, blocks, n, out, stream)
        o_pin.copy_(out, non_blocking=True)
        stream.synchronize()
    e2e_s = (time.perf_counter() - te) / E
    return {"total_ms": t0.elapsed_time(t1), "launch_ms": [a.elapsed_time(b) for a, b in evs],
            "abytes": dequant_bytes(qtype, n), "clocks": clocks, "e2e_s": e2e_s,
            "h2d": b_pin.numel(), "d2h": 4 * n, "launches": K}


def dequant_cpu_baseline(workload: str, budget_s: float = 8.0) -> dict:
    """The oracle's dequantisation on the host, one thread, on 2^22-weight samples."""
    import oracle
    orc = oracle.get()
    qtype = DEQUANT_TYPES[workload]
    n = 1 << 22
    blocks = synth.gen_blocks(qtype, n // synth.BLOCK_WEIGHTS[qtype], np.random.default_rng(0))
    spent, reps = 0.0, 0
    while spent < budget_s:
        ts = time.perf_counter()
        orc.dequant(qtype, blocks, n)
        spent += time.perf_counter() - ts
        reps += 1
    return {"value": round(reps * dequant_bytes(qtype, n) / spent / 1e9, 4), "unit": "GB/s", "cores": 1,
            "kind": "oracle", **host_cpu(),
            "sample": f"{reps} dequantisations of 2^22 weights ({spent:.1f} s), plain C oracle, one thread"}


TOKEN_POS0 = 64  # the timed token steps start at this cache position (earlier rows filled in warm-up)


def token_bytes(layers: int, pos: int) -> int:
    """Algorithmic bytes of one token step at cache position pos: every GEMV's
    weights, the embedding row, the fp16 key/value rows read (positions 0..pos of
    every layer), the norm vectors, and the activation vectors each level reads
    and writes once."""
    L = synth.LLAMA_1B
    dim, hid, kv, vocab = L["hidden"], L["ffn"], L["n_kv_heads"] * L["head_dim"], L["vocab"]
    w = synth.step_weight_bytes(synth.llama_1b_step(layers))
    embd = synth.row_bytes(synth.Q4_K, dim)
    cache = layers * 2 * (pos + 1) * kv * 2
    norms = (2 * layers + 1) * dim * 4
    act = layers * 4 * (3 * dim + 2 * kv + 3 * hid + dim + dim) + 4 * (dim + vocab)
    return w + embd + cache + norms + act


def run_token(args, device):
    """Greedy decoding through qdq_llama_forward: each timed step is one token at
    the next cache position; the token fed is the previous step's argmax."""
    import torch
    from quant_dequant_gemv_gb300 import build, qdq

    build.build()
    L = synth.LLAMA_1B
    cfg = dict(dim=L["hidden"], hidden=L["ffn"], n_layers=args.layers, n_heads=L["n_heads"],
               n_kv_heads=L["n_kv_heads"], vocab=L["vocab"])
    m = synth.gen_llama_model(seed=0, **cfg)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(device)
    layers = []
    for lw in m["layers"]:
        d = {name: (lw[name][0], t(lw[name][3])) for name in synth.LAYER_TENSORS}
        d["attn_norm"], d["ffn_norm"] = t(lw["attn_norm"]), t(lw["ffn_norm"])
        layers.append(d)
    e, o = m["token_embd"], m["output"]
    max_seq = TOKEN_POS0 + 2 * (args.steps + args.warmup) + 8
    model = qdq.Llama(max_seq=max_seq, embd=(e[0], t(e[3])), layers=layers, output_norm=t(m["output_norm"]),
                      output=(o[0], t(o[3])), **cfg)
    stream = torch.cuda.current_stream(device)
    pos = 0
    while pos < TOKEN_POS0 + args.warmup:  # fill the cache up to the timed positions
        model.forward(pos % cfg["vocab"], pos, stream)
        pos += 1
    torch.cuda.synchronize(device)
    sampler = ClockSampler(device.index if device.index is not None else 0)
    sampler.start()
    K = args.steps
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    p0 = pos
    t0.record(stream)
    for i, ev in enumerate(evs):
        ev[0].record(stream)
        model.forward(int(i * 7919 % cfg["vocab"]), p0 + i, stream)
        ev[1].record(stream)
    t1.record(stream)
    torch.cuda.synchronize(device)
    clocks = sampler.stop()
    rc = qdq.get_device_status(stream)
    if rc != 0:
        raise SystemExit(f"device status after timing: {qdq.status_string(rc)}")
    # end to end: greedy decoding, the argmax read back to the host each step
    # and fed as the next token
    am = torch.empty(1, dtype=torch.int64).pin_memory()
    pos = p0 + K
    tok = 1
    E = K
    te = time.perf_counter()
    for i in range(E):
        model.forward(tok, pos + i, stream)
        am.copy_(model.argmax, non_blocking=True)
        stream.synchronize()
        tok = int(am.item())
    e2e_s = (time.perf_counter() - te) / E
    launches = model.launches
    abytes = token_bytes(args.layers, p0 + K // 2)
    model.close()
    return {"total_ms": t0.elapsed_time(t1), "launch_ms": [a.elapsed_time(b) for a, b in evs], "abytes": abytes,
            "clocks": clocks, "e2e_s": e2e_s, "h2d": 0, "d2h": 8, "launches": K * launches}


def run_ours(args, rank, world, device):
    import torch
    from quant_dequant_gemv_gb300 import build, qdq

    build.build()
    levels = workload_levels(args.workload, args.layers)
    batch = args.batch
    stream = torch.cuda.current_stream(device)
    abytes = algorithmic_bytes(levels, batch)
    use_plan = args.workload == "step"
    if use_plan:
        items, lv, xs_host = build_inputs(levels, batch, device)
        plan = qdq.Plan(items, lv, batch)
        launches_per_step = plan.launches

        def steps(i, n):
            for _ in range(n):
                plan.run(stream)
    else:
        # single GEMVs: rotate enough weight copies that W streams from HBM, not L2
        wbytes = sum(g.weight_bytes for lv_ in levels for g in lv_)
        ncopy = max(1, -(-4 * L2_BYTES // wbytes))
        ncopy = -(-ncopy // GROUP) * GROUP  # whole groups of weight copies
        copies, xs_dev, ys, xs_host = [], [], [], []
        for li, level in enumerate(levels):
            x = synth.gen_x(batch, level[0].cols, 1000 + li)
            xs_host.append(x)
            xs_dev.append(torch.from_numpy(x).to(device))
        for c in range(ncopy):
            copies.append([[torch.from_numpy(synth.gen_matrix(g.qtype, g.rows, g.cols, 10 * li + gi)).to(device)
                            for gi, g in enumerate(level)] for li, level in enumerate(levels)])
        ys = [[torch.empty(batch, g.rows, dtype=torch.float32, device=device) for g in level] for level in levels]

        def step_api(i, st):
            cw = copies[i % ncopy]
            for li, level in enumerate(levels):
                for gi, g in enumerate(level):
                    qdq.gemv(g.qtype, cw[li][gi], g.rows, g.cols, xs_dev[li], ys[li][gi], batch, st)
        launches_per_step = sum(gemv_launches(g, batch) for lv_ in levels for g in lv_)
        # The timed steps replay CUDA graphs of the same calls: groups of GROUP
        # consecutive steps (different weight copies) per graph, and single-step
        # graphs for a remainder. Calls then run back to back on the device, as in
        # a serving loop that captures its GEMVs, instead of each step waiting for
        # its own graph launch.
        for i in range(3):
            step_api(i, stream)
        torch.cuda.synchronize(device)
        single, grouped = [], []
        for c in range(ncopy):
            g_ = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g_):
                step_api(c, torch.cuda.current_stream(device))
            single.append(g_)
        for c0 in range(0, ncopy, GROUP):
            g_ = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g_):
                for c in range(c0, c0 + GROUP):
                    step_api(c, torch.cuda.current_stream(device))
            grouped.append(g_)
        torch.cuda.synchronize(device)

        def steps(i, n):
            if n == GROUP:
                grouped[(i % ncopy) // GROUP].replay()
            else:
                single[i % ncopy].replay()

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()

    def group_len(i, left):  # steps run together from step i (a graph group when aligned)
        return GROUP if (not use_plan and i % GROUP == 0 and left >= GROUP) else 1

    i = 0
    while i < args.warmup:
        n = group_len(i, args.warmup - i)
        steps(i, n)
        i += n
    torch.cuda.synchronize(device)
    rc = qdq.get_device_status(stream)
    if rc != 0:
        raise SystemExit(f"device status after warm-up: {qdq.status_string(rc)}")

    sampler = ClockSampler(device.index if device.index is not None else 0)
    sampler.start()
    t_load = time.perf_counter()
    i = 0
    while time.perf_counter() - t_load < 1.0:  # untimed load so the clock samples see a busy GPU
        for _ in range(50):
            steps(i, 1)
            i += 1
        torch.cuda.synchronize(device)

    K = args.steps
    runs = []  # (steps, events) of each replay in the timed region
    barrier()
    torch.cuda.synchronize(device)
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    i = 0
    while i < K:
        n = group_len(i, K - i)
        e = (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
        e[0].record(stream)
        steps(i, n)
        e[1].record(stream)
        runs.append((n, e))
        i += n
    t1.record(stream)
    torch.cuda.synchronize(device)
    barrier()
    clocks = sampler.stop()
    total_ms = t0.elapsed_time(t1)
    launch_ms = [e[0].elapsed_time(e[1]) / n for n, e in runs for _ in range(n)]  # per step
    rc = qdq.get_device_status(stream)
    if rc != 0:
        raise SystemExit(f"device status after timing: {qdq.status_string(rc)}")

    # end to end through the C ABI: pinned host x in, every y out, each step
    E = max(3, K // 2)
    if use_plan:
        x_host = torch.from_numpy(np.concatenate([a.reshape(-1) for a in xs_host])).pin_memory()
        y_host = torch.empty(sum(batch * it[2] for it in items), dtype=torch.float32).pin_memory()
        for _ in range(3):
            plan.run_io(x_host, y_host, stream)
        torch.cuda.synchronize(device)
        barrier()
        te = time.perf_counter()
        h2d = d2h = 0
        for _ in range(E):
            h2d, d2h = plan.run_io(x_host, y_host, stream)
            stream.synchronize()
        e2e_s = (time.perf_counter() - te) / E
        plan.close()
    else:
        x_pin = [torch.from_numpy(a).pin_memory() for a in xs_host]
        y_pin = [[torch.empty(batch, g.rows, dtype=torch.float32).pin_memory() for g in level] for level in levels]
        h2d = sum(t.numel() * 4 for t in x_pin)
        d2h = sum(t.numel() * 4 for row in y_pin for t in row)

        def step_io(i):
            for li in range(len(levels)):
                xs_dev[li].copy_(x_pin[li], non_blocking=True)
            step_api(i, stream)
            for li, level in enumerate(levels):
                for gi in range(len(level)):
                    y_pin[li][gi].copy_(ys[li][gi], non_blocking=True)
        for i in range(3):
            step_io(i)
        torch.cuda.synchronize(device)
        barrier()
        te = time.perf_counter()
        for i in range(E):
            step_io(i)
            stream.synchronize()
        e2e_s = (time.perf_counter() - te) / E
    barrier()
    return {"total_ms": total_ms, "launch_ms": launch_ms, "abytes": abytes, "clocks": clocks,
            "e2e_s": e2e_s, "h2d": h2d, "d2h": d2h, "launches": K * launches_per_step}


def host_cpu() -> dict:
    """Host core count and CPU model, for the CPU baseline record."""
    model = None
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.split(":", 1)[0].strip() == "Model name":
                model = line.split(":", 1)[1].strip()
                break
    except (OSError, subprocess.SubprocessError):
        pass
    if model is None:
        try:
            for line in Path("/proc/cpuinfo").read_text().splitlines():
                if line.lower().startswith("model name"):
                    model = line.split(":", 1)[1].strip()
                    break
        except OSError:
            pass
    import platform
    return {"host_cores": os.cpu_count(), "cpu_model": model or platform.processor() or platform.machine()}


def time_oracle(levels, batch, budget_s, mode="single", threads=1):
    """Time the CPU baseline on the workload's GEMVs in step order, until budget_s
    of measured time is spent (input generation excluded). Modes:
      single  -- the C oracle, one thread (dequantise a row, dot in double);
      threads -- the same C oracle, the rows of each GEMV split over `threads`
                 host threads (ctypes releases the GIL during the C call);
      numpy   -- unfused: the C oracle dequantises the whole matrix to fp32, then
                 a NumPy matmul (BLAS) multiplies it by x, the dequantise-per-call
                 structure of the NumPy port the pages describe.
    Returns (seconds, bytes of the GEMVs done, GEMVs done)."""
    import oracle
    from concurrent.futures import ThreadPoolExecutor
    orc = oracle.get()
    pool = ThreadPoolExecutor(max_workers=threads) if mode == "threads" else None
    spent, done_bytes, n = 0.0, 0, 0
    try:
        for li, level in enumerate(levels):
            x = synth.gen_x(batch, level[0].cols, 1000 + li)
            for gi, g in enumerate(level):
                W = synth.gen_matrix(g.qtype, g.rows, g.cols, 10 * li + gi)
                ts = time.perf_counter()
                if mode == "single":
                    orc.gemv(g.qtype, W, g.rows, g.cols, x)
                elif mode == "threads":
                    bounds = [g.rows * t // threads for t in range(threads + 1)]
                    list(pool.map(lambda t: orc.gemv(g.qtype, W, g.rows, g.cols, x, bounds[t], bounds[t + 1]),
                                  range(threads)))
                else:
                    Wf = orc.dequant(g.qtype, W, g.rows * g.cols).reshape(g.rows, g.cols)
                    np.matmul(x, Wf.T)
                spent += time.perf_counter() - ts
                done_bytes += g.weight_bytes + 4 * batch * (g.cols + g.rows)
                n += 1
            if spent > budget_s:
                break
    finally:
        if pool is not None:
            pool.shutdown()
    return spent, done_bytes, n


def cpu_baselines(levels, batch, budget_single=10.0, budget_other=5.0) -> dict:
    """The three CPU baselines side by side (reported only, never targets)."""
    cpu = host_cpu()
    threads = cpu["host_cores"] or 1
    legs = {}
    for name, mode, th, budget in (("oracle_1_thread", "single", 1, budget_single),
                                   ("oracle_all_cores", "threads", threads, budget_other),
                                   ("numpy_unfused", "numpy", 1, budget_other)):
        spent, done, n = time_oracle(levels, batch, budget, mode, th)
        legs[name] = {"value": round(done / spent / 1e9, 4), "unit": "GB/s",
                      "threads": th if mode != "numpy" else "dequantise: 1; matmul: NumPy's BLAS threads",
                      "sample": f"first {n} GEMVs of the workload in step order ({done / 1e6:.0f} MB of weights, "
                                f"{spent:.1f} s)"}
    first = legs["oracle_1_thread"]
    return {"value": first["value"], "unit": "GB/s", "cores": 1, "kind": "oracle",
            "sample": "oracle_1_thread leg: " + first["sample"] + "; plain C oracle, one thread",
            **cpu, "legs": legs}


def slowest_replica(total_ms: float, e2e_s: float, world: int, device) -> tuple[float, float]:
    """Replicas (one process per GPU, no data exchange): the job's time is the
    slowest rank's. Uses the initialised process group (NCCL on GPUs, gloo in tests)."""
    if world <= 1:
        return total_ms, e2e_s
    import torch
    import torch.distributed as dist
    t = torch.tensor([total_ms, e2e_s], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t[0]), float(t[1])


def replicas_gbs(step_bytes: int, world: int, ms_step: float) -> float:
    """Whole-job throughput: every replica moves step_bytes per step."""
    return world * step_bytes / (ms_step * 1e-3) / 1e9


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="step", choices=sorted(WORKLOADS))
    ap.add_argument("--batch", type=int, default=1)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--layers", type=int, default=22,
                    help="layers of the decode-step workload (a shorter step for profiling captures)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    levels = workload_levels(args.workload, args.layers)
    abytes = (dequant_bytes(DEQUANT_TYPES[args.workload], DEQUANT_N) if args.workload in DEQUANT_TYPES
              else token_bytes(args.layers, TOKEN_POS0 + args.warmup + args.steps // 2) if args.workload == "token"
              else algorithmic_bytes(levels, args.batch))
    step_bytes = abytes
    wname = WORKLOADS[args.workload]
    tkey = args.workload
    if args.workload == "step" and args.layers != 22:
        wname = f"{args.layers}-layer variant of the " + wname
        tkey = f"step{args.layers}"

    if args.impl == "reference":
        # The reference arm is the CPU oracle, as it stands, on the host cores:
        # each step is a bounded sample of the workload (its first GEMVs in step
        # order, about 1 s of work); the metric is extrapolated per byte.
        if rank != 0:
            return
        if args.workload in DEQUANT_TYPES:
            cpu = dequant_cpu_baseline(args.workload, budget_s=0.5 * args.steps)
            line = {"impl": "reference", "metric": METRIC, "value": cpu["value"], "unit": "GB/s",
                    "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
                    "ms_per_step": round(1e3 * step_bytes / (cpu["value"] * 1e9), 3), "higher_is_better": True,
                    "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
                    "config": {"workload": wname, "l2": "n/a (CPU)"}, "cpu_baseline": cpu,
                    "e2e": {"value": cpu["value"], "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
            print(json.dumps(line))
            return
        budget = 0.8
        for _ in range(args.warmup):
            time_oracle(levels, args.batch, 0.05)
        spent = done = 0
        n_last = 0
        for _ in range(args.steps):
            s, d, n_last = time_oracle(levels, args.batch, budget)
            spent += s
            done += d
        gbs = done / spent / 1e9
        line = {
            "impl": "reference", "metric": METRIC, "value": round(gbs, 4), "unit": "GB/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(1e3 * spent / args.steps, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32 (oracle: f64 sums)",
            "data": "synthetic", "tok_s": round(gbs * 1e9 / step_bytes, 4),
            "config": {"workload": wname, "batch": args.batch,
                       "l2": "n/a (CPU)"},
            "cpu_baseline": {"value": round(gbs, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
                             "sample": f"first {n_last} GEMVs of the workload in step order per step "
                                       f"(~{budget:.1f} s of oracle time), plain C, one thread"},
            "e2e": {"value": round(gbs, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        }
        print(json.dumps(line))
        return

    import torch
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    device = torch.device(f"cuda:{local}")
    torch.cuda.set_device(device)
    if args.workload == "token" and args.batch != 1:
        raise SystemExit("the token workload is batch 1")
    r = (run_dequant(args, device) if args.workload in DEQUANT_TYPES
         else run_token(args, device) if args.workload == "token" else run_ours(args, rank, world, device))

    total_ms, e2e_s = slowest_replica(r["total_ms"], r["e2e_s"], world, device)
    ms_step = total_ms / args.steps
    value = replicas_gbs(abytes, world, ms_step)
    avg_launch_ms = statistics.mean(r["launch_ms"])
    achieved = abytes / (avg_launch_ms * 1e-3) / 1e9
    peaks = load_peaks()
    traffic = recorded_traffic(tkey, args.batch)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        if args.workload.startswith("dequant_"):
            cpu = dequant_cpu_baseline(args.workload)
        else:
            cpu = cpu_baselines(levels, args.batch)

    if rank == 0:
        line = {
            "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(ms_step, 5), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "tok_s": round(world * 1e3 / ms_step, 1),
            "config": {"workload": wname, "batch": args.batch,
                       "step_bytes": abytes,
                       "l2": ("inputs larger than L2 (weights per step exceed 129 MB)"
                              if args.workload in ("step", "token")
                              else "inputs larger than L2 (blocks in + fp32 out exceed 129 MB)"
                              if args.workload in DEQUANT_TYPES
                              else "weights rotate over copies totalling at least 4x the 129 MB L2; "
                                   f"timed steps replay CUDA graphs of the qdq_gemv calls, {GROUP} steps "
                                   "(weight copies) per graph"),
                       "parallelism": "replicas" if world > 1 else "single GPU"},
            "roofline": {"bound": "hbm", "achieved": round(achieved, 2), "peak": peaks["hbm_gbs"],
                         "unit": "GB/s", "frac": round(achieved / peaks["hbm_gbs"], 4),
                         "traffic": traffic, "peak_source": peaks["source"],
                         "kernel": ("stream1_kernel (persistent plan launch)" if args.workload == "step"
                                    else "whole token step (plan launches + attention + embedding decode)"
                                    if args.workload == "token"
                                    else "dequant_kernel" if args.workload in DEQUANT_TYPES
                                    else "mma_gemv_kernel (tensor cores)"
                                    if args.batch >= mma_min_batch(levels[0][0].qtype)
                                    else "gemv_more_kernel (exact per-weight decode)"
                                    if args.workload in MORE_GEMV
                                    else "stream1_kernel (one GEMV per launch)")},
            "e2e": {"value": round(world * abytes / e2e_s / 1e9, 2), "unit": "GB/s", "tok_s": round(world / e2e_s, 1),
                    "h2d_bytes_per_step": r["h2d"], "d2h_bytes_per_step": r["d2h"]},
            "gpu_launches": r["launches"],
            "clocks": r["clocks"],
            "cpu_baseline": cpu,
        }
        print(json.dumps(line))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
