"""Closed-form checks of the block formats against the figures the pages print
(tests/golden/page_figures.json, each with its page and section)."""
import json
from pathlib import Path

from quant_dequant_gemv_gb300 import synth

FIG = json.loads((Path(__file__).parent / "golden" / "page_figures.json").read_text())


def test_bits_per_weight_match_printed_figures():
    for name, f in FIG["bits_per_weight"].items():
        bpw = f["bytes"] * 8 / f["weights"]
        assert abs(bpw - f["printed"]) <= 0.005 + 1e-12, name


def test_library_block_sizes_match_the_pages():
    bpw = FIG["bits_per_weight"]
    assert synth.BLOCK_BYTES[synth.Q4_K] == bpw["Q4_K"]["bytes"]
    assert synth.BLOCK_BYTES[synth.Q6_K] == bpw["Q6_K"]["bytes"]
    assert synth.BLOCK_BYTES[synth.Q4_0] == bpw["q4_0"]["bytes"]
    assert synth.BLOCK_BYTES[synth.Q8_0] == FIG["q8_0_block"]["bytes"] == 4 + 32
    assert synth.BLOCK_WEIGHTS[synth.Q4_K] == 8 * FIG["q4k_subblocks"]["weights_per_subblock"]
    q6 = FIG["q6k_scales_per_block"]
    assert synth.BLOCK_WEIGHTS[synth.Q6_K] == q6["printed"] * q6["weights_per_scale"]
    # Q6_K struct: ql[128] + qh[64] + scales[16] + fp16 d
    assert 128 + 64 + 16 + 2 == synth.BLOCK_BYTES[synth.Q6_K]
    # Q4_K: fp16 d + fp16 dmin + 12 packed bytes + 128 nibble bytes
    assert 2 + 2 + 12 + 128 == synth.BLOCK_BYTES[synth.Q4_K]


def test_memory_ratios_vs_fp32():
    ratio_q8 = 32 * 4 / synth.BLOCK_BYTES[synth.Q8_0]
    ratio_q4 = 32 * 4 / synth.BLOCK_BYTES[synth.Q4_0]
    assert round(ratio_q8) == 4 and round(ratio_q4) == 7


def test_decode_step_weight_bytes_near_printed_model_size():
    # The step's GEMV weights (no token embedding, no norms) against the printed
    # mapped size of the whole Q4_K_M file: close, and a little below it.
    step = synth.step_weight_bytes(synth.llama_1b_step())
    assert step == 667_152_384
    mib = step / 2 ** 20
    assert 0.95 * FIG["tinyllama_q4_k_m_mapped_mb"]["printed"] <= mib <= FIG["tinyllama_q4_k_m_mapped_mb"]["printed"]
    shape = FIG["llama_1b_shape"]
    assert synth.LLAMA_1B["n_layers"] == shape["n_layers"]
    assert synth.LLAMA_1B["n_kv_heads"] == shape["n_kv_heads"]
    assert synth.LLAMA_1B["head_dim"] == shape["head_dim"]
