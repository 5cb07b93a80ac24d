"""GB300-native fused dequant-GEMV over block-quantised weights.

The compute path is the C-ABI library ``libqdq.so`` (hand-written CUDA for
sm_103a, declared in ``include/qdq.h``); ``quant_dequant_gemv_gb300.qdq`` is its
thin ctypes binding. ``synth`` holds the seeded input generators.
Importing this package loads nothing; the library is loaded on first use.
"""
from .synth import Q4_0, Q8_0, Q4_K, Q6_K, BLOCK_BYTES, BLOCK_WEIGHTS  # noqa: F401
