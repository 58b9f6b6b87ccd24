"""Oracle work for the full-size tests, run in spawned worker processes.

This module imports only numpy and the oracle, so a worker starts quickly and
never touches CUDA (the pool is created with the spawn method, because the test
process has already initialised the GPU).
"""
from __future__ import annotations

import numpy as np

from oracle import kvq_oracle as O


def check_stream(args):
    """One (sequence, kv-head) stream: the oracle's cache state from the source
    rows, its dequantized keys and values against the library's (bit-exact), and
    its attention for the stream's query heads against the library's output.

    Returns (key, dequantize_exact, relative L2 of each query head)."""
    key, cfg, K, V, q_heads, k_deq, v_deq, out_heads, k_scale, v_scale = args
    st = O.quantize_stream(cfg, K.astype(np.float64), V.astype(np.float64), k_scale, v_scale)
    ko, vo = O.dequantize_stream(cfg, st, k_scale, v_scale)
    exact = bool(np.array_equal(k_deq.astype(np.float64), ko) and np.array_equal(v_deq.astype(np.float64), vo))
    ref = O.decode_head(cfg, st, q_heads.astype(np.float64), k_scale, v_scale)
    got = out_heads.astype(np.float64)
    err = np.linalg.norm(got - ref, axis=1) / np.maximum(np.linalg.norm(ref, axis=1), 1e-30)
    return key, exact, err.tolist()
