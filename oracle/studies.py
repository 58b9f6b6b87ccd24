"""Accuracy studies on top of the CPU oracle (float64 numpy).

TEST INFRASTRUCTURE ONLY, like the rest of oracle/: only tests/ may import it.

Two studies the pages call for, written as plain functions of the oracle's
quantizers:

* Pre-RoPE versus post-RoPE per-channel keys ("KV Cache Quantization: Why Keys
  and Values Need Different Axes", section "Where does RoPE break this?", and
  "FP8 KV Cache Quantization: Why Keys Break Before Values", section "Should you
  quantize keys pre-RoPE or post-RoPE?"): rotary embedding mixes each channel
  with its pair partner by a position-dependent angle, so an outlier channel
  that is steady before rotation becomes a rotating mixture after it, and a
  per-channel scale fitted over a token group fits it worse.  pre: quantize the
  raw keys, dequantize, rotate.  post: rotate, quantize, dequantize.
* Attention agreement between a full-precision and a quantized cache (the same
  page as the second above, section "Why doesn't perplexity catch KV cache
  quantization damage?": per-head attention KL and rank agreement of the top-k
  attention indices).  Definitions used here (the page names the quantities but
  not their formulas):
    KL(p || q) = sum_i p_i (ln p_i - ln q_i), terms with p_i = 0 are 0;
    top-k overlap = |topk(p) and topk(q)| / k;
    top-k rank agreement = over the pairs i != j of topk(p) with p_i != p_j,
      the fraction ordered the same way by q (1 when no such pair).
  topk(x) is the k indices of the largest values, ties to the lower index.
"""
from __future__ import annotations

import numpy as np

from . import kvq_oracle as O


def dequantized_keys(K, spec: O.QSpec) -> np.ndarray:
    """Keys [T, D] after quantization with `spec` and dequantization, every token
    quantized (per-channel: T a multiple of the group G)."""
    K = np.asarray(K, dtype=np.float64)
    T, D = K.shape
    residual = spec.group if spec.axis == O.PER_CHANNEL else 0
    cfg = O.Config(1, 1, D, spec, O.QSpec(O.INT8, O.SYM, O.PER_TOKEN, 0), residual=residual, page_size=16)
    st = O.quantize_stream(cfg, K, np.zeros_like(K))
    assert st.n_q == T
    return O.dequantize_stream(cfg, st)[0]


def rope_keys_pre(K, positions, theta: float, spec: O.QSpec) -> np.ndarray:
    """Pre-RoPE cache: quantize the raw keys, dequantize, then rotate."""
    return O.rope(dequantized_keys(K, spec), positions, theta)


def rope_keys_post(K, positions, theta: float, spec: O.QSpec) -> np.ndarray:
    """Post-RoPE cache: rotate the raw keys, then quantize and dequantize."""
    return dequantized_keys(O.rope(K, positions, theta), spec)


def logit_errors(q, K_ref, K_test, scale=None) -> tuple[float, float]:
    """(mean |logit error|, relative Frobenius logit error) of q K_test^T * scale
    against q K_ref^T * scale."""
    q = np.asarray(q, dtype=np.float64)
    if scale is None:
        scale = 1.0 / np.sqrt(q.shape[-1])
    ref = (q @ np.asarray(K_ref, np.float64).T) * scale
    got = (q @ np.asarray(K_test, np.float64).T) * scale
    d = got - ref
    return float(np.abs(d).mean()), float(np.linalg.norm(d) / np.linalg.norm(ref))


def attention_probs(q, K, scale=None) -> np.ndarray:
    """Softmax attention weights [H, T] of the query rows q [H, D] over K [T, D]."""
    q = np.asarray(q, dtype=np.float64)
    if scale is None:
        scale = 1.0 / np.sqrt(q.shape[-1])
    return O.softmax((q @ np.asarray(K, np.float64).T) * scale)


def kl_rows(p, q) -> np.ndarray:
    """KL(p_r || q_r) for each row r of two probability arrays [H, T]."""
    p = np.asarray(p, dtype=np.float64)
    q = np.asarray(q, dtype=np.float64)
    with np.errstate(divide="ignore", invalid="ignore"):
        t = np.where(p > 0.0, p * (np.log(p) - np.log(q)), 0.0)
    return t.sum(axis=-1)


def topk_indices(x, k: int) -> np.ndarray:
    """Indices of the k largest entries of each row, largest first; equal values
    in index order."""
    x = np.asarray(x, dtype=np.float64)
    return np.argsort(-x, axis=-1, kind="stable")[..., :k]


def topk_overlap(p, q, k: int) -> np.ndarray:
    """|topk(p_r) and topk(q_r)| / k for each row r."""
    a, b = topk_indices(p, k), topk_indices(q, k)
    return np.array([len(set(x.tolist()) & set(y.tolist())) / k for x, y in zip(a, b)])


def topk_rank_agreement(p, q, k: int) -> np.ndarray:
    """For each row: over the pairs (i, j), i < j, of topk(p) with p_i != p_j, the
    fraction with sign(q_i - q_j) == sign(p_i - p_j); 1 when there is no pair."""
    p = np.asarray(p, dtype=np.float64)
    q = np.asarray(q, dtype=np.float64)
    out = []
    for pr, qr, idx in zip(p, q, topk_indices(p, k)):
        same = total = 0
        for a in range(len(idx)):
            for b in range(a + 1, len(idx)):
                i, j = idx[a], idx[b]
                sp = np.sign(pr[i] - pr[j])
                if sp == 0:
                    continue
                total += 1
                same += int(np.sign(qr[i] - qr[j]) == sp)
        out.append(same / total if total else 1.0)
    return np.array(out)
