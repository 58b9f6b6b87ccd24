"""Seeded synthetic inputs for the quantized-KV decode-attention workloads.

This module is shared by the CPU oracle's tests and by the CUDA path's tests and
benchmark.  It holds only input generation (random draws, outlier planting, bf16
storage rounding, ragged lengths, page permutations) and the workload shapes; none
of the quantization or attention arithmetic lives here.

Every stream is generated block-wise: the values of tokens [t0, t1) of one
(config, sequence, kv-head, tensor) stream come from numpy ``default_rng`` seeded
with ``SeedSequence([config, seq, head, kind, block])`` for 1024-token blocks, so
any token range of any stream can be regenerated without the rest.

Workloads (shapes and distributions follow the synthetic experiments of
"FP8 KV Cache Quantization: Why Keys Break Before Values", section "Why does the
K cache break before the V cache?" and "KV Cache Quantization: Why Keys and Values
Need Different Axes", section "Why does per-token key quantization destroy
accuracy?", scaled up to Llama-3.1-8B / 70B decode layers):

 1. single head, T=4096, D=128, fp32; K channels 7, 23, 88 scaled x20.
 2. single head, T=512, D=128, fp32; K channels 3, 17, 44, 91 scaled x60;
    64 query vectors.
 3. B=16, Hq=32, Hkv=8, D=128, bf16, T=32768 quantized + 127 window tokens;
    4 random K outlier channels per kv-head scaled by U(20, 60).
 4. B=8, Hq=64, Hkv=8, D=128, bf16, T=131072; 4 random K outlier channels per
    kv-head scaled x30.
 5. B=64, Hq=32, Hkv=8, D=128, bf16, ragged T ~ floor(exp(U(ln 1024, ln 65536)));
    16-token pages in a randomly permuted physical order; 4 random K outlier
    channels per kv-head scaled by U(20, 60).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

BLOCK = 1024  # tokens per independently seeded block

KIND_K, KIND_V, KIND_Q = 0, 1, 2


@dataclass(frozen=True)
class Workload:
    cid: int
    batch: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    src_dtype: str  # "f32" or "bf16"
    fixed_len: int = 0  # tokens per sequence (0: ragged, see lengths())
    fixed_outliers: tuple = ()  # same K outlier channels for every head, fixed factor
    fixed_factor: float = 1.0
    n_random_outliers: int = 0  # per kv-head random outlier channels
    factor_lo: float = 1.0
    factor_hi: float = 1.0
    ragged_lo: int = 0
    ragged_hi: int = 0
    extra: dict = field(default_factory=dict)


WORKLOADS = {
    1: Workload(1, 1, 1, 1, 128, "f32", fixed_len=4096, fixed_outliers=(7, 23, 88), fixed_factor=20.0),
    2: Workload(2, 1, 64, 1, 128, "f32", fixed_len=512, fixed_outliers=(3, 17, 44, 91), fixed_factor=60.0),
    3: Workload(3, 16, 32, 8, 128, "bf16", fixed_len=32768 + 127, n_random_outliers=4,
                factor_lo=20.0, factor_hi=60.0),
    4: Workload(4, 8, 64, 8, 128, "bf16", fixed_len=131072, n_random_outliers=4,
                factor_lo=30.0, factor_hi=30.0),
    5: Workload(5, 64, 32, 8, 128, "bf16", n_random_outliers=4, factor_lo=20.0, factor_hi=60.0,
                ragged_lo=1024, ragged_hi=65536),
}


def _rng(*key: int) -> np.random.Generator:
    return np.random.default_rng(np.random.SeedSequence([int(k) for k in key]))


def bf16_round(x: np.ndarray) -> tuple[np.ndarray, np.ndarray]:
    """Round float32 values to bfloat16 storage (nearest, ties to even).

    Returns (bits uint16, values float32 holding the exact bf16 values)."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32).astype(np.uint64)
    lsb = (u >> 16) & 1
    r = ((u + 0x7FFF + lsb) >> 16).astype(np.uint16)
    vals = (r.astype(np.uint32) << 16).view(np.float32)
    return r, vals


def outliers(w: Workload, seq: int, head: int) -> tuple[np.ndarray, np.ndarray]:
    """K outlier channels and their factors for one (sequence, kv-head).

    The channels are the same for every token of the stream (the outliers are
    channel-consistent).  Random channels are drawn per kv-head and shared by all
    sequences, as a model's heads would be."""
    if w.fixed_outliers:
        ch = np.array(w.fixed_outliers, dtype=np.int64)
        return ch, np.full(len(ch), w.fixed_factor, dtype=np.float32)
    if w.n_random_outliers == 0:
        return np.zeros(0, np.int64), np.zeros(0, np.float32)
    g = _rng(w.cid, 7777, head)
    ch = np.sort(g.choice(w.head_dim, size=w.n_random_outliers, replace=False))
    f = g.uniform(w.factor_lo, w.factor_hi, size=w.n_random_outliers).astype(np.float32)
    return ch.astype(np.int64), f


def lengths(w: Workload) -> np.ndarray:
    """Tokens per sequence.  Ragged: floor(exp(U(ln lo, ln hi))) with seed 5."""
    if w.fixed_len:
        return np.full(w.batch, w.fixed_len, dtype=np.int64)
    g = _rng(w.cid, 5)
    u = g.uniform(math.log(w.ragged_lo), math.log(w.ragged_hi), size=w.batch)
    return np.floor(np.exp(u)).astype(np.int64)


def kv_block(w: Workload, seq: int, head: int, kind: int, t0: int, t1: int) -> np.ndarray:
    """Source K (kind=0) or V (kind=1) values of tokens [t0, t1) of one stream.

    float32 [t1-t0, D]; for bf16 workloads the values are already bf16-exact."""
    D = w.head_dim
    out = np.empty((max(t1 - t0, 0), D), dtype=np.float32)
    if t1 <= t0:
        return out
    b0, b1 = t0 // BLOCK, (t1 - 1) // BLOCK
    for blk in range(b0, b1 + 1):
        g = _rng(w.cid, seq, head, kind, blk)
        x = g.standard_normal((BLOCK, D), dtype=np.float32)
        lo, hi = max(t0, blk * BLOCK), min(t1, (blk + 1) * BLOCK)
        out[lo - t0:hi - t0] = x[lo - blk * BLOCK:hi - blk * BLOCK]
    if kind == KIND_K:
        ch, f = outliers(w, seq, head)
        if len(ch):
            out[:, ch] *= f[None, :]
    if w.src_dtype == "bf16":
        out = bf16_round(out)[1]
    return out


def queries(w: Workload, step: int) -> np.ndarray:
    """Query vectors [B, Hq, D] (float32; bf16-exact for bf16 workloads)."""
    g = _rng(w.cid, 4242, step)
    q = g.standard_normal((w.batch, w.num_q_heads, w.head_dim), dtype=np.float32)
    if w.src_dtype == "bf16":
        q = bf16_round(q)[1]
    return q


def new_tokens(w: Workload, step: int, n: int) -> tuple[np.ndarray, np.ndarray]:
    """Fresh K, V tokens for decode step `step` (appended after the prefill):
    float32 [B, n, Hkv, D] each, drawn from the same distributions."""
    B, H, D = w.batch, w.num_kv_heads, w.head_dim
    k = np.empty((B, n, H, D), np.float32)
    v = np.empty((B, n, H, D), np.float32)
    for b in range(B):
        for h in range(H):
            g = _rng(w.cid, 9090, step, b, h)
            kk = g.standard_normal((n, D), dtype=np.float32)
            ch, f = outliers(w, b, h)
            if len(ch):
                kk[:, ch] *= f[None, :]
            k[b, :, h] = kk
            v[b, :, h] = g.standard_normal((n, D), dtype=np.float32)
    if w.src_dtype == "bf16":
        k, v = bf16_round(k)[1], bf16_round(v)[1]
    return k, v


def page_permutation(n_pages: int, seed: int) -> np.ndarray:
    """A random physical order for the cache pages."""
    return _rng(seed, 31337).permutation(n_pages).astype(np.int32)


def small_stream(seed: int, T: int, D: int, outlier_ch=(), factor=1.0, bf16=False) -> np.ndarray:
    """A free-form [T, D] N(0,1) stream for small tests (seeded, optional outliers)."""
    x = _rng(seed, 555, T, D).standard_normal((T, D), dtype=np.float32)
    if len(outlier_ch):
        x[:, list(outlier_ch)] *= np.float32(factor)
    if bf16:
        x = bf16_round(x)[1]
    return x


# ---------------------------------------------------------------- device-side draws

def torch_outlier_scale(w: Workload, device):
    """[Hkv, D] float32 torch tensor: 1 except the K outlier channels of each
    kv-head, which hold their factors (outliers() of sequence 0: the random
    channels are per kv-head and shared by all sequences)."""
    import torch
    scale = torch.ones(w.num_kv_heads, w.head_dim, device=device)
    for h in range(w.num_kv_heads):
        ch, f = outliers(w, 0, h)
        if len(ch):
            scale[h, torch.as_tensor(ch, device=device)] = torch.as_tensor(f, device=device)
    return scale


def torch_kv_chunk(w: Workload, gen, batch: int, n: int, scale, device):
    """The next n tokens of every stream as bf16 torch tensors [batch, n, Hkv, D]:
    K ~ N(0,1) times the outlier scale, V ~ N(0,1), drawn from the seeded torch
    generator `gen` (large workloads are generated on the device this way)."""
    import torch
    H, D = w.num_kv_heads, w.head_dim
    k = (torch.randn(batch, n, H, D, generator=gen, device=device) * scale).to(torch.bfloat16)
    v = torch.randn(batch, n, H, D, generator=gen, device=device).to(torch.bfloat16)
    return k, v
