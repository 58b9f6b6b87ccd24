"""GPU side of the accuracy studies.

Pre-/post-RoPE keys ("KV Cache Quantization: Why Keys and Values Need Different
Axes", section "Where does RoPE break this?"):
The same keys, with a steady offset on four fast-rotating channels, go through
two caches of the library: a pre-RoPE cache (raw keys stored, rotated after
dequantization inside the attention kernel) and a post-RoPE cache (keys rotated
on the host and stored in bf16).  Both use INT4 per-channel keys in 64-token
groups, INT8 per-token values and a 64-token window.  Each cache's attention
matches its own oracle to the parity tolerance, and measured against float64
attention over the unquantized rotated keys the post-RoPE cache's error is the
larger one, as the oracle study finds.

FP8 scales ("FP8 KV Cache Quantization: Why Keys Break Before Values", section
"Why do per-tensor scales waste bits on the K cache?", failure mode 1): keys
whose outlier channels reach about +-1000 go through E4M3 and E5M2 caches at
the unit scale (no calibration) and an E4M3 cache with calibrated scales.  Each
matches its own oracle (bytes and attention), and against float64 attention the
clipping E4M3 cache is far worse than the coarse E5M2 one, which is worse than
the calibrated E4M3 one.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import kvq_inputs as W  # noqa: E402
from oracle import kvq_oracle as O  # noqa: E402

if not torch.cuda.is_available():  # pragma: no cover
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

from kvq_testlib import Case, torch_src  # noqa: E402

THETA = 500000.0
FAST = [2, 9, 17, 30]


def test_pre_rope_cache_beats_post_rope_cache_on_the_gpu():
    T, D, B = 4096 + 37, 128, 2
    base = dict(num_q_heads=4, num_kv_heads=1, head_dim=D, v=O.QSpec(O.INT8, O.SYM, O.PER_TOKEN, 0),
                residual=64, page_size=16, rope_theta=THETA, src_dtype=O.BF16,
                k=O.QSpec(O.INT4, O.ASYM, O.PER_CHANNEL, 64))
    pre_cfg, post_cfg = O.Config(rope_pre=1, **base), O.Config(rope_pre=0, **base)
    K, Kpost, Kref, V = [], [], [], []
    for b in range(B):
        k = W.small_stream(900 + b, T, D).astype(np.float64)
        k[:, FAST] += 30.0
        k = W.bf16_round(k.astype(np.float32))[1]
        kr = O.rope(k.astype(np.float64), np.arange(T), THETA)
        K.append([k])
        Kref.append(kr)
        Kpost.append([W.bf16_round(kr.astype(np.float32))[1]])
        V.append([W.small_stream(950 + b, T, D, bf16=True)])
    pre = Case(pre_cfg, [T] * B, seed=3, streams=(K, V))
    post = Case(post_cfg, [T] * B, seed=3, streams=(Kpost, V))
    q = pre.queries(seed=11)
    pre.check_attention(q)
    post.check_attention(q)
    errs = {}
    for name, case in (("pre", pre), ("post", post)):
        out = case.cache.attention(torch_src(q, case.cfg)).cpu().numpy().astype(np.float64)
        e = []
        for b in range(B):
            ref = O.attention(q[b].astype(np.float64), Kref[b], V[b][0].astype(np.float64))
            e.append(np.linalg.norm(out[b] - ref, axis=1) / np.linalg.norm(ref, axis=1))
        errs[name] = float(np.mean(e))
    assert errs["post"] >= 1.8 * errs["pre"], errs


def test_fp8_unit_scale_clipping_on_the_gpu():
    T, D, B = 2048, 128, 2
    K, V, Q = [], [], []
    for b in range(B):
        k = W.small_stream(b, T, D).astype(np.float64)
        k[:, [3, 17, 44, 91]] *= 1000.0 / 3.0
        K.append([W.bf16_round(k.astype(np.float32))[1]])
        V.append([W.small_stream(b + 50, T, D, bf16=True)])
        Q.append(W.bf16_round(np.random.default_rng(b).standard_normal((8, D)).astype(np.float32) * 0.05)[1])
    q = np.stack(Q)
    errs = {}
    for name, fmt, unit in (("e4m3_unit", O.FP8_E4M3, True), ("e5m2_unit", O.FP8_E5M2, True),
                            ("e4m3_calibrated", O.FP8_E4M3, False)):
        spec = O.QSpec(fmt, O.SYM, O.PER_TENSOR)
        cfg = O.Config(8, 1, D, spec, spec, 0, 256, 0, 1e4, O.BF16)
        case = Case(cfg, [T] * B, seed=5, streams=(K, V), static_scales=([1.0], [1.0]) if unit else None)
        case.check_pages()
        case.check_attention(q)
        out = case.cache.attention(torch_src(q, cfg)).cpu().numpy().astype(np.float64)
        e = []
        for b in range(B):
            ref = O.attention(q[b].astype(np.float64), K[b][0].astype(np.float64), V[b][0].astype(np.float64))
            e.append(np.linalg.norm(out[b] - ref, axis=1) / np.linalg.norm(ref, axis=1))
        errs[name] = float(np.mean(e))
    assert errs["e4m3_unit"] > 2.0 * errs["e5m2_unit"], errs
    assert errs["e5m2_unit"] > errs["e4m3_calibrated"], errs
