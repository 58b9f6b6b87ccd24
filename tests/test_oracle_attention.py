"""Pins of the oracle's cache model, RoPE and attention.

Window bookkeeping (token-at-a-time model vs closed form, chunking invariance),
RoPE against complex multiplication and its invariants, attention against
explicit loops and its special cases, split-K combine against one pass, the
pages' printed figures and the orderings of their synthetic-head experiments.
"""
import json
import math
import os

import numpy as np
import pytest

import kvq_inputs as W
from oracle import kvq_oracle as O

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _claims():
    with open(os.path.join(GOLD, "page_claims.json")) as f:
        return json.load(f)


CFGS = {
    "int2_kivi": O.Config(4, 2, 64, O.QSpec(O.INT2, O.ASYM, O.PER_CHANNEL, 8),
                          O.QSpec(O.INT2, O.ASYM, O.PER_TOKEN, 16), residual=16, page_size=16),
    "int8k_int4v": O.Config(4, 1, 64, O.QSpec(O.INT8, O.SYM, O.PER_CHANNEL, 16),
                            O.QSpec(O.INT4, O.ASYM, O.PER_TOKEN, 0), residual=32, page_size=16,
                            rope_pre=1, rope_theta=500000.0),
    "pertoken_r0": O.Config(2, 1, 64, O.QSpec(O.INT4, O.ASYM, O.PER_TOKEN, 0),
                            O.QSpec(O.INT4, O.SYM, O.PER_TOKEN, 32), residual=0, page_size=16),
    "fp8": O.Config(8, 1, 64, O.QSpec(O.FP8_E4M3, 0, O.PER_TENSOR), O.QSpec(O.FP8_E4M3, 0, O.PER_TENSOR),
                    residual=0, page_size=16),
}


def _eq_state(a, b):
    for f in ["T", "n_q"]:
        assert getattr(a, f) == getattr(b, f)
    for f in ["kc", "ks", "km", "vc", "vs", "vm", "k_win", "v_win"]:
        x, y = getattr(a, f), getattr(b, f)
        if x is None or y is None:
            assert (x is None or x.size == 0) and (y is None or y.size == 0), f
        else:
            assert np.array_equal(x, y), f


@pytest.mark.parametrize("name", sorted(CFGS))
@pytest.mark.parametrize("T", [0, 1, 7, 8, 15, 16, 17, 31, 32, 33, 70])
def test_window_model_matches_closed_form_and_chunking(name, T):
    cfg = CFGS[name]
    K = W.small_stream(1, T, cfg.head_dim, (3, 9), 30.0)
    V = W.small_stream(2, T, cfg.head_dim)
    ks, vs = O.calibrate_absmax(K, 448.0), O.calibrate_absmax(V, 448.0)
    closed = O.quantize_stream(cfg, K, V, ks, vs)
    assert closed.n_q == O.n_quantized(T, cfg.residual)
    g = np.random.default_rng(T)
    for split in range(3):
        sc = O.StreamCache(cfg, ks, vs)
        t = 0
        while t < T:
            n = 1 if split == 0 else int(g.integers(1, 12))
            sc.append(K[t:t + n], V[t:t + n])
            t += n
        _eq_state(sc.state(), closed)


def test_window_holds_everything_below_R():
    cfg = CFGS["int8k_int4v"]
    T = cfg.residual - 1
    K = W.small_stream(3, T, 64)
    V = W.small_stream(4, T, 64)
    st = O.quantize_stream(cfg, K, V)
    assert st.n_q == 0
    q = W.small_stream(5, 4, 64)
    Kr = O.rope(K, np.arange(T), cfg.rope_theta)
    assert np.allclose(O.decode_head(cfg, st, q), O.attention(q, Kr, V), rtol=0, atol=1e-14)


def test_per_channel_groups_are_token_aligned():
    cfg = CFGS["int2_kivi"]
    K = W.small_stream(6, 48, 64, (5,), 40.0)
    V = W.small_stream(7, 48, 64)
    st = O.quantize_stream(cfg, K, V)
    assert st.n_q == 48 and st.ks.shape == (6, 64)
    for j in range(6):  # group j's range is exactly tokens 8j..8j+7
        blk = K[8 * j:8 * j + 8]
        assert np.array_equal(st.km[j], blk.min(axis=0))
        assert np.array_equal(st.ks[j], O.fl32(np.maximum(O.fl32(blk.max(0) - blk.min(0)), O.FL32_1EM8) / 3))


def test_dequantize_roundtrip_bound():
    cfg = CFGS["int8k_int4v"]
    K = W.small_stream(8, 96, 64, (1, 40), 50.0)
    V = W.small_stream(9, 96, 64)
    st = O.quantize_stream(cfg, K, V)
    Kh, Vh = O.dequantize_stream(cfg, st)
    for j in range(96 // 16):
        s = st.ks[j]
        assert np.all(np.abs(Kh[16 * j:16 * j + 16] - K[16 * j:16 * j + 16]) <= s / 2 * (1 + 1e-6) + 1e-30)
    assert np.all(np.abs(Vh - V) <= st.vs[:, :1] / 2 * (1 + 1e-6))


def test_rope_against_complex_multiplication():
    g = np.random.default_rng(10)
    D, n = 128, 50
    x = g.standard_normal((n, D))
    pos = g.integers(0, 70000, n)
    z = x[:, 0::2] + 1j * x[:, 1::2]
    theta = 500000.0
    freqs = np.array([theta ** (-(2.0 * i) / D) for i in range(D // 2)])
    zr = z * np.exp(1j * pos[:, None] * freqs[None, :])
    r = O.rope(x, pos, theta)
    assert np.allclose(r[:, 0::2], zr.real, atol=1e-12) and np.allclose(r[:, 1::2], zr.imag, atol=1e-12)


def test_rope_invariants():
    g = np.random.default_rng(11)
    D = 64
    q, k = g.standard_normal((1, D)), g.standard_normal((1, D))
    assert np.array_equal(O.rope(k, [0], 1e4), k)
    for m, n in [(0, 5), (100, 37), (65535, 1), (12345, 54321)]:
        rq, rk = O.rope(q, [m], 5e5), O.rope(k, [n], 5e5)
        assert abs(np.linalg.norm(rk) - np.linalg.norm(k)) < 1e-12
        rel = O.rope(k, [n - m], 5e5)  # (R(m)q).(R(n)k) = q.(R(n-m)k)
        assert abs((rq @ rk.T)[0, 0] - (q @ rel.T)[0, 0]) < 1e-10


def _brute_attention(q, K, V, scale):
    out = []
    for h in range(q.shape[0]):
        lg = [sum(q[h, d] * K[j, d] for d in range(K.shape[1])) * scale for j in range(K.shape[0])]
        m = max(lg)
        w = [math.exp(x - m) for x in lg]
        z = sum(w)
        out.append([sum(w[j] * V[j, d] for j in range(K.shape[0])) / z for d in range(V.shape[1])])
    return np.array(out)


@pytest.mark.parametrize("T", [1, 2, 5, 8])
def test_attention_brute_force(T):
    g = np.random.default_rng(T)
    q, K, V = g.standard_normal((3, 4)), g.standard_normal((T, 4)), g.standard_normal((T, 4))
    assert np.allclose(O.attention(q, K, V), _brute_attention(q, K, V, 0.5), rtol=0, atol=1e-13)


def test_attention_special_cases():
    g = np.random.default_rng(12)
    K, V = g.standard_normal((40, 16)), g.standard_normal((40, 16))
    q = g.standard_normal((2, 16))
    lg = (q @ K.T) / 4.0
    assert np.allclose(O.softmax(lg).sum(axis=1), 1.0, atol=1e-12)
    assert np.allclose(O.attention(q, K[:1], V[:1]), np.repeat(V[:1], 2, 0), atol=1e-15)
    assert np.allclose(O.attention(q, np.repeat(K[:1], 40, 0), V), V.mean(0), atol=1e-13)
    assert np.allclose(O.attention(np.zeros((1, 16)), K, V), V.mean(0), atol=1e-13)
    assert np.all(O.attention(q, K[:0], V[:0]) == 0)


@pytest.mark.parametrize("bounds", [[0, 40], [0, 1, 40], [0, 13, 14, 27, 40], list(range(0, 41, 4))])
def test_split_combine_equals_single_pass(bounds):
    g = np.random.default_rng(13)
    K, V = g.standard_normal((40, 16)) * 3, g.standard_normal((40, 16))
    q = g.standard_normal((4, 16))
    assert np.allclose(O.split_combine(q, K, V, bounds), O.attention(q, K, V), rtol=0, atol=1e-13)


def test_byte_accounting_matches_pages():
    c = _claims()
    b = c["kv_bytes_per_token_llama31_70b_fp16"]
    per_tok = O.kv_bytes_per_token(b["layers"], b["kv_heads"], b["head_dim"], b["dtype_bytes"])
    assert per_tok == b["value"] == 320 * 1024
    assert per_tok * 131072 / 2 ** 30 == c["kv_gib_128k_fp16"]["value"]
    assert O.kv_bytes_per_token(80, 8, 128, 1) * 131072 / 2 ** 30 == c["kv_gib_128k_fp8"]["value"]
    f = c["logit_error_weight_factor"]
    assert round(math.exp(f["logit_error"]), 1) == f["factor"]


def _rel(a, b):
    return float(np.linalg.norm(a - b) / np.linalg.norm(b))


def _synthetic_head_errors(seed):
    """The first page's synthetic head (T=4096, D=128, K channels 7/23/88 x20),
    INT8 symmetric absmax, four schemes; returns {name: (out_err, max_logit_err)}."""
    w = W.WORKLOADS[1]
    T, D = 4096, 128
    K = W.small_stream(seed, T, D, w.fixed_outliers, w.fixed_factor).astype(np.float64)
    V = W.small_stream(seed + 1000, T, D).astype(np.float64)
    q = W.small_stream(seed + 2000, 1, D).astype(np.float64)

    def per_tensor(x):
        c, s = O.quant_sym(x, np.max(np.abs(x)), 8)
        return O.dequant_sym(c, s)

    def per_axis(x, axis):
        c, s = O.quant_sym(x, np.max(np.abs(x), axis=axis, keepdims=True), 8)
        return O.dequant_sym(c, s)

    scale = 1 / math.sqrt(D)
    ref = O.attention(q, K, V)
    ref_lg = (q @ K.T) * scale
    out = {}
    for name, (Kq, Vq) in {"per_tensor_kv": (per_tensor(K), per_tensor(V)),
                           "per_channel_k_per_token_v": (per_axis(K, 0), per_axis(V, 1)),
                           "v_only": (K, per_axis(V, 1)),
                           "k_only": (per_tensor(K), V)}.items():
        o = O.attention(q, Kq, Vq)
        out[name] = (_rel(o, ref), float(np.max(np.abs((q @ Kq.T) * scale - ref_lg))))
    return out, float(np.max(np.abs(K)) / np.median(np.abs(K)))


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_synthetic_head_ordering(seed):
    e, headroom = _synthetic_head_errors(seed)
    pt, pc, vo, ko = (e[k][0] for k in ["per_tensor_kv", "per_channel_k_per_token_v", "v_only", "k_only"])
    assert pt > pc > vo  # K error dominates; per-channel K + per-token V cuts it
    assert abs(ko - pt) < 0.2 * pt  # "the combined error is essentially all K"
    assert e["v_only"][1] == 0.0  # V-only leaves the logits exact
    # magnitudes in the spread the page's table falls in (its RNG draws cannot be reproduced)
    assert 0.02 < pt < 0.6 and 0.005 < pc < 0.06 and 0.004 < vo < 0.012
    assert 50 < headroom < 250  # the page: absmax / median|K| ~ 130


def test_per_channel_beats_per_token_keys():
    # the fourth page's experiment: T=512, D=128, channels 3/17/44/91 x60, asym INT4
    w = W.WORKLOADS[2]
    K = W.small_stream(0, 512, 128, w.fixed_outliers, w.fixed_factor).astype(np.float64)
    q = W.small_stream(1, 8, 128).astype(np.float64)
    tok = O.dequant_asym(*O.quant_asym(K, K.min(1, keepdims=True), K.max(1, keepdims=True), 4))
    ch = O.dequant_asym(*O.quant_asym(K, K.min(0, keepdims=True), K.max(0, keepdims=True), 4))
    assert _rel(ch, K) < _rel(tok, K)
    assert _rel(q @ ch.T, q @ K.T) < _rel(q @ tok.T, q @ K.T)
