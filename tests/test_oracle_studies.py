"""Pins of the accuracy studies (oracle/studies.py) and the orderings they show.

Metric definitions against hand-worked values, Gibbs' inequality and their
invariances; the pre-/post-RoPE key study against its identity case and the
orderings "KV Cache Quantization: Why Keys and Values Need Different Axes",
section "Where does RoPE break this?" describes; the attention-agreement study
(per-head KL, top-k overlap and rank agreement, "FP8 KV Cache Quantization: Why
Keys Break Before Values", section "Why doesn't perplexity catch KV cache
quantization damage?") on the seeded streams of the benchmark workloads.

`python -m pytest tests/test_oracle_studies.py -k table -s` prints the study
tables quoted in the design notes.
"""
import math

import numpy as np
import pytest

import kvq_inputs as W
from oracle import kvq_oracle as O
from oracle import studies as S

THETA = 500000.0
FAST = (2, 9, 17, 30)  # pairs 1, 4, 8, 15: theta^(-2i/D) = 0.82 .. 0.03 rad per token
SLOW = (100, 110, 118, 126)  # pairs 50 .. 63: below 4e-5 rad per token


# ------------------------------------------------------------------ metric pins

def test_kl_hand_values_and_gibbs():
    p = np.array([[0.5, 0.5]])
    q = np.array([[0.25, 0.75]])
    want = 0.5 * math.log(0.5 / 0.25) + 0.5 * math.log(0.5 / 0.75)
    assert S.kl_rows(p, q)[0] == pytest.approx(want, rel=1e-15)
    assert S.kl_rows(p, p)[0] == 0.0
    # a zero in p contributes nothing; a zero in q under mass of p is infinite
    assert S.kl_rows(np.array([[1.0, 0.0]]), np.array([[0.5, 0.5]]))[0] == pytest.approx(math.log(2.0))
    assert S.kl_rows(np.array([[0.5, 0.5]]), np.array([[1.0, 0.0]]))[0] == math.inf
    g = np.random.default_rng(3)
    for _ in range(20):
        a = g.random((4, 37)); a /= a.sum(1, keepdims=True)
        b = g.random((4, 37)); b /= b.sum(1, keepdims=True)
        assert np.all(S.kl_rows(a, b) > 0.0)


def test_topk_indices_ties_and_order():
    x = np.array([[1.0, 3.0, 3.0, 2.0, 0.5]])
    assert S.topk_indices(x, 3).tolist() == [[1, 2, 3]]
    assert S.topk_indices(x, 1).tolist() == [[1]]


def test_topk_overlap_hand_values_and_invariance():
    p = np.array([[0.4, 0.3, 0.2, 0.1]])
    assert S.topk_overlap(p, p, 2)[0] == 1.0
    assert S.topk_overlap(p, p[:, ::-1], 2)[0] == 0.0
    assert S.topk_overlap(p, np.array([[0.4, 0.1, 0.3, 0.2]]), 2)[0] == 0.5
    g = np.random.default_rng(4)
    a, b = g.random((3, 50)), g.random((3, 50))
    perm = g.permutation(50)
    assert np.array_equal(S.topk_overlap(a, b, 8), S.topk_overlap(a[:, perm], b[:, perm], 8))


def test_topk_rank_agreement_hand_values():
    p = np.array([[0.4, 0.3, 0.2, 0.1]])
    assert S.topk_rank_agreement(p, p, 4)[0] == 1.0
    assert S.topk_rank_agreement(p, p[:, ::-1], 4)[0] == 0.0
    # one adjacent swap: 5 of the 6 pairs keep their order
    assert S.topk_rank_agreement(p, np.array([[0.3, 0.4, 0.2, 0.1]]), 4)[0] == pytest.approx(5 / 6)
    # pairs tied in p are skipped; no untied pair gives 1
    assert S.topk_rank_agreement(np.array([[0.5, 0.5]]), np.array([[0.2, 0.8]]), 2)[0] == 1.0


# ----------------------------------------------------- pre- versus post-RoPE keys

def _offset_head(seed, T, channels, offset=30.0):
    """N(0,1) keys whose `channels` carry a steady offset: the clean, persistent
    outlier structure the pages describe ("channel 44 is always huge")."""
    K = W.small_stream(seed, T, 128).astype(np.float64)
    K[:, list(channels)] += offset
    return W.bf16_round(K.astype(np.float32))[1].astype(np.float64)


def _pre_post_logit_err(K, bits, G=64, theta=THETA, seed=0):
    T = K.shape[0]
    pos = np.arange(T)
    spec = O.QSpec(bits, O.ASYM, O.PER_CHANNEL, G)
    Kr = O.rope(K, pos, theta)
    q = np.random.default_rng(100 + seed).standard_normal((4, 128))
    pre = S.logit_errors(q, Kr, S.rope_keys_pre(K, pos, theta, spec))[0]
    post = S.logit_errors(q, Kr, S.rope_keys_post(K, pos, theta, spec))[0]
    return pre, post


def test_rope_schemes_agree_without_rotation():
    K = _offset_head(1, 256, FAST)
    spec = O.QSpec(O.INT4, O.ASYM, O.PER_CHANNEL, 64)
    zero = np.zeros(256, dtype=np.int64)
    assert np.array_equal(S.rope_keys_pre(K, zero, THETA, spec), S.rope_keys_post(K, zero, THETA, spec))


@pytest.mark.parametrize("bits", [O.INT2, O.INT4, O.INT8])
def test_post_rope_smears_fast_pair_outliers(bits):
    r = [_pre_post_logit_err(_offset_head(s, 2048, FAST), bits, seed=s) for s in range(3)]
    pre, post = np.mean([x[0] for x in r]), np.mean([x[1] for x in r])
    assert post >= 2.0 * pre, (pre, post)


@pytest.mark.parametrize("bits", [O.INT2, O.INT4])
def test_slow_pairs_keep_their_channel_structure(bits):
    r = [_pre_post_logit_err(_offset_head(s, 2048, SLOW), bits, seed=s) for s in range(3)]
    pre, post = np.mean([x[0] for x in r]), np.mean([x[1] for x in r])
    assert 0.95 * pre <= post <= 1.05 * pre, (pre, post)


def test_scaled_outliers_on_fast_pairs_still_favour_pre_rope():
    r = []
    for s in range(3):
        K = W.small_stream(s, 2048, 128, FAST, 30.0, True).astype(np.float64)
        r.append(_pre_post_logit_err(K, O.INT4, seed=s))
    assert np.mean([x[1] for x in r]) >= 1.05 * np.mean([x[0] for x in r])


def test_post_rope_attention_error_at_output():
    """The same ordering after softmax and P.V: a pre-RoPE cache against a cache
    holding bf16 post-RoPE keys, both INT4 per-channel keys (G 64) with INT8
    per-token values and a 64-token window, against float64 attention over the
    unquantized rotated keys."""
    T = 4096 + 37
    base = dict(num_q_heads=4, num_kv_heads=1, head_dim=128, v=O.QSpec(O.INT8, O.SYM, O.PER_TOKEN, 0),
                residual=64, page_size=16, rope_theta=THETA, src_dtype=O.BF16,
                k=O.QSpec(O.INT4, O.ASYM, O.PER_CHANNEL, 64))
    pre_cfg, post_cfg = O.Config(rope_pre=1, **base), O.Config(rope_pre=0, **base)
    ep, eq = [], []
    for b in range(2):
        K = _offset_head(900 + b, T, FAST)
        V = W.small_stream(950 + b, T, 128, bf16=True).astype(np.float64)
        Kr = O.rope(K, np.arange(T), THETA)
        Kpost = W.bf16_round(Kr.astype(np.float32))[1].astype(np.float64)
        q = W.bf16_round(np.random.default_rng(7 + b).standard_normal((4, 128)).astype(np.float32))[1]
        ref = O.attention(q, Kr, V)
        for cfg, Ks, acc in ((pre_cfg, K, ep), (post_cfg, Kpost, eq)):
            out = O.decode_head(cfg, O.quantize_stream(cfg, Ks, V), q.astype(np.float64))
            acc.append(np.linalg.norm(out - ref, axis=1) / np.linalg.norm(ref, axis=1))
    assert np.mean(eq) >= 1.8 * np.mean(ep), (np.mean(ep), np.mean(eq))


# -------------------------------------------------- attention agreement (KL, top-k)

def _agreement(cid, seq, head, T, spec, rope_theta=None, k=32):
    w = W.WORKLOADS[cid]
    rep = w.num_q_heads // w.num_kv_heads
    K = W.kv_block(w, seq, head, W.KIND_K, 0, T).astype(np.float64)
    q = W.queries(w, 0)[seq, head * rep:(head + 1) * rep].astype(np.float64)
    pos = np.arange(T)
    Kref = O.rope(K, pos, rope_theta) if rope_theta else K
    Kq = S.dequantized_keys(K, spec)
    if rope_theta:
        Kq = O.rope(Kq, pos, rope_theta)
    p, pq = S.attention_probs(q, Kref), S.attention_probs(q, Kq)
    return S.kl_rows(p, pq).mean(), S.topk_overlap(p, pq, k).mean(), S.topk_rank_agreement(p, pq, k).mean()


HEADS = {3: [(0, 0), (1, 5), (7, 2)], 5: [(0, 0), (3, 2), (9, 6)]}


@pytest.mark.parametrize("cid", [3, 5])
@pytest.mark.parametrize("bits", [O.INT2, O.INT4])
def test_per_channel_keys_keep_attention_closer(cid, bits):
    theta = THETA if cid == 5 else None
    g = 32 if cid == 3 else 64
    for seq, head in HEADS[cid]:
        ch = _agreement(cid, seq, head, 4096, O.QSpec(bits, O.ASYM, O.PER_CHANNEL, g), theta)
        tok = _agreement(cid, seq, head, 4096, O.QSpec(bits, O.ASYM, O.PER_TOKEN, 32 if cid == 3 else 0), theta)
        assert ch[0] < tok[0], (seq, head, ch, tok)  # KL
        assert ch[1] > tok[1], (seq, head, ch, tok)  # top-32 overlap


def test_attention_kl_falls_with_bits():
    for seq, head in HEADS[3]:
        kl = [_agreement(3, seq, head, 4096, O.QSpec(b, O.ASYM if b < 8 else O.SYM, O.PER_CHANNEL, 32))[0]
              for b in (O.INT2, O.INT4, O.INT8)]
        assert kl[0] > kl[1] > kl[2] > 0.0, kl
        ov = _agreement(3, seq, head, 4096, O.QSpec(O.INT8, O.SYM, O.PER_CHANNEL, 32))[1]
        assert ov >= 0.95


# ------------------------------------------- FP8 formats, calibrated and unit scales

def fp8_head(seed, T=2048, reach=1000.0):
    """A synthetic head for the FP8 comparison ("FP8 KV Cache Quantization: Why
    Keys Break Before Values", section "Why do per-tensor scales waste bits on
    the K cache?", failure mode 1): N(0,1) keys whose channels 3, 17, 44 and 91
    are scaled by reach / 3 (so they reach about +-reach), N(0,1) values and 8
    queries N(0, 0.05^2); all bf16."""
    K = W.small_stream(seed, T, 128).astype(np.float64)
    K[:, [3, 17, 44, 91]] *= reach / 3.0
    K = W.bf16_round(K.astype(np.float32))[1].astype(np.float64)
    V = W.small_stream(seed + 50, T, 128, bf16=True).astype(np.float64)
    q = W.bf16_round(np.random.default_rng(seed).standard_normal((8, 128)).astype(np.float32) * 0.05)[1]
    return K, V, q.astype(np.float64)


FP8_SCHEMES = (("E4M3, unit scale", O.FP8_E4M3, None), ("E5M2, unit scale", O.FP8_E5M2, None),
               ("E4M3, calibrated", O.FP8_E4M3, 448.0), ("E5M2, calibrated", O.FP8_E5M2, 57344.0))


def fp8_errors(reach, seeds=(0, 1, 2)):
    """Mean relative L2 attention error of each FP8 key scheme (values kept
    exact) against float64 attention over the bf16 keys."""
    out = {}
    for seed in seeds:
        K, V, q = fp8_head(seed, reach=reach)
        ref = O.attention(q, K, V)
        for name, fmt, qmax in FP8_SCHEMES:
            s = 1.0 if qmax is None else O.calibrate_absmax(K, qmax)
            Kq = O.dequant_fp8(O.quant_fp8(K, s, fmt), s, fmt)
            e = np.linalg.norm(O.attention(q, Kq, V) - ref, axis=1) / np.linalg.norm(ref, axis=1)
            out.setdefault(name, []).append(e.mean())
    return {k: float(np.mean(v)) for k, v in out.items()}


def test_unit_scale_clipping_is_worse_than_coarse_e5m2():
    e = fp8_errors(1000.0)
    assert e["E4M3, unit scale"] > 2.0 * e["E5M2, unit scale"], e  # clipping deletes the channel
    assert e["E5M2, unit scale"] > e["E4M3, calibrated"], e
    assert e["E4M3, calibrated"] < e["E5M2, calibrated"], e  # 3 mantissa bits beat 2 once nothing clips


def test_unit_scale_costs_little_in_range():
    e = fp8_errors(250.0)  # below 448: nothing clips; calibration only moves values to finer binades
    assert e["E4M3, unit scale"] <= 1.3 * e["E4M3, calibrated"], e
    assert e["E4M3, unit scale"] < 0.1 * fp8_errors(1000.0)["E4M3, unit scale"], e


# --------------------------------------------------------------------- the tables

def test_study_tables():
    print("\npre- vs post-RoPE per-channel keys (asym, G 64, theta 5e5, T 2048, 3 heads):"
          " mean |logit error| pre / post")
    for name, ch in (("steady offset +30 on fast pairs", FAST), ("steady offset +30 on slow pairs", SLOW)):
        row = []
        for bits in (O.INT2, O.INT4, O.INT8):
            r = [_pre_post_logit_err(_offset_head(s, 2048, ch), bits, seed=s) for s in range(3)]
            row.append(f"INT{bits} {np.mean([x[0] for x in r]):.4f} / {np.mean([x[1] for x in r]):.4f}")
        print(f"  {name:34s} " + "   ".join(row))
    print("attention agreement, 4096 tokens, mean over 3 (seq, kv-head): KL / top-32 overlap / rank agreement")
    for cid, theta, g in ((3, None, 32), (5, THETA, 64)):
        for label, spec in (("INT2 per-channel", O.QSpec(O.INT2, O.ASYM, O.PER_CHANNEL, g)),
                            ("INT2 per-token", O.QSpec(O.INT2, O.ASYM, O.PER_TOKEN, 32 if cid == 3 else 0)),
                            ("INT4 per-channel", O.QSpec(O.INT4, O.ASYM, O.PER_CHANNEL, g)),
                            ("INT4 per-token", O.QSpec(O.INT4, O.ASYM, O.PER_TOKEN, 32 if cid == 3 else 0)),
                            ("INT8 per-channel", O.QSpec(O.INT8, O.SYM, O.PER_CHANNEL, g))):
            r = np.array([_agreement(cid, s, h, 4096, spec, theta) for s, h in HEADS[cid]])
            print(f"  workload {cid} {label:18s} {r[:, 0].mean():9.3g} {r[:, 1].mean():6.3f} {r[:, 2].mean():6.3f}")
    print("FP8 keys, attention rel L2 error (values exact), keys reaching ~250 / ~1000:")
    lo, hi = fp8_errors(250.0), fp8_errors(1000.0)
    for name, _, _ in FP8_SCHEMES:
        print(f"  {name:18s} {lo[name]:.4f} / {hi[name]:.4f}")
