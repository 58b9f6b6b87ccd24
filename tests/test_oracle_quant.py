"""Pins of the oracle's quantizers against what the pages and the mathematics fix.

Hand-worked examples (tests/golden/quantizer_examples.json), the E4M3 format
definition (tests/golden/e4m3_points.json and torch's float8_e4m3fn), the
quantization error bound, exact reconstruction of constant groups, code ranges,
and per-tensor codes worked by hand.
"""
import json
import os

import numpy as np
import pytest
import torch

import kvq_inputs as W
from oracle import kvq_oracle as O

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _gold(name):
    with open(os.path.join(GOLD, name)) as f:
        return json.load(f)


def test_fl32_matches_ieee_float32_ops():
    g = np.random.default_rng(1)
    a = g.standard_normal(20000).astype(np.float32) * np.float32(7.0)
    b = g.standard_normal(20000).astype(np.float32) + np.float32(0.01)
    a64, b64 = a.astype(np.float64), b.astype(np.float64)
    assert np.array_equal(O.fl32(a64 / b64), (a / b).astype(np.float64))
    assert np.array_equal(O.fl32(a64 * b64), (a * b).astype(np.float64))
    assert np.array_equal(O.fl32(a64 - b64), (a - b).astype(np.float64))
    assert np.array_equal(O.fl32(a64 + b64), (a + b).astype(np.float64))


@pytest.mark.parametrize("case", _gold("quantizer_examples.json")["sym"])
def test_sym_hand_examples(case):
    x = np.array(case["x"])
    c, s = O.quant_sym(x, np.max(np.abs(x)), case["bits"])
    assert float(s) == case["scale"]
    assert c.tolist() == case["codes"]
    assert O.dequant_sym(c, s).tolist() == case["deq"]


@pytest.mark.parametrize("case", _gold("quantizer_examples.json")["asym"])
def test_asym_hand_examples(case):
    x = np.array(case["x"])
    c, s, m = O.quant_asym(x, x.min(), x.max(), case["bits"])
    assert float(s) == case["scale"] and float(m) == case["min"]
    assert c.tolist() == case["codes"]
    assert O.dequant_asym(c, s, m).tolist() == case["deq"]


# Per-tensor symmetric INT (a static per-head scale, the first page's per-tensor
# case of its synthetic head): codes = clamp(round_half_even(x / s), -qmax, qmax).
# Worked by hand with s = 0.5, so every quotient is exact:
#   x      3.0  -0.25  0.75  1.25  100.0  -100.0  0.2   -3.5
#   x/s    6    -0.5   1.5   2.5   200    -200    0.4   -7
#   INT8   6     0     2     2     127    -127    0     -7
#   INT4   6     0     2     2     7      -7      0     -7
_PT_X = [3.0, -0.25, 0.75, 1.25, 100.0, -100.0, 0.2, -3.5]


@pytest.mark.parametrize("fmt,codes", [(O.INT8, [6, 0, 2, 2, 127, -127, 0, -7]),
                                       (O.INT4, [6, 0, 2, 2, 7, -7, 0, -7]),
                                       (O.INT2, [1, 0, 1, 1, 1, -1, 0, -1])])
def test_per_tensor_codes_by_hand(fmt, codes):
    x = O.fl32(np.array(_PT_X)).reshape(1, 8)
    c, s, m = O._quant_tokens(x, O.QSpec(fmt, O.SYM, O.PER_TENSOR), 0.5, 8)
    assert s is None and m is None
    assert c[0].tolist() == codes
    assert O._dequant_tokens(c, None, None, O.QSpec(fmt, O.SYM, O.PER_TENSOR), 0.5, 8)[0].tolist() == \
        [0.5 * k for k in codes]


def test_per_tensor_zero_scale_gives_zero_codes():
    x = np.zeros((3, 8))
    c, _, _ = O._quant_tokens(x, O.QSpec(O.INT8, O.SYM, O.PER_TENSOR), 0.0, 8)
    assert np.all(c == 0)


def test_per_tensor_with_the_tensor_absmax_equals_one_group():
    """With the static scale taken over the whole tensor, the per-tensor branch is
    the symmetric quantizer applied to the tensor as a single group (pinned above
    by hand examples and its bound)."""
    g = np.random.default_rng(12)
    x = O.fl32(g.standard_normal((300, 64)) * np.where(np.arange(64) % 17 == 3, 25.0, 1.0))
    for bits in (2, 4, 8):
        s = O.calibrate_absmax(x, O.sym_qmax(bits))
        c, _, _ = O._quant_tokens(x, O.QSpec(bits, O.SYM, O.PER_TENSOR), s, 64)
        c1, s1 = O.quant_sym(x, np.max(np.abs(x)), bits)
        assert float(s1) == s and np.array_equal(c, c1)


@pytest.mark.parametrize("bits", [2, 4, 8])
def test_error_bound_and_code_ranges(bits):
    g = np.random.default_rng(bits)
    for trial in range(200):
        n = int(g.integers(1, 70))
        x = O.fl32(g.standard_normal(n) * 10.0 ** g.uniform(-3, 3) + g.uniform(-5, 5))
        # asymmetric: |x - x^| <= s/2 (+ a few ulp of the operands), codes in [0, qmax]
        c, s, m = O.quant_asym(x, x.min(), x.max(), bits)
        xh = O.dequant_asym(c, s, m)
        slack = 4 * np.spacing(np.float32(np.max(np.abs(x)) + s * O.asym_qmax(bits)))
        assert np.all(np.abs(x - xh) <= s / 2 + slack)
        assert c.min() >= 0 and c.max() <= O.asym_qmax(bits)
        assert c[np.argmin(x)] == 0
        if O.fl32(x.max() - x.min()) > O.FL32_1EM8:  # the range is not clamped
            assert c[np.argmax(x)] == O.asym_qmax(bits)
        # symmetric: |x - x^| <= s/2 (+ slack), codes in [-qmax, qmax], never -qmax-1
        a = np.max(np.abs(x))
        c, s = O.quant_sym(x, a, bits)
        xh = O.dequant_sym(c, s)
        slack = 4 * np.spacing(np.float32(a))
        assert np.all(np.abs(x - xh) <= s / 2 + slack)
        q = O.sym_qmax(bits)
        assert c.min() >= -q and c.max() <= q
        assert abs(c[np.argmax(np.abs(x))]) == q


@pytest.mark.parametrize("bits", [2, 4, 8])
def test_constant_groups(bits):
    for v in [0.0, 1.0, -3.25, 1e-20, 12345.678]:
        x = O.fl32(np.full(33, v))
        c, s, m = O.quant_asym(x, x.min(), x.max(), bits)
        assert np.all(c == 0) and np.array_equal(O.dequant_asym(c, s, m), x)
        c, s = O.quant_sym(x, np.max(np.abs(x)), bits)
        xh = O.dequant_sym(c, s)
        if v == 0.0:
            assert np.all(xh == 0.0)
        else:  # 127*fl32(a/127) need not equal a: within one float32 ulp
            assert np.all(np.abs(xh - x) <= np.spacing(np.float32(abs(v))))


def test_e4m3_points():
    d = _gold("e4m3_points.json")
    for k, v in d["decode"].items():
        got = O.e4m3_decode(int(k))
        assert got == v and np.signbit(got) == np.signbit(v)
    for b in d["nan_bytes"]:
        assert np.isnan(O.e4m3_decode(b))
    for y, byte in d["encode"]:
        assert int(O.e4m3_encode(y)) == byte, (y, byte)


def test_e4m3_table_against_torch_float8():
    all_bytes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    t = all_bytes.view(torch.float8_e4m3fn).float().double().numpy()
    mine = O.e4m3_decode_table()
    nan = np.isnan(t)
    assert np.array_equal(nan, np.isnan(mine))
    assert np.array_equal(t[~nan], mine[~nan])


def test_e4m3_encode_against_torch_below_saturation():
    g = np.random.default_rng(7)
    y = np.concatenate([
        g.standard_normal(50000) * 10.0 ** g.uniform(-4, 2.6, 50000),
        O.e4m3_decode_table()[:0x7E] * (1 + g.uniform(-0.07, 0.07, 0x7E)),
    ])
    y = O.fl32(y[np.abs(y) < 464.0])
    ref = torch.from_numpy(y.astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(O.e4m3_encode(y), ref.astype(np.int64))


def test_e4m3_midpoints_ties_to_even_and_saturation():
    pos = O.e4m3_decode_table()[:0x7F]
    mids = (pos[:-1] + pos[1:]) / 2
    enc = O.e4m3_encode(mids)
    lo = np.arange(0x7E)
    assert np.all(enc == np.where(lo % 2 == 0, lo, lo + 1))
    assert np.all(O.e4m3_encode(-mids) == (enc | 0x80))
    assert np.all(O.e4m3_encode([448.0, 463.9, 464.0, 1e9]) == 0x7E)
    assert np.all(O.e4m3_encode([-448.0, -1e9]) == 0xFE)


def test_e4m3_relative_error_in_normal_range():
    # the first page: ~3 mantissa bits, <= 6.25% step error across binades
    g = np.random.default_rng(9)
    y = O.fl32(np.exp(g.uniform(np.log(2.0 ** -6), np.log(448.0), 100000)))
    rel = np.abs(O.e4m3_decode(O.e4m3_encode(y)) - y) / y
    assert rel.max() <= 2.0 ** -4


def test_e5m2_table_is_the_top_byte_of_ieee_half():
    # E5M2 shares IEEE binary16's sign, exponent field and bias; its two mantissa
    # bits are the top two of binary16's ten, so byte b is the half with bits b << 8
    halves = (np.arange(256, dtype=np.uint16) << 8).view(np.float16).astype(np.float64)
    mine = O.e5m2_decode_table()
    nan = np.isnan(halves)
    assert np.array_equal(nan, np.isnan(mine))
    assert np.array_equal(halves[~nan], mine[~nan])
    assert O.e5m2_decode(0x7B) == O.E5M2_MAX == 57344.0  # the first page: E5M2 saturates at +-57344
    assert O.e5m2_decode(0x01) == 2.0 ** -16 and O.e5m2_decode(0x04) == 2.0 ** -14


def test_e5m2_encode_is_nearest_with_ties_to_even_over_all_halves():
    # every finite half below saturation, against a brute-force nearest search
    h = np.arange(0, 0x7C00, dtype=np.uint16).view(np.float16).astype(np.float64)
    h = h[h < O.E5M2_MAX]
    pos = O.e5m2_decode_table()[:0x7C]
    d = np.abs(h[:, None] - pos[None, :])
    best = d.min(axis=1, keepdims=True)
    cand = d == best
    # ties: the even byte (even mantissa)
    want = np.where(cand.sum(1) > 1, np.argmax(cand & (np.arange(0x7C) % 2 == 0)[None, :], axis=1),
                    np.argmax(cand, axis=1))
    assert np.array_equal(O.e5m2_encode(h), want)
    assert np.array_equal(O.e5m2_encode(-h[h > 0]), want[h > 0] | 0x80)


def test_e5m2_midpoints_saturation_and_torch():
    pos = O.e5m2_decode_table()[:0x7C]
    mids = (pos[:-1] + pos[1:]) / 2
    lo = np.arange(0x7B)
    assert np.all(O.e5m2_encode(mids) == np.where(lo % 2 == 0, lo, lo + 1))
    assert np.all(O.e5m2_encode([57344.0, 61439.0, 61440.0, 1e9]) == 0x7B)
    assert np.all(O.e5m2_encode([-57344.0, -1e9]) == 0xFB)
    all_bytes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    t = all_bytes.view(torch.float8_e5m2).float().double().numpy()
    nan = np.isnan(t)
    assert np.array_equal(nan, np.isnan(O.e5m2_decode_table()))
    assert np.array_equal(t[~nan], O.e5m2_decode_table()[~nan])
    g = np.random.default_rng(13)
    y = O.fl32(g.standard_normal(50000) * 10.0 ** g.uniform(-5, 4.6, 50000))
    y = y[np.abs(y) < 57344.0]
    ref = torch.from_numpy(y.astype(np.float32)).to(torch.float8_e5m2).view(torch.uint8).numpy()
    assert np.array_equal(O.e5m2_encode(y), ref.astype(np.int64))


def test_e5m2_relative_error_in_normal_range():
    # the first page: E5M2 has only 2 mantissa bits: <= 12.5% step error
    g = np.random.default_rng(10)
    y = O.fl32(np.exp(g.uniform(np.log(2.0 ** -14), np.log(57344.0), 100000)))
    rel = np.abs(O.e5m2_decode(O.e5m2_encode(y)) - y) / y
    assert rel.max() <= 2.0 ** -3
    assert rel.max() > 2.0 ** -4  # coarser than E4M3


def test_fp8_formats_quantize_with_their_own_tables():
    g = np.random.default_rng(12)
    x = O.fl32(g.standard_normal(4096) * 30)
    for fmt, qmax, dec in ((O.FP8_E4M3, 448.0, O.e4m3_decode), (O.FP8_E5M2, 57344.0, O.e5m2_decode)):
        s = O.calibrate_absmax(x, qmax)
        b = O.quant_fp8(x, s, fmt)
        assert np.array_equal(O.dequant_fp8(b, s, fmt), O.fl32(dec(b) * s))
        assert np.array_equal(b, O.fp8_encode(O.fl32(x / s), fmt))


# ---------------------------------------------------------- fp16 scale/min storage

_H16 = np.arange(0, 0x10000, dtype=np.uint16).view(np.float16)
_HALVES = np.unique(_H16[np.isfinite(_H16)].astype(np.float64))  # every finite binary16 value, increasing


def test_f16_directed_rounding_against_every_half():
    g = np.random.default_rng(21)
    x = np.concatenate([g.standard_normal(20000) * 10.0 ** g.uniform(-9, 4.9, 20000),
                        _HALVES[::97], [0.0, -0.0, 65504.0, -65504.0, 6.0e-8, 3.0e-8]])
    x = O.fl32(x)
    x = x[np.abs(x) <= 65504.0]  # beyond: saturation, checked below
    up = _HALVES[np.searchsorted(_HALVES, x, side="left")]
    down = _HALVES[np.searchsorted(_HALVES, x, side="right") - 1]
    assert np.array_equal(O.f16_up(x), up)
    assert np.array_equal(O.f16_down(x), down)
    assert np.all(O.f16_up([7e4, 1e9]) == 65504.0) and np.all(O.f16_down([-7e4, -1e9]) == -65504.0)


@pytest.mark.parametrize("bits", [2, 4, 8])
def test_fp16_meta_keeps_the_half_step_bound(bits):
    g = np.random.default_rng(22 + bits)
    for trial in range(200):
        scale = 10.0 ** g.uniform(-3, 3)
        x = O.fl32(g.standard_normal(64) * scale + g.uniform(-3, 3) * scale)
        mn, mx = x.min(), x.max()
        c, s, m = O.quant_asym16(x, mn, mx, bits)
        c32, s32, _ = O.quant_asym(x, mn, mx, bits)
        assert s == O.f16_up(s) and m == O.f16_down(m) and m <= mn and s >= s32 * (1 - 2.0 ** -23)
        assert c.min() >= 0 and c.max() <= O.asym_qmax(bits)
        err = np.abs(O.dequant_asym(c, s, m) - x)
        assert np.all(err <= s / 2 * (1 + 2.0 ** -20) + 4 * np.spacing(np.float32(np.abs(x).max())))
        a = np.max(np.abs(x))
        c, s = O.quant_sym16(x, a, bits)
        assert s == O.f16_up(s) and s >= float(O.fl32(a / O.sym_qmax(bits)))
        assert np.abs(c).max() <= O.sym_qmax(bits)
        err = np.abs(O.dequant_sym(c, s) - x)
        assert np.all(err <= s / 2 * (1 + 2.0 ** -20) + 4 * np.spacing(np.float32(a)))


def test_fp16_meta_zero_and_constant_groups():
    z = np.zeros(16)
    c, s = O.quant_sym16(z, 0.0, 4)
    assert s == 0.0 and np.all(c == 0)
    x = np.full(16, 3.25)  # a binary16 value: the minimum is stored exactly
    c, s, m = O.quant_asym16(x, x.min(), x.max(), 4)
    assert np.all(c == 0) and m == 3.25 and np.all(O.dequant_asym(c, s, m) == x)


def test_fp16_meta_halves_the_metadata_of_the_2bit_layer():
    # the 8B layer's formats: 2-bit codes (32 B K + 32 B V per token and kv-head), key
    # scale+min per (32-token group, channel), value scale+min per (token, 32-channel group)
    base = dict(num_q_heads=32, num_kv_heads=8, head_dim=128, k=O.QSpec(O.INT2, O.ASYM, O.PER_CHANNEL, 32),
                v=O.QSpec(O.INT2, O.ASYM, O.PER_TOKEN, 32), residual=128, page_size=256)
    L32, L16 = O.layout(O.Config(**base)), O.layout(O.Config(meta_dtype=O.F16, **base))
    per_tok = lambda L: (L["head"] - 0) / 256
    assert per_tok(L32) == 64 + 32 + 32 and per_tok(L16) == 64 + 16 + 16
    # 16 sequences x 8 kv-heads x 32768 quantized tokens, + 127 bf16 window rows of K and V, + q/out
    nq = 16 * 8 * 32768
    extra = 16 * 8 * 127 * 128 * 2 * 2 + 16 * 32 * 128 * (2 + 4)
    assert round((nq * per_tok(L32) + extra) / 1e6, 1) == 545.6
    assert round((nq * per_tok(L16) + extra) / 1e6, 1) == 411.4


def test_fp16_meta_chunking_invariance():
    cfg = O.Config(4, 1, 64, O.QSpec(O.INT4, O.ASYM, O.PER_CHANNEL, 16), O.QSpec(O.INT2, O.SYM, O.PER_TOKEN, 32),
                   residual=32, page_size=16, meta_dtype=O.F16)
    K = W.small_stream(31, 200, 64, (3, 9), 40.0)
    V = W.small_stream(32, 200, 64)
    sc = O.StreamCache(cfg)
    for a, b in ((0, 1), (1, 40), (40, 41), (41, 200)):
        sc.append(K[a:b], V[a:b])
    st, ref = sc.state(), O.quantize_stream(cfg, K, V)
    for f in ("kc", "ks", "km", "vc", "vs"):
        assert np.array_equal(getattr(st, f), getattr(ref, f)), f


def test_fp8_scale_roundtrip_and_zero_scale():
    g = np.random.default_rng(11)
    x = O.fl32(g.standard_normal(4096) * 30)
    s = O.calibrate_absmax(x, 448.0)
    assert s == float(np.float32(np.float32(np.max(np.abs(x))) / np.float32(448.0)))
    b = O.quant_fp8(x, s)
    xh = O.dequant_fp8(b, s)
    assert np.all(np.abs(xh) <= 448.0 * s * (1 + 2 ** -23))
    assert np.max(np.abs(xh - x) / np.maximum(np.abs(x), 2.0 ** -6 * s)) <= 2.0 ** -4 + 1e-6
    assert np.all(O.quant_fp8(x, 0.0) == 0) and np.all(O.dequant_fp8(O.quant_fp8(x, 0.0), 0.0) == 0)
