"""CPU oracle for quantized-KV decode attention (float64 numpy).

TEST INFRASTRUCTURE ONLY.  Only the tests under tests/, the smoke check in
__graft_entry__.smoke() and bench.py's cpu_baseline / reference leg may import,
call or execute anything under oracle/.  The product path (the CUDA library and
its Python binding) never does, and this module imports nothing from it.

Everything here is the plain definition, written for a reader to check by eye:

* fl32(x) rounds a float64 value to the nearest float32 (ties to even).  One
  IEEE fp32 +, -, *, / is emulated exactly as fl32 of the float64 operation on
  fp32 inputs (53 >= 2*24 + 2, so the double rounding is harmless).
* Symmetric absmax INT-b -- "FP8 KV Cache Quantization: Why Keys Break Before
  Values", section "Why does the K cache break before the V cache?", `qint8`
  listing: s = amax|x|/qmax, c = clamp(round(x/s), -qmax, qmax), x^ = c*s.
  qmax = 2^(b-1)-1 (127 for INT8; 7 for INT4 as "KV Cache Quantization: Why
  Keys and Values Need Different Axes", section "Why does per-token key
  quantization destroy accuracy?" states).  Reading where the page is silent:
  an all-zero group has s = 0 and codes 0.
* Asymmetric min-max INT-b -- "KV Cache Quantization: Why Keys and Values Need
  Different Axes", same section, `quant_dequant` listing: qmax = 2^b-1,
  scale = max(mx-mn, 1e-8)/qmax, c = clamp(round((x-mn)/scale), 0, qmax),
  x^ = c*scale + mn; the zero point is the float minimum.
* FP8 E4M3 with a static per-head scale -- "FP8 KV Cache Quantization: Why Keys
  Break Before Values", section "Why do per-tensor scales waste bits on the K
  cache?" (E4M3 saturates at +-448, ~3 mantissa bits).  The encoder below is
  written from the OCP E4M3FN format definition (bias 7, subnormal step 2^-9,
  no infinities, 0x7F/0xFF NaN): round to nearest, ties to even, saturate.
  FP8 E5M2 (the same page and section: saturates at +-57344, 2 mantissa bits)
  is written from its format definition (bias 15, subnormal step 2^-16,
  exponent 31 for infinities and NaN): round to nearest, ties to even,
  saturating at 57344; an uncalibrated cache uses the unit scale (the same page,
  section "Why do per-tensor scales waste bits on the K cache?", failure mode
  1), which the static-scale path covers with scale 1.
* fp16 scale/min storage (optional): the scale is stored rounded up to the next
  binary16 value and the minimum rounded down, and the codes are computed from
  the stored values, so the +-s/2 error bound of the fp32 rule still holds.
  Reading: the asymmetric range is taken from the stored (rounded-down) minimum,
  d = max(mx - mn16, 1e-8), so the top code never clips.  Values beyond the
  binary16 range saturate (scale 65504, minimum -65504).
* Axes: K per channel over G-token groups, V per token ("Why Keys Are More
  Sensitive Than Values in INT8 KV Cache Quantization", section "Outlier
  Distribution in Key Channels"; fourth page, "What should I actually turn on
  in production?" checklist).
* Residual window: the newest tokens stay unquantized and are folded into the
  quantized cache in blocks (first page, section "Should you quantize keys
  pre-RoPE or post-RoPE?"; fourth page checklist).  Reading: the window holds R
  tokens; when it fills, all R are quantized and it empties.
* RoPE on pre-RoPE keys after dequantization: pairs (2i, 2i+1) rotated by the
  absolute position times theta^(-2i/D) (fourth page, section "Where does RoPE
  break this?").
* Attention: logits = q.k/sqrt(d), softmax, out = sum p_j v_j (first page,
  section "Why does the K cache break before the V cache?").

Every function is pinned by the tests in tests/test_oracle_*.py against values
the pages print, closed forms, invariants and brute force.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np

INT2, INT4, INT8, FP8_E4M3, FP8_E5M2 = 2, 4, 8, 9, 10
SYM, ASYM = 0, 1
PER_TENSOR, PER_TOKEN, PER_CHANNEL = 0, 1, 2
F32, BF16, F16 = 0, 1, 2  # source dtypes; F16 also names fp16 scale/min storage

FL32_1EM8 = float(np.float32(1e-8))
E4M3_MAX = 448.0
E5M2_MAX = 57344.0


def fl32(x):
    """Round float64 values to the nearest float32 (ties to even), as float64."""
    return np.asarray(x, dtype=np.float64).astype(np.float32).astype(np.float64)


# ----------------------------------------------------------------------------- formats

def is_fp8(fmt: int) -> bool:
    return fmt in (FP8_E4M3, FP8_E5M2)


def bits_of(fmt: int) -> int:
    return 8 if is_fp8(fmt) else int(fmt)


def sym_qmax(bits: int) -> int:
    return 2 ** (bits - 1) - 1


def asym_qmax(bits: int) -> int:
    return 2 ** bits - 1


def e4m3_decode_table() -> np.ndarray:
    """Value of every E4M3FN byte (NaN for 0x7F and 0xFF)."""
    t = np.empty(256, dtype=np.float64)
    for byte in range(256):
        sign = -1.0 if byte & 0x80 else 1.0
        e = (byte >> 3) & 0xF
        m = byte & 0x7
        if e == 0xF and m == 0x7:
            t[byte] = np.nan
        elif e == 0:
            t[byte] = sign * m * 2.0 ** -9
        else:
            t[byte] = sign * (1.0 + m / 8.0) * 2.0 ** (e - 7)
    return t


_E4M3 = e4m3_decode_table()
_E4M3_POS = _E4M3[:0x7F]  # bytes 0x00..0x7E: every finite non-negative value, increasing


def e4m3_encode(y) -> np.ndarray:
    """Encode float values to E4M3FN bytes: nearest value, ties to the even
    mantissa (the even byte), magnitudes >= 448 saturate to 448 (0x7E)."""
    y = np.asarray(y, dtype=np.float64)
    a = np.abs(y)
    sat = a >= E4M3_MAX
    ac = np.where(sat, 0.0, a)
    idx = np.searchsorted(_E4M3_POS, ac, side="right") - 1  # _E4M3_POS[idx] <= a
    idx = np.clip(idx, 0, 0x7D)
    lo = _E4M3_POS[idx]
    hi = _E4M3_POS[idx + 1]
    dlo = ac - lo
    dhi = hi - ac
    up = (dhi < dlo) | ((dhi == dlo) & (idx % 2 == 1))
    mag = np.where(up, idx + 1, idx)
    mag = np.where(sat, 0x7E, mag)
    out = mag.astype(np.int64) | np.where(np.signbit(y), 0x80, 0)
    out = np.where(np.isnan(y), 0x7F, out)
    return out.astype(np.int64)


def e4m3_decode(byte) -> np.ndarray:
    return _E4M3[np.asarray(byte, dtype=np.int64)]


def e5m2_decode_table() -> np.ndarray:
    """Value of every E5M2 byte (+-inf for 0x7C/0xFC, NaN for 0x7D..0x7F and
    0xFD..0xFF)."""
    t = np.empty(256, dtype=np.float64)
    for byte in range(256):
        sign = -1.0 if byte & 0x80 else 1.0
        e = (byte >> 2) & 0x1F
        m = byte & 0x3
        if e == 0x1F:
            t[byte] = sign * np.inf if m == 0 else np.nan
        elif e == 0:
            t[byte] = sign * m * 2.0 ** -16
        else:
            t[byte] = sign * (1.0 + m / 4.0) * 2.0 ** (e - 15)
    return t


_E5M2 = e5m2_decode_table()
_E5M2_POS = _E5M2[:0x7C]  # bytes 0x00..0x7B: every finite non-negative value, increasing


def e5m2_encode(y) -> np.ndarray:
    """Encode float values to E5M2 bytes: nearest value, ties to the even
    mantissa (the even byte), magnitudes >= 57344 saturate to 57344 (0x7B)."""
    y = np.asarray(y, dtype=np.float64)
    a = np.abs(y)
    sat = a >= E5M2_MAX
    ac = np.where(sat | np.isnan(y), 0.0, a)
    idx = np.searchsorted(_E5M2_POS, ac, side="right") - 1  # _E5M2_POS[idx] <= a
    idx = np.clip(idx, 0, 0x7A)
    lo = _E5M2_POS[idx]
    hi = _E5M2_POS[idx + 1]
    dlo = ac - lo
    dhi = hi - ac
    up = (dhi < dlo) | ((dhi == dlo) & (idx % 2 == 1))
    mag = np.where(up, idx + 1, idx)
    mag = np.where(sat, 0x7B, mag)
    out = mag.astype(np.int64) | np.where(np.signbit(y), 0x80, 0)
    out = np.where(np.isnan(y), 0x7F, out)
    return out.astype(np.int64)


def e5m2_decode(byte) -> np.ndarray:
    return _E5M2[np.asarray(byte, dtype=np.int64)]


def fp8_max(fmt: int) -> float:
    return E5M2_MAX if fmt == FP8_E5M2 else E4M3_MAX


def fp8_encode(y, fmt: int) -> np.ndarray:
    return e5m2_encode(y) if fmt == FP8_E5M2 else e4m3_encode(y)


def fp8_decode(byte, fmt: int) -> np.ndarray:
    return e5m2_decode(byte) if fmt == FP8_E5M2 else e4m3_decode(byte)


# ------------------------------------------------------------------------- quantizers

def quant_sym(x, absmax, bits: int):
    """Symmetric absmax INT-b of fp32-exact values x against the group absmax.

    Returns (codes int64, scale)."""
    qmax = sym_qmax(bits)
    s = fl32(np.asarray(absmax, dtype=np.float64) / qmax)
    with np.errstate(divide="ignore", invalid="ignore"):
        y = fl32(np.asarray(x, dtype=np.float64) / s)
    c = np.clip(np.rint(y), -qmax, qmax)
    c = np.where(s == 0.0, 0.0, c)
    return c.astype(np.int64), s


F16_MAX = 65504.0


def f16_up(x) -> np.ndarray:
    """Smallest binary16 value >= x (as float64), saturating at +-65504."""
    x = np.asarray(x, dtype=np.float64)
    h = np.clip(x, -F16_MAX, F16_MAX).astype(np.float16)  # nearest
    with np.errstate(over="ignore"):  # stepping past 65504 gives inf, saturated below
        h = np.where(h.astype(np.float64) < x, np.nextafter(h, np.float16(np.inf)), h)
    return np.minimum(h.astype(np.float64), F16_MAX)


def f16_down(x) -> np.ndarray:
    """Largest binary16 value <= x (as float64), saturating at +-65504."""
    x = np.asarray(x, dtype=np.float64)
    h = np.clip(x, -F16_MAX, F16_MAX).astype(np.float16)
    with np.errstate(over="ignore"):
        h = np.where(h.astype(np.float64) > x, np.nextafter(h, np.float16(-np.inf)), h)
    return np.maximum(h.astype(np.float64), -F16_MAX)


def quant_sym16(x, absmax, bits: int):
    """Symmetric INT-b with the scale stored as binary16 rounded up:
    s = f16_up(fl32(a / qmax)), c = clamp(rint(fl32(x / s)), -qmax, qmax)."""
    qmax = sym_qmax(bits)
    s = f16_up(fl32(np.asarray(absmax, dtype=np.float64) / qmax))
    with np.errstate(divide="ignore", invalid="ignore"):
        y = fl32(np.asarray(x, dtype=np.float64) / s)
    c = np.clip(np.rint(y), -qmax, qmax)
    c = np.where(s == 0.0, 0.0, c)
    return c.astype(np.int64), s


def quant_asym16(x, mn, mx, bits: int):
    """Asymmetric INT-b with binary16 storage: mn16 = f16_down(mn),
    d = max(fl32(mx - mn16), 1e-8f), s = f16_up(fl32(d / qmax)),
    c = clamp(rint(fl32(fl32(x - mn16) / s)), 0, qmax).  Returns (codes, s, mn16)."""
    qmax = asym_qmax(bits)
    mn16 = f16_down(np.asarray(mn, dtype=np.float64))
    d = np.maximum(fl32(np.asarray(mx, dtype=np.float64) - mn16), FL32_1EM8)
    s = f16_up(fl32(d / qmax))
    t = fl32(np.asarray(x, dtype=np.float64) - mn16)
    c = np.clip(np.rint(fl32(t / s)), 0, qmax)
    return c.astype(np.int64), s, mn16


def dequant_sym(c, s):
    return fl32(np.asarray(c, dtype=np.float64) * s)


def quant_asym(x, mn, mx, bits: int):
    """Asymmetric min-max INT-b.  Returns (codes int64, scale, min)."""
    qmax = asym_qmax(bits)
    mn = np.asarray(mn, dtype=np.float64)
    d = fl32(np.asarray(mx, dtype=np.float64) - mn)
    d = np.maximum(d, FL32_1EM8)
    s = fl32(d / qmax)
    t = fl32(np.asarray(x, dtype=np.float64) - mn)
    c = np.clip(np.rint(fl32(t / s)), 0, qmax)
    return c.astype(np.int64), s, mn


def dequant_asym(c, s, mn):
    return fl32(fl32(np.asarray(c, dtype=np.float64) * s) + mn)


def quant_fp8(x, scale, fmt: int = FP8_E4M3):
    """FP8 bytes (E4M3 or E5M2) of x/scale (scale 0 gives byte 0)."""
    scale = np.asarray(scale, dtype=np.float64)
    with np.errstate(divide="ignore", invalid="ignore"):
        y = fl32(np.asarray(x, dtype=np.float64) / scale)
    b = fp8_encode(np.where(scale == 0.0, 0.0, y), fmt)
    return np.where(scale == 0.0, 0, b).astype(np.int64)


def dequant_fp8(byte, scale, fmt: int = FP8_E4M3):
    return fl32(fp8_decode(byte, fmt) * np.asarray(scale, dtype=np.float64))


def calibrate_absmax(x, qmax: float) -> float:
    """Static scale of one head: max|x| / qmax in fp32 (0 when all zero)."""
    a = float(np.max(np.abs(np.asarray(x, dtype=np.float64)))) if np.size(x) else 0.0
    return float(fl32(a / float(fl32(qmax))))


# --------------------------------------------------------------------------- configs

@dataclass(frozen=True)
class QSpec:
    fmt: int
    mode: int
    axis: int
    group: int = 0


@dataclass(frozen=True)
class Config:
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    k: QSpec
    v: QSpec
    residual: int
    page_size: int
    rope_pre: int = 0
    rope_theta: float = 10000.0
    src_dtype: int = F32
    meta_dtype: int = F32  # stored scales / minima: F32 or F16

    @property
    def n_rep(self) -> int:
        return self.num_q_heads // self.num_kv_heads


def _tok_group(spec: QSpec, D: int) -> int:
    return spec.group if spec.group else D


def _n_meta(spec: QSpec) -> int:
    return 2 if (spec.mode == ASYM and not is_fp8(spec.fmt)) else 1


def meta_bytes(cfg: Config) -> int:
    """Bytes of one stored scale or minimum."""
    return 2 if cfg.meta_dtype == F16 else 4


def _align16(n: int) -> int:
    return (n + 15) // 16 * 16


def layout(cfg: Config) -> dict:
    """Byte offsets of the sections of one head block and the page size, as the
    library header documents the page layout."""
    D, P = cfg.head_dim, cfg.page_size
    krow = D * bits_of(cfg.k.fmt) // 8
    vrow = D * bits_of(cfg.v.fmt) // 8
    kc = 0
    vc = _align16(kc + P * krow)
    vm = _align16(vc + P * vrow)
    mb = meta_bytes(cfg)
    vm_bytes = P * (D // _tok_group(cfg.v, D)) * _n_meta(cfg.v) * mb if cfg.v.axis == PER_TOKEN else 0
    km = _align16(vm + vm_bytes)
    if cfg.k.axis == PER_CHANNEL:
        km_bytes = max(1, P // cfg.k.group) * D * _n_meta(cfg.k) * mb
    elif cfg.k.axis == PER_TOKEN:
        km_bytes = P * (D // _tok_group(cfg.k, D)) * _n_meta(cfg.k) * mb
    else:
        km_bytes = 0
    head = _align16(km + km_bytes)
    return dict(krow=krow, vrow=vrow, kc=kc, vc=vc, vm=vm, km=km, head=head,
                page=head * cfg.num_kv_heads)


# -------------------------------------------------------------- one (seq, kv-head) stream

def _quant_tokens(x, spec: QSpec, static_scale, D, meta16=False):
    """Quantize rows x [n, D] along a per-token / per-tensor / FP8 axis.

    Returns (codes [n, D], scales [n, ng] or None, mins [n, ng] or None)."""
    bits = bits_of(spec.fmt)
    if is_fp8(spec.fmt):
        return quant_fp8(x, static_scale, spec.fmt), None, None
    if spec.axis == PER_TENSOR:
        # static symmetric scale: the same rounding rule as quant_sym, with s given
        s = np.float64(static_scale)
        with np.errstate(divide="ignore", invalid="ignore"):
            y = fl32(x / s)
        qmax = sym_qmax(bits)
        c = np.where(s == 0.0, 0.0, np.clip(np.rint(y), -qmax, qmax)).astype(np.int64)
        return c, None, None
    g = _tok_group(spec, D)
    n = x.shape[0]
    xg = x.reshape(n, D // g, g)
    if spec.mode == SYM:
        a = np.max(np.abs(xg), axis=2, keepdims=True)
        c, s = (quant_sym16 if meta16 else quant_sym)(xg, a, bits)
        return c.reshape(n, D), s[..., 0], None
    mn = np.min(xg, axis=2, keepdims=True)
    mx = np.max(xg, axis=2, keepdims=True)
    c, s, m = (quant_asym16 if meta16 else quant_asym)(xg, mn, mx, bits)
    return c.reshape(n, D), s[..., 0], m[..., 0]


def _quant_k_channel(x, spec: QSpec, meta16=False):
    """Per-channel K over groups of G consecutive tokens: x [n, D], n % G == 0.

    Returns (codes [n, D], scales [n/G, D], mins [n/G, D] or None)."""
    bits = bits_of(spec.fmt)
    G = spec.group
    n, D = x.shape
    xg = x.reshape(n // G, G, D)
    if spec.mode == SYM:
        a = np.max(np.abs(xg), axis=1, keepdims=True)
        c, s = (quant_sym16 if meta16 else quant_sym)(xg, a, bits)
        return c.reshape(n, D), s[:, 0, :], None
    mn = np.min(xg, axis=1, keepdims=True)
    mx = np.max(xg, axis=1, keepdims=True)
    c, s, m = (quant_asym16 if meta16 else quant_asym)(xg, mn, mx, bits)
    return c.reshape(n, D), s[:, 0, :], m[:, 0, :]


@dataclass
class HeadState:
    """Quantized state of one (sequence, kv-head) stream after T tokens."""
    T: int
    n_q: int
    kc: np.ndarray  # [n_q, D] int64 signed codes (FP8: bytes)
    ks: np.ndarray | None  # PER_CHANNEL [n_q/G, D]; PER_TOKEN [n_q, D/g]
    km: np.ndarray | None
    vc: np.ndarray
    vs: np.ndarray | None
    vm: np.ndarray | None
    k_win: np.ndarray  # [T - n_q, D] source values
    v_win: np.ndarray


def n_quantized(T: int, R: int) -> int:
    return T if R == 0 else R * (T // R)


def quantize_stream(cfg: Config, K, V, k_scale=0.0, v_scale=0.0) -> HeadState:
    """Closed form of the cache state after appending the T rows of K and V
    (fp32-exact source values, [T, D]) to an empty (sequence, kv-head)."""
    K = np.asarray(K, dtype=np.float64)
    V = np.asarray(V, dtype=np.float64)
    T, D = K.shape
    nq = n_quantized(T, cfg.residual)
    m16 = cfg.meta_dtype == F16
    if cfg.k.axis == PER_CHANNEL:
        kc, ks, km = _quant_k_channel(K[:nq], cfg.k, m16)
    else:
        kc, ks, km = _quant_tokens(K[:nq], cfg.k, k_scale, D, m16)
    vc, vs, vm = _quant_tokens(V[:nq], cfg.v, v_scale, D, m16)
    return HeadState(T, nq, kc, ks, km, vc, vs, vm, K[nq:].copy(), V[nq:].copy())


class StreamCache:
    """Token-at-a-time model of one (sequence, kv-head) cache: each token goes
    into the window; when the window holds R tokens they are quantized together
    and the window empties (R = 0: each token is quantized on arrival)."""

    def __init__(self, cfg: Config, k_scale=0.0, v_scale=0.0):
        self.cfg, self.k_scale, self.v_scale = cfg, k_scale, v_scale
        self.blocks = []  # list of HeadState-like tuples per quantized block
        self.win_k, self.win_v = [], []
        self.T = 0

    def append(self, k_rows, v_rows):
        cfg = self.cfg
        for kr, vr in zip(np.asarray(k_rows, np.float64), np.asarray(v_rows, np.float64)):
            self.T += 1
            if cfg.residual == 0:
                self.blocks.append(quantize_stream(cfg, kr[None], vr[None], self.k_scale, self.v_scale))
                continue
            self.win_k.append(kr)
            self.win_v.append(vr)
            if len(self.win_k) == cfg.residual:
                self.blocks.append(quantize_stream(cfg, np.stack(self.win_k), np.stack(self.win_v),
                                                   self.k_scale, self.v_scale))
                self.win_k, self.win_v = [], []

    def state(self) -> HeadState:
        D = self.cfg.head_dim
        cat = lambda xs: (np.concatenate(xs) if xs and xs[0] is not None else None)
        b = self.blocks
        nq = sum(x.n_q for x in b)
        kc = np.concatenate([x.kc for x in b]) if b else np.zeros((0, D), np.int64)
        vc = np.concatenate([x.vc for x in b]) if b else np.zeros((0, D), np.int64)
        kw = np.stack(self.win_k) if self.win_k else np.zeros((0, D))
        vw = np.stack(self.win_v) if self.win_v else np.zeros((0, D))
        return HeadState(self.T, nq, kc, cat([x.ks for x in b]), cat([x.km for x in b]), vc,
                         cat([x.vs for x in b]), cat([x.vm for x in b]), kw, vw)


def _dequant_tokens(c, s, m, spec: QSpec, static_scale, D):
    if is_fp8(spec.fmt):
        return dequant_fp8(c, static_scale, spec.fmt)
    if spec.axis == PER_TENSOR:
        return dequant_sym(c, np.float64(static_scale))
    g = _tok_group(spec, D)
    n = c.shape[0]
    cg = c.reshape(n, D // g, g)
    if spec.mode == SYM:
        return dequant_sym(cg, s[..., None]).reshape(n, D)
    return dequant_asym(cg, s[..., None], m[..., None]).reshape(n, D)


def dequantize_stream(cfg: Config, st: HeadState, k_scale=0.0, v_scale=0.0):
    """Dequantized K, V [T, D] (float64 holding fp32 values); window rows are the
    stored source values.  Keys are as stored (pre-RoPE when rope_pre)."""
    D = cfg.head_dim
    if cfg.k.axis == PER_CHANNEL:
        G = cfg.k.group
        n = st.n_q
        cg = st.kc.reshape(n // G, G, D)
        if cfg.k.mode == SYM:
            kq = dequant_sym(cg, st.ks[:, None, :]).reshape(n, D)
        else:
            kq = dequant_asym(cg, st.ks[:, None, :], st.km[:, None, :]).reshape(n, D)
    else:
        kq = _dequant_tokens(st.kc, st.ks, st.km, cfg.k, k_scale, D)
    vq = _dequant_tokens(st.vc, st.vs, st.vm, cfg.v, v_scale, D)
    return np.concatenate([kq, st.k_win]), np.concatenate([vq, st.v_win])


# -------------------------------------------------------------------- RoPE, attention

def rope_angles(positions, D: int, theta: float):
    """Angle p * theta^(-2i/D) for each position p and pair i (float64)."""
    i = np.arange(D // 2, dtype=np.float64)
    inv = float(theta) ** (-(2.0 * i) / D)
    return np.asarray(positions, dtype=np.float64)[:, None] * inv[None, :]


def rope(x, positions, theta: float):
    """Rotate pairs (2i, 2i+1) of each row of x [n, D] by its position's angle."""
    x = np.asarray(x, dtype=np.float64)
    ang = rope_angles(positions, x.shape[1], theta)
    c, s = np.cos(ang), np.sin(ang)
    out = np.empty_like(x)
    out[:, 0::2] = x[:, 0::2] * c - x[:, 1::2] * s
    out[:, 1::2] = x[:, 0::2] * s + x[:, 1::2] * c
    return out


def attention(q, K, V, scale=None):
    """Single-query attention for each row of q [H, D] over K, V [T, D]:
    softmax(q K^T * scale) V, scale = 1/sqrt(D) by default.  T = 0 gives 0."""
    q = np.asarray(q, dtype=np.float64)
    K = np.asarray(K, dtype=np.float64)
    V = np.asarray(V, dtype=np.float64)
    if scale is None:
        scale = 1.0 / np.sqrt(q.shape[-1])
    if K.shape[0] == 0:
        return np.zeros((q.shape[0], V.shape[1]))
    logits = (q @ K.T) * scale
    m = logits.max(axis=1, keepdims=True)
    p = np.exp(logits - m)
    p /= p.sum(axis=1, keepdims=True)
    return p @ V


def softmax(logits):
    logits = np.asarray(logits, dtype=np.float64)
    m = logits.max(axis=-1, keepdims=True)
    p = np.exp(logits - m)
    return p / p.sum(axis=-1, keepdims=True)


def decode_head(cfg: Config, st: HeadState, q_heads, k_scale=0.0, v_scale=0.0, scale=None):
    """Attention output of the query heads q_heads [n_rep, D] that share this
    kv-head, over its dequantized (and, for pre-RoPE caches, rotated) keys."""
    K, V = dequantize_stream(cfg, st, k_scale, v_scale)
    if cfg.rope_pre:
        K = rope(K, np.arange(K.shape[0]), cfg.rope_theta)
    return attention(q_heads, K, V, scale)


def split_combine(q, K, V, bounds, scale=None):
    """Attention computed as independent chunks [bounds[i], bounds[i+1]) whose
    partial (max, sum, unnormalised output) are merged afterwards."""
    q = np.asarray(q, dtype=np.float64)
    if scale is None:
        scale = 1.0 / np.sqrt(q.shape[-1])
    parts = []
    for a, b in zip(bounds[:-1], bounds[1:]):
        if b <= a:
            continue
        lg = (q @ np.asarray(K[a:b], np.float64).T) * scale
        m = lg.max(axis=1)
        p = np.exp(lg - m[:, None])
        parts.append((m, p.sum(axis=1), p @ np.asarray(V[a:b], np.float64)))
    M = np.max(np.stack([p[0] for p in parts]), axis=0)
    L = sum(np.exp(p[0] - M) * p[1] for p in parts)
    O = sum(np.exp(p[0] - M)[:, None] * p[2] for p in parts)
    return O / L[:, None]


# ------------------------------------------------------------------------ page bytes

def _code_bytes(c, spec: QSpec):
    """Unsigned stored code values from signed codes."""
    bits = bits_of(spec.fmt)
    c = np.asarray(c, dtype=np.int64)
    if is_fp8(spec.fmt) or spec.mode == ASYM:
        return c
    if bits == 8:
        return c & 0xFF
    return c + 2 ** (bits - 1)


def pack_rows(u, bits: int) -> np.ndarray:
    """Pack unsigned codes [n, D] along D: channel c at bit (c*bits) % 8 of
    byte (c*bits)//8."""
    u = np.asarray(u, dtype=np.int64)
    n, D = u.shape
    if bits == 8:
        return u.astype(np.uint8)
    per = 8 // bits
    g = u.reshape(n, D // per, per)
    out = np.zeros((n, D // per), dtype=np.int64)
    for j in range(per):
        out |= g[:, :, j] << (j * bits)
    return out.astype(np.uint8)


def write_head_pages(cfg: Config, pages: np.ndarray, defined: np.ndarray, block_table,
                     b: int, h: int, st: HeadState):
    """Write the quantized part of one (sequence b, kv-head h) state into the
    page bytes `pages` [n_pages, page_bytes] through block_table [B][maxp],
    marking every byte the layout defines in `defined`."""
    L = layout(cfg)
    D, P = cfg.head_dim, cfg.page_size
    kb, vb = bits_of(cfg.k.fmt), bits_of(cfg.v.fmt)
    kpack = pack_rows(_code_bytes(st.kc, cfg.k), kb) if st.n_q else np.zeros((0, L["krow"]), np.uint8)
    vpack = pack_rows(_code_bytes(st.vc, cfg.v), vb) if st.n_q else np.zeros((0, L["vrow"]), np.uint8)
    mb = meta_bytes(cfg)
    f32 = lambda a: np.asarray(a, dtype=np.float16 if mb == 2 else np.float32).view(np.uint8)

    def put(page, off, data):
        base = h * L["head"] + off
        pages[page, base:base + len(data)] = data
        defined[page, base:base + len(data)] = True

    for t in range(st.n_q):
        page = int(block_table[b][t // P])
        slot = t % P
        put(page, L["kc"] + slot * L["krow"], kpack[t])
        put(page, L["vc"] + slot * L["vrow"], vpack[t])
        if cfg.v.axis == PER_TOKEN:
            ng = D // _tok_group(cfg.v, D)
            row = [st.vs[t]] + ([st.vm[t]] if _n_meta(cfg.v) == 2 else [])
            put(page, L["vm"] + slot * ng * _n_meta(cfg.v) * mb, f32(np.concatenate(row)))
        if cfg.k.axis == PER_TOKEN:
            ng = D // _tok_group(cfg.k, D)
            row = [st.ks[t]] + ([st.km[t]] if _n_meta(cfg.k) == 2 else [])
            put(page, L["km"] + slot * ng * _n_meta(cfg.k) * mb, f32(np.concatenate(row)))
    if cfg.k.axis == PER_CHANNEL:
        G = cfg.k.group
        for j in range(st.n_q // G):
            t0 = j * G
            page = int(block_table[b][t0 // P])
            slot = (t0 % P) // G
            row = [st.ks[j]] + ([st.km[j]] if _n_meta(cfg.k) == 2 else [])
            put(page, L["km"] + slot * D * _n_meta(cfg.k) * mb, f32(np.concatenate(row)))


def kv_bytes_per_token(n_layers: int, n_kv_heads: int, head_dim: int, dtype_bytes: float) -> float:
    """KV-cache bytes per token: 2 (K and V) x layers x kv-heads x head_dim x
    bytes per element ("KV Cache Quantization: Why Keys and Values Need
    Different Axes", section "Why is the KV cache the thing that actually runs
    out of memory?")."""
    return 2 * n_layers * n_kv_heads * head_dim * dtype_bytes
