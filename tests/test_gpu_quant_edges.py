"""Quantize-append edge cases on the GPU, bit-exact against the oracle.

The append kernels compute x / scale as x * (1 / scale) and fall back to the
exact IEEE division only when the product is within 2^-16 of a rounding half
point.  These streams put quotients exactly on ties (power-of-two scales,
values at k + 1/2: round half to even must decide) and within 2^-20 of them,
plus constant and all-zero groups, for every integer format and both modes.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

from oracle import kvq_oracle as O  # noqa: E402

if not torch.cuda.is_available():  # pragma: no cover
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

from kvq_testlib import Case  # noqa: E402


def tie_stream(rng, T, D, bits, mode, axis_tokens, near):
    """Values whose quotient by the group scale is k + 1/2 (times 1 +- 2^-20 when near)."""
    qmax = 2 ** (bits - 1) - 1 if mode == O.SYM else 2 ** bits - 1
    e = rng.integers(-3, 4)
    s = 2.0 ** int(e)
    if mode == O.SYM:
        k = rng.integers(-qmax, qmax, size=(T, D)).astype(np.float64) + 0.5
    else:
        k = rng.integers(0, qmax, size=(T, D)).astype(np.float64) + 0.5
    if near:
        k = k * (1.0 + rng.choice([-1.0, 1.0], size=(T, D)) * 2.0 ** -20)
    x = k * s
    # pin each group's range so that the scale is exactly s
    if axis_tokens:  # groups along channels of a token: set channel 0 / 1 extremes
        x[:, 0] = qmax * s if mode == O.SYM else 0.0
        if mode == O.ASYM:
            x[:, 1] = qmax * s
    else:  # per-channel groups along tokens
        x[0, :] = qmax * s if mode == O.SYM else 0.0
        if mode == O.ASYM:
            x[1, :] = qmax * s
    x[:, 5] = 0.0 if mode == O.SYM else x[:, 5]  # a zero channel
    return O.fl32(x).astype(np.float32)


@pytest.mark.parametrize("bits", [2, 4, 8])
@pytest.mark.parametrize("mode", [O.SYM, O.ASYM])
@pytest.mark.parametrize("near", [False, True])
def test_ties_and_near_ties_bit_exact(bits, mode, near):
    rng = np.random.default_rng(bits * 10 + mode * 3 + near)
    D, G, R = 64, 16, 32
    cfg = O.Config(2, 1, D, O.QSpec(bits, mode, O.PER_CHANNEL, G), O.QSpec(bits, mode, O.PER_TOKEN, 16),
                   residual=R, page_size=16, src_dtype=O.F32)
    lens = [96, 64]
    Ks, Vs = [], []
    for T in lens:
        K = np.concatenate([tie_stream(rng, G, D, bits, mode, False, near) for _ in range(T // G)])
        V = tie_stream(rng, T, D, bits, mode, True, near)
        Ks.append([K])
        Vs.append([V])
    c = Case(cfg, lens, seed=1, streams=(Ks, Vs))
    c.check_pages()
    c.check_dequantize()


def test_constant_and_zero_groups_bit_exact():
    D, G = 64, 16
    cfg = O.Config(2, 1, D, O.QSpec(O.INT4, O.ASYM, O.PER_CHANNEL, G), O.QSpec(O.INT8, O.SYM, O.PER_TOKEN, 0),
                   residual=32, page_size=16, src_dtype=O.F32)
    K = np.full((64, D), 3.25, np.float32)
    K[16:32] = 0.0
    V = np.zeros((64, D), np.float32)
    V[:8] = -1.5
    c = Case(cfg, [64], seed=2, streams=([[K]], [[V]]))
    c.check_pages()
    c.check_dequantize()
