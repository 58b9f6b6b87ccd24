"""Seeded random format mixes through the whole CUDA path against the oracle.

Each draw picks key and value formats (INT2/4/8 symmetric or asymmetric, FP8
E4M3/E5M2), axes and group sizes, head_dim, the GQA ratio, the window, the page
size, pre-RoPE keys, the source and metadata dtypes and a few ragged sequence
lengths; draws the library rejects (kvq_validate) are drawn again.  Every case
checks the page bytes bit for bit, the dequantized cache bit for bit and the
attention within the parity tolerance, on whichever decode kernel the call
takes.  The draws are fixed by the seed, so a failure names a reproducible
configuration.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

from oracle import kvq_oracle as O  # noqa: E402

if not torch.cuda.is_available():  # pragma: no cover
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

from kvq_testlib import Case, to_c  # noqa: E402

N_DRAWS = 64
INTS = (O.INT2, O.INT4, O.INT8)
FP8S = (O.FP8_E4M3, O.FP8_E5M2)


def _spec(rng, D, is_key):
    if rng.random() < 0.2:
        return O.QSpec(FP8S[rng.integers(2)], O.SYM, O.PER_TENSOR, 0)
    fmt = INTS[rng.integers(3)]
    axes = [O.PER_TENSOR, O.PER_TOKEN] + ([O.PER_CHANNEL] * 2 if is_key else [])
    axis = axes[rng.integers(len(axes))]
    if axis == O.PER_TENSOR:
        return O.QSpec(fmt, O.SYM, axis, 0)
    mode = (O.SYM, O.ASYM)[rng.integers(2)]
    if axis == O.PER_CHANNEL:
        return O.QSpec(fmt, mode, axis, int((16, 32, 64)[rng.integers(3)]))
    groups = [g for g in (0, 16, 32, 64) if g == 0 or D % g == 0]
    return O.QSpec(fmt, mode, axis, int(groups[rng.integers(len(groups))]))


def _draw(rng):
    import asymmetric_quantized_kv_gb300 as K
    while True:
        D = int((64, 128, 256)[rng.integers(3)])
        hkv = int((1, 2, 4)[rng.integers(3)])
        n_rep = int((1, 2, 3, 4, 8, 12)[rng.integers(6)])
        k, v = _spec(rng, D, True), _spec(rng, D, False)
        if k.axis == O.PER_CHANNEL:
            R = k.group * int(rng.integers(1, 3))
        else:
            R = int((0, 16, 32, 64)[rng.integers(4)])
        P = int((16, 32, 64, 128, 256)[rng.integers(5)])
        rope = int(rng.random() < 0.3)
        src = (O.F32, O.BF16)[rng.integers(2)]
        meta = (O.F32, O.F16)[rng.integers(2)]
        cfg = O.Config(hkv * n_rep, hkv, D, k, v, R, P, rope, float((1e4, 5e5)[rng.integers(2)]), src,
                       meta_dtype=meta)
        if K.kvq_validate(to_c(cfg)) != K.KVQ_OK:
            continue
        lens = [int(x) for x in rng.integers(0, 261, size=int(rng.integers(1, 4)))]
        return cfg, lens


def _draws():
    rng = np.random.default_rng(20261203)
    return [_draw(rng) for _ in range(N_DRAWS)]


@pytest.mark.parametrize("i", range(N_DRAWS))
def test_random_format_mix(i):
    cfg, lens = _draws()[i]
    c = Case(cfg, lens, seed=100 + i)
    c.check_pages()
    c.check_dequantize()
    c.check_attention()
