"""CUDA path vs oracle on small cases that span several tiles and ragged tails.

Bit-exact: page bytes (codes and scale/min metadata), window contents, lengths,
static scales and kvq_dequantize.  Attention: relative L2 <= 1e-3 per
(sequence, query head) against the oracle on the same dequantized values.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

from oracle import kvq_oracle as O  # noqa: E402

if not torch.cuda.is_available():  # pragma: no cover
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

from kvq_testlib import Case, to_c, torch_src  # noqa: E402

Q = O.QSpec
A, S = O.ASYM, O.SYM
CH, TOK, TEN = O.PER_CHANNEL, O.PER_TOKEN, O.PER_TENSOR

CASES = {
    # KIVI-style 2-bit (the Llama-3.1-8B layer's formats), contiguous pages
    "int2_kivi": (O.Config(8, 2, 128, Q(O.INT2, A, CH, 32), Q(O.INT2, A, TOK, 32), 128, 256, 0, 1e4, O.BF16),
                  [0, 1, 127, 128, 129, 300, 1000]),
    # the same formats with the 8B layer's heads (32 query / 8 kv) in 16-token pages
    "int2_kivi_p16": (O.Config(32, 8, 128, Q(O.INT2, A, CH, 32), Q(O.INT2, A, TOK, 32), 128, 16, 0, 1e4, O.BF16),
                      [129, 1000, 2200]),
    # 64-token key groups, fp32 sources
    "int2_g64_f32": (O.Config(8, 2, 128, Q(O.INT2, A, CH, 64), Q(O.INT2, A, TOK, 32), 128, 64, 0, 1e4, O.F32),
                     [63, 64, 65, 700]),
    # 32-token tiles of the 2-bit kernel across pages: 64-token key groups in 16-token pages (a group
    # spans two tiles and four pages), 128-token groups in 32-token pages, both metadata types
    "int2_g64_p16": (O.Config(16, 4, 128, Q(O.INT2, A, CH, 64), Q(O.INT2, A, TOK, 32), 128, 16, 0, 1e4, O.BF16),
                     [63, 64, 128, 129, 1100]),
    "m16_int2_g64_p16": (O.Config(16, 4, 128, Q(O.INT2, A, CH, 64), Q(O.INT2, A, TOK, 32), 128, 16, 0, 1e4,
                                  O.BF16, meta_dtype=O.F16), [63, 64, 128, 129, 1100]),
    "int2_g128_p32": (O.Config(8, 2, 128, Q(O.INT2, A, CH, 128), Q(O.INT2, A, TOK, 32), 256, 32, 0, 1e4, O.F32),
                      [255, 256, 257, 900]),
    # INT8 per-channel pre-RoPE keys + INT4 per-token values in 16-token pages
    "int8k_rope_int4v": (O.Config(8, 2, 128, Q(O.INT8, S, CH, 64), Q(O.INT4, A, TOK, 128), 64, 16, 1, 5e5, O.BF16),
                         [1, 63, 64, 65, 700, 2100]),
    # FP8 E4M3 with calibrated per-head scales, 8 query heads per kv-head
    "fp8": (O.Config(16, 2, 128, Q(O.FP8_E4M3, S, TEN), Q(O.FP8_E4M3, S, TEN), 0, 256, 0, 1e4, O.BF16),
            [1, 255, 256, 900]),
    # FP8 in 16-token pages (partial last tiles, permuted pages), fp32 sources
    "fp8_p16_f32": (O.Config(16, 2, 128, Q(O.FP8_E4M3, S, TEN), Q(O.FP8_E4M3, S, TEN), 0, 16, 0, 1e4, O.F32),
                    [1, 15, 16, 17, 300, 1000]),
    # FP8 with the 70B layer's heads: 64 query heads on 8 kv-heads
    "fp8_64q8kv": (O.Config(64, 8, 128, Q(O.FP8_E4M3, S, TEN), Q(O.FP8_E4M3, S, TEN), 0, 256, 0, 1e4, O.BF16),
                   [700, 33]),
    # FP8 E5M2 (2 mantissa bits, saturating at 57344) through the tensor-core kernel
    "fp8_e5m2": (O.Config(16, 2, 128, Q(O.FP8_E5M2, S, TEN), Q(O.FP8_E5M2, S, TEN), 0, 256, 0, 1e4, O.BF16),
                 [1, 255, 256, 900]),
    "fp8_e5m2_p16_f32": (O.Config(16, 2, 128, Q(O.FP8_E5M2, S, TEN), Q(O.FP8_E5M2, S, TEN), 0, 16, 0, 1e4, O.F32),
                         [1, 15, 16, 17, 300, 1000]),
    # E4M3 keys with E5M2 values, 4 query heads per kv-head (the generic kernel)
    "fp8_mixed": (O.Config(8, 2, 128, Q(O.FP8_E4M3, S, TEN), Q(O.FP8_E5M2, S, TEN), 0, 64, 0, 1e4, O.BF16),
                  [5, 64, 333]),
    # per-tensor INT8 (the synthetic head's failing baseline), fp32 sources
    "int8_tensor": (O.Config(1, 1, 128, Q(O.INT8, S, TEN), Q(O.INT8, S, TEN), 0, 256, 0, 1e4, O.F32), [4096]),
    # per-channel K over one 4096-token group + per-token V, fp32
    "int8_channel_4096": (O.Config(1, 1, 128, Q(O.INT8, S, CH, 4096), Q(O.INT8, S, TOK, 0), 4096, 4096, 0, 1e4,
                                   O.F32), [4096]),
    # asymmetric INT4 per-token keys, 64 query heads on one kv-head
    "int4_token_64q": (O.Config(64, 1, 128, Q(O.INT4, A, TOK, 0), Q(O.INT4, A, TOK, 0), 0, 512, 0, 1e4, O.F32),
                       [512]),
    "int4_channel_64q": (O.Config(64, 1, 128, Q(O.INT4, A, CH, 512), Q(O.INT4, A, TOK, 0), 512, 512, 0, 1e4,
                                  O.F32), [512]),
    # the tensor-core kernel's formats: 8 kv-heads x 4 query heads, pre-RoPE INT8 keys, INT4 values
    "fast_rope_i8i4_p16": (O.Config(32, 8, 128, Q(O.INT8, S, CH, 64), Q(O.INT4, A, TOK, 128), 64, 16, 1, 5e5,
                                    O.BF16), [1, 63, 64, 65, 700, 2100, 3000, 777]),
    "fast_rope_i8i4_p64": (O.Config(32, 8, 128, Q(O.INT8, S, CH, 64), Q(O.INT4, A, TOK, 128), 64, 64, 1, 5e5,
                                    O.BF16), [5, 130, 1500]),
    "fast_rope_i8i4_g128": (O.Config(32, 8, 128, Q(O.INT8, S, CH, 128), Q(O.INT4, A, TOK, 0), 128, 16, 1, 1e4,
                                     O.BF16), [128, 129, 1000, 4100]),
    # fp16 scale/min storage: the 8B layer's formats, pre-RoPE INT8 keys + INT4 values,
    # per-channel keys folded through the sub-chunk path (R 512), grouped per-token encodings
    "m16_int2_kivi": (O.Config(8, 2, 128, Q(O.INT2, A, CH, 32), Q(O.INT2, A, TOK, 32), 128, 256, 0, 1e4, O.BF16,
                               meta_dtype=O.F16), [0, 1, 127, 128, 129, 300, 1000]),
    "m16_int2_kivi_p16": (O.Config(32, 8, 128, Q(O.INT2, A, CH, 32), Q(O.INT2, A, TOK, 32), 128, 16, 0, 1e4,
                                   O.BF16, meta_dtype=O.F16), [129, 1000, 2200]),
    "m16_rope_i8i4": (O.Config(8, 2, 128, Q(O.INT8, S, CH, 64), Q(O.INT4, A, TOK, 128), 64, 16, 1, 5e5, O.BF16,
                               meta_dtype=O.F16), [1, 63, 64, 65, 700, 2100]),
    # the pre-RoPE tensor-core kernel's binary16 instance: whole-page and per-section copies
    "m16_fast_rope_p16": (O.Config(32, 8, 128, Q(O.INT8, S, CH, 64), Q(O.INT4, A, TOK, 128), 64, 16, 1, 5e5,
                                   O.BF16, meta_dtype=O.F16), [1, 63, 64, 65, 700, 2100, 3000, 777]),
    "m16_fast_rope_p64": (O.Config(32, 8, 128, Q(O.INT8, S, CH, 64), Q(O.INT4, A, TOK, 128), 64, 64, 1, 5e5,
                                   O.BF16, meta_dtype=O.F16), [5, 130, 1500]),
    "m16_int4_channel_r512": (O.Config(8, 1, 128, Q(O.INT4, A, CH, 512), Q(O.INT4, A, TOK, 0), 512, 512, 0, 1e4,
                                       O.F32, meta_dtype=O.F16), [512, 1100]),
    "m16_d64_grouped": (O.Config(4, 4, 64, Q(O.INT4, S, TOK, 32), Q(O.INT8, A, TOK, 16), 32, 32, 1, 1e4, O.F32,
                                 meta_dtype=O.F16), [5, 33, 64, 99]),
    # other head sizes and mixed encodings
    "d64_int4sym": (O.Config(4, 4, 64, Q(O.INT4, S, TOK, 32), Q(O.INT8, A, TOK, 16), 32, 32, 1, 1e4, O.F32),
                    [5, 33, 64, 99]),
    "d256_int8asym": (O.Config(6, 2, 256, Q(O.INT8, A, CH, 16), Q(O.INT2, S, TOK, 64), 48, 16, 0, 1e4, O.BF16),
                      [47, 48, 49, 400]),
    # the generic kernel's other per-item head counts and encodings: 2 query heads per
    # kv-head with per-tensor INT4/INT2; 8 with 2-bit asymmetric per-token keys, D 64
    "int4_tensor_nrep2": (O.Config(4, 2, 128, Q(O.INT4, S, TEN), Q(O.INT2, S, TEN), 0, 32, 0, 1e4, O.BF16),
                          [1, 31, 32, 33, 250]),
    "int2_token_nrep8_d64": (O.Config(16, 2, 64, Q(O.INT2, A, TOK, 32), Q(O.INT4, A, TOK, 64), 64, 16, 0, 1e4,
                                      O.BF16), [0, 7, 64, 65, 190]),
    # per-token scale/min entries the generic kernel reads from the pages instead of
    # staging them: 128 bytes a token (D 256, 16-channel groups, asymmetric fp32),
    # and 2 bytes a token (one binary16 scale per row)
    "d256_token_g16": (O.Config(4, 2, 256, Q(O.INT4, A, TOK, 16), Q(O.INT8, A, TOK, 16), 32, 32, 0, 1e4, O.F32),
                       [1, 31, 32, 33, 150]),
    "m16_int8_token_row": (O.Config(4, 4, 128, Q(O.INT8, S, TOK, 0), Q(O.INT4, S, TOK, 0), 0, 16, 0, 1e4, O.BF16,
                                    meta_dtype=O.F16), [1, 17, 200]),
    # the generic kernel's remaining (query heads per item, D) instances: 8 heads at D 256,
    # 1 head at D 256, 2 and 4 heads at D 64 (pre-RoPE), and 12 query heads per kv-head
    # (a full block of 8, then a block of 4)
    "nrep8_d256": (O.Config(16, 2, 256, Q(O.INT4, A, CH, 32), Q(O.INT4, A, TOK, 64), 32, 32, 0, 1e4, O.BF16),
                   [1, 40, 300]),
    "nrep1_d256": (O.Config(2, 2, 256, Q(O.INT8, S, TOK, 0), Q(O.INT8, A, TOK, 128), 0, 64, 0, 1e4, O.F32),
                   [5, 200]),
    "nrep2_d64_int2": (O.Config(4, 2, 64, Q(O.INT2, A, CH, 16), Q(O.INT2, A, TOK, 32), 32, 16, 0, 1e4, O.BF16),
                       [3, 77]),
    "nrep4_d64_rope": (O.Config(8, 2, 64, Q(O.INT8, S, CH, 16), Q(O.INT4, S, TOK, 0), 16, 16, 1, 1e4, O.BF16),
                       [17, 150]),
    "nrep12": (O.Config(12, 1, 128, Q(O.INT4, A, CH, 16), Q(O.INT8, S, TOK, 0), 16, 32, 0, 1e4, O.F32), [33, 100]),
}


# The decode kernel each case must run on (kvq_decode_kernel); every other case
# runs on the generic kernel.  A tensor-core kernel that stopped taking its
# format mix (a shape test, or the driver's tensor-map encoder missing) would
# otherwise leave the suite green on the generic kernel.
TC_KERNEL = {
    "int2_kivi": "INT2", "int2_kivi_p16": "INT2", "int2_g64_f32": "INT2", "m16_int2_kivi": "INT2",
    "m16_int2_kivi_p16": "INT2", "int2_g64_p16": "INT2", "m16_int2_g64_p16": "INT2", "int2_g128_p32": "INT2",
    "fp8": "FP8", "fp8_p16_f32": "FP8", "fp8_64q8kv": "FP8", "fp8_e5m2": "FP8", "fp8_e5m2_p16_f32": "FP8",
    "fast_rope_i8i4_p16": "ROPE_I8I4", "fast_rope_i8i4_p64": "ROPE_I8I4", "fast_rope_i8i4_g128": "ROPE_I8I4",
    "m16_fast_rope_p16": "ROPE_I8I4", "m16_fast_rope_p64": "ROPE_I8I4",
}


@pytest.fixture(scope="module", params=sorted(CASES))
def case(request):
    cfg, lens = CASES[request.param]
    c = Case(cfg, lens, seed=sorted(CASES).index(request.param))
    c.name = request.param
    return c


def test_decode_kernel_choice(case):
    import asymmetric_quantized_kv_gb300 as K
    want = getattr(K, "KVQ_KERNEL_" + TC_KERNEL.get(case.name, "GENERIC"))
    assert case.cache.decode_kernel() == want


def test_pages_bit_exact(case):
    case.check_pages()


def test_lengths_window_scales(case):
    case.check_lengths_and_window()
    case.check_scales()


def test_dequantize_bit_exact(case):
    case.check_dequantize()


def test_attention_within_tolerance(case):
    case.check_attention()


def test_attention_custom_scale(case):
    case.check_attention(scale=0.05)


@pytest.mark.parametrize("name", ["fast_rope_i8i4_p16", "m16_fast_rope_p16", "fast_rope_i8i4_g128"])
def test_rope_table_paths(name):
    """The pre-RoPE tensor-core kernel with the cos/sin computed in the kernel
    (no table, and a table too short for the cache, which the kernel then does
    not use) and copied from a table of every position: each within the
    tolerance of the oracle, and the outputs within 5e-5 of each other (the
    kernel's own cos/sin follow a recurrence reseeded every 512 tokens; the
    table's are computed per position)."""
    import asymmetric_quantized_kv_gb300 as K
    cfg, lens = CASES[name]
    outs = []
    for rope_table in (False, 200, True):
        c = Case(cfg, lens, seed=5, rope_table=rope_table)
        assert c.cache.decode_kernel() == K.KVQ_KERNEL_ROPE_I8I4
        c.check_attention()
        q = c.queries()
        outs.append(c.cache.attention(torch_src(q, cfg)).cpu().numpy().astype(np.float64))
    for o in outs[:2]:
        err = np.linalg.norm(o - outs[2], axis=-1) / np.maximum(np.linalg.norm(outs[2], axis=-1), 1e-30)
        assert float(err.max()) <= 5e-5, float(err.max())


@pytest.mark.parametrize("rope_table", [80, 96, True])
def test_rope_table_on_a_full_cache_of_80_positions(rope_table):
    """A cache of 5 pages of 16 tokens (80 positions, not a whole number of the
    kernel's 32-position tables) filled to capacity: a table of exactly 80
    positions is not used (the last table's copy would read past its end), one
    of 96 is, and the cache wrapper rounds its own table up to 96; all within
    tolerance of the oracle."""
    cfg, _ = CASES["fast_rope_i8i4_p16"]
    c = Case(cfg, [80, 33, 64], seed=6, extra_pages=0, rope_table=rope_table)
    assert c.maxp * cfg.page_size == 80
    if rope_table is True:
        assert c.cache.rope_positions == 96
    c.check_attention()


def test_rope_table_values():
    """kvq_rope_table_init against the oracle's rotation angles (float64 cos and
    sin of p * theta^(-2i/D)): every (position, pair) of 70,000 positions to
    2e-6, read through the table's private arrangement (row p holds pairs
    (2u, 2u+1) as (cos, cos, sin, sin) at slot u ^ ((2 (u / 8) + p % 2) % 8))."""
    import asymmetric_quantized_kv_gb300 as K
    for D, theta in ((128, 5e5), (64, 1e4)):
        cfg = to_c(O.Config(8, 2, D, Q(O.INT8, S, CH, 64), Q(O.INT4, A, TOK, 0), 64, 16, 1, theta, O.BF16))
        n = 70000
        table = torch.empty(K.kvq_rope_table_bytes(cfg, n), dtype=torch.uint8, device="cuda")
        K.kvq_rope_table_init(cfg, n, table)
        t = table.view(torch.float32).view(n, D // 4, 4).cpu().numpy().astype(np.float64)
        U = D // 4
        p = np.arange(n)[:, None]
        u = np.arange(U)[None, :]
        slot = u ^ (((2 * (u >> 3)) | (p & 1)) & 7)
        got = np.take_along_axis(t, np.broadcast_to(slot[..., None], (n, U, 4)), axis=1)
        ang = O.rope_angles(np.arange(n), D, theta)  # [n, D/2]
        want = np.stack([np.cos(ang[:, 0::2]), np.cos(ang[:, 1::2]), np.sin(ang[:, 0::2]), np.sin(ang[:, 1::2])], -1)
        assert float(np.abs(got - want).max()) <= 2e-6, (D, float(np.abs(got - want).max()))


@pytest.mark.parametrize("chunking", ["all", "one"])
def test_chunking_invariance(chunking):
    cfg, lens = CASES["int8k_rope_int4v"]
    a = Case(cfg, lens, seed=3, chunking="random")
    b = Case(cfg, lens, seed=3, chunking=chunking)
    pa, pb = a.cache.page_view().cpu().numpy(), b.cache.page_view().cpu().numpy()
    _, defined = a.oracle_pages()
    assert np.array_equal(pa[defined], pb[defined])
    ka, kb = a.cache.k_win.cpu().float().numpy(), b.cache.k_win.cpu().float().numpy()
    for i, T in enumerate(lens):  # only the live window slots [0, T mod R) are defined
        r = T % cfg.residual
        assert np.array_equal(ka[i, :r], kb[i, :r])


def test_empty_cache_outputs_zero():
    cfg, _ = CASES["int2_kivi"]
    c = Case(cfg, [0, 0], seed=1)
    c.check_attention()
