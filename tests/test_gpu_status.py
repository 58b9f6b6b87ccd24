"""Device-side status through every decode kernel: a block-table entry outside
[0, n_pages) is never dereferenced, sets KVQ_DEV_BAD_PAGE in the caller's status
word, and leaves the other sequences' attention exact; with the entry restored
the same cache gives the oracle's attention everywhere again.  (The sequence
that holds the bad entry has no defined output: which of its tokens drop out
depends on the kernel.)"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

from oracle import kvq_oracle as O  # noqa: E402

if not torch.cuda.is_available():  # pragma: no cover
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

from kvq_testlib import ATT_TOL, Case, torch_src  # noqa: E402

Q = O.QSpec
S, A = O.SYM, O.ASYM
TEN, TOK, CH = O.PER_TENSOR, O.PER_TOKEN, O.PER_CHANNEL
BAD_PAGE = 0x1

CASES = {
    # pre-RoPE INT8 keys + INT4 values (the CTA-level tensor-core kernel)
    "rope_i8i4": (O.Config(32, 8, 128, Q(O.INT8, S, CH, 64), Q(O.INT4, A, TOK, 128), 64, 16, 1, 5e5, O.BF16),
                  [700, 2100, 64]),
    # FP8 (the warp-level tensor-core kernel), 16-token pages
    "fp8": (O.Config(16, 2, 128, Q(O.FP8_E4M3, S, TEN), Q(O.FP8_E4M3, S, TEN), 0, 16, 0, 1e4, O.F32), [300, 1000, 17]),
    # 2-bit KIVI (tensor copies of whole page sections)
    "int2": (O.Config(32, 8, 128, Q(O.INT2, A, CH, 32), Q(O.INT2, A, TOK, 32), 128, 16, 0, 1e4, O.BF16),
             [1000, 2200, 129]),
    # the generic kernel
    "generic": (O.Config(4, 4, 64, Q(O.INT4, S, TOK, 32), Q(O.INT8, A, TOK, 16), 32, 32, 1, 1e4, O.F32),
                [99, 400, 33]),
    # the generic kernel with per-channel keys: 32-token key groups over 16-token pages
    # (the tokens of the bad page lose their rows, their group's scales are elsewhere)
    "generic_channel": (O.Config(8, 2, 128, Q(O.INT8, A, CH, 32), Q(O.INT4, A, TOK, 0), 32, 16, 0, 1e4, O.BF16),
                        [99, 400, 33]),
}


@pytest.mark.parametrize("name", sorted(CASES))
def test_bad_block_table_entry(name):
    cfg, lens = CASES[name]
    case = Case(cfg, lens, seed=11)
    q = case.queries(seed=5)
    b_bad = int(np.argmax(lens))
    cache = case.cache
    good = int(cache.block_table[b_bad, 1].item())
    cache.block_table[b_bad, 1] = cache.n_pages + 7
    out = cache.attention(torch_src(q, cfg)).cpu().numpy().astype(np.float64)
    assert int(cache.status.item()) & BAD_PAGE
    for b in range(len(lens)):
        if b == b_bad:
            continue
        for h in range(cfg.num_kv_heads):
            heads = slice(h * cfg.n_rep, (h + 1) * cfg.n_rep)
            ref = O.decode_head(cfg, case.states[b][h], q[b, heads].astype(np.float64), case.k_scale[h],
                                case.v_scale[h])
            err = np.linalg.norm(out[b, heads] - ref, axis=1) / np.linalg.norm(ref, axis=1)
            assert float(err.max()) <= ATT_TOL, (b, h, float(err.max()))
    cache.block_table[b_bad, 1] = good
    cache.status.zero_()
    case.check_attention(q)


def test_bounded_wait_gives_up_and_reports_timeout():
    """A pipeline wait that can never complete (a barrier phase nothing finishes,
    nothing in flight) gives up after the decode kernels' poll limit and reports
    KVQ_DEV_TIMEOUT in the status word; the context stays usable: a decode call
    right after it is exact."""
    import time
    import asymmetric_quantized_kv_gb300 as K
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    t0 = time.perf_counter()
    K.kvq_selftest_bounded_wait(status)
    torch.cuda.synchronize()
    waited = time.perf_counter() - t0
    assert int(status.item()) == K.KVQ_DEV_TIMEOUT
    assert waited < 30.0, waited
    cfg, lens = CASES["int2"]
    c = Case(cfg, lens, seed=4)
    c.check_attention()


@pytest.mark.parametrize("D,fits,too_many", [(128, 41_000, 43_000), (256, 30_000, 32_000)])
def test_generic_kernel_batch_limit(D, fits, too_many):
    """The generic kernel's shared memory grows with the batch (the plan's
    per-sequence prefix): the header gives about 42,000 sequences at head_dim
    128 and 30,000 at 256.  A batch below that runs (every sequence empty: out is
    0); one above returns KVQ_ERR_CAPACITY with nothing launched (out untouched)."""
    import asymmetric_quantized_kv_gb300 as K
    from kvq_testlib import to_c
    cfg = to_c(O.Config(4, 4, D, Q(O.INT8, S, TOK, 0), Q(O.INT8, S, TOK, 0), 0, 16, 0, 1e4, O.F32))
    for batch, ok in ((fits, True), (too_many, False)):
        cache = K.PagedKVCache(cfg, batch, 1, n_pages=1, block_table=torch.zeros(batch, 1, dtype=torch.int32))
        assert cache.decode_kernel() == K.KVQ_KERNEL_GENERIC
        q = torch.randn(batch, 4, D, device="cuda")
        out = torch.full((batch, 4, D), 7.0, device="cuda")
        if ok:
            cache.attention(q, out)
            torch.cuda.synchronize()
            assert float(out.abs().max()) == 0.0
        else:
            with pytest.raises(K.KvqError) as e:
                cache.attention(q, out)
            assert e.value.code == K.KVQ_ERR_CAPACITY
            torch.cuda.synchronize()
            assert bool((out == 7.0).all())
        assert int(cache.status.item()) == 0
        del cache, q, out
        torch.cuda.empty_cache()
