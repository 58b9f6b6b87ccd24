"""kvq_decode_attention_noalloc: decode attention for callers that cannot
allocate device memory (for instance a plugin inside a serving process whose
memory pool already owns the GPU, or a loop that must not call cudaMalloc).
It uses a fixed scratch array inside the library instead of a caller workspace.

Checked through the C ABI against kvq_decode_attention on two calls in a row
(the second with another query, so leftovers of the first call in the shared
array cannot leak into it): within the attention tolerance the other tests use,
and in fact bit for bit, since both entry points run the same kernels with the
same split plan.  Also its size limit.  This file sorts last so that a run stopping at the
first failure has already run every other test.
"""
import ctypes

import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import asymmetric_quantized_kv_gb300 as K  # noqa: E402

TOL = 1e-3  # relative L2 per (sequence, query head), as in the parity tests


def _filled_cache(batch=3, lens=(300, 1, 777)):
    cfg = K.make_config(8, 2, 128, (K.KVQ_INT8, K.KVQ_SYM_ABSMAX, K.KVQ_PER_CHANNEL, 64),
                        (K.KVQ_INT4, K.KVQ_ASYM_MINMAX, K.KVQ_PER_TOKEN, 0), 64, 16, 1, 500000.0, K.KVQ_BF16)
    maxp = max(lens) // 16 + 2
    cache = K.PagedKVCache(cfg, batch, maxp)
    g = torch.Generator(device="cuda")
    g.manual_seed(11)
    n = max(lens)
    k = torch.randn(batch, n, 2, 128, generator=g, device="cuda").to(torch.bfloat16)
    v = torch.randn(batch, n, 2, 128, generator=g, device="cuda").to(torch.bfloat16)
    cache.append(k, v, torch.tensor(lens, dtype=torch.int32, device="cuda"))
    return cfg, cache, g


def _rel(a, b):
    a, b = a.double().cpu().numpy(), b.double().cpu().numpy()
    return float((np.linalg.norm(a - b, axis=-1) / np.linalg.norm(b, axis=-1)).max())


def test_noalloc_matches_workspace_entry_point_on_two_calls():
    cfg, cache, g = _filled_cache()
    for call in range(2):
        q = torch.randn(3, 8, 128, generator=g, device="cuda").to(torch.bfloat16)
        ref = torch.empty(3, 8, 128, dtype=torch.float32, device="cuda")
        K.kvq_decode_attention(cfg, cache.c, q, ref, 0.0, cache.workspace)
        out = torch.full_like(ref, float("nan"))
        K.kvq_decode_attention_noalloc(cfg, cache.c, q, out, 0.0)
        torch.cuda.synchronize()
        assert torch.isfinite(out).all(), call
        assert _rel(out, ref) <= TOL, call
        # same kernels, same split plan, same merge order: the outputs are the same bits
        assert torch.equal(out, ref), call
    assert int(cache.status.item()) == 0


def test_noalloc_rejects_calls_beyond_the_scratch_size():
    cfg = K.make_config(8, 8, 128, (K.KVQ_INT8, K.KVQ_SYM_ABSMAX, K.KVQ_PER_CHANNEL, 64),
                        (K.KVQ_INT4, K.KVQ_ASYM_MINMAX, K.KVQ_PER_TOKEN, 0), 64, 16, 0, 1e4, K.KVQ_BF16)
    batch = 4096
    assert K.kvq_workspace_bytes(cfg, batch, 16) > K.KVQ_NOALLOC_SCRATCH_BYTES
    cache = K.PagedKVCache(cfg, batch, 1)
    q = torch.zeros(batch, 8, 128, dtype=torch.bfloat16, device="cuda")
    out = torch.zeros(batch, 8, 128, dtype=torch.float32, device="cuda")
    code = K.binding.LIB.kvq_decode_attention_noalloc(ctypes.byref(cfg), ctypes.byref(cache.c),
                                                      ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(out.data_ptr()),
                                                      0.0, None)
    assert code == K.KVQ_ERR_CAPACITY
