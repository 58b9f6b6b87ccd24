"""The library's calls inside a CUDA graph: decode attention captured with
torch.cuda.graph and replayed gives the eager call's output bit for bit, for
every decode kernel; an append captured in the same graph advances the cache on
every replay exactly as eager appends do (the benchmark's end-to-end loop relies
on both)."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

from oracle import kvq_oracle as O  # noqa: E402
from kvq_testlib import Case, torch_src  # noqa: E402
from test_gpu_parity import CASES  # noqa: E402


@pytest.mark.parametrize("name", ["fast_rope_i8i4_p16", "fp8", "int2_kivi_p16", "int8k_rope_int4v"])
def test_decode_in_a_cuda_graph_is_bit_identical(name):
    import asymmetric_quantized_kv_gb300 as K
    cfg, lens = CASES[name]
    c = Case(cfg, lens, seed=3)
    q = torch_src(c.queries(), cfg)
    eager = c.cache.attention(q)
    out = torch.zeros_like(eager)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        K.kvq_decode_attention(c.cache.cfg, c.cache.c, q, out, 0.0, c.cache.workspace, s)
    torch.cuda.synchronize()
    for _ in range(2):
        out.zero_()
        graph.replay()
        torch.cuda.synchronize()
        assert torch.equal(out, eager), name
    assert int(c.cache.status.item()) == 0


def test_append_and_decode_replayed_in_a_graph_match_eager_steps():
    """Two identical caches: one advanced by three eager (append, decode) steps,
    the other by three replays of the same two calls captured in a graph; every
    step's output and the final lengths agree bit for bit."""
    import asymmetric_quantized_kv_gb300 as K
    cfg, lens = CASES["fast_rope_i8i4_p16"]
    a = Case(cfg, lens, seed=4, extra_pages=2)
    b = Case(cfg, lens, seed=4, extra_pages=2)
    Bn, H, D = len(lens), cfg.num_kv_heads, cfg.head_dim
    g = torch.Generator(device="cuda").manual_seed(9)
    steps = [(torch.randn(Bn, 1, H, D, generator=g, device="cuda").to(torch.bfloat16),
              torch.randn(Bn, 1, H, D, generator=g, device="cuda").to(torch.bfloat16),
              torch.randn(Bn, cfg.num_q_heads, D, generator=g, device="cuda").to(torch.bfloat16)) for _ in range(3)]
    want = []
    for k, v, q in steps:
        a.cache.append(k, v)
        want.append(a.cache.attention(q).clone())
    kb, vb, qb = (torch.empty_like(x) for x in steps[0])
    out = torch.zeros_like(want[0])
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        K.kvq_quantize_append(b.cache.cfg, b.cache.c, kb, vb, 1, None, s)
        K.kvq_decode_attention(b.cache.cfg, b.cache.c, qb, out, 0.0, b.cache.workspace, s)
    torch.cuda.synchronize()
    for (k, v, q), w in zip(steps, want):
        kb.copy_(k); vb.copy_(v); qb.copy_(q)
        graph.replay()
        torch.cuda.synchronize()
        assert torch.equal(out, w)
    assert torch.equal(a.cache.seq_lens, b.cache.seq_lens)
    assert torch.equal(a.cache.pages, b.cache.pages)
    assert int(b.cache.status.item()) == 0
