"""The benchmark's byte accounting (host logic, no GPU): the algorithmic bytes
of one decode call for each workload, against closed forms written out from the
formats (codes at b bits per element, fp32 or binary16 scale/min entries,
bf16/fp32 window rows, q in and fp32 out)."""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
import kvq_inputs as W  # noqa: E402


def _call_bytes(cid, **kw):
    spec = bench.workload_spec(cid, **kw)
    return bench.attention_bytes(spec, [int(T) for T in W.lengths(spec["w"])])


def test_single_head_int8_workloads():
    codes = 4096 * 128 * 2                  # INT8 K and V
    qo = 128 * (4 + 4)                      # fp32 q in, fp32 out
    # one 4096-token key group: 128 scales; values: one scale per token
    assert _call_bytes(1) == codes + 128 * 4 + 4096 * 4 + qo
    assert _call_bytes(1, k_axis="tensor") == codes + qo  # static scales are not per-call bytes


def test_64_query_int4_workloads():
    codes = 512 * 128 // 2 * 2              # INT4 K and V
    qo = 64 * 128 * (4 + 4)
    vmeta = 512 * 2 * 4                     # asym: scale + min per token
    assert _call_bytes(2) == codes + 128 * 2 * 4 + vmeta + qo       # one 512-token key group
    assert _call_bytes(2, k_axis="token") == codes + 512 * 2 * 4 + vmeta + qo


@pytest.mark.parametrize("meta,per_token", [("f32", 64 + 32 + 32), ("f16", 64 + 16 + 16)])
def test_2bit_8b_layer(meta, per_token):
    nq = 16 * 8 * 32768
    window = 16 * 8 * 127 * 128 * 2 * 2     # bf16 K and V rows
    qo = 16 * 32 * 128 * (2 + 4)
    assert _call_bytes(3, meta=meta) == nq * per_token + window + qo


@pytest.mark.parametrize("fp8", ["e4m3", "e5m2"])
def test_fp8_70b_layer(fp8):
    assert _call_bytes(4, fp8=fp8) == 8 * 8 * 131072 * 128 * 2 + 8 * 64 * 128 * (2 + 4)


def test_paged_ragged_layer():
    lens = [int(T) for T in W.lengths(W.WORKLOADS[5])]
    total = 0
    for T in lens:
        nq = 64 * (T // 64)
        # INT8 K + INT4 V codes, one fp32 scale per (64-token group, channel), V scale + min per token
        total += 8 * (nq * (128 + 64) + (nq // 64) * 128 * 4 + nq * 2 * 4 + (T - nq) * 128 * 2 * 2)
    assert _call_bytes(5) == total + 64 * 32 * 128 * (2 + 4)


def test_key_axis_is_only_for_the_single_head_workloads():
    with pytest.raises(SystemExit):
        bench.workload_spec(1, k_axis="token")
    with pytest.raises(SystemExit):
        bench.workload_spec(2, k_axis="tensor")


def test_append_bytes_window_write_and_fold():
    # paged layer: 8 kv-heads x 128 channels, bf16 sources, 64-token window.
    # A sequence at 10 tokens reads the new K/V row and writes it to the window; one
    # at 63 fills the window with it, reads the 63 older rows back and writes 64
    # tokens' codes (INT8 K, INT4 V, V scale+min per token) and the group's key scales.
    spec = bench.workload_spec(5)
    row = 2 * 8 * 128 * 2                        # one token's K and V rows, all heads
    plain = row + row
    fold = row + 63 * row + 8 * 64 * (128 + 64 + 8) + 8 * 128 * 4
    assert bench.append_bytes(spec, [10]) == plain
    assert bench.append_bytes(spec, [63]) == fold
    assert bench.append_bytes(spec, [63, 10]) == fold + plain


def test_paged_layer_inputs():
    lens = W.lengths(W.WORKLOADS[5])
    assert len(lens) == 64 and int(lens.sum()) == 1051067
    assert lens.min() >= 1024 and lens.max() < 65536
    perm = W.page_permutation(4099, 5)
    assert sorted(perm.tolist()) == list(range(4099))
