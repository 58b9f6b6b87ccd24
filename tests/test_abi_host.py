"""Host-side checks of the C ABI (no GPU needed): the library builds, loads and
exports every function include/kvq.h declares; validation and layout arithmetic
agree with the oracle's independent reading of the documented layout; bad
arguments are rejected before anything is launched."""
import ctypes
import os
import re

import pytest

from oracle import kvq_oracle as O

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def K():
    import __graft_entry__
    __graft_entry__.build()
    import asymmetric_quantized_kv_gb300 as K
    return K


def declared_functions():
    text = open(os.path.join(ROOT, "include", "kvq.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(kvq_[a-z_]+)\s*\(", text)))


def test_every_declared_symbol_is_exported(K):
    names = declared_functions()
    assert len(names) >= 10
    lib = ctypes.CDLL(K.binding.LIB_PATH)
    for n in names:
        assert hasattr(lib, n), n


def test_status_strings(K):
    for code in range(6):
        assert K.status_string(code) not in ("", "unknown status")
    assert K.status_string(99) == "unknown status"


SPECS = [(O.INT2, O.ASYM, O.PER_CHANNEL, 32), (O.INT8, O.SYM, O.PER_CHANNEL, 64), (O.INT4, O.ASYM, O.PER_TOKEN, 0),
         (O.INT4, O.SYM, O.PER_TOKEN, 32), (O.INT8, O.SYM, O.PER_TENSOR, 0), (O.FP8_E4M3, 0, O.PER_TENSOR, 0),
         (O.FP8_E5M2, 0, O.PER_TENSOR, 0)]


@pytest.mark.parametrize("D", [64, 128, 256])
@pytest.mark.parametrize("P", [16, 64, 256])
@pytest.mark.parametrize("meta", [O.F32, O.F16])
def test_layout_agrees_with_oracle(K, D, P, meta):
    for ks in SPECS:
        for vs in SPECS:
            if vs[2] == O.PER_CHANNEL:
                continue
            R = 64 if ks[2] == O.PER_CHANNEL else 0
            if ks[2] == O.PER_CHANNEL and (P % ks[3] and ks[3] % P):
                continue
            cfg = O.Config(8, 2, D, O.QSpec(*ks), O.QSpec(*vs), R, P, meta_dtype=meta)
            c = K.kvq_config(8, 2, D, K.kvq_qspec(*ks), K.kvq_qspec(*vs), R, P, 0, 1e4, 0, meta)
            assert K.kvq_validate(c) == 0
            L = O.layout(cfg)
            assert K.kvq_page_bytes(c) == L["page"]
            assert K.kvq_head_block_bytes(c) == L["head"]
            assert K.kvq_head_block_offsets(c) == [L["kc"], L["vc"], L["vm"], L["km"]]


def _cfg(K, **kw):
    base = dict(num_q_heads=32, num_kv_heads=8, head_dim=128, k=K.kvq_qspec(8, 0, 2, 64),
                v=K.kvq_qspec(4, 1, 1, 0), residual=64, page_size=16, rope_pre=1, rope_theta=5e5, src_dtype=1)
    base.update(kw)
    return K.kvq_config(**base)


def test_validation_rejects_bad_configs(K):
    E, U = K.KVQ_ERR_INVALID_ARG, K.KVQ_ERR_UNSUPPORTED
    assert K.kvq_validate(_cfg(K)) == 0
    assert K.kvq_validate(_cfg(K, num_q_heads=30)) == E
    assert K.kvq_validate(_cfg(K, head_dim=96)) == U
    assert K.kvq_validate(_cfg(K, residual=60)) == E            # R % G != 0
    assert K.kvq_validate(_cfg(K, meta_dtype=1)) == E           # scales/minima: F32 or F16 only
    assert K.kvq_validate(_cfg(K, meta_dtype=2)) == 0
    assert K.kvq_validate(_cfg(K, residual=0)) == E             # per-channel keys need a window
    assert K.kvq_validate(_cfg(K, page_size=24)) == E
    assert K.kvq_validate(_cfg(K, k=K.kvq_qspec(3, 0, 2, 64))) == E
    assert K.kvq_validate(_cfg(K, k=K.kvq_qspec(8, 0, 2, 40))) == E
    assert K.kvq_validate(_cfg(K, v=K.kvq_qspec(4, 1, 2, 64))) == U   # per-channel values
    assert K.kvq_validate(_cfg(K, v=K.kvq_qspec(9, 0, 1, 0))) == U    # FP8 is per-tensor only
    assert K.kvq_validate(_cfg(K, v=K.kvq_qspec(4, 1, 0, 0))) == U    # asym per-tensor
    assert K.kvq_validate(_cfg(K, v=K.kvq_qspec(4, 1, 1, 48))) == E   # group must divide D
    assert K.kvq_validate(_cfg(K, rope_theta=0.0)) == E
    assert K.kvq_validate(_cfg(K, src_dtype=3)) == E
    assert K.kvq_page_bytes(_cfg(K, head_dim=96)) == 0
    assert K.kvq_workspace_bytes(_cfg(K), 0, 100) == 0


def test_entry_points_reject_bad_arguments_before_launch(K):
    c = _cfg(K)
    L = K.binding.LIB
    cache = K.kvq_cache(None, None, None, None, None, None, None, 1, 1, 1, None)
    by = ctypes.byref
    assert L.kvq_quantize_append(by(c), by(cache), None, None, 1, None, None) == K.KVQ_ERR_INVALID_ARG
    assert L.kvq_decode_attention(by(c), by(cache), None, None, 0.0, None, 0, None) == K.KVQ_ERR_INVALID_ARG
    assert L.kvq_dequantize(by(c), by(cache), 0, 0, 1, None, None, None) == K.KVQ_ERR_INVALID_ARG
    # a plausible-looking cache (fake, never dereferenced): the checks still fire first
    fake = K.kvq_cache(4096, 4096, 4096, 4096, 4096, 4096, 4096, 2, 4, 8, 4096)
    assert L.kvq_quantize_append(by(c), by(fake), None, None, 5, None, None) == K.KVQ_ERR_INVALID_ARG
    assert L.kvq_quantize_append(by(c), by(fake), 4096, 4096, -1, None, None) == K.KVQ_ERR_INVALID_ARG
    assert L.kvq_quantize_append(by(c), by(fake), 4096, 4096, 10 ** 6, None, None) == K.KVQ_ERR_CAPACITY
    assert L.kvq_decode_attention(by(c), by(fake), 4096, 4096, 0.0, 4096, 10, None) == K.KVQ_ERR_WORKSPACE
    assert L.kvq_decode_attention(by(c), by(fake), 4096, 4096, 0.0, 4097, 1 << 30, None) == K.KVQ_ERR_WORKSPACE
    assert L.kvq_decode_attention(by(c), by(fake), 4096, 4096, -1.0, 4096, 1 << 30, None) == K.KVQ_ERR_INVALID_ARG
    assert L.kvq_dequantize(by(c), by(fake), 2, 0, 1, 4096, 4096, None) == K.KVQ_ERR_INVALID_ARG
    assert L.kvq_dequantize(by(c), by(fake), 0, 5, 1, 4096, 4096, None) == K.KVQ_ERR_INVALID_ARG
    assert L.kvq_dequantize(by(c), by(fake), 0, 0, 65, 4096, 4096, None) == K.KVQ_ERR_CAPACITY
    assert L.kvq_dequantize(by(c), by(fake), 0, 3, 3, None, None, None) == K.KVQ_OK  # empty range: no launch
    assert L.kvq_calibrate_absmax(by(c), None, 10, 448.0, None, None) == K.KVQ_ERR_INVALID_ARG
    assert L.kvq_calibrate_absmax(by(c), 4096, 10, 0.0, 4096, None) == K.KVQ_ERR_INVALID_ARG


def test_decode_kernel_query_on_the_host(K):
    """kvq_decode_kernel answers from the configuration and the cache struct
    alone (the pointers are never dereferenced): the pre-RoPE INT8/INT4 mix with
    8 kv-heads x 4 query heads goes to its tensor-core kernel, the same mix with
    2 kv-heads to the generic kernel; bad arguments give the decode call's errors."""
    L = K.binding.LIB
    by = ctypes.byref
    spec_k = (O.INT8, O.SYM, O.PER_CHANNEL, 64)
    spec_v = (O.INT4, O.ASYM, O.PER_TOKEN, 0)
    fast = K.make_config(32, 8, 128, spec_k, spec_v, 64, 16, 1, 5e5, K.KVQ_BF16)
    small = K.make_config(8, 2, 128, spec_k, spec_v, 64, 16, 1, 5e5, K.KVQ_BF16)
    fake = K.kvq_cache(4096, 4096, 4096, 4096, 4096, 4096, 4096, 2, 4, 8, 4096)
    out = ctypes.c_int32(-1)
    assert L.kvq_decode_kernel(by(fast), by(fake), by(out)) == K.KVQ_OK and out.value == K.KVQ_KERNEL_ROPE_I8I4
    assert L.kvq_decode_kernel(by(small), by(fake), by(out)) == K.KVQ_OK and out.value == K.KVQ_KERNEL_GENERIC
    assert L.kvq_decode_kernel(by(fast), by(fake), None) == K.KVQ_ERR_INVALID_ARG
    empty = K.kvq_cache(None, None, None, None, None, None, None, 1, 1, 1, None)
    assert L.kvq_decode_kernel(by(fast), by(empty), by(out)) == K.KVQ_ERR_INVALID_ARG


def test_no_process_wide_unique_symbols(K):
    """The library's per-device launch settings live in tables with internal
    linkage.  A GNU unique symbol (what a function-local static of an ordinary
    inline function becomes) would be shared by every copy of the library loaded
    into one process, and a second build would then skip kernel attributes that
    only its own kernels carry."""
    import shutil
    import subprocess
    nm = shutil.which("nm")
    if nm is None:
        pytest.skip("nm not available")
    out = subprocess.run([nm, "-D", K.binding.LIB_PATH], capture_output=True, text=True, check=True).stdout
    unique = [line for line in out.splitlines() if " u " in line]
    assert not unique, unique[:5]


def test_decode_kernel_batch_limit_on_the_host(K):
    """The tensor-core kernels keep the plan's per-sequence prefix in shared
    memory and take at most 4096 sequences; a larger batch runs on the generic
    kernel (the pre-RoPE kernel's shape test needs no device, so the host can
    check both sides of the limit)."""
    L = K.binding.LIB
    by = ctypes.byref
    cfg = K.make_config(32, 8, 128, (O.INT8, O.SYM, O.PER_CHANNEL, 64), (O.INT4, O.ASYM, O.PER_TOKEN, 0), 64, 16,
                        1, 5e5, K.KVQ_BF16)
    out = ctypes.c_int32(-1)
    for batch, want in ((4096, K.KVQ_KERNEL_ROPE_I8I4), (4097, K.KVQ_KERNEL_GENERIC)):
        fake = K.kvq_cache(4096, 4096, 4096, 4096, 4096, 4096, 4096, batch, 4, 8 * batch, 4096)
        assert L.kvq_decode_kernel(by(cfg), by(fake), by(out)) == K.KVQ_OK
        assert out.value == want, (batch, out.value)


def test_rope_table_arguments_on_the_host(K):
    """kvq_rope_table_bytes / kvq_rope_table_init argument checks, and the cache
    struct's optional table (checked before anything is launched: a misaligned
    table, a table on a config without pre-RoPE keys, or no positions)."""
    L = K.binding.LIB
    by = ctypes.byref
    rope = _cfg(K)
    plain = _cfg(K, rope_pre=0)
    assert K.kvq_rope_table_bytes(rope, 100) == 100 * 128 * 4
    assert K.kvq_rope_table_bytes(_cfg(K, head_dim=64, k=K.kvq_qspec(8, 0, 2, 64)), 3) == 3 * 64 * 4
    assert K.kvq_rope_table_bytes(rope, 0) == 0
    assert K.kvq_rope_table_bytes(plain, 100) == 0
    assert L.kvq_rope_table_init(by(rope), 100, None, None) == K.KVQ_ERR_INVALID_ARG
    assert L.kvq_rope_table_init(by(rope), 100, 4100, None) == K.KVQ_ERR_INVALID_ARG   # not 16-byte aligned
    assert L.kvq_rope_table_init(by(rope), 0, 4096, None) == K.KVQ_ERR_INVALID_ARG
    assert L.kvq_rope_table_init(by(plain), 100, 4096, None) == K.KVQ_ERR_INVALID_ARG
    assert L.kvq_rope_table_init(by(rope), (1 << 24) + 1, 4096, None) == K.KVQ_ERR_CAPACITY
    out = ctypes.c_int32(-1)
    ok = K.kvq_cache(4096, 4096, 4096, 4096, 4096, 4096, 4096, 2, 4, 8, 4096, 8192, 64)
    assert L.kvq_decode_kernel(by(rope), by(ok), by(out)) == K.KVQ_OK and out.value == K.KVQ_KERNEL_ROPE_I8I4
    for table, n, cfg in ((8200, 64, rope), (8192, 0, rope), (8192, 64, plain)):
        bad = K.kvq_cache(4096, 4096, 4096, 4096, 4096, 4096, 4096, 2, 4, 8, 4096, table, n)
        assert L.kvq_decode_kernel(by(cfg), by(bad), by(out)) == K.KVQ_ERR_INVALID_ARG, (table, n)
        assert L.kvq_decode_attention(by(cfg), by(bad), 4096, 4096, 0.0, 4096, 1 << 30, None) == \
            K.KVQ_ERR_INVALID_ARG
    # no table: rope_positions is ignored
    none = K.kvq_cache(4096, 4096, 4096, 4096, 4096, 4096, 4096, 2, 4, 8, 4096, None, -5)
    assert L.kvq_decode_kernel(by(rope), by(none), by(out)) == K.KVQ_OK
