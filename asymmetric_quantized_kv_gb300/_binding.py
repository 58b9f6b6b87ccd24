"""ctypes binding of libkvq's C ABI (include/kvq.h).

Argument marshalling only: every step of the hot path runs in the CUDA library.
The functions keep the C names; tensors are torch CUDA tensors whose data
pointers are passed through, streams default to torch's current stream.
Importing this module raises when libkvq.so has not been built.
"""
from __future__ import annotations

import ctypes
import os
from ctypes import c_float, c_int32, c_int64, c_size_t, c_void_p

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libkvq.so")

KVQ_OK, KVQ_ERR_INVALID_ARG, KVQ_ERR_UNSUPPORTED, KVQ_ERR_CUDA, KVQ_ERR_CAPACITY, KVQ_ERR_WORKSPACE = range(6)
KVQ_INT2, KVQ_INT4, KVQ_INT8, KVQ_FP8_E4M3, KVQ_FP8_E5M2 = 2, 4, 8, 9, 10
KVQ_SYM_ABSMAX, KVQ_ASYM_MINMAX = 0, 1
KVQ_PER_TENSOR, KVQ_PER_TOKEN, KVQ_PER_CHANNEL = 0, 1, 2
KVQ_F32, KVQ_BF16, KVQ_F16 = 0, 1, 2
KVQ_DEV_BAD_PAGE, KVQ_DEV_OVERFLOW, KVQ_DEV_TIMEOUT, KVQ_DEV_BAD_LENGTH = 1, 2, 4, 8
KVQ_NOALLOC_SCRATCH_BYTES = 32 * 1024 * 1024
KVQ_KERNEL_GENERIC, KVQ_KERNEL_ROPE_I8I4, KVQ_KERNEL_FP8, KVQ_KERNEL_INT2 = 0, 1, 2, 3


class kvq_qspec(ctypes.Structure):
    _fields_ = [("fmt", c_int32), ("mode", c_int32), ("axis", c_int32), ("group", c_int32)]


class kvq_config(ctypes.Structure):
    _fields_ = [("num_q_heads", c_int32), ("num_kv_heads", c_int32), ("head_dim", c_int32),
                ("k", kvq_qspec), ("v", kvq_qspec), ("residual", c_int32), ("page_size", c_int32),
                ("rope_pre", c_int32), ("rope_theta", c_float), ("src_dtype", c_int32),
                ("meta_dtype", c_int32)]


class kvq_cache(ctypes.Structure):
    _fields_ = [("pages", c_void_p), ("block_table", c_void_p), ("seq_lens", c_void_p),
                ("k_win", c_void_p), ("v_win", c_void_p), ("k_scale", c_void_p), ("v_scale", c_void_p),
                ("batch", c_int32), ("max_pages_per_seq", c_int32), ("n_pages", c_int32),
                ("status", c_void_p), ("rope_table", c_void_p), ("rope_positions", c_int32)]


class KvqError(RuntimeError):
    def __init__(self, fn, code):
        super().__init__(f"{fn} failed: {status_string(code)} ({code})")
        self.code = code


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is missing: build it with asymmetric_quantized_kv_gb300.build.build()")
    lib = ctypes.CDLL(LIB_PATH)
    P = ctypes.POINTER
    sig = {
        "kvq_layout_version": (c_int32, []),
        "kvq_rope_table_bytes": (c_size_t, [P(kvq_config), c_int32]),
        "kvq_rope_table_init": (c_int32, [P(kvq_config), c_int32, c_void_p, c_void_p]),
        "kvq_validate": (c_int32, [P(kvq_config)]),
        "kvq_head_block_bytes": (c_size_t, [P(kvq_config)]),
        "kvq_page_bytes": (c_size_t, [P(kvq_config)]),
        "kvq_head_block_offsets": (c_int32, [P(kvq_config), P(c_size_t)]),
        "kvq_workspace_bytes": (c_size_t, [P(kvq_config), c_int32, c_int32]),
        "kvq_calibrate_absmax": (c_int32, [P(kvq_config), c_void_p, c_int64, c_float, c_void_p, c_void_p]),
        "kvq_quantize_append": (c_int32, [P(kvq_config), P(kvq_cache), c_void_p, c_void_p, c_int32,
                                          c_void_p, c_void_p]),
        "kvq_decode_attention": (c_int32, [P(kvq_config), P(kvq_cache), c_void_p, c_void_p, c_float,
                                           c_void_p, c_size_t, c_void_p]),
        "kvq_decode_attention_noalloc": (c_int32, [P(kvq_config), P(kvq_cache), c_void_p, c_void_p, c_float,
                                                   c_void_p]),
        "kvq_dequantize": (c_int32, [P(kvq_config), P(kvq_cache), c_int32, c_int32, c_int32, c_void_p,
                                     c_void_p, c_void_p]),
        "kvq_decode_kernel": (c_int32, [P(kvq_config), P(kvq_cache), P(c_int32)]),
        "kvq_selftest_bounded_wait": (c_int32, [c_void_p, c_void_p]),
        "kvq_status_string": (ctypes.c_char_p, [c_int32]),
    }
    for name, (res, args) in sig.items():
        f = getattr(lib, name)
        f.restype, f.argtypes = res, args
    return lib


LIB = _load()


def status_string(code: int) -> str:
    return LIB.kvq_status_string(int(code)).decode()


def _check(fn, code):
    if code != KVQ_OK:
        raise KvqError(fn, code)


def _ptr(t):
    return None if t is None else c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        import torch
        stream = torch.cuda.current_stream()
    return c_void_p(getattr(stream, "cuda_stream", stream))


def kvq_validate(cfg: kvq_config) -> int:
    return LIB.kvq_validate(ctypes.byref(cfg))


def kvq_page_bytes(cfg: kvq_config) -> int:
    return LIB.kvq_page_bytes(ctypes.byref(cfg))


def kvq_head_block_bytes(cfg: kvq_config) -> int:
    return LIB.kvq_head_block_bytes(ctypes.byref(cfg))


def kvq_head_block_offsets(cfg: kvq_config) -> list[int]:
    out = (c_size_t * 4)()
    _check("kvq_head_block_offsets", LIB.kvq_head_block_offsets(ctypes.byref(cfg), out))
    return list(out)


def kvq_workspace_bytes(cfg: kvq_config, batch: int, max_seq_len: int) -> int:
    return LIB.kvq_workspace_bytes(ctypes.byref(cfg), batch, max_seq_len)


def kvq_rope_table_bytes(cfg: kvq_config, positions: int) -> int:
    return LIB.kvq_rope_table_bytes(ctypes.byref(cfg), int(positions))


def kvq_rope_table_init(cfg, positions, table, stream=None):
    _check("kvq_rope_table_init",
           LIB.kvq_rope_table_init(ctypes.byref(cfg), int(positions), _ptr(table), _stream(stream)))


def kvq_calibrate_absmax(cfg, src, n_tokens, qmax, scale_out, stream=None):
    _check("kvq_calibrate_absmax",
           LIB.kvq_calibrate_absmax(ctypes.byref(cfg), _ptr(src), int(n_tokens), float(qmax), _ptr(scale_out),
                                    _stream(stream)))


def kvq_quantize_append(cfg, cache: kvq_cache, k_new, v_new, n_new, n_new_per_seq=None, stream=None):
    _check("kvq_quantize_append",
           LIB.kvq_quantize_append(ctypes.byref(cfg), ctypes.byref(cache), _ptr(k_new), _ptr(v_new), int(n_new),
                                   _ptr(n_new_per_seq), _stream(stream)))


def kvq_decode_attention(cfg, cache: kvq_cache, q, out, softmax_scale, workspace, stream=None):
    nbytes = workspace.numel() * workspace.element_size()
    _check("kvq_decode_attention",
           LIB.kvq_decode_attention(ctypes.byref(cfg), ctypes.byref(cache), _ptr(q), _ptr(out),
                                    float(softmax_scale), _ptr(workspace), nbytes, _stream(stream)))


def kvq_decode_attention_noalloc(cfg, cache: kvq_cache, q, out, softmax_scale, stream=None):
    """kvq_decode_attention with the library's own fixed scratch array instead of
    a caller workspace, for callers that cannot allocate device memory."""
    _check("kvq_decode_attention_noalloc",
           LIB.kvq_decode_attention_noalloc(ctypes.byref(cfg), ctypes.byref(cache), _ptr(q), _ptr(out),
                                            float(softmax_scale), _stream(stream)))


def kvq_decode_kernel(cfg, cache: kvq_cache) -> int:
    """The decode kernel (KVQ_KERNEL_*) kvq_decode_attention launches for this cache."""
    k = c_int32(-1)
    _check("kvq_decode_kernel", LIB.kvq_decode_kernel(ctypes.byref(cfg), ctypes.byref(cache), ctypes.byref(k)))
    return k.value


def kvq_selftest_bounded_wait(status, stream=None):
    """Run the bounded-wait self-test: `status` (an int32 device tensor) gets
    KVQ_DEV_TIMEOUT when the deliberately unfinished wait gives up."""
    _check("kvq_selftest_bounded_wait", LIB.kvq_selftest_bounded_wait(_ptr(status), _stream(stream)))


def kvq_dequantize(cfg, cache: kvq_cache, seq, tok_begin, tok_end, k_out, v_out, stream=None):
    _check("kvq_dequantize",
           LIB.kvq_dequantize(ctypes.byref(cfg), ctypes.byref(cache), int(seq), int(tok_begin), int(tok_end),
                              _ptr(k_out), _ptr(v_out), _stream(stream)))
