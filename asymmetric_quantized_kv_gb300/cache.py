"""Device-memory plumbing around the C ABI: a paged quantized KV cache whose
buffers are torch CUDA tensors.  Every computation is a libkvq call."""
from __future__ import annotations

import ctypes

import torch

from . import _binding as B


def make_config(num_q_heads, num_kv_heads, head_dim, k, v, residual, page_size, rope_pre=0,
                rope_theta=10000.0, src_dtype=B.KVQ_F32, meta_dtype=B.KVQ_F32) -> B.kvq_config:
    """k, v: (fmt, mode, axis, group) tuples; meta_dtype: stored scales / minima (F32 or F16)."""
    cfg = B.kvq_config(num_q_heads, num_kv_heads, head_dim, B.kvq_qspec(*k), B.kvq_qspec(*v), residual,
                       page_size, rope_pre, rope_theta, src_dtype, meta_dtype)
    code = B.kvq_validate(cfg)
    if code != B.KVQ_OK:
        raise B.KvqError("kvq_validate", code)
    return cfg


def src_torch_dtype(cfg) -> torch.dtype:
    return torch.bfloat16 if cfg.src_dtype == B.KVQ_BF16 else torch.float32


class PagedKVCache:
    """Caller-owned buffers of one cache (pages, block table, lengths, window,
    static scales, status word) and the kvq_cache struct pointing at them."""

    def __init__(self, cfg, batch, max_pages_per_seq, n_pages=None, block_table=None, device="cuda",
                 rope_table=True):
        """rope_table (pre-RoPE keys only): True builds a table for every position the
        pages can hold (rounded up to a multiple of 32, as the kernel reads whole
        32-position tables), False leaves the decode kernel to compute the cos/sin,
        and a (tensor, positions) pair shares a table built by kvq_rope_table_init."""
        self.cfg = cfg
        self.batch = batch
        self.max_pages = max_pages_per_seq
        self.n_pages = n_pages if n_pages is not None else batch * max_pages_per_seq
        self.page_bytes = B.kvq_page_bytes(cfg)
        dev = torch.device(device)
        self.pages = torch.zeros(self.n_pages * self.page_bytes, dtype=torch.uint8, device=dev)
        if block_table is None:
            block_table = torch.arange(batch * max_pages_per_seq, dtype=torch.int32).reshape(batch, -1)
        self.block_table = torch.as_tensor(block_table, dtype=torch.int32).reshape(batch, max_pages_per_seq).to(dev)
        self.seq_lens = torch.zeros(batch, dtype=torch.int32, device=dev)
        R, H, D = cfg.residual, cfg.num_kv_heads, cfg.head_dim
        dt = src_torch_dtype(cfg)
        self.k_win = torch.zeros(batch, max(R, 1), H, D, dtype=dt, device=dev) if R else None
        self.v_win = torch.zeros(batch, max(R, 1), H, D, dtype=dt, device=dev) if R else None
        self.k_scale = torch.zeros(H, dtype=torch.float32, device=dev)
        self.v_scale = torch.zeros(H, dtype=torch.float32, device=dev)
        self.status = torch.zeros(1, dtype=torch.int32, device=dev)
        self.workspace = torch.empty(
            max(B.kvq_workspace_bytes(cfg, batch, max_pages_per_seq * cfg.page_size), 256),
            dtype=torch.uint8, device=dev)
        self.rope_table, self.rope_positions = None, 0
        if cfg.rope_pre and rope_table is not False:
            if rope_table is True:
                n = (max_pages_per_seq * cfg.page_size + 31) // 32 * 32  # whole 32-position tables
                self.rope_table = torch.empty(B.kvq_rope_table_bytes(cfg, n), dtype=torch.uint8, device=dev)
                self.rope_positions = n
                B.kvq_rope_table_init(cfg, n, self.rope_table)
            else:
                self.rope_table, self.rope_positions = rope_table
        p = lambda t: None if t is None else t.data_ptr()
        self.c = B.kvq_cache(p(self.pages), p(self.block_table), p(self.seq_lens), p(self.k_win), p(self.v_win),
                             p(self.k_scale), p(self.v_scale), batch, max_pages_per_seq, self.n_pages,
                             p(self.status), p(self.rope_table), self.rope_positions)

    # --- thin wrappers over the C ABI
    def append(self, k_new, v_new, n_new_per_seq=None, stream=None):
        n = k_new.shape[1]
        B.kvq_quantize_append(self.cfg, self.c, k_new, v_new, n, n_new_per_seq, stream)

    def attention(self, q, out=None, softmax_scale=0.0, stream=None):
        if out is None:
            out = torch.empty(q.shape, dtype=torch.float32, device=q.device)
        B.kvq_decode_attention(self.cfg, self.c, q, out, softmax_scale, self.workspace, stream)
        return out

    def decode_kernel(self) -> int:
        """The decode kernel (KVQ_KERNEL_*) attention() launches for this cache."""
        return B.kvq_decode_kernel(self.cfg, self.c)

    def dequantize(self, seq, tok_begin, tok_end, stream=None):
        n = tok_end - tok_begin
        k = torch.empty(n, self.cfg.num_kv_heads, self.cfg.head_dim, dtype=torch.float32, device=self.pages.device)
        v = torch.empty_like(k)
        B.kvq_dequantize(self.cfg, self.c, seq, tok_begin, tok_end, k, v, stream)
        return k, v

    def calibrate(self, k_src, v_src, k_qmax, v_qmax, stream=None):
        """Set the static per-head scales from [N, Hkv, D] source tensors."""
        B.kvq_calibrate_absmax(self.cfg, k_src, k_src.shape[0], k_qmax, self.k_scale, stream)
        B.kvq_calibrate_absmax(self.cfg, v_src, v_src.shape[0], v_qmax, self.v_scale, stream)

    def page_view(self):
        return self.pages.view(self.n_pages, self.page_bytes)
