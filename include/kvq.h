/*
 * kvq.h — C ABI of libkvq: single-query (decode) attention over an
 * asymmetrically quantized KV cache, for one NVIDIA GB300 (sm_103a).
 *
 * What is computed (sources are the web pages this library restates):
 *   - Attention: logits = q.k_j / sqrt(d) -> softmax -> out = sum_j p_j v_j
 *     ("FP8 KV Cache Quantization: Why Keys Break Before Values", section
 *     "Why does the K cache break before the V cache?", attention formula;
 *     "Why Keys Are More Sensitive Than Values in INT8 KV Cache Quantization",
 *     section "Computational Paths for Key and Value", Score/Output equations).
 *   - Symmetric absmax quantization s = amax|x| / qmax, c = clamp(round(x/s)),
 *     x^ = c*s (first page, same section, `qint8` listing; qmax = 7 for INT4
 *     from "KV Cache Quantization: Why Keys and Values Need Different Axes",
 *     section "Why does per-token key quantization destroy accuracy?").
 *   - Asymmetric min-max quantization qmax = 2^b-1, s = max(mx-mn, 1e-8)/qmax,
 *     c = clamp(round((x-mn)/s), 0, qmax), x^ = c*s + mn (fourth page, same
 *     section, `quant_dequant` listing).
 *   - K quantized per channel over fixed token groups, V per token, a
 *     full-precision residual window of the newest tokens folded into the
 *     quantized cache in blocks (first page, section "Should you quantize keys
 *     pre-RoPE or post-RoPE?"; fourth page, section "What should I actually
 *     turn on in production?", checklist).
 *   - Pre-RoPE keys, rotated after dequantization: pairs (2i, 2i+1) rotated
 *     by an angle that depends on the absolute position (fourth page, section
 *     "Where does RoPE break this?").
 *   - FP8 E4M3 with calibrated per-head k_scale / v_scale, saturating at
 *     +-448, and FP8 E5M2, saturating at +-57344 with 2 mantissa bits (first
 *     page, section "Why do per-tensor scales waste bits on the K cache?").
 *     A cache without calibrated scales holds 1.0 in k_scale / v_scale (the
 *     unit scale of that section's first failure mode): raw magnitudes are
 *     then clipped at the format's maximum.
 *
 * Conventions for every entry point
 *   - All tensor pointers are DEVICE pointers unless stated otherwise; the
 *     caller owns every buffer.  The library never allocates, frees or
 *     synchronises; it only enqueues kernels on `stream` (a cudaStream_t
 *     passed as void*, NULL = legacy default stream).
 *   - Host-side argument checks return a kvq_status synchronously and launch
 *     nothing.  A launch failure returns KVQ_ERR_CUDA (cudaGetLastError).
 *   - Problems only visible on the device (a block-table entry outside
 *     [0, n_pages), a sequence that would outgrow its pages, a pipeline wait
 *     that timed out) set bits in the caller's `*status` word with atomicOr
 *     and skip the affected work; kernels never trap and never spin without
 *     an iteration limit.  Read the word when convenient.
 *   - Every call that enqueues work (calibrate, append, decode, dequantize)
 *     opens an NVTX range named after itself in the "libkvq" domain, so a
 *     profiler can attribute the kernels to the call; with no profiler
 *     attached a range costs a pointer test.
 *   - Those calls can be captured into a CUDA graph (stream capture) once the
 *     same call has run uncaptured on the device: the first call of a kernel
 *     on a device sets its launch attributes.  A replay re-reads the cache
 *     struct's device buffers (lengths, block table), so replaying an append
 *     and a decode advances the cache exactly as eager calls do.
 *
 * Quantization rules (bit-exact; all arithmetic IEEE fp32 round-to-nearest-
 * even, no fused multiply-add, in exactly this order):
 *   sym  INT-b: qmax = 2^(b-1)-1; a = max|x| over the group; s = a/qmax;
 *               c = clamp(rint(x/s), -qmax, qmax) (c = 0 when s == 0);
 *               x^ = c*s.
 *   asym INT-b: qmax = 2^b-1; mn, mx = min, max over the group;
 *               d = max(mx-mn, 1e-8f); s = d/qmax;
 *               c = clamp(rint((x-mn)/s), 0, qmax); x^ = (c*s) + mn.
 *   FP8 E4M3:   s = k_scale[h] (or v_scale[h]); y = x/s; byte = E4M3FN
 *               encoding of y, round-to-nearest-even, saturating to +-448
 *               (byte 0 when s == 0); x^ = decode(byte)*s.
 *   FP8 E5M2:   the same with the E5M2 encoding (bias 15, 2 mantissa bits,
 *               subnormal step 2^-16), saturating to +-57344.
 *   rint() is round-half-to-even.
 *   fp16 scale/min storage (meta_dtype = KVQ_F16; the pages leave the dtype of
 *   the metadata open): the scale is stored rounded up to a binary16 value and
 *   the minimum rounded down, and the codes use the stored values:
 *     sym:  s = f16_up(a/qmax);
 *     asym: m = f16_down(mn); d = max(mx-m, 1e-8f); s = f16_up(d/qmax);
 *           c = clamp(rint((x-m)/s), 0, qmax); x^ = (c*s) + m;
 *   so |x - x^| <= s/2 still holds.  f16_up / f16_down saturate at +-65504.
 *
 * Axes (kvq_qspec.axis):
 *   PER_CHANNEL (K only): one group per (channel, block of `group` tokens),
 *               blocks aligned to absolute token index multiples of `group`.
 *   PER_TOKEN:  one group per (token, `group` consecutive channels);
 *               group 0 means head_dim.
 *   PER_TENSOR: the static per-head scale k_scale[h] / v_scale[h]
 *               (symmetric INT-b or FP8 only).
 *
 * Residual window (`residual` = R tokens, per sequence and kv-head): new
 * tokens are written unquantized (source dtype) into the window; when an
 * append makes the window hold R tokens, all R are quantized together (R/G
 * key groups, R value rows) and the window empties.  So after T tokens,
 * n_q = R*floor(T/R) tokens are quantized and T - n_q sit in the window.
 * Appending n tokens in one call gives the same bytes as n single appends.
 * R = 0 quantizes every token on append (not allowed with PER_CHANNEL keys).
 *
 * Page layout (stable; version KVQ_LAYOUT_VERSION).  Tokens of sequence b
 * live in pages block_table[b][t / P] at slot t % P (P = page_size).  A page
 * is num_kv_heads consecutive head blocks of kvq_head_block_bytes() bytes.
 * Each head block holds, each section starting on a 16-byte boundary:
 *   K codes  [P][D*bk/8]   bk = bits (8 for FP8)
 *   V codes  [P][D*bv/8]
 *   V meta   [P][ {D/gv scales} {D/gv mins (asym only)} ]  PER_TOKEN V
 *   K meta   PER_CHANNEL: [max(1, P/G)][ {D scales} {D mins (asym)} ];
 *            key group j is stored in the page holding token j*G, in slot
 *            (j*G % P) / G;
 *            PER_TOKEN:   [P][ {D/gk scales} {D/gk mins (asym)} ]
 *            (scales and minima: fp32, or binary16 with meta_dtype = KVQ_F16)
 * Codes are packed along D: channel c's code occupies bits (c*b) % 8 ..
 * of byte (c*b)/8 of the token's row (little-endian bit order).  Code values:
 * sym INT8 two's complement; sym INT2/INT4 offset binary c + 2^(b-1);
 * asym unsigned 0..2^b-1; FP8 the raw E4M3 or E5M2 byte.
 *
 * Residual window buffers k_win / v_win: [batch][R][num_kv_heads][head_dim]
 * in the source dtype; window slot j of sequence b holds token n_q + j.
 */
#ifndef KVQ_H_
#define KVQ_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define KVQ_LAYOUT_VERSION 1

typedef enum {
  KVQ_OK = 0,
  KVQ_ERR_INVALID_ARG = 1, /* null pointer, bad size, inconsistent config  */
  KVQ_ERR_UNSUPPORTED = 2, /* valid but not implemented combination         */
  KVQ_ERR_CUDA = 3,        /* a CUDA runtime call or launch failed          */
  KVQ_ERR_CAPACITY = 4,    /* a size exceeds a documented maximum           */
  KVQ_ERR_WORKSPACE = 5    /* workspace missing, too small or misaligned    */
} kvq_status;

typedef enum { KVQ_INT2 = 2, KVQ_INT4 = 4, KVQ_INT8 = 8, KVQ_FP8_E4M3 = 9, KVQ_FP8_E5M2 = 10 } kvq_format;
typedef enum { KVQ_SYM_ABSMAX = 0, KVQ_ASYM_MINMAX = 1 } kvq_mode; /* ignored for FP8 */
typedef enum { KVQ_PER_TENSOR = 0, KVQ_PER_TOKEN = 1, KVQ_PER_CHANNEL = 2 } kvq_axis;
typedef enum { KVQ_F32 = 0, KVQ_BF16 = 1, KVQ_F16 = 2 } kvq_dtype; /* source/window/q: F32, BF16;
                                                                 stored scales/minima: F32, F16 */

/* Device-side status bits (OR-ed into *kvq_cache.status). */
#define KVQ_DEV_BAD_PAGE 0x1      /* block-table entry outside [0, n_pages)          */
#define KVQ_DEV_OVERFLOW 0x2      /* append would exceed max_pages_per_seq * P tokens */
#define KVQ_DEV_TIMEOUT 0x4       /* a bounded pipeline wait gave up                  */
#define KVQ_DEV_BAD_LENGTH 0x8    /* seq_lens[b] < 0 or beyond the pages              */

typedef struct {
  int32_t fmt;   /* kvq_format */
  int32_t mode;  /* kvq_mode   */
  int32_t axis;  /* kvq_axis   */
  int32_t group; /* PER_CHANNEL: G tokens; PER_TOKEN: g channels (0 = D); else 0 */
} kvq_qspec;

typedef struct {
  int32_t num_q_heads;  /* Hq; a multiple of num_kv_heads                        */
  int32_t num_kv_heads; /* Hkv; query head h reads kv-head h / (Hq/Hkv) (GQA)    */
  int32_t head_dim;     /* D in {64, 128, 256}                                    */
  kvq_qspec k, v;       /* key and value quantization                              */
  int32_t residual;     /* R: window tokens; R % G == 0 when keys are PER_CHANNEL  */
  int32_t page_size;    /* P tokens per page, a multiple of 16; P % G == 0 or G % P == 0 */
  int32_t rope_pre;     /* 1: the cache holds pre-RoPE keys, rotated after dequant */
  float rope_theta;     /* RoPE base; angle of pair i at position p = p*theta^(-2i/D) */
  int32_t src_dtype;    /* kvq_dtype of appended K/V, the window and q            */
  int32_t meta_dtype;   /* stored scales / minima: KVQ_F32 (0) or KVQ_F16 (2)     */
} kvq_config;

typedef struct {
  void* pages;                /* n_pages * kvq_page_bytes(cfg) bytes, 16-byte aligned */
  const int32_t* block_table; /* [batch][max_pages_per_seq] physical page ids        */
  int32_t* seq_lens;          /* [batch] tokens per sequence; advanced by append      */
  void* k_win;                /* [batch][R][Hkv][D] src dtype (NULL when R == 0)      */
  void* v_win;                /* same                                                  */
  const float* k_scale;       /* [Hkv] static scales (PER_TENSOR / FP8 keys), or NULL */
  const float* v_scale;       /* [Hkv] same for values                                */
  int32_t batch;
  int32_t max_pages_per_seq;
  int32_t n_pages;
  int32_t* status;            /* one device int32; error bits are OR-ed in            */
  /* Optional RoPE table, pre-RoPE keys only (NULL otherwise, and then
   * rope_positions is ignored): the output of kvq_rope_table_init for this
   * config, covering positions [0, rope_positions), rope_positions >= 1.
   * Device, 16-byte aligned, owned by the caller, read only, and shareable by
   * every cache with the same head_dim and rope_theta.  When it covers every
   * position the pages can hold, rounded up to a multiple of 32
   * (rope_positions >= max_pages_per_seq * page_size rounded up), the pre-RoPE
   * tensor-core decode kernel copies the cos/sin from it, 32 positions at a
   * time, instead of computing them; otherwise the kernel computes them (same
   * results to ~1e-6 relative).  KVQ_ERR_INVALID_ARG for a table that is
   * misaligned, set for a config without pre-RoPE keys, or with
   * rope_positions < 1. */
  const void* rope_table;
  int32_t rope_positions;
} kvq_cache;

/* Library layout version (KVQ_LAYOUT_VERSION). */
int32_t kvq_layout_version(void);

/* Bytes of a RoPE table for `positions` positions: positions * head_dim * 4
 * (the cos and sin of every (position, pair) in fp32); 0 when cfg is invalid,
 * does not hold pre-RoPE keys, or positions < 1. */
size_t kvq_rope_table_bytes(const kvq_config* cfg, int32_t positions);

/* Fill a RoPE table (kvq_cache.rope_table): the rotation of pair i at position
 * p, angle p * theta^(-2i/D) ("KV Cache Quantization: Why Keys and Values Need
 * Different Axes", "Where does RoPE break this?"; interleaved pairs (2i, 2i+1)),
 * for p in [0, positions).  The values are those the decode kernel computes
 * itself (the same angle reduction and sincospi); the arrangement inside the
 * table is private to the library.  table: device, kvq_rope_table_bytes bytes,
 * 16-byte aligned, overwritten.  Enqueued on `stream`; no synchronisation.
 * KVQ_ERR_INVALID_ARG for a null or misaligned table, positions < 1, or a
 * config without pre-RoPE keys; KVQ_ERR_CAPACITY above 2^24 positions (the
 * angle reduction, here and in the kernel, is exact below that). */
kvq_status kvq_rope_table_init(const kvq_config* cfg, int32_t positions, void* table, void* stream);

/* KVQ_OK when the configuration is consistent and supported, else the reason. */
kvq_status kvq_validate(const kvq_config* cfg);

/* Bytes of one head block and of one page (0 when cfg is invalid). */
size_t kvq_head_block_bytes(const kvq_config* cfg);
size_t kvq_page_bytes(const kvq_config* cfg);

/* Offsets inside a head block: out[0..3] = K codes, V codes, V meta, K meta. */
kvq_status kvq_head_block_offsets(const kvq_config* cfg, size_t out[4]);

/* Workspace bytes kvq_decode_attention needs for `batch` sequences of at most
 * `max_seq_len` tokens (0 when cfg is invalid). */
size_t kvq_workspace_bytes(const kvq_config* cfg, int32_t batch, int32_t max_seq_len);

/* Static per-head scale: scale_out[h] = (max over the n_tokens x D values of
 * head h of |src|) / qmax, fp32; 0 when all are 0.  src: [n_tokens][Hkv][D]
 * device, src dtype.  qmax: 448 for FP8 E4M3, 57344 for FP8 E5M2, 2^(b-1)-1
 * for sym INT-b.
 * scale_out: [Hkv] device fp32, overwritten (also used as the reduction
 * buffer, so it must not alias src). */
kvq_status kvq_calibrate_absmax(const kvq_config* cfg, const void* src, int64_t n_tokens,
                                float qmax, float* scale_out, void* stream);

/* Append tokens to every sequence of the cache.
 * k_new, v_new: [batch][n_new][Hkv][D] device, src dtype; sequence b appends
 * its first n_new_per_seq[b] rows (n_new_per_seq: [batch] device int32, or
 * NULL for n_new each).  Copies inputs: they may be reused once the stream
 * has passed this call.  Writes the window and, for every window that fills
 * (or every token when R == 0), quantizes and packs into the pages; then
 * advances seq_lens.  A sequence that would exceed max_pages_per_seq * P
 * tokens is left unchanged and sets KVQ_DEV_OVERFLOW. */
kvq_status kvq_quantize_append(const kvq_config* cfg, const kvq_cache* cache, const void* k_new,
                               const void* v_new, int32_t n_new, const int32_t* n_new_per_seq,
                               void* stream);

/* Decode attention for one query per (sequence, query head).
 * q: [batch][Hq][D] device, src dtype, already rotated to its own position
 * (post-RoPE q).  out: [batch][Hq][D] device fp32.  softmax_scale: logit
 * multiplier, 0 means 1/sqrt(D).  Attention covers all seq_lens[b] tokens
 * (quantized pages and window); a sequence with 0 tokens gets out = 0.
 * Split-K flash decoding: partial (max, sum, output) per token chunk in
 * `workspace` (device, >= kvq_workspace_bytes(cfg, batch, max_pages_per_seq*P)
 * bytes, 256-byte aligned, contents need no initialisation), then a combine.
 * Returns KVQ_ERR_CAPACITY (nothing launched) when the format mix runs on the
 * generic kernel and its shared memory (the plan's per-sequence prefix grows
 * with the batch) exceeds the device's per-block limit: above about 42,000
 * sequences at head_dim 128, 30,000 at 256. */
kvq_status kvq_decode_attention(const kvq_config* cfg, const kvq_cache* cache, const void* q,
                                float* out, float softmax_scale, void* workspace,
                                size_t ws_bytes, void* stream);

/* The decode kernels kvq_decode_attention chooses between (the pages give no
 * kernel design; these are this library's).  Each tensor-core kernel handles one
 * format mix at head_dim 128 and takes the call when its shape and pointer tests
 * pass; every other call runs on the generic kernel. */
typedef enum {
  KVQ_KERNEL_GENERIC = 0,   /* any format mix, head_dim 64/128/256, any GQA ratio */
  KVQ_KERNEL_ROPE_I8I4 = 1, /* sym INT8 per-channel pre-RoPE K + asym INT4 per-token V,
                               8 kv-heads x 4 query heads, power-of-two G and P */
  KVQ_KERNEL_FP8 = 2,       /* FP8 (E4M3 or E5M2) K and V, 8 query heads per kv-head */
  KVQ_KERNEL_INT2 = 3       /* asym 2-bit per-channel K + asym 2-bit per-token V (g = 32),
                               4 query heads per kv-head, bf16 or fp32 window */
} kvq_kernel;

/* Which kvq_kernel kvq_decode_attention launches for these arguments.  Host
 * only: nothing is enqueued and no device memory is read.  Returns the same
 * argument errors kvq_decode_attention would (before its q/out/workspace
 * checks); *kernel is written on KVQ_OK. */
kvq_status kvq_decode_kernel(const kvq_config* cfg, const kvq_cache* cache, int32_t* kernel);

/* Size of the scratch array kvq_decode_attention_noalloc uses (32 MiB). */
#define KVQ_NOALLOC_SCRATCH_BYTES (32u * 1024u * 1024u)

/* kvq_decode_attention for callers that cannot allocate device memory; the
 * pages have no counterpart to this entry point.  Examples: a plugin inside a
 * serving process whose memory pool already owns the GPU's memory, or a
 * latency-critical loop that must not call cudaMalloc (it can synchronise the
 * device).  Arguments and results are those of kvq_decode_attention without
 * the workspace: the split-K partials go to a KVQ_NOALLOC_SCRATCH_BYTES array
 * inside the library, which every GPU that loads the library holds until the
 * process exits.  It allocates nothing and calls no allocating routine.
 * - Returns KVQ_ERR_CAPACITY (nothing launched) when the call would need more
 *   than KVQ_NOALLOC_SCRATCH_BYTES, i.e. when
 *   kvq_workspace_bytes(cfg, batch, max_pages_per_seq * page_size) exceeds it.
 * - The first call on a device (the calling thread's current device, which
 *   must be the cache's) looks up the array's device address and keeps it for
 *   the process; make that first call before any stream capture.  The address
 *   belongs to the device's primary context: using the library across a
 *   cudaDeviceReset() is not supported.
 * - All calls on a device share the one array: calls that overlap on the GPU
 *   (other streams, other host threads) race and corrupt each other's results.
 *   Calls ordered on one stream are safe; nothing needs clearing between them. */
kvq_status kvq_decode_attention_noalloc(const kvq_config* cfg, const kvq_cache* cache,
                                        const void* q, float* out, float softmax_scale,
                                        void* stream);

/* Dequantize tokens [tok_begin, tok_end) of sequence `seq` to fp32:
 * k_out, v_out: [tok_end - tok_begin][Hkv][D] device.  Quantized tokens use
 * the rules above (bit-exact); window tokens are the stored source values.
 * Keys are returned as stored (pre-RoPE when rope_pre).  Tokens at or
 * beyond seq_lens[seq] are written as 0. */
kvq_status kvq_dequantize(const kvq_config* cfg, const kvq_cache* cache, int32_t seq,
                          int32_t tok_begin, int32_t tok_end, float* k_out, float* v_out,
                          void* stream);

/* Self-test of the device-side failure detection (the pages have no
 * counterpart: it checks this library's own mechanism).  Every pipeline wait of
 * the decode kernels gives up after a fixed number of polls (well under a few
 * seconds), sets KVQ_DEV_TIMEOUT in the status word and lets the kernel finish.
 * This call launches one warp that runs that bounded wait on a barrier phase
 * that nothing completes, so *status (device int32, OR-ed into) gets
 * KVQ_DEV_TIMEOUT once the wait gives up; the context stays usable.  Takes up to
 * about a second of GPU time.  Returns KVQ_ERR_INVALID_ARG for a null status. */
kvq_status kvq_selftest_bounded_wait(int32_t* status, void* stream);

/* Human-readable name of a status code (static storage). */
const char* kvq_status_string(kvq_status s);

#ifdef __cplusplus
}
#endif

#endif /* KVQ_H_ */
