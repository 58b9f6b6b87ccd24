// C ABI of libkvq: argument validation, page-layout arithmetic and the
// extern "C" entry points declared in include/kvq.h.  Kernels live in the
// other translation units; nothing here allocates, frees or synchronises.
#include <math.h>
#include <string.h>

#include "kvq_host.h"
#include "kvq_internal.cuh"

namespace {

inline bool fmt_is_fp8(int fmt) { return fmt == KVQ_FP8_E4M3 || fmt == KVQ_FP8_E5M2; }
inline int bits_of(int fmt) { return fmt_is_fp8(fmt) ? 8 : fmt; }
inline bool fmt_ok(int fmt) {
  return fmt == KVQ_INT2 || fmt == KVQ_INT4 || fmt == KVQ_INT8 || fmt_is_fp8(fmt);
}
inline size_t align16(size_t n) { return (n + 15) & ~size_t(15); }

int tok_group(const kvq_qspec& s, int D) { return s.group ? s.group : D; }

int n_meta(const kvq_qspec& s) {
  return (s.mode == KVQ_ASYM_MINMAX && !fmt_is_fp8(s.fmt)) ? 2 : 1;
}

kvq_status check_spec(const kvq_qspec& s, int D, bool is_key) {
  if (!fmt_ok(s.fmt)) return KVQ_ERR_INVALID_ARG;
  if (s.mode != KVQ_SYM_ABSMAX && s.mode != KVQ_ASYM_MINMAX) return KVQ_ERR_INVALID_ARG;
  if (s.axis != KVQ_PER_TENSOR && s.axis != KVQ_PER_TOKEN && s.axis != KVQ_PER_CHANNEL)
    return KVQ_ERR_INVALID_ARG;
  if (fmt_is_fp8(s.fmt)) return s.axis == KVQ_PER_TENSOR ? KVQ_OK : KVQ_ERR_UNSUPPORTED;
  if (s.axis == KVQ_PER_TENSOR) return s.mode == KVQ_SYM_ABSMAX ? KVQ_OK : KVQ_ERR_UNSUPPORTED;
  if (s.axis == KVQ_PER_CHANNEL) {
    if (!is_key) return KVQ_ERR_UNSUPPORTED;
    if (s.group < 16 || s.group % 16) return KVQ_ERR_INVALID_ARG;
    return KVQ_OK;
  }
  const int g = tok_group(s, D);
  if (g < 16 || g % 16 || D % g) return KVQ_ERR_INVALID_ARG;
  return KVQ_OK;
}

struct Layout {
  size_t krow, vrow, kc, vc, vm, km, head, page;
};

bool layout_of(const kvq_config* c, Layout* L) {
  if (kvq_validate(c) != KVQ_OK) return false;
  const size_t D = c->head_dim, P = c->page_size;
  const size_t mb = c->meta_dtype == KVQ_F16 ? 2 : 4;  // bytes per stored scale / minimum
  L->krow = D * bits_of(c->k.fmt) / 8;
  L->vrow = D * bits_of(c->v.fmt) / 8;
  L->kc = 0;
  L->vc = align16(L->kc + P * L->krow);
  L->vm = align16(L->vc + P * L->vrow);
  size_t vm_bytes = 0;
  if (c->v.axis == KVQ_PER_TOKEN) vm_bytes = P * (D / tok_group(c->v, D)) * n_meta(c->v) * mb;
  L->km = align16(L->vm + vm_bytes);
  size_t km_bytes = 0;
  if (c->k.axis == KVQ_PER_CHANNEL) {
    const size_t G = c->k.group;
    km_bytes = (P >= G ? P / G : 1) * D * n_meta(c->k) * mb;
  } else if (c->k.axis == KVQ_PER_TOKEN) {
    km_bytes = P * (D / tok_group(c->k, D)) * n_meta(c->k) * mb;
  }
  L->head = align16(L->km + km_bytes);
  L->page = L->head * c->num_kv_heads;
  return true;
}

kvq_status check_cache(const kvq_config* c, const kvq_cache* k) {
  if (!k || !k->pages || !k->block_table || !k->seq_lens || !k->status) return KVQ_ERR_INVALID_ARG;
  if (k->batch < 1 || k->max_pages_per_seq < 1 || k->n_pages < 1) return KVQ_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(k->pages) & 15) return KVQ_ERR_INVALID_ARG;
  if (c->residual > 0 && (!k->k_win || !k->v_win)) return KVQ_ERR_INVALID_ARG;
  if ((c->k.axis == KVQ_PER_TENSOR) && !k->k_scale) return KVQ_ERR_INVALID_ARG;
  if ((c->v.axis == KVQ_PER_TENSOR) && !k->v_scale) return KVQ_ERR_INVALID_ARG;
  if ((long long)k->max_pages_per_seq * c->page_size > (1LL << 30)) return KVQ_ERR_CAPACITY;
  if (k->rope_table) {
    if (!c->rope_pre || k->rope_positions < 1 || (reinterpret_cast<uintptr_t>(k->rope_table) & 15))
      return KVQ_ERR_INVALID_ARG;
  }
  return KVQ_OK;
}

}  // namespace

namespace kvq {

bool make_view(const kvq_config* c, const kvq_cache* k, KvqView* v) {
  Layout L;
  if (!layout_of(c, &L)) return false;
  memset(v, 0, sizeof(*v));
  v->Hq = c->num_q_heads;
  v->Hkv = c->num_kv_heads;
  v->D = c->head_dim;
  v->n_rep = c->num_q_heads / c->num_kv_heads;
  v->kfmt = c->k.fmt;
  v->kmode = fmt_is_fp8(c->k.fmt) ? KVQ_SYM_ABSMAX : c->k.mode;
  v->kaxis = c->k.axis;
  v->kgroup = c->k.axis == KVQ_PER_CHANNEL ? c->k.group
              : c->k.axis == KVQ_PER_TOKEN ? tok_group(c->k, c->head_dim) : 0;
  v->vfmt = c->v.fmt;
  v->vmode = fmt_is_fp8(c->v.fmt) ? KVQ_SYM_ABSMAX : c->v.mode;
  v->vaxis = c->v.axis;
  v->vgroup = c->v.axis == KVQ_PER_TOKEN ? tok_group(c->v, c->head_dim) : 0;
  v->kbits = bits_of(c->k.fmt);
  v->vbits = bits_of(c->v.fmt);
  v->R = c->residual;
  v->P = c->page_size;
  v->rope_pre = c->rope_pre;
  v->rope_theta = c->rope_theta;
  v->src_bf16 = c->src_dtype == KVQ_BF16;
  v->krow = (int)L.krow;
  v->vrow = (int)L.vrow;
  v->off_vc = (int)L.vc;
  v->off_vm = (int)L.vm;
  v->off_km = (int)L.km;
  v->meta16 = c->meta_dtype == KVQ_F16;
  v->mb = v->meta16 ? 2 : 4;
  v->k_nmeta = n_meta(c->k);
  v->v_nmeta = n_meta(c->v);
  v->k_ng = c->k.axis == KVQ_PER_TOKEN ? c->head_dim / v->kgroup : 0;
  v->v_ng = c->v.axis == KVQ_PER_TOKEN ? c->head_dim / v->vgroup : 0;
  v->head_bytes = (int)L.head;
  v->page_bytes = (long long)L.page;
  if (k) {
    v->pages = static_cast<uint8_t*>(k->pages);
    v->block_table = k->block_table;
    v->seq_lens = k->seq_lens;
    v->k_win = k->k_win;
    v->v_win = k->v_win;
    v->k_scale = k->k_scale;
    v->v_scale = k->v_scale;
    v->batch = k->batch;
    v->max_pages = k->max_pages_per_seq;
    v->n_pages = k->n_pages;
    v->status = k->status;
    v->rope_table = k->rope_table;
    v->rope_positions = k->rope_table ? k->rope_positions : 0;
  }
  return true;
}

}  // namespace kvq

extern "C" {

int32_t kvq_layout_version(void) { return KVQ_LAYOUT_VERSION; }

size_t kvq_rope_table_bytes(const kvq_config* c, int32_t positions) {
  if (!c || kvq_validate(c) != KVQ_OK || !c->rope_pre || positions < 1) return 0;
  return (size_t)positions * (size_t)c->head_dim * sizeof(float);
}

kvq_status kvq_rope_table_init(const kvq_config* c, int32_t positions, void* table, void* stream) {
  const kvq::NvtxRange range("kvq_rope_table_init");
  kvq::KvqView v;
  if (!kvq::make_view(c, nullptr, &v)) return kvq_validate(c);
  if (!c->rope_pre || positions < 1 || !table || (reinterpret_cast<uintptr_t>(table) & 15))
    return KVQ_ERR_INVALID_ARG;
  if (positions > (1 << 24)) return KVQ_ERR_CAPACITY;
  return kvq::launch_rope_table(v, positions, table, (cudaStream_t)stream);
}

kvq_status kvq_validate(const kvq_config* c) {
  if (!c) return KVQ_ERR_INVALID_ARG;
  if (c->num_kv_heads < 1 || c->num_q_heads < c->num_kv_heads ||
      c->num_q_heads % c->num_kv_heads)
    return KVQ_ERR_INVALID_ARG;
  if (c->head_dim != 64 && c->head_dim != 128 && c->head_dim != 256) return KVQ_ERR_UNSUPPORTED;
  kvq_status s = check_spec(c->k, c->head_dim, true);
  if (s != KVQ_OK) return s;
  s = check_spec(c->v, c->head_dim, false);
  if (s != KVQ_OK) return s;
  if (c->residual < 0 || c->page_size < 16 || c->page_size % 16) return KVQ_ERR_INVALID_ARG;
  if (c->k.axis == KVQ_PER_CHANNEL) {
    const int G = c->k.group;
    if (c->residual == 0 || c->residual % G) return KVQ_ERR_INVALID_ARG;
    if (c->page_size % G && G % c->page_size) return KVQ_ERR_INVALID_ARG;
  }
  if (c->rope_pre != 0 && c->rope_pre != 1) return KVQ_ERR_INVALID_ARG;
  if (c->rope_pre && !(c->rope_theta > 1.0f && isfinite(c->rope_theta))) return KVQ_ERR_INVALID_ARG;
  if (c->src_dtype != KVQ_F32 && c->src_dtype != KVQ_BF16) return KVQ_ERR_INVALID_ARG;
  if (c->meta_dtype != KVQ_F32 && c->meta_dtype != KVQ_F16) return KVQ_ERR_INVALID_ARG;
  return KVQ_OK;
}

size_t kvq_head_block_bytes(const kvq_config* c) {
  Layout L;
  return layout_of(c, &L) ? L.head : 0;
}

size_t kvq_page_bytes(const kvq_config* c) {
  Layout L;
  return layout_of(c, &L) ? L.page : 0;
}

kvq_status kvq_head_block_offsets(const kvq_config* c, size_t out[4]) {
  Layout L;
  if (!out) return KVQ_ERR_INVALID_ARG;
  if (!layout_of(c, &L)) return kvq_validate(c);
  out[0] = L.kc;
  out[1] = L.vc;
  out[2] = L.vm;
  out[3] = L.km;
  return KVQ_OK;
}

size_t kvq_workspace_bytes(const kvq_config* c, int32_t batch, int32_t max_seq_len) {
  kvq::KvqView v;
  if (batch < 1 || max_seq_len < 0 || !kvq::make_view(c, nullptr, &v)) return 0;
  return kvq::attention_workspace_bytes(v, batch);
}

kvq_status kvq_calibrate_absmax(const kvq_config* c, const void* src, int64_t n_tokens, float qmax,
                                float* scale_out, void* stream) {
  const kvq::NvtxRange range("kvq_calibrate_absmax");
  kvq::KvqView v;
  if (!kvq::make_view(c, nullptr, &v)) return kvq_validate(c);
  if (!src || !scale_out || n_tokens < 0 || !(qmax > 0.f) || !isfinite(qmax))
    return KVQ_ERR_INVALID_ARG;
  return kvq::launch_calibrate(v, src, n_tokens, qmax, scale_out, (cudaStream_t)stream);
}

kvq_status kvq_quantize_append(const kvq_config* c, const kvq_cache* cache, const void* k_new,
                               const void* v_new, int32_t n_new, const int32_t* n_new_per_seq,
                               void* stream) {
  const kvq::NvtxRange range("kvq_quantize_append");
  kvq::KvqView v;
  if (!kvq::make_view(c, cache, &v)) return kvq_validate(c);
  kvq_status s = check_cache(c, cache);
  if (s != KVQ_OK) return s;
  if (n_new < 0) return KVQ_ERR_INVALID_ARG;
  if ((long long)n_new > (long long)cache->max_pages_per_seq * c->page_size) return KVQ_ERR_CAPACITY;
  if (n_new == 0) return KVQ_OK;
  if (!k_new || !v_new) return KVQ_ERR_INVALID_ARG;
  return kvq::launch_append(v, k_new, v_new, n_new, n_new_per_seq, (cudaStream_t)stream);
}

kvq_status kvq_decode_attention(const kvq_config* c, const kvq_cache* cache, const void* q,
                                float* out, float softmax_scale, void* workspace, size_t ws_bytes,
                                void* stream) {
  const kvq::NvtxRange range("kvq_decode_attention");
  kvq::KvqView v;
  if (!kvq::make_view(c, cache, &v)) return kvq_validate(c);
  kvq_status s = check_cache(c, cache);
  if (s != KVQ_OK) return s;
  if (!q || !out || !(softmax_scale >= 0.f) || !isfinite(softmax_scale)) return KVQ_ERR_INVALID_ARG;
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255)) return KVQ_ERR_WORKSPACE;
  if (ws_bytes < kvq::attention_workspace_bytes(v, cache->batch)) return KVQ_ERR_WORKSPACE;
  const float scale = softmax_scale > 0.f ? softmax_scale : 1.0f / sqrtf((float)c->head_dim);
  return kvq::launch_attention(v, q, out, scale, workspace, ws_bytes, (cudaStream_t)stream);
}

kvq_status kvq_dequantize(const kvq_config* c, const kvq_cache* cache, int32_t seq,
                          int32_t tok_begin, int32_t tok_end, float* k_out, float* v_out,
                          void* stream) {
  const kvq::NvtxRange range("kvq_dequantize");
  kvq::KvqView v;
  if (!kvq::make_view(c, cache, &v)) return kvq_validate(c);
  kvq_status s = check_cache(c, cache);
  if (s != KVQ_OK) return s;
  if (seq < 0 || seq >= cache->batch || tok_begin < 0 || tok_end < tok_begin) return KVQ_ERR_INVALID_ARG;
  if ((long long)tok_end > (long long)cache->max_pages_per_seq * c->page_size) return KVQ_ERR_CAPACITY;
  if (tok_end == tok_begin) return KVQ_OK;
  if (!k_out || !v_out) return KVQ_ERR_INVALID_ARG;
  return kvq::launch_dequantize(v, seq, tok_begin, tok_end, k_out, v_out, (cudaStream_t)stream);
}

kvq_status kvq_decode_kernel(const kvq_config* c, const kvq_cache* cache, int32_t* kernel) {
  kvq::KvqView v;
  if (!kernel) return KVQ_ERR_INVALID_ARG;
  if (!kvq::make_view(c, cache, &v)) return kvq_validate(c);
  const kvq_status s = check_cache(c, cache);
  if (s != KVQ_OK) return s;
  *kernel = kvq::pick_decode_kernel(v);
  return KVQ_OK;
}

const char* kvq_status_string(kvq_status s) {
  switch (s) {
    case KVQ_OK: return "ok";
    case KVQ_ERR_INVALID_ARG: return "invalid argument";
    case KVQ_ERR_UNSUPPORTED: return "unsupported configuration";
    case KVQ_ERR_CUDA: return "CUDA error";
    case KVQ_ERR_CAPACITY: return "capacity exceeded";
    case KVQ_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
  }
  return "unknown status";
}

}  // extern "C"
