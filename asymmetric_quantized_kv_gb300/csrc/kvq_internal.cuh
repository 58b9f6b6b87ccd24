// Internal declarations shared by the libkvq translation units.
//
// KvqView is the resolved, by-value description of one cache (configuration,
// page layout and caller pointers) that every kernel receives.  The helpers
// below implement the bit-exact quantization steps of include/kvq.h with
// explicit IEEE round-to-nearest intrinsics (no FMA contraction).
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "../../include/kvq.h"

namespace kvq {

struct KvqView {
  // configuration
  int Hq, Hkv, D, n_rep;
  int kfmt, kmode, kaxis, kgroup;  // kgroup: G (PER_CHANNEL) or g (PER_TOKEN, resolved)
  int vfmt, vmode, vaxis, vgroup;
  int kbits, vbits;
  int R, P;
  int rope_pre;
  float rope_theta;
  int src_bf16;
  // layout of one head block
  int krow, vrow;                    // bytes per packed token row
  int off_vc, off_vm, off_km;        // section offsets (K codes at 0)
  int k_nmeta, v_nmeta;              // values per group entry: 2 asym (scale, min), 1 sym
  int meta16, mb;                    // stored scales / minima binary16 (mb = 2 bytes) or fp32 (4)
  int k_ng, v_ng;                    // PER_TOKEN groups per token
  int head_bytes;
  long long page_bytes;
  // caller's cache
  uint8_t* pages;
  const int32_t* block_table;
  int32_t* seq_lens;
  void* k_win;
  void* v_win;
  const float* k_scale;
  const float* v_scale;
  int batch, max_pages, n_pages;
  int32_t* status;
  const void* rope_table;  // optional: kvq_rope_table_init output for positions [0, rope_positions)
  int rope_positions;
};

// Host: resolve a validated config + cache into a view (false when invalid).
bool make_view(const kvq_config* cfg, const kvq_cache* cache, KvqView* out);

// Host launchers (each returns KVQ_OK or KVQ_ERR_CUDA).
kvq_status launch_append(const KvqView& v, const void* k_new, const void* v_new, int n_new,
                         const int32_t* n_new_per_seq, cudaStream_t st);
kvq_status launch_dequantize(const KvqView& v, int seq, int t0, int t1, float* k_out,
                             float* v_out, cudaStream_t st);
kvq_status launch_calibrate(const KvqView& v, const void* src, long long n_tokens, float qmax,
                            float* scale_out, cudaStream_t st);
size_t attention_workspace_bytes(const KvqView& v, int batch);
// Fill a RoPE table (kvq_rope_table_init): positions rows of D/4 float4.
kvq_status launch_rope_table(const KvqView& v, int positions, void* table, cudaStream_t st);
// Tensor-core decode kernel for INT8 per-channel pre-RoPE keys + INT4 per-token values.
bool fast_eligible(const KvqView& v);
size_t fast_workspace_bytes(const KvqView& v, int batch);
kvq_status launch_fast(const KvqView& v, const void* q, float* out, float scale, void* ws,
                       cudaStream_t st);
// Tensor-core decode kernel for FP8 E4M3 keys and values, 8 query heads per kv-head.
bool fp8_shape_eligible(const KvqView& v);  // config only: sizes the workspace
bool fp8_eligible(const KvqView& v);        // config, cache pointers and pool size
kvq_status launch_fp8(const KvqView& v, const void* q, float* out, float scale, void* ws, cudaStream_t st);
// Tensor-core decode kernel for 2-bit asymmetric per-channel keys + per-token values (g = 32).
bool int2_shape_eligible(const KvqView& v);  // config only: sizes the workspace
bool int2_eligible(const KvqView& v);        // config, cache pointers and pool size
kvq_status launch_int2(const KvqView& v, const void* q, float* out, float scale, void* ws, cudaStream_t st);
// The decode kernel launch_attention runs for a resolved cache (a kvq_kernel value):
// the first tensor-core kernel whose shape and pointer tests pass, else the generic one.
int pick_decode_kernel(const KvqView& v);
kvq_status launch_attention(const KvqView& v, const void* q, float* out, float scale,
                            void* ws, size_t ws_bytes, cudaStream_t st);

// ------------------------------------------------------------------ device helpers

__device__ __forceinline__ float load_src(const void* base, long long idx, int bf16) {
  if (bf16) {
    const unsigned short u = reinterpret_cast<const unsigned short*>(base)[idx];
    return __uint_as_float(static_cast<unsigned>(u) << 16);
  }
  return reinterpret_cast<const float*>(base)[idx];
}

__device__ __forceinline__ void store_src(void* base, long long idx, float x, int bf16) {
  if (bf16) {
    // x already holds a bf16-exact value (it came from bf16 storage)
    reinterpret_cast<unsigned short*>(base)[idx] =
        static_cast<unsigned short>(__float_as_uint(x) >> 16);
  } else {
    reinterpret_cast<float*>(base)[idx] = x;
  }
}

// Physical page of token t of sequence b, or nullptr (and a status bit) when the
// block-table entry is out of range.
__device__ __forceinline__ uint8_t* page_of(const KvqView& v, int b, int t) {
  const int pid = v.block_table[(long long)b * v.max_pages + t / v.P];
  if (pid < 0 || pid >= v.n_pages) {
    atomicOr(v.status, KVQ_DEV_BAD_PAGE);
    return nullptr;
  }
  return v.pages + (long long)pid * v.page_bytes;
}

__device__ __forceinline__ int n_quantized(int T, int R) { return R > 0 ? R * (T / R) : T; }

// Unsigned code of channel c in a packed row of `bits`-bit codes.
__device__ __forceinline__ unsigned get_code(const uint8_t* row, int c, int bits) {
  if (bits == 8) return row[c];
  const int bit = c * bits;
  return (row[bit >> 3] >> (bit & 7)) & ((1u << bits) - 1u);
}

// Signed code value from the stored unsigned code (sym / asym encodings).
__device__ __forceinline__ int signed_code(unsigned u, int bits, int mode) {
  if (mode == KVQ_ASYM_MINMAX) return static_cast<int>(u);
  if (bits == 8) return static_cast<int>(static_cast<int8_t>(u));
  return static_cast<int>(u) - (1 << (bits - 1));
}

__device__ __forceinline__ unsigned stored_code(int c, int bits, int mode) {
  if (mode == KVQ_ASYM_MINMAX) return static_cast<unsigned>(c);
  if (bits == 8) return static_cast<unsigned>(c) & 0xFFu;
  return static_cast<unsigned>(c + (1 << (bits - 1)));
}

__device__ __forceinline__ bool is_fp8(int fmt) { return fmt == KVQ_FP8_E4M3 || fmt == KVQ_FP8_E5M2; }

// Value of an FP8 byte of format fmt (E4M3 or E5M2); exact in f16 and fp32.
__device__ __forceinline__ float fp8_to_float(unsigned byte, int fmt) {
  const __half_raw h = __nv_cvt_fp8_to_halfraw(static_cast<__nv_fp8_storage_t>(byte),
                                               fmt == KVQ_FP8_E5M2 ? __NV_E5M2 : __NV_E4M3);
  return __half2float(__half(h));
}

// FP8 byte of y: nearest value, ties to even, saturating at the format's maximum.
__device__ __forceinline__ unsigned float_to_fp8(float y, int fmt) {
  return static_cast<unsigned>(
      __nv_cvt_float_to_fp8(y, __NV_SATFINITE, fmt == KVQ_FP8_E5M2 ? __NV_E5M2 : __NV_E4M3));
}

// ---- the exact quantization steps of include/kvq.h

__device__ __forceinline__ int sym_qmax(int bits) { return (1 << (bits - 1)) - 1; }
__device__ __forceinline__ int asym_qmax(int bits) { return (1 << bits) - 1; }

__device__ __forceinline__ float sym_scale(float absmax, int bits) {
  return __fdiv_rn(absmax, static_cast<float>(sym_qmax(bits)));
}

__device__ __forceinline__ int sym_code(float x, float s, int bits) {
  if (s == 0.f) return 0;
  const float q = static_cast<float>(sym_qmax(bits));
  const float r = rintf(__fdiv_rn(x, s));
  return static_cast<int>(fminf(fmaxf(r, -q), q));
}

__device__ __forceinline__ float asym_scale(float mn, float mx, int bits) {
  const float d = fmaxf(__fsub_rn(mx, mn), 1e-8f);
  return __fdiv_rn(d, static_cast<float>(asym_qmax(bits)));
}

__device__ __forceinline__ int asym_code(float x, float mn, float s, int bits) {
  const float r = rintf(__fdiv_rn(__fsub_rn(x, mn), s));
  return static_cast<int>(fminf(fmaxf(r, 0.f), static_cast<float>(asym_qmax(bits))));
}

// rint(fl32(x / s)) without a division per element: r = 1/s rounded to nearest,
// so fl32(x * r) lies within 2^-23 (relative) of x / s, as does fl32(x / s).  The
// two round to the same integer unless the product is near a half-integer; those
// rare cases (and non-finite r) take the exact IEEE division.
// The exact path, kept out of line: it is rare, and inlining the IEEE division at
// every quantizer call site would bloat the code a short kernel has to fetch.
static __device__ __noinline__ float rint_div_exact(float x, float s) { return rintf(__fdiv_rn(x, s)); }

// True when the product q = fl32(x * r) may round to another integer than x / s
// (near a half-integer, or not a number).
__device__ __forceinline__ bool quot_near_half(float q) {
  const float f = q - floorf(q);
  return !(fabsf(f - 0.5f) > 1.52587890625e-05f * fmaxf(1.f, fabsf(q)));
}

__device__ __forceinline__ float rint_quot(float x, float s, float r) {
  const float q = __fmul_rn(x, r);
  if (quot_near_half(q)) return rint_div_exact(x, s);
  return rintf(q);
}

__device__ __forceinline__ int sym_code_r(float x, float s, float r, int bits) {
  if (s == 0.f) return 0;
  const float q = static_cast<float>(sym_qmax(bits));
  return static_cast<int>(fminf(fmaxf(rint_quot(x, s, r), -q), q));
}

__device__ __forceinline__ int asym_code_r(float x, float mn, float s, float r, int bits) {
  const float c = rint_quot(__fsub_rn(x, mn), s, r);
  return static_cast<int>(fminf(fmaxf(c, 0.f), static_cast<float>(asym_qmax(bits))));
}

__device__ __forceinline__ unsigned fp8_code(float x, float s, int fmt) {
  if (s == 0.f) return 0u;
  return float_to_fp8(__fdiv_rn(x, s), fmt);
}

// ---- binary16 storage of scales and minima (meta_dtype KVQ_F16): the scale
// rounded up, the minimum rounded down, saturating at +-65504
__device__ __forceinline__ float f16_up(float x) { return fminf(__half2float(__float2half_ru(x)), 65504.f); }
__device__ __forceinline__ float f16_down(float x) { return fmaxf(__half2float(__float2half_rd(x)), -65504.f); }

__device__ __forceinline__ float load_meta(const uint8_t* p, int i, int m16) {
  return m16 ? __half2float(reinterpret_cast<const __half*>(p)[i]) : reinterpret_cast<const float*>(p)[i];
}
__device__ __forceinline__ void store_meta(uint8_t* p, int i, float x, int m16) {
  if (m16) {
    reinterpret_cast<__half*>(p)[i] = __float2half_rn(x);  // x is a binary16 value already
  } else {
    reinterpret_cast<float*>(p)[i] = x;
  }
}

// Scale s and minimum m of one group as stored (include/kvq.h): from the group's
// min / max (asym) or absmax (sym), fp32 or binary16 storage.
__device__ __forceinline__ void group_scale(float mn, float mx, float amax, bool asym, int bits, int m16,
                                            float& s, float& m) {
  if (asym) {
    if (m16) {
      m = f16_down(mn);
      s = f16_up(__fdiv_rn(fmaxf(__fsub_rn(mx, m), 1e-8f), static_cast<float>(asym_qmax(bits))));
    } else {
      s = asym_scale(mn, mx, bits);
      m = mn;
    }
  } else {
    s = sym_scale(amax, bits);
    if (m16) s = f16_up(s);
    m = 0.f;
  }
}

__device__ __forceinline__ float dequant_sym(int c, float s) {
  return __fmul_rn(static_cast<float>(c), s);
}
__device__ __forceinline__ float dequant_asym(int c, float s, float mn) {
  return __fadd_rn(__fmul_rn(static_cast<float>(c), s), mn);
}

// ---- RoPE angle (turns) of position p for pair i, accurate for p < 2^24:
// omega_i = theta^(-2i/D) / (2 pi) is held as a two-float hi + lo; p*hi is split
// exactly with an FMA (TwoProduct), its integer part dropped, and the rest summed.
__device__ __forceinline__ float rope_turns(int p, float w_hi, float w_lo) {
  const float pf = static_cast<float>(p);
  const float P = __fmul_rn(pf, w_hi);
  const float E = fmaf(pf, w_hi, -P);
  const float F = __fsub_rn(P, rintf(P));
  return F + (E + pf * w_lo);
}

}  // namespace kvq
