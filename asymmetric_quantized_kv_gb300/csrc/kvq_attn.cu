// Split-K decode attention over the quantized cache: the generic kernel (every
// format, axis, window and pre-RoPE combination), the work plan and the combine.
//
// What is computed: for each sequence b and query head h, over all T tokens,
// logits_j = (q_h . k_j) * scale, p = softmax(logits), out = sum_j p_j v_j
// ("FP8 KV Cache Quantization: Why Keys Break Before Values", section "Why does
// the K cache break before the V cache?", attention formula), with k_j, v_j
// dequantized by the rules of include/kvq.h and, for a pre-RoPE cache, k_j
// rotated by its absolute position after dequantization ("KV Cache
// Quantization: Why Keys and Values Need Different Axes", section "Where does
// RoPE break this?").  Query head h reads kv-head h / (Hq/Hkv).
//
// Split-K: the tokens of each (sequence, kv-head) are cut into chunks of C
// tokens (plus one item for the residual window); every chunk produces a
// partial (max, sum, unnormalised output) per query head in base-2 exponent
// form, and a combine kernel merges the partials exactly:
//   M = max m_i,  L = sum l_i 2^(m_i - M),  out = sum o_i 2^(m_i - M) / L.
#include <math.h>

#include "kvq_attn_plan.cuh"

namespace kvq {
namespace {

constexpr int kWarps = 4;
constexpr int kThreads = kWarps * 32;
constexpr float kLog2e = 1.4426950408889634f;

struct TileKeys {
  const uint8_t* hb;     // head block of the token's page (quantized tokens)
  const uint8_t* kmeta;  // PER_CHANNEL: group meta; PER_TOKEN: token meta (fp32 or binary16 entries)
  int slot;
};

__device__ __forceinline__ float deq_key(const KvqView& v, const TileKeys& tk, int h, int c) {
  const unsigned u = get_code(tk.hb + tk.slot * v.krow, c, v.kbits);
  if (is_fp8(v.kfmt)) return __fmul_rn(fp8_to_float(u, v.kfmt), v.k_scale[h]);
  if (v.kaxis == KVQ_PER_TENSOR) return dequant_sym(signed_code(u, v.kbits, KVQ_SYM_ABSMAX), v.k_scale[h]);
  const int code = signed_code(u, v.kbits, v.kmode);
  float s, mn = 0.f;
  if (v.kaxis == KVQ_PER_TOKEN) {
    const int grp = c / v.kgroup;
    s = load_meta(tk.kmeta, grp, v.meta16);
    if (v.k_nmeta == 2) mn = load_meta(tk.kmeta, v.k_ng + grp, v.meta16);
  } else {
    s = load_meta(tk.kmeta, c, v.meta16);
    if (v.k_nmeta == 2) mn = load_meta(tk.kmeta, v.D + c, v.meta16);
  }
  return v.kmode == KVQ_ASYM_MINMAX ? dequant_asym(code, s, mn) : dequant_sym(code, s);
}

__device__ __forceinline__ float deq_value(const KvqView& v, const uint8_t* hb, int slot, int h, int c) {
  const unsigned u = get_code(hb + v.off_vc + slot * v.vrow, c, v.vbits);
  if (is_fp8(v.vfmt)) return __fmul_rn(fp8_to_float(u, v.vfmt), v.v_scale[h]);
  if (v.vaxis == KVQ_PER_TENSOR) return dequant_sym(signed_code(u, v.vbits, KVQ_SYM_ABSMAX), v.v_scale[h]);
  const uint8_t* meta = hb + v.off_vm + slot * v.v_ng * v.v_nmeta * v.mb;
  const int grp = c / v.vgroup;
  const int code = signed_code(u, v.vbits, v.vmode);
  const float s = load_meta(meta, grp, v.meta16);
  return v.vmode == KVQ_ASYM_MINMAX ? dequant_asym(code, s, load_meta(meta, v.v_ng + grp, v.meta16))
                                    : dequant_sym(code, s);
}

__device__ __forceinline__ float warp_max(float x) {
  for (int o = 16; o; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
  return x;
}
__device__ __forceinline__ float warp_sum(float x) {
  for (int o = 16; o; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

struct GenericSmem {
  float qs[kHB][kMaxHeadDim];
  float ps[kWarps][kHB][32];
  float wm[kWarps][kHB];
  float wl[kWarps][kHB];
  float wo[kWarps][kHB][kMaxHeadDim];
  float rope_hi[kMaxHeadDim / 2];
  float rope_lo[kMaxHeadDim / 2];
};

__global__ void __launch_bounds__(kThreads) split_generic_kernel(KvqView v, const void* q, float scale,
                                                                  float* ws) {
  extern __shared__ __align__(16) unsigned char dyn[];
  GenericSmem& sm = *reinterpret_cast<GenericSmem*>(dyn);
  int* pref = reinterpret_cast<int*>(dyn + sizeof(GenericSmem));
  const int HB = (v.n_rep + kHB - 1) / kHB;
  __shared__ int s_C, s_items;
  plan_items(v, HB, pref, &s_C, &s_items);
  if (blockIdx.x == 0) store_plan(v, ws, pref, s_C, s_items);
  const int C = s_C, n_items = s_items;
  const int D = v.D;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (v.rope_pre) {
    for (int i = threadIdx.x; i < D / 2; i += kThreads) rope_split(v, i, &sm.rope_hi[i], &sm.rope_lo[i]);
  }
  float* part = plan_partials(ws, v.batch);
  for (int item = blockIdx.x; item < n_items; item += gridDim.x) {
    ItemInfo it = decode_item(v, pref, C, HB, item);
    const int nh = min(kHB, v.n_rep - it.hb * kHB);
    __syncthreads();  // smem of the previous item is free
    for (int e = threadIdx.x; e < kHB * D; e += kThreads) {
      const int hh = e / D, c = e % D;
      float x = 0.f;
      if (hh < nh) {
        const int hq = it.kvh * v.n_rep + it.hb * kHB + hh;
        x = load_src(q, ((long long)it.b * v.Hq + hq) * D + c, v.src_bf16) * scale * kLog2e;
      }
      sm.qs[hh][c] = x;
    }
    __syncthreads();
    float m_run[kHB], l_run[kHB], o[kHB][kMaxHeadDim / 32];
#pragma unroll
    for (int hh = 0; hh < kHB; ++hh) {
      m_run[hh] = -INFINITY;
      l_run[hh] = 0.f;
#pragma unroll
      for (int j = 0; j < kMaxHeadDim / 32; ++j) o[hh][j] = 0.f;
    }
    const int nj = D / 32;
    for (int tile = it.t0 + warp * 32; tile < it.t1; tile += kWarps * 32) {
      const int t = tile + lane;
      bool valid = t < it.t1;
      TileKeys tk{nullptr, nullptr, 0};
      long long wrow = 0;
      if (valid && !it.window) {
        const uint8_t* page = page_of(v, it.b, t);
        valid = page != nullptr;
        if (valid) {
          tk.hb = page + (long long)it.kvh * v.head_bytes;
          tk.slot = t % v.P;
          if (v.kaxis == KVQ_PER_TOKEN) {
            tk.kmeta = tk.hb + v.off_km + tk.slot * v.k_ng * v.k_nmeta * v.mb;
          } else if (v.kaxis == KVQ_PER_CHANNEL) {
            const int g0 = (t / v.kgroup) * v.kgroup;
            const uint8_t* gp = page_of(v, it.b, g0);
            valid = gp != nullptr;
            if (valid)
              tk.kmeta = gp + (long long)it.kvh * v.head_bytes + v.off_km +
                         (long long)((g0 % v.P) / v.kgroup) * D * v.k_nmeta * v.mb;
          }
        }
      } else if (valid) {
        wrow = (((long long)it.b * v.R + (t - it.t0)) * v.Hkv + it.kvh) * D;
      }
      float acc[kHB];
#pragma unroll
      for (int hh = 0; hh < kHB; ++hh) acc[hh] = 0.f;
      if (valid) {
        for (int c = 0; c < D; c += 2) {
          float k0, k1;
          if (it.window) {
            k0 = load_src(v.k_win, wrow + c, v.src_bf16);
            k1 = load_src(v.k_win, wrow + c + 1, v.src_bf16);
          } else {
            k0 = deq_key(v, tk, it.kvh, c);
            k1 = deq_key(v, tk, it.kvh, c + 1);
          }
          if (v.rope_pre) {
            float sn, cs;
            sincospif(2.f * rope_turns(t, sm.rope_hi[c / 2], sm.rope_lo[c / 2]), &sn, &cs);
            const float r0 = k0 * cs - k1 * sn;
            const float r1 = k0 * sn + k1 * cs;
            k0 = r0;
            k1 = r1;
          }
#pragma unroll
          for (int hh = 0; hh < kHB; ++hh) acc[hh] += sm.qs[hh][c] * k0 + sm.qs[hh][c + 1] * k1;
        }
      }
#pragma unroll
      for (int hh = 0; hh < kHB; ++hh) {
        const float lg = valid ? acc[hh] : -INFINITY;
        const float m_new = fmaxf(m_run[hh], warp_max(lg));
        const float alpha = m_new == -INFINITY ? 1.f : exp2f(m_run[hh] - m_new);
        const float p = valid ? exp2f(lg - m_new) : 0.f;
        l_run[hh] = l_run[hh] * alpha + warp_sum(p);
        m_run[hh] = m_new;
#pragma unroll
        for (int j = 0; j < kMaxHeadDim / 32; ++j) o[hh][j] *= alpha;
        sm.ps[warp][hh][lane] = p;
      }
      __syncwarp();
      const int nt = min(32, it.t1 - tile);
      for (int tt = 0; tt < nt; ++tt) {
        const int tok = tile + tt;
        const uint8_t* hb = nullptr;
        long long vrow = 0;
        if (!it.window) {
          const uint8_t* page = page_of(v, it.b, tok);
          if (!page) continue;
          hb = page + (long long)it.kvh * v.head_bytes;
        } else {
          vrow = (((long long)it.b * v.R + (tok - it.t0)) * v.Hkv + it.kvh) * D;
        }
        for (int j = 0; j < nj; ++j) {
          const int c = lane + 32 * j;
          const float vx = it.window ? load_src(v.v_win, vrow + c, v.src_bf16)
                                     : deq_value(v, hb, tok % v.P, it.kvh, c);
#pragma unroll
          for (int hh = 0; hh < kHB; ++hh) o[hh][j] += sm.ps[warp][hh][tt] * vx;
        }
      }
      __syncwarp();
    }
    // merge the warps of this CTA
#pragma unroll
    for (int hh = 0; hh < kHB; ++hh) {
      if (lane == 0) {
        sm.wm[warp][hh] = m_run[hh];
        sm.wl[warp][hh] = l_run[hh];
      }
      for (int j = 0; j < nj; ++j) sm.wo[warp][hh][lane + 32 * j] = o[hh][j];
    }
    __syncthreads();
    float* dst = part + (long long)item * kHB * (D + 2);
    for (int e = threadIdx.x; e < nh * D; e += kThreads) {
      const int hh = e / D, c = e % D;
      float M = -INFINITY;
      for (int w = 0; w < kWarps; ++w) M = fmaxf(M, sm.wm[w][hh]);
      float L = 0.f, O = 0.f;
      for (int w = 0; w < kWarps; ++w) {
        const float f = sm.wm[w][hh] == -INFINITY ? 0.f : exp2f(sm.wm[w][hh] - M);
        L += sm.wl[w][hh] * f;
        O += sm.wo[w][hh][c] * f;
      }
      if (c == 0) {
        dst[hh * (D + 2) + 0] = M;
        dst[hh * (D + 2) + 1] = L;
      }
      dst[hh * (D + 2) + 2 + c] = O;
    }
  }
}

}  // namespace

__global__ void combine_kernel(KvqView v, float* ws, float* out) {
  const int hq = blockIdx.x, b = blockIdx.y;
  const int D = v.D;
  const int HB = (v.n_rep + kHB - 1) / kHB;
  const int* pref = plan_prefix(ws);
  const float* part = plan_partials(ws, v.batch);
  const int kvh = hq / v.n_rep, hr = hq % v.n_rep, hb = hr / kHB, hh = hr % kHB;
  const int nc = (pref[b + 1] - pref[b]) / (v.Hkv * HB);
  const long long item0 = pref[b] + (long long)(kvh * HB + hb) * nc;
  float M = -INFINITY;
  for (int i = 0; i < nc; ++i) M = fmaxf(M, part[(item0 + i) * kHB * (D + 2) + hh * (D + 2)]);
  float L = 0.f;
  for (int i = 0; i < nc; ++i) {
    const float* p = part + (item0 + i) * kHB * (D + 2) + hh * (D + 2);
    L += p[0] == -INFINITY ? 0.f : p[1] * exp2f(p[0] - M);
  }
  const float invL = L > 0.f ? 1.f / L : 0.f;
  for (int c = threadIdx.x; c < D; c += blockDim.x) {
    float O = 0.f;
    for (int i = 0; i < nc; ++i) {
      const float* p = part + (item0 + i) * kHB * (D + 2) + hh * (D + 2);
      if (p[0] != -INFINITY) O += p[2 + c] * exp2f(p[0] - M);
    }
    out[((long long)b * v.Hq + hq) * D + c] = O * invL;
  }
}

size_t attention_workspace_bytes(const KvqView& v, int batch) {
  const int HB = (v.n_rep + kHB - 1) / kHB;
  const long long items = kTargetItems + 2LL * batch * v.Hkv * HB;
  const size_t generic = plan_header_bytes(batch) + (size_t)items * kHB * (v.D + 2) * sizeof(float);
  KvqView b = v;
  b.batch = batch;
  const size_t split = fast_workspace_bytes(v, batch);  // layout of the tensor-core kernels
  return (fast_eligible(b) || fp8_shape_eligible(b) || int2_shape_eligible(b)) && split > generic ? split : generic;
}

kvq_status launch_attention(const KvqView& v, const void* q, float* out, float scale, void* ws,
                            size_t ws_bytes, cudaStream_t st) {
  (void)ws_bytes;
  if (fast_eligible(v)) return launch_fast(v, q, out, scale, ws, st);
  if (fp8_eligible(v)) return launch_fp8(v, q, out, scale, ws, st);
  if (int2_eligible(v)) return launch_int2(v, q, out, scale, ws, st);
  const size_t smem = sizeof(GenericSmem) + sizeof(int) * (v.batch + 1);
  static bool attr_set = false;
  if (!attr_set) {
    if (cudaFuncSetAttribute(split_generic_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             160 * 1024) != cudaSuccess)
      return KVQ_ERR_CUDA;
    attr_set = true;
  }
  if (smem > 160 * 1024) return KVQ_ERR_CAPACITY;
  const int grid = num_sms() * 2;
  split_generic_kernel<<<grid, kThreads, smem, st>>>(v, q, scale, static_cast<float*>(ws));
  combine_kernel<<<dim3(v.Hq, v.batch), 128, 0, st>>>(v, static_cast<float*>(ws), out);
  return cudaGetLastError() == cudaSuccess ? KVQ_OK : KVQ_ERR_CUDA;
}

}  // namespace kvq
