// Quantize-append, dequantize and absmax calibration kernels.
//
// Append follows the residual-window rule of include/kvq.h: new tokens go to the
// window; every window that fills is quantized as one block of R tokens (R/G
// per-channel key groups, R per-token value rows) and packed into the pages.
// ("FP8 KV Cache Quantization: Why Keys Break Before Values", section "Should
// you quantize keys pre-RoPE or post-RoPE?": grouping within fixed-size blocks
// plus a full-precision window of recent tokens; "KV Cache Quantization: Why
// Keys and Values Need Different Axes", section "What should I actually turn on
// in production?", checklist.)
//
// One CTA per (flush block, kv-head, sequence).  CTA 0 of a sequence also owns
// the window: it first quantizes the block that may read the old window, then
// (after a barrier) writes the remaining new tokens into the window, so one
// launch never reads and overwrites the same window slots out of order.
#include "kvq_internal.cuh"

namespace kvq {
namespace {

constexpr int kThreads = 256;
constexpr int kSub = 32;        // tokens staged per sub-chunk
constexpr int kUnitTok = 64;    // tokens per CTA when R == 0
constexpr int kMaxD = 256;
constexpr int kMaxGroups = 16;  // PER_TOKEN groups per token (D/g with g >= 16)

struct Src {
  const void* win;    // [B][R][Hkv][D]
  const void* fresh;  // [B][n_new][Hkv][D]
};

struct TQ {  // one tensor's quantization parameters
  int fmt, mode, axis, group, bits, nmeta, ng, off_codes, off_meta, row;
  const float* static_scale;
};

struct AppendCtx {
  int b, h, T0, wbase, n_stride;
};

__device__ __forceinline__ float src_value(const KvqView& v, const Src& s, const AppendCtx& a,
                                           int t, int c) {
  if (t < a.T0) {
    const long long i = (((long long)a.b * v.R + (t - a.wbase)) * v.Hkv + a.h) * v.D + c;
    return load_src(s.win, i, v.src_bf16);
  }
  const long long i = (((long long)a.b * a.n_stride + (t - a.T0)) * v.Hkv + a.h) * v.D + c;
  return load_src(s.fresh, i, v.src_bf16);
}

struct Smem {
  float xs[kSub][kMaxD];
  uint32_t stage[kSub][kMaxD * 8 / 32];
  float gs[kSub][kMaxGroups];
  float gm[kSub][kMaxGroups];
  float cmin[kThreads];
  float cmax[kThreads];
  float ch_s[kMaxD];
  float ch_m[kMaxD];
};

// Pack the codes of rows [t0, t0+n) staged in sm.stage into the pages.
__device__ void flush_stage(const KvqView& v, const AppendCtx& a, const TQ& q, Smem& sm, int t0,
                            int n) {
  const int wpr = q.row / 4;
  for (int w = threadIdx.x; w < n * wpr; w += kThreads) {
    const int r = w / wpr, k = w % wpr;
    const int t = t0 + r;
    uint8_t* page = page_of(v, a.b, t);
    if (!page) continue;
    uint8_t* dst = page + (long long)a.h * v.head_bytes + q.off_codes + (t % v.P) * q.row;
    reinterpret_cast<uint32_t*>(dst)[k] = sm.stage[r][k];
  }
}

__device__ __forceinline__ void stage_code(Smem& sm, int r, int c, int bits, unsigned u) {
  const int bit = c * bits;
  atomicOr(&sm.stage[r][bit >> 5], u << (bit & 31));
}

__device__ void clear_stage(Smem& sm, const TQ& q, int n) {
  const int wpr = q.row / 4;
  for (int w = threadIdx.x; w < n * wpr; w += kThreads) sm.stage[w / wpr][w % wpr] = 0u;
}

// Tokens [t_begin, t_begin + count) of one tensor, quantized along a per-token,
// per-tensor or FP8 axis.
__device__ void quantize_rows(const KvqView& v, const Src& s, const AppendCtx& a, const TQ& q,
                              Smem& sm, int t_begin, int count) {
  const int D = v.D;
  for (int sub = 0; sub < count; sub += kSub) {
    const int n = min(kSub, count - sub);
    const int t0 = t_begin + sub;
    for (int e = threadIdx.x; e < n * D; e += kThreads) sm.xs[e / D][e % D] = src_value(v, s, a, t0 + e / D, e % D);
    clear_stage(sm, q, n);
    __syncthreads();
    if (q.axis == KVQ_PER_TOKEN) {
      const int g = q.group;
      for (int e = threadIdx.x; e < n * q.ng; e += kThreads) {
        const int r = e / q.ng, grp = e % q.ng;
        float mn = sm.xs[r][grp * g], mx = mn, am = fabsf(mn);
        for (int c = grp * g + 1; c < (grp + 1) * g; ++c) {
          const float x = sm.xs[r][c];
          mn = fminf(mn, x);
          mx = fmaxf(mx, x);
          am = fmaxf(am, fabsf(x));
        }
        float sc;
        if (q.mode == KVQ_ASYM_MINMAX) {
          sc = asym_scale(mn, mx, q.bits);
        } else {
          sc = sym_scale(am, q.bits);
          mn = 0.f;
        }
        sm.gs[r][grp] = sc;
        sm.gm[r][grp] = mn;
        uint8_t* page = page_of(v, a.b, t0 + r);
        if (page) {
          float* meta = reinterpret_cast<float*>(page + (long long)a.h * v.head_bytes + q.off_meta +
                                                 ((t0 + r) % v.P) * q.ng * q.nmeta * 4);
          meta[grp] = sc;
          if (q.nmeta == 2) meta[q.ng + grp] = mn;
        }
      }
      __syncthreads();
    }
    for (int e = threadIdx.x; e < n * D; e += kThreads) {
      const int r = e / D, c = e % D;
      const float x = sm.xs[r][c];
      unsigned u;
      if (q.fmt == KVQ_FP8_E4M3) {
        u = fp8_code(x, q.static_scale[a.h]);
      } else if (q.axis == KVQ_PER_TENSOR) {
        u = stored_code(sym_code(x, q.static_scale[a.h], q.bits), q.bits, KVQ_SYM_ABSMAX);
      } else {
        const int grp = c / q.group;
        const int code = q.mode == KVQ_ASYM_MINMAX ? asym_code(x, sm.gm[r][grp], sm.gs[r][grp], q.bits)
                                                   : sym_code(x, sm.gs[r][grp], q.bits);
        u = stored_code(code, q.bits, q.mode);
      }
      stage_code(sm, r, c, q.bits, u);
    }
    __syncthreads();
    flush_stage(v, a, q, sm, t0, n);
    __syncthreads();
  }
}

// Keys of tokens [t_begin, t_begin + count), count a multiple of G, quantized per
// channel over groups of G tokens aligned to multiples of G.
__device__ void quantize_key_channels(const KvqView& v, const Src& s, const AppendCtx& a,
                                      const TQ& q, Smem& sm, int t_begin, int count) {
  const int D = v.D, G = q.group;
  const int lanes = kThreads / D;
  const int c = threadIdx.x % D, lane = threadIdx.x / D;
  for (int g0 = t_begin; g0 < t_begin + count; g0 += G) {
    float mn = INFINITY, mx = -INFINITY;
    for (int t = g0 + lane; t < g0 + G; t += lanes) {
      const float x = src_value(v, s, a, t, c);
      mn = fminf(mn, x);
      mx = fmaxf(mx, x);
    }
    sm.cmin[threadIdx.x] = mn;
    sm.cmax[threadIdx.x] = mx;
    __syncthreads();
    if (lane == 0) {
      for (int l = 1; l < lanes; ++l) {
        mn = fminf(mn, sm.cmin[l * D + c]);
        mx = fmaxf(mx, sm.cmax[l * D + c]);
      }
      float sc;
      if (q.mode == KVQ_ASYM_MINMAX) {
        sc = asym_scale(mn, mx, q.bits);
      } else {
        sc = sym_scale(fmaxf(fabsf(mn), fabsf(mx)), q.bits);
        mn = 0.f;
      }
      sm.ch_s[c] = sc;
      sm.ch_m[c] = mn;
      uint8_t* page = page_of(v, a.b, g0);
      if (page) {
        const int slot = (g0 % v.P) / G;
        float* meta = reinterpret_cast<float*>(page + (long long)a.h * v.head_bytes + q.off_meta +
                                               (long long)slot * D * q.nmeta * 4);
        meta[c] = sc;
        if (q.nmeta == 2) meta[D + c] = mn;
      }
    }
    __syncthreads();
    for (int sub = 0; sub < G; sub += kSub) {
      const int n = min(kSub, G - sub);
      const int t0 = g0 + sub;
      clear_stage(sm, q, n);
      __syncthreads();
      for (int e = threadIdx.x; e < n * D; e += kThreads) {
        const int r = e / D, cc = e % D;
        const float x = src_value(v, s, a, t0 + r, cc);
        const int code = q.mode == KVQ_ASYM_MINMAX ? asym_code(x, sm.ch_m[cc], sm.ch_s[cc], q.bits)
                                                   : sym_code(x, sm.ch_s[cc], q.bits);
        stage_code(sm, r, cc, q.bits, stored_code(code, q.bits, q.mode));
      }
      __syncthreads();
      flush_stage(v, a, q, sm, t0, n);
      __syncthreads();
    }
  }
}

__device__ TQ key_q(const KvqView& v) {
  TQ q;
  q.fmt = v.kfmt; q.mode = v.kmode; q.axis = v.kaxis; q.group = v.kgroup; q.bits = v.kbits;
  q.nmeta = v.k_nmeta; q.ng = v.k_ng; q.off_codes = 0; q.off_meta = v.off_km; q.row = v.krow;
  q.static_scale = v.k_scale;
  return q;
}

__device__ TQ value_q(const KvqView& v) {
  TQ q;
  q.fmt = v.vfmt; q.mode = v.vmode; q.axis = v.vaxis; q.group = v.vgroup; q.bits = v.vbits;
  q.nmeta = v.v_nmeta; q.ng = v.v_ng; q.off_codes = v.off_vc; q.off_meta = v.off_vm; q.row = v.vrow;
  q.static_scale = v.v_scale;
  return q;
}

__device__ void quantize_block(const KvqView& v, const Src& ks, const Src& vs, const AppendCtx& a,
                               Smem& sm, int t_begin, int count) {
  const TQ kq = key_q(v), vq = value_q(v);
  if (kq.axis == KVQ_PER_CHANNEL) {
    quantize_key_channels(v, ks, a, kq, sm, t_begin, count);
  } else {
    quantize_rows(v, ks, a, kq, sm, t_begin, count);
  }
  quantize_rows(v, vs, a, vq, sm, t_begin, count);
}

__global__ void __launch_bounds__(kThreads) append_kernel(KvqView v, const void* k_new,
                                                           const void* v_new, int n_stride,
                                                           const int32_t* n_per_seq) {
  __shared__ Smem sm;
  const int unit = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int T0 = v.seq_lens[b];
  const int n = n_per_seq ? n_per_seq[b] : n_stride;
  if (n <= 0) return;
  const long long cap = (long long)v.max_pages * v.P;
  if (T0 < 0 || n > n_stride || (long long)T0 + n > cap) {
    if (unit == 0 && h == 0 && threadIdx.x == 0) atomicOr(v.status, KVQ_DEV_OVERFLOW);
    return;
  }
  const int T1 = T0 + n;
  AppendCtx a;
  a.b = b;
  a.h = h;
  a.T0 = T0;
  a.n_stride = n_stride;
  const Src ks{v.k_win, k_new}, vs{v.v_win, v_new};
  if (v.R > 0) {
    const int jb0 = T0 / v.R, jb1 = T1 / v.R;
    a.wbase = jb0 * v.R;
    if (unit < jb1 - jb0) quantize_block(v, ks, vs, a, sm, (jb0 + unit) * v.R, v.R);
    if (unit == 0) {
      __syncthreads();
      const int base = jb1 * v.R;
      const int t_lo = max(base, T0);
      const int D = v.D;
      for (int e = threadIdx.x; e < (T1 - t_lo) * D; e += kThreads) {
        const int t = t_lo + e / D, c = e % D;
        const long long si = (((long long)b * n_stride + (t - T0)) * v.Hkv + h) * D + c;
        const long long di = (((long long)b * v.R + (t - base)) * v.Hkv + h) * D + c;
        store_src(v.k_win, di, load_src(k_new, si, v.src_bf16), v.src_bf16);
        store_src(v.v_win, di, load_src(v_new, si, v.src_bf16), v.src_bf16);
      }
    }
  } else {
    a.wbase = 0;
    const int t_lo = T0 + unit * kUnitTok;
    if (t_lo < T1) quantize_block(v, ks, vs, a, sm, t_lo, min(kUnitTok, T1 - t_lo));
  }
}

__global__ void advance_lengths_kernel(KvqView v, int n_stride, const int32_t* n_per_seq) {
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= v.batch) return;
  const int T0 = v.seq_lens[b];
  const int n = n_per_seq ? n_per_seq[b] : n_stride;
  if (n <= 0 || T0 < 0 || n > n_stride || (long long)T0 + n > (long long)v.max_pages * v.P) return;
  v.seq_lens[b] = T0 + n;
}

// ------------------------------------------------------------------- dequantize

__global__ void dequantize_kernel(KvqView v, int seq, int t0, float* k_out, float* v_out) {
  const int t = t0 + blockIdx.x, h = blockIdx.y;
  const int T = v.seq_lens[seq];
  const int nq = n_quantized(T, v.R);
  for (int c = threadIdx.x; c < v.D; c += blockDim.x) {
    const long long o = ((long long)blockIdx.x * v.Hkv + h) * v.D + c;
    float kx = 0.f, vx = 0.f;
    if (t < T && t >= nq) {
      const long long wi = (((long long)seq * v.R + (t - nq)) * v.Hkv + h) * v.D + c;
      kx = load_src(v.k_win, wi, v.src_bf16);
      vx = load_src(v.v_win, wi, v.src_bf16);
    } else if (t < T) {
      const uint8_t* page = page_of(v, seq, t);
      if (page) {
        const uint8_t* hb = page + (long long)h * v.head_bytes;
        const int slot = t % v.P;
        const unsigned ku = get_code(hb + slot * v.krow, c, v.kbits);
        if (v.kfmt == KVQ_FP8_E4M3) {
          kx = __fmul_rn(fp8_e4m3_to_float(ku), v.k_scale[h]);
        } else if (v.kaxis == KVQ_PER_TENSOR) {
          kx = dequant_sym(signed_code(ku, v.kbits, KVQ_SYM_ABSMAX), v.k_scale[h]);
        } else {
          const float* meta;
          float s, mn = 0.f;
          if (v.kaxis == KVQ_PER_TOKEN) {
            meta = reinterpret_cast<const float*>(hb + v.off_km + slot * v.k_ng * v.k_nmeta * 4);
            const int grp = c / v.kgroup;
            s = meta[grp];
            if (v.k_nmeta == 2) mn = meta[v.k_ng + grp];
          } else {
            const int g0 = (t / v.kgroup) * v.kgroup;
            const uint8_t* gp = page_of(v, seq, g0);
            meta = gp ? reinterpret_cast<const float*>(gp + (long long)h * v.head_bytes + v.off_km +
                                                       (long long)((g0 % v.P) / v.kgroup) * v.D * v.k_nmeta * 4)
                      : nullptr;
            s = meta ? meta[c] : 0.f;
            if (meta && v.k_nmeta == 2) mn = meta[v.D + c];
          }
          const int code = signed_code(ku, v.kbits, v.kmode);
          kx = v.kmode == KVQ_ASYM_MINMAX ? dequant_asym(code, s, mn) : dequant_sym(code, s);
        }
        const unsigned vu = get_code(hb + v.off_vc + slot * v.vrow, c, v.vbits);
        if (v.vfmt == KVQ_FP8_E4M3) {
          vx = __fmul_rn(fp8_e4m3_to_float(vu), v.v_scale[h]);
        } else if (v.vaxis == KVQ_PER_TENSOR) {
          vx = dequant_sym(signed_code(vu, v.vbits, KVQ_SYM_ABSMAX), v.v_scale[h]);
        } else {
          const float* meta = reinterpret_cast<const float*>(hb + v.off_vm + slot * v.v_ng * v.v_nmeta * 4);
          const int grp = c / v.vgroup;
          const int code = signed_code(vu, v.vbits, v.vmode);
          vx = v.vmode == KVQ_ASYM_MINMAX ? dequant_asym(code, meta[grp], meta[v.v_ng + grp])
                                          : dequant_sym(code, meta[grp]);
        }
      }
    }
    k_out[o] = kx;
    v_out[o] = vx;
  }
}

// -------------------------------------------------------------------- calibrate

__global__ void absmax_kernel(const void* src, long long n_tokens, int Hkv, int D, int bf16,
                              unsigned* acc) {
  __shared__ float red[32];
  const int h = blockIdx.y;
  float m = 0.f;
  const long long n = n_tokens * D;
  for (long long e = (long long)blockIdx.x * blockDim.x + threadIdx.x; e < n;
       e += (long long)gridDim.x * blockDim.x) {
    const long long t = e / D, c = e % D;
    m = fmaxf(m, fabsf(load_src(src, (t * Hkv + h) * D + c, bf16)));
  }
  for (int o = 16; o; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
  __syncthreads();
  if (threadIdx.x < 32) {
    m = threadIdx.x < (blockDim.x >> 5) ? red[threadIdx.x] : 0.f;
    for (int o = 16; o; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    if (threadIdx.x == 0) atomicMax(acc + h, __float_as_uint(m));  // m >= 0: bit order = value order
  }
}

__global__ void scale_finalize_kernel(float* scale, int Hkv, float qmax) {
  const int h = blockIdx.x * blockDim.x + threadIdx.x;
  if (h < Hkv) scale[h] = __fdiv_rn(scale[h], qmax);
}

}  // namespace

kvq_status launch_append(const KvqView& v, const void* k_new, const void* v_new, int n_new,
                         const int32_t* n_new_per_seq, cudaStream_t st) {
  const int units = v.R > 0 ? n_new / v.R + 1 : (n_new + kUnitTok - 1) / kUnitTok;
  dim3 grid(units, v.Hkv, v.batch);
  append_kernel<<<grid, kThreads, 0, st>>>(v, k_new, v_new, n_new, n_new_per_seq);
  advance_lengths_kernel<<<(v.batch + 127) / 128, 128, 0, st>>>(v, n_new, n_new_per_seq);
  return cudaGetLastError() == cudaSuccess ? KVQ_OK : KVQ_ERR_CUDA;
}

kvq_status launch_dequantize(const KvqView& v, int seq, int t0, int t1, float* k_out, float* v_out,
                             cudaStream_t st) {
  dim3 grid(t1 - t0, v.Hkv);
  dequantize_kernel<<<grid, 128, 0, st>>>(v, seq, t0, k_out, v_out);
  return cudaGetLastError() == cudaSuccess ? KVQ_OK : KVQ_ERR_CUDA;
}

kvq_status launch_calibrate(const KvqView& v, const void* src, long long n_tokens, float qmax,
                            float* scale_out, cudaStream_t st) {
  if (cudaMemsetAsync(scale_out, 0, sizeof(float) * v.Hkv, st) != cudaSuccess) return KVQ_ERR_CUDA;
  if (n_tokens > 0) {
    const long long n = n_tokens * v.D;
    const int blocks = (int)min((n + 255) / 256, 1024LL);
    absmax_kernel<<<dim3(blocks, v.Hkv), 256, 0, st>>>(src, n_tokens, v.Hkv, v.D, v.src_bf16,
                                                       reinterpret_cast<unsigned*>(scale_out));
  }
  scale_finalize_kernel<<<(v.Hkv + 127) / 128, 128, 0, st>>>(scale_out, v.Hkv, qmax);
  return cudaGetLastError() == cudaSuccess ? KVQ_OK : KVQ_ERR_CUDA;
}

}  // namespace kvq
