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
// Two launches: the fold kernel, one CTA per (fold block, kv-head, sequence),
// quantizes every window that fills (reading the old window and the new rows);
// then one CTA per sequence writes the remaining new tokens into the window and
// advances seq_lens, so window slots are never read and overwritten out of order.
#include "kvq_host.h"
#include "kvq_internal.cuh"

namespace kvq {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kSub = 16;        // tokens staged per sub-chunk
constexpr int kUnitTok = 64;    // tokens per CTA when R == 0
constexpr int kMaxD = 256;
constexpr int kMaxGroups = 16;  // PER_TOKEN groups per token (D/g with g >= 16)
constexpr int kStageMax = 64 * 1024;  // shared-memory staging of one fold block

struct Src {
  const void* win;    // [B][R][Hkv][D]
  const void* fresh;  // [B][n_new][Hkv][D]
  const void* staged; // the block's rows [count][D] in shared memory, or nullptr
};

struct TQ {  // one tensor's quantization parameters
  int fmt, mode, axis, group, bits, nmeta, ng, off_codes, off_meta, row;
  const float* static_scale;
};

struct AppendCtx {
  int b, h, T0, wbase, n_stride, st_t0;
};

__device__ __forceinline__ float src_value(const KvqView& v, const Src& s, const AppendCtx& a,
                                           int t, int c) {
  if (s.staged) return load_src(s.staged, (long long)(t - a.st_t0) * v.D + c, v.src_bf16);
  if (t < a.T0) {
    const long long i = (((long long)a.b * v.R + (t - a.wbase)) * v.Hkv + a.h) * v.D + c;
    return load_src(s.win, i, v.src_bf16);
  }
  const long long i = (((long long)a.b * a.n_stride + (t - a.T0)) * v.Hkv + a.h) * v.D + c;
  return load_src(s.fresh, i, v.src_bf16);
}

struct Smem {
  float xs[kSub][kMaxD + 1];  // +1: a thread per row reads a column without bank conflicts
  uint32_t stage[kSub][kMaxD * 8 / 32];
  float gs[kSub][kMaxGroups];
  float gr[kSub][kMaxGroups];  // 1 / scale, rounded to nearest
  float gm[kSub][kMaxGroups];
  float cmin[kThreads];
  float cmax[kThreads];
  uint8_t* rowp[kSub];  // head block of each staged row (nullptr: bad page)
  int rslot[kSub];      // its slot within the page
  float ch_s[kMaxD];
  float ch_r[kMaxD];
  float ch_m[kMaxD];
};

__device__ __forceinline__ int log2i(int x) { return __ffs(x) - 1; }  // x a power of two

// Head-block address and page slot of each of the n rows of a sub-chunk, once.
__device__ void load_rows(const KvqView& v, const AppendCtx& a, Smem& sm, int t0, int n) {
  if (threadIdx.x < n) {
    const int t = t0 + threadIdx.x;
    uint8_t* page = page_of(v, a.b, t);
    sm.rowp[threadIdx.x] = page ? page + (long long)a.h * v.head_bytes : nullptr;
    sm.rslot[threadIdx.x] = t % v.P;
  }
}

// Pack the codes of the n rows staged in sm.stage into the pages.
__device__ void flush_stage(const KvqView& v, const TQ& q, Smem& sm, int n) {
  const int wpr = q.row >> 2, lw = log2i(wpr);
  for (int w = threadIdx.x; w < (n << lw); w += kThreads) {
    const int r = w >> lw, k = w & (wpr - 1);
    uint8_t* hb = sm.rowp[r];
    if (!hb) continue;
    reinterpret_cast<uint32_t*>(hb + q.off_codes + sm.rslot[r] * q.row)[k] = sm.stage[r][k];
  }
}

__device__ __forceinline__ void stage_code(Smem& sm, int r, int c, int bits, unsigned u) {
  const int bit = c * bits;
  atomicOr(&sm.stage[r][bit >> 5], u << (bit & 31));
}

__device__ void clear_stage(Smem& sm, const TQ& q, int n) {
  const int wpr = q.row >> 2, lw = log2i(wpr);
  for (int w = threadIdx.x; w < (n << lw); w += kThreads) sm.stage[w >> lw][w & (wpr - 1)] = 0u;
}

// Tokens [t_begin, t_begin + count) of one tensor, quantized along a per-token,
// per-tensor or FP8 axis.  D and the group sizes are powers of two.
__device__ void quantize_rows(const KvqView& v, const Src& s, const AppendCtx& a, const TQ& q,
                              Smem& sm, int t_begin, int count) {
  const int D = v.D, lD = log2i(D);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int sub = 0; sub < count; sub += kSub) {
    const int n = min(kSub, count - sub);
    const int t0 = t_begin + sub;
    for (int e = threadIdx.x; e < (n << lD); e += kThreads)
      sm.xs[e >> lD][e & (D - 1)] = src_value(v, s, a, t0 + (e >> lD), e & (D - 1));
    clear_stage(sm, q, n);
    load_rows(v, a, sm, t0, n);
    __syncthreads();
    if (q.axis == KVQ_PER_TOKEN) {
      // one warp per row: lanes scan the group's channels, shuffles reduce
      const int g = q.group, lg = log2i(g);
      const int width = g < 32 ? g : 32;  // lanes sharing one group
      for (int r = warp; r < n; r += kThreads / 32) {
        for (int grp0 = 0; grp0 < q.ng; grp0 += 32 / width) {
          const int grp = grp0 + lane / width;
          float mn = INFINITY, mx = -INFINITY, am = 0.f;
          if (grp < q.ng) {
            for (int c = (grp << lg) + (lane & (width - 1)); c < ((grp + 1) << lg); c += width) {
              const float x = sm.xs[r][c];
              mn = fminf(mn, x);
              mx = fmaxf(mx, x);
              am = fmaxf(am, fabsf(x));
            }
          }
          for (int o = width >> 1; o; o >>= 1) {
            mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, o));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
            am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, o));
          }
          if ((lane & (width - 1)) == 0 && grp < q.ng) {
            float sc, gm;
            group_scale(mn, mx, am, q.mode == KVQ_ASYM_MINMAX, q.bits, v.meta16, sc, gm);
            sm.gs[r][grp] = sc;
            sm.gr[r][grp] = sc > 0.f ? __frcp_rn(sc) : 0.f;
            sm.gm[r][grp] = gm;
            uint8_t* hb = sm.rowp[r];
            if (hb) {
              uint8_t* meta = hb + q.off_meta + sm.rslot[r] * q.ng * q.nmeta * v.mb;
              store_meta(meta, grp, sc, v.meta16);
              if (q.nmeta == 2) store_meta(meta, q.ng + grp, gm, v.meta16);
            }
          }
        }
      }
      __syncthreads();
    }
    const int lg = q.axis == KVQ_PER_TOKEN ? log2i(q.group) : 0;
    const float ss = q.axis == KVQ_PER_TENSOR || is_fp8(q.fmt) ? q.static_scale[a.h] : 0.f;
    const float sr = ss > 0.f ? __frcp_rn(ss) : 0.f;
    for (int e = threadIdx.x; e < (n << lD); e += kThreads) {
      const int r = e >> lD, c = e & (D - 1);
      const float x = sm.xs[r][c];
      unsigned u;
      if (is_fp8(q.fmt)) {
        u = fp8_code(x, ss, q.fmt);
      } else if (q.axis == KVQ_PER_TENSOR) {
        u = stored_code(sym_code_r(x, ss, sr, q.bits), q.bits, KVQ_SYM_ABSMAX);
      } else {
        const int grp = c >> lg;
        const int code = q.mode == KVQ_ASYM_MINMAX
                             ? asym_code_r(x, sm.gm[r][grp], sm.gs[r][grp], sm.gr[r][grp], q.bits)
                             : sym_code_r(x, sm.gs[r][grp], sm.gr[r][grp], q.bits);
        u = stored_code(code, q.bits, q.mode);
      }
      stage_code(sm, r, c, q.bits, u);
    }
    __syncthreads();
    flush_stage(v, q, sm, n);
    __syncthreads();
  }
}

// Keys of tokens [t_begin, t_begin + count), count a multiple of G, quantized per
// channel over groups of G tokens aligned to multiples of G.
__device__ void quantize_key_channels(const KvqView& v, const Src& s, const AppendCtx& a,
                                      const TQ& q, Smem& sm, int t_begin, int count) {
  const int D = v.D, G = q.group, lD = log2i(D);
  const int lanes = kThreads >> lD;
  const int c = threadIdx.x & (D - 1), lane = threadIdx.x >> lD;
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
      group_scale(mn, mx, fmaxf(fabsf(mn), fabsf(mx)), q.mode == KVQ_ASYM_MINMAX, q.bits, v.meta16, sc, mn);
      sm.ch_s[c] = sc;
      sm.ch_r[c] = sc > 0.f ? __frcp_rn(sc) : 0.f;
      sm.ch_m[c] = mn;
      uint8_t* page = page_of(v, a.b, g0);
      if (page) {
        const int slot = (g0 % v.P) / G;
        uint8_t* meta = page + (long long)a.h * v.head_bytes + q.off_meta + (long long)slot * D * q.nmeta * v.mb;
        store_meta(meta, c, sc, v.meta16);
        if (q.nmeta == 2) store_meta(meta, D + c, mn, v.meta16);
      }
    }
    __syncthreads();
    for (int sub = 0; sub < G; sub += kSub) {
      const int n = min(kSub, G - sub);
      const int t0 = g0 + sub;
      clear_stage(sm, q, n);
      load_rows(v, a, sm, t0, n);
      __syncthreads();
      for (int e = threadIdx.x; e < (n << lD); e += kThreads) {
        const int r = e >> lD, cc = e & (D - 1);
        const float x = src_value(v, s, a, t0 + r, cc);
        const int code = q.mode == KVQ_ASYM_MINMAX
                             ? asym_code_r(x, sm.ch_m[cc], sm.ch_s[cc], sm.ch_r[cc], q.bits)
                             : sym_code_r(x, sm.ch_s[cc], sm.ch_r[cc], q.bits);
        stage_code(sm, r, cc, q.bits, stored_code(code, q.bits, q.mode));
      }
      __syncthreads();
      flush_stage(v, q, sm, n);
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

// 16-byte global -> shared copy that completes asynchronously (cp.async, sm_80+);
// cp.async.wait_all makes the thread's copies visible to itself.
__device__ __forceinline__ void cp_async16(void* smem_dst, const void* gsrc) {
  const unsigned d = static_cast<unsigned>(__cvta_generic_to_shared(smem_dst));
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(d), "l"(gsrc) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;\n" ::: "memory"); }

// Copy the source rows (window or new tokens) of tokens [t_begin, t_begin + count)
// of one head into shared memory as 16-byte asynchronous copies, K rows then V
// rows.  `between` runs while the copies are in flight, so the global reads it
// makes overlap theirs.  The loop stays rolled: a launch runs this code once, so
// its size, not its instruction count, sets its cost.
template <typename Between>
__device__ void stage_block(const KvqView& v, const AppendCtx& a, const void* k_new, const void* v_new,
                            int t_begin, int count, unsigned char* dst, Between&& between) {
  const int row = v.D * (v.src_bf16 ? 2 : 4);
  const int lp = log2i(row >> 4);  // 16-byte pieces per row: 2^lp
  const int per_tensor = count << lp;
  const int n = 2 * per_tensor;
#pragma unroll 1
  for (int e = threadIdx.x; e < n; e += kThreads) {
    const int tensor = e >= per_tensor;
    const int rem = tensor ? e - per_tensor : e;
    const int r = rem >> lp, k = rem & ((1 << lp) - 1);
    const int t = t_begin + r;
    const unsigned char* src;
    if (t < a.T0) {
      const long long i = (((long long)a.b * v.R + (t - a.wbase)) * v.Hkv + a.h) * row;
      src = static_cast<const unsigned char*>(tensor ? v.v_win : v.k_win) + i;
    } else {
      const long long i = (((long long)a.b * a.n_stride + (t - a.T0)) * v.Hkv + a.h) * row;
      src = static_cast<const unsigned char*>(tensor ? v_new : k_new) + i;
    }
    cp_async16(dst + 16 * e, src + 16 * k);  // piece e of the block sits at byte 16 e
  }
  between();
  cp_async_wait_all();
  __syncthreads();
}

// ---- parallel fold of one R-token block of one kv-head (R <= kMaxFold)
//
// The block's K rows then V rows are staged in shared memory in the source dtype,
// with the page address of every token looked up while the rows are in flight.
// Per-channel keys: each key group's channel scales, then the code words, one
// thread per word column with its channels' parameters in registers across the
// group's tokens.  Rows (values, per-token keys, per-tensor and FP8 tensors):
// D/16 lanes per token, 16 consecutive channels per lane, one code word at a time.
// A launch runs this code about once, from cold instruction caches, so loops stay
// rolled.  Scales and codes follow the rules of the sub-chunk path exactly, so the
// bytes are identical.
constexpr int kMaxFold = 256;
constexpr int kCPL = 16;  // channels per lane in the row fold (every token group holds whole lanes)

struct FoldSmem {
  uint8_t* rowp[kMaxFold];  // head block of each token of the block (nullptr: bad page)
  int rslot[kMaxFold];      // its slot within the page
  float cmin[kThreads], cmax[kThreads];
  float ch_s[kMaxD], ch_r[kMaxD], ch_m[kMaxD];
};

template <bool BF16>
__device__ __forceinline__ float staged_value(const unsigned char* rows, int t, int c, int D) {
  if constexpr (BF16) {
    const unsigned short u = reinterpret_cast<const unsigned short*>(rows)[t * D + c];
    return __uint_as_float(static_cast<unsigned>(u) << 16);
  } else {
    return reinterpret_cast<const float*>(rows)[t * D + c];
  }
}

// N consecutive source values of staged row t from channel c0 (the address is a
// multiple of N * 2 bytes for bf16, N * 4 for fp32).
template <int N, bool BF16>
__device__ __forceinline__ void load_chunk(const unsigned char* rows, int t, int c0, int D, float (&x)[N]) {
  if constexpr (BF16) {
    const unsigned char* p = rows + (t * D + c0) * 2;
    if constexpr (N == 4) {
      const uint2 u = *reinterpret_cast<const uint2*>(p);
      x[0] = __uint_as_float(u.x << 16);
      x[1] = __uint_as_float(u.x & 0xffff0000u);
      x[2] = __uint_as_float(u.y << 16);
      x[3] = __uint_as_float(u.y & 0xffff0000u);
    } else {
#pragma unroll
      for (int j = 0; j < N / 8; ++j) {
        const uint4 u = reinterpret_cast<const uint4*>(p)[j];
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          x[8 * j + 2 * i] = __uint_as_float(w[i] << 16);
          x[8 * j + 2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
        }
      }
    }
  } else {
    const float4* p = reinterpret_cast<const float4*>(rows + (t * D + c0) * 4);
#pragma unroll
    for (int j = 0; j < N / 4; ++j) {
      const float4 f = p[j];
      x[4 * j] = f.x;
      x[4 * j + 1] = f.y;
      x[4 * j + 2] = f.z;
      x[4 * j + 3] = f.w;
    }
  }
}

// rint(fl32(y * r)) with r = fl32(1 / s) equals rint(fl32(y / s)) unless a
// half-integer lies between the two: both are within 3 * 2^-24 |y / s| of the exact
// quotient.  A product farther than kNearHalf |q| (over five times that distance) from
// every half-integer is therefore safe; a nearer one, or one that is not a finite
// number, takes the exact rule.  Besides the band's own width, bf16 sources put x / s
// exactly on a half-integer fairly often (about 0.4% of the codes of normal data).
constexpr float kNearHalf = 9.5367431640625e-07f;  // 2^-20

// One code word: the BITS-bit stored codes of N elements with scales s,
// reciprocals r and minimums m, equal to those of sym_code_r / asym_code_r.  The
// quotient comes from the reciprocal; the few elements within kNearHalf |q| of a
// half-integer (or not finite) take the IEEE division, inline, so a warp pays for
// it only at the element positions where one of its lanes needs it.
template <int N, int BITS>
__device__ __forceinline__ uint32_t pack_codes(const float (&x)[N], const float (&s)[N], const float (&r)[N],
                                               const float (&m)[N], bool asym) {
  const float hi = static_cast<float>(asym ? (1 << BITS) - 1 : (1 << (BITS - 1)) - 1);
  const float lo = asym ? 0.f : -hi;
  const unsigned off = (asym || BITS == 8) ? 0u : (1u << (BITS - 1));  // offset binary for sym INT2 / INT4
  uint32_t w = 0u;
#pragma unroll
  for (int i = 0; i < N; ++i) {
    const float y = asym ? __fsub_rn(x[i], m[i]) : x[i];
    const float q = __fmul_rn(y, r[i]);
    float c = rintf(q);
    if (!(fabsf(__fsub_rn(fabsf(__fsub_rn(q, c)), 0.5f)) > __fmul_rn(kNearHalf, fabsf(q))))
      c = rintf(__fdiv_rn(y, s[i]));
    const int code = (!asym && s[i] == 0.f) ? 0 : static_cast<int>(fminf(fmaxf(c, lo), hi));
    w |= ((static_cast<unsigned>(code) + off) & ((1u << BITS) - 1u)) << (i * BITS);
  }
  return w;
}

template <int N>
__device__ __forceinline__ void tree_minmax(const float (&x)[N], float& mn, float& mx, float& am) {
  float a[N / 2], b[N / 2], c[N / 2];
#pragma unroll
  for (int i = 0; i < N / 2; ++i) {
    a[i] = fminf(x[i], x[i + N / 2]);
    b[i] = fmaxf(x[i], x[i + N / 2]);
    c[i] = fmaxf(fabsf(x[i]), fabsf(x[i + N / 2]));
  }
#pragma unroll
  for (int w = N / 4; w >= 1; w >>= 1) {
#pragma unroll
    for (int i = 0; i < w; ++i) {
      a[i] = fminf(a[i], a[i + w]);
      b[i] = fmaxf(b[i], b[i + w]);
      c[i] = fmaxf(c[i], c[i + w]);
    }
  }
  mn = a[0];
  mx = b[0];
  am = c[0];
}

// Rows of one tensor with BITS-bit codes (8 for FP8).
template <int BITS, bool BF16>
__device__ __forceinline__ void fold_rows_t(const KvqView& v, const TQ& q, const unsigned char* rows,
                                            FoldSmem& fs, int R) {
  constexpr int kCPW = 32 / BITS;       // codes per word
  constexpr int kWords = kCPL / kCPW;   // words per lane: 1, 2 or 4
  const int D = v.D, lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int lpt = D / kCPL, tpw = 32 / lpt;  // lanes per token, tokens per warp
  const int sub = lane % lpt, tok = lane / lpt;
  const bool fp8 = is_fp8(q.fmt);
  const bool stat = fp8 || q.axis == KVQ_PER_TENSOR;
  const bool asym = !stat && q.mode == KVQ_ASYM_MINMAX;
  const float ss = stat ? q.static_scale[0] : 0.f;
  const float sr = ss > 0.f ? __frcp_rn(ss) : 0.f;
  const int lpg = stat ? 1 : q.group / kCPL;  // lanes per group (group = lpg * 16 channels)
#pragma unroll 1
  for (int t0 = warp * tpw; t0 < R; t0 += kWarps * tpw) {
    const int t = t0 + tok;
    const bool ok = t < R;
    float gs = ss, gr = sr, gm = 0.f;
    if (!stat) {
      float x[kCPL];
      if (ok) {
        load_chunk<kCPL, BF16>(rows, t, sub * kCPL, D, x);
      } else {
#pragma unroll
        for (int i = 0; i < kCPL; ++i) x[i] = 0.f;
      }
      float mn, mx, am;
      tree_minmax<kCPL>(x, mn, mx, am);
      for (int o = 1; o < lpg; o <<= 1) {
        mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, o));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, o));
      }
      group_scale(mn, mx, am, asym, BITS, v.meta16, gs, gm);
      gr = gs > 0.f ? __frcp_rn(gs) : 0.f;
    }
    uint8_t* hb = ok ? fs.rowp[t] : nullptr;
    if (!hb) continue;
    const int slot = fs.rslot[t];
    if (!stat && sub % lpg == 0) {
      uint8_t* meta = hb + q.off_meta + slot * q.ng * q.nmeta * v.mb;
      store_meta(meta, sub / lpg, gs, v.meta16);
      if (q.nmeta == 2) store_meta(meta, q.ng + sub / lpg, gm, v.meta16);
    }
    uint32_t* dst = reinterpret_cast<uint32_t*>(hb + q.off_codes + slot * q.row) + sub * kWords;
    float sc[kCPW], r[kCPW], m[kCPW];
#pragma unroll
    for (int i = 0; i < kCPW; ++i) {
      sc[i] = gs;
      r[i] = gr;
      m[i] = gm;
    }
#pragma unroll 1
    for (int j = 0; j < kWords; ++j) {
      const int c0 = sub * kCPL + j * kCPW;
      float x[kCPW];
      load_chunk<kCPW, BF16>(rows, t, c0, D, x);
      uint32_t w = 0u;
      if (fp8) {
#pragma unroll
        for (int i = 0; i < kCPW; ++i) w |= fp8_code(x[i], ss, q.fmt) << (8 * i);
      } else {
        w = pack_codes<kCPW, BITS>(x, sc, r, m, asym);
      }
      dst[j] = w;
    }
  }
}

template <bool BF16>
__device__ __forceinline__ void fold_rows(const KvqView& v, const TQ& q, const unsigned char* rows, FoldSmem& fs,
                                          int R) {
  if (q.bits == 2) {
    fold_rows_t<2, BF16>(v, q, rows, fs, R);
  } else if (q.bits == 4) {
    fold_rows_t<4, BF16>(v, q, rows, fs, R);
  } else {
    fold_rows_t<8, BF16>(v, q, rows, fs, R);
  }
}

// Keys per channel over groups of G tokens of the block, BITS-bit codes.
template <int BITS, bool BF16>
__device__ __forceinline__ void fold_key_channels_t(const KvqView& v, const TQ& q, const unsigned char* rows,
                                                    FoldSmem& fs, int tb, int R) {
  constexpr int kCPW = 32 / BITS;  // channels per code word
  const int D = v.D, G = q.group;
  const int parts = kThreads / D;  // threads per channel for the scans (1, 2 or 4)
  const int c = threadIdx.x % D, part = threadIdx.x / D;
  const int wpr = D / kCPW;        // code words per row
  const int k = threadIdx.x % wpr, tl = threadIdx.x / wpr, ntl = kThreads / wpr;
  const bool asym = q.mode == KVQ_ASYM_MINMAX;
#pragma unroll 1
  for (int g0 = 0; g0 < R; g0 += G) {
    // min and max of channel c over the group's tokens, two chains per thread
    float mn0 = INFINITY, mx0 = -INFINITY, mn1 = INFINITY, mx1 = -INFINITY;
    int t = g0 + part;
#pragma unroll 2
    for (; t + parts < g0 + G; t += 2 * parts) {
      const float x0 = staged_value<BF16>(rows, t, c, D), x1 = staged_value<BF16>(rows, t + parts, c, D);
      mn0 = fminf(mn0, x0);
      mx0 = fmaxf(mx0, x0);
      mn1 = fminf(mn1, x1);
      mx1 = fmaxf(mx1, x1);
    }
    if (t < g0 + G) {
      const float x0 = staged_value<BF16>(rows, t, c, D);
      mn0 = fminf(mn0, x0);
      mx0 = fmaxf(mx0, x0);
    }
    float mn = fminf(mn0, mn1), mx = fmaxf(mx0, mx1);
    fs.cmin[threadIdx.x] = mn;
    fs.cmax[threadIdx.x] = mx;
    __syncthreads();
    if (threadIdx.x < D) {
      for (int p = 1; p < parts; ++p) {
        mn = fminf(mn, fs.cmin[p * D + c]);
        mx = fmaxf(mx, fs.cmax[p * D + c]);
      }
      float sc;
      group_scale(mn, mx, fmaxf(fabsf(mn), fabsf(mx)), asym, BITS, v.meta16, sc, mn);
      fs.ch_s[c] = sc;
      fs.ch_r[c] = sc > 0.f ? __frcp_rn(sc) : 0.f;
      fs.ch_m[c] = mn;
      uint8_t* hb0 = fs.rowp[g0];  // head block of the page holding the group's first token
      if (hb0) {
        const int slot = ((tb + g0) % v.P) / G;
        uint8_t* meta = hb0 + q.off_meta + (long long)slot * D * q.nmeta * v.mb;
        store_meta(meta, c, sc, v.meta16);
        if (q.nmeta == 2) store_meta(meta, D + c, mn, v.meta16);
      }
    }
    __syncthreads();
    // word column k (channels k * kCPW ..) of the group's tokens tl, tl + ntl, ...
    float cs[kCPW], cr[kCPW], cm[kCPW];
#pragma unroll
    for (int i = 0; i < kCPW; i += 4) {
      const float4 s4 = *reinterpret_cast<const float4*>(&fs.ch_s[k * kCPW + i]);
      const float4 r4 = *reinterpret_cast<const float4*>(&fs.ch_r[k * kCPW + i]);
      const float4 m4 = *reinterpret_cast<const float4*>(&fs.ch_m[k * kCPW + i]);
      cs[i] = s4.x; cs[i + 1] = s4.y; cs[i + 2] = s4.z; cs[i + 3] = s4.w;
      cr[i] = r4.x; cr[i + 1] = r4.y; cr[i + 2] = r4.z; cr[i + 3] = r4.w;
      cm[i] = m4.x; cm[i + 1] = m4.y; cm[i + 2] = m4.z; cm[i + 3] = m4.w;
    }
#pragma unroll 1
    for (int tt = g0 + tl; tt < g0 + G; tt += ntl) {
      float x[kCPW];
      load_chunk<kCPW, BF16>(rows, tt, k * kCPW, D, x);
      const uint32_t w = pack_codes<kCPW, BITS>(x, cs, cr, cm, asym);
      uint8_t* hb = fs.rowp[tt];
      if (hb) reinterpret_cast<uint32_t*>(hb + q.off_codes + fs.rslot[tt] * q.row)[k] = w;
    }
    __syncthreads();
  }
}

// Stage the block, look up its pages meanwhile, then fold keys and values.
template <bool BF16>
__device__ __forceinline__ void fold_block(const KvqView& v, const AppendCtx& a, const void* k_new,
                                           const void* v_new, int tb, unsigned char* staged, FoldSmem& fs) {
  const int R = v.R;
  stage_block(v, a, k_new, v_new, tb, R, staged, [&] {
    if (threadIdx.x < R) {
      const int t = tb + threadIdx.x;
      uint8_t* page = page_of(v, a.b, t);
      fs.rowp[threadIdx.x] = page ? page + (long long)a.h * v.head_bytes : nullptr;
      fs.rslot[threadIdx.x] = t % v.P;
    }
  });
  const int row = v.D * (BF16 ? 2 : 4);
  TQ kq = key_q(v), vq = value_q(v);
  kq.static_scale = v.k_scale + a.h;
  vq.static_scale = v.v_scale + a.h;
  if (kq.axis == KVQ_PER_CHANNEL) {
    if (kq.bits == 2) {
      fold_key_channels_t<2, BF16>(v, kq, staged, fs, tb, R);
    } else if (kq.bits == 4) {
      fold_key_channels_t<4, BF16>(v, kq, staged, fs, tb, R);
    } else {
      fold_key_channels_t<8, BF16>(v, kq, staged, fs, tb, R);
    }
  }
#pragma unroll 1
  for (int tensor = kq.axis == KVQ_PER_CHANNEL ? 1 : 0; tensor < 2; ++tensor)
    fold_rows<BF16>(v, tensor ? vq : kq, staged + tensor * R * row, fs, R);
}

__global__ void __launch_bounds__(kThreads) append_kernel(KvqView v, const void* k_new,
                                                           const void* v_new, int n_stride,
                                                           const int32_t* n_per_seq, int stage_ok) {
  __shared__ Smem sm;
  extern __shared__ __align__(16) unsigned char staged[];
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
  a.st_t0 = 0;
  const Src ks{v.k_win, k_new, nullptr}, vs{v.v_win, v_new, nullptr};
  if (v.R > 0) {
    const int jb0 = T0 / v.R, jb1 = T1 / v.R;
    a.wbase = jb0 * v.R;
    if (unit < jb1 - jb0) {
      const int tb = (jb0 + unit) * v.R;
      if (stage_ok) {
        // the whole R-token block fits in shared memory: one parallel pass of loads,
        // then every quantizer pass reads shared memory
        if (v.R <= kMaxFold) {
          __shared__ FoldSmem fs;
          if (v.src_bf16) {
            fold_block<true>(v, a, k_new, v_new, tb, staged, fs);
          } else {
            fold_block<false>(v, a, k_new, v_new, tb, staged, fs);
          }
        } else {
          stage_block(v, a, k_new, v_new, tb, v.R, staged, [] {});
          a.st_t0 = tb;
          const int row = v.D * (v.src_bf16 ? 2 : 4);
          const Src kss{v.k_win, k_new, staged}, vss{v.v_win, v_new, staged + (long long)v.R * row};
          quantize_block(v, kss, vss, a, sm, tb, v.R);
        }
      } else {
        quantize_block(v, ks, vs, a, sm, tb, v.R);
      }
    }
  } else {
    a.wbase = 0;
    const int t_lo = T0 + unit * kUnitTok;
    if (t_lo < T1) quantize_block(v, ks, vs, a, sm, t_lo, min(kUnitTok, T1 - t_lo));
  }
}

// After the folds: write each sequence's remaining new tokens into its window
// (slots from the last fold boundary) and advance seq_lens.  One CTA per
// sequence, so the CTA that updates seq_lens[b] is the only one that reads it.
__global__ void __launch_bounds__(kThreads) window_lengths_kernel(KvqView v, const void* k_new,
                                                                   const void* v_new, int n_stride,
                                                                   const int32_t* n_per_seq) {
  const int b = blockIdx.x;
  const int T0 = v.seq_lens[b];
  const int n = n_per_seq ? n_per_seq[b] : n_stride;
  if (n <= 0 || T0 < 0 || n > n_stride || (long long)T0 + n > (long long)v.max_pages * v.P) return;
  const int T1 = T0 + n;
  if (v.R > 0) {
    const int base = (T1 / v.R) * v.R;
    const int t_lo = max(base, T0);
    const int row = v.Hkv * v.D;  // elements of one token (all heads)
    const int esz = v.src_bf16 ? 2 : 4;
    const uintptr_t al = reinterpret_cast<uintptr_t>(k_new) | reinterpret_cast<uintptr_t>(v_new) |
                         reinterpret_cast<uintptr_t>(v.k_win) | reinterpret_cast<uintptr_t>(v.v_win);
    if ((al & 15) == 0 && (row * esz) % 16 == 0) {
      // 16-byte chunks: a token's row of all heads is contiguous in both tensors
      const int cpr = row * esz / 16;
      for (int e = threadIdx.x; e < (T1 - t_lo) * cpr; e += kThreads) {
        const int t = t_lo + e / cpr, k = e % cpr;
        const long long si = ((long long)b * n_stride + (t - T0)) * cpr + k;
        const long long di = ((long long)b * v.R + (t - base)) * cpr + k;
        const uint4 kx = reinterpret_cast<const uint4*>(k_new)[si];
        const uint4 vx = reinterpret_cast<const uint4*>(v_new)[si];
        reinterpret_cast<uint4*>(v.k_win)[di] = kx;
        reinterpret_cast<uint4*>(v.v_win)[di] = vx;
      }
    } else {
      for (int e = threadIdx.x; e < (T1 - t_lo) * row; e += kThreads) {
        const int t = t_lo + e / row, c = e % row;
        const long long si = ((long long)b * n_stride + (t - T0)) * row + c;
        const long long di = ((long long)b * v.R + (t - base)) * row + c;
        store_src(v.k_win, di, load_src(k_new, si, v.src_bf16), v.src_bf16);
        store_src(v.v_win, di, load_src(v_new, si, v.src_bf16), v.src_bf16);
      }
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) v.seq_lens[b] = T1;
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
        if (is_fp8(v.kfmt)) {
          kx = __fmul_rn(fp8_to_float(ku, v.kfmt), v.k_scale[h]);
        } else if (v.kaxis == KVQ_PER_TENSOR) {
          kx = dequant_sym(signed_code(ku, v.kbits, KVQ_SYM_ABSMAX), v.k_scale[h]);
        } else {
          const uint8_t* meta;
          float s, mn = 0.f;
          if (v.kaxis == KVQ_PER_TOKEN) {
            meta = hb + v.off_km + slot * v.k_ng * v.k_nmeta * v.mb;
            const int grp = c / v.kgroup;
            s = load_meta(meta, grp, v.meta16);
            if (v.k_nmeta == 2) mn = load_meta(meta, v.k_ng + grp, v.meta16);
          } else {
            const int g0 = (t / v.kgroup) * v.kgroup;
            const uint8_t* gp = page_of(v, seq, g0);
            meta = gp ? gp + (long long)h * v.head_bytes + v.off_km +
                            (long long)((g0 % v.P) / v.kgroup) * v.D * v.k_nmeta * v.mb
                      : nullptr;
            s = meta ? load_meta(meta, c, v.meta16) : 0.f;
            if (meta && v.k_nmeta == 2) mn = load_meta(meta, v.D + c, v.meta16);
          }
          const int code = signed_code(ku, v.kbits, v.kmode);
          kx = v.kmode == KVQ_ASYM_MINMAX ? dequant_asym(code, s, mn) : dequant_sym(code, s);
        }
        const unsigned vu = get_code(hb + v.off_vc + slot * v.vrow, c, v.vbits);
        if (is_fp8(v.vfmt)) {
          vx = __fmul_rn(fp8_to_float(vu, v.vfmt), v.v_scale[h]);
        } else if (v.vaxis == KVQ_PER_TENSOR) {
          vx = dequant_sym(signed_code(vu, v.vbits, KVQ_SYM_ABSMAX), v.v_scale[h]);
        } else {
          const uint8_t* meta = hb + v.off_vm + slot * v.v_ng * v.v_nmeta * v.mb;
          const int grp = c / v.vgroup;
          const int code = signed_code(vu, v.vbits, v.vmode);
          const float vs = load_meta(meta, grp, v.meta16);
          vx = v.vmode == KVQ_ASYM_MINMAX ? dequant_asym(code, vs, load_meta(meta, v.v_ng + grp, v.meta16))
                                          : dequant_sym(code, vs);
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
  const size_t stage_bytes = v.R > 0 ? 2ull * v.R * v.D * (v.src_bf16 ? 2 : 4) : 0;
  const uintptr_t align_bits = reinterpret_cast<uintptr_t>(k_new) | reinterpret_cast<uintptr_t>(v_new) |
                               reinterpret_cast<uintptr_t>(v.k_win) | reinterpret_cast<uintptr_t>(v.v_win);
  const int stage_ok = stage_bytes > 0 && stage_bytes <= kStageMax && (align_bits & 15) == 0;
  if (stage_ok) {
    const kvq_status ss = ensure_dynamic_smem(kSlotAppend, append_kernel, kStageMax);
    if (ss != KVQ_OK) return ss == KVQ_ERR_CAPACITY ? KVQ_ERR_CUDA : ss;
  }
  append_kernel<<<grid, kThreads, stage_ok ? stage_bytes : 0, st>>>(v, k_new, v_new, n_new, n_new_per_seq,
                                                                    stage_ok);
  window_lengths_kernel<<<v.batch, kThreads, 0, st>>>(v, k_new, v_new, n_new, n_new_per_seq);
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
