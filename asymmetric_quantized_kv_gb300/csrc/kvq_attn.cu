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
#include "kvq_ptx.cuh"

namespace kvq {
namespace {

constexpr int kWarps = 4;
constexpr int kThreads = kWarps * 32;
constexpr float kLog2e = 1.4426950408889634f;

// Work split: an item (sequence, kv-head, head block, chunk of C tokens) runs on
// one CTA of 4 warps; each warp takes sub-tiles of kST tokens.  Per sub-tile the
// warp dequantizes the K rows into shared memory (lanes over 32-bit code words;
// rows of fewer than 32 words share a pass), computes the logits with the lanes
// over (token, head group or channel part), dequantizes the V rows into the same
// buffer and accumulates P*V with lanes over channels.  Short sub-tiles keep the
// serial path of a warp short: small calls are latency-bound, and C shrinks to 32
// tokens there.
constexpr int kST = 8;
// The sub-tile's packed K and V rows (with per-token scale/min entries of up to
// kMetaStage bytes a token, and the key group's per-channel entries when the
// sub-tile lies in one group) are copied to shared memory with cp.async before
// any is dequantized: all the sub-tile's reads are in flight at once.  A warp's
// first sub-tile is requested right after the query's loads are issued (q goes
// to shared memory after the requests), each later one as soon as the previous
// sub-tile's V rows are dequantized (its P*V and the next logits overlap the
// copies).
constexpr int kMetaStage = 64;

// Dequantization rule of one side (K or V) for a call, resolved once.
struct DeqRule {
  int kind;        // kFp8, kTensor, kChannel, kToken
  int bits, fmt;   // code bits; FP8 format
  bool asym;
  uint32_t xw;     // word ^ xw, then code - sub = the signed code value (sym INT8: 0x80 per byte / 128)
  float bias;      // 2^23 + sub
  int lg, ng;      // PER_TOKEN: log2(group), groups per token
};
constexpr int kFp8 = 0, kTensor = 1, kChannel = 2, kToken = 3;

__device__ __forceinline__ DeqRule make_rule(int fmt, int mode, int axis, int group, int bits, int ng) {
  DeqRule r;
  r.fmt = fmt;
  r.bits = bits;
  r.kind = is_fp8(fmt) ? kFp8 : axis == KVQ_PER_TENSOR ? kTensor : axis == KVQ_PER_CHANNEL ? kChannel : kToken;
  r.asym = !is_fp8(fmt) && axis != KVQ_PER_TENSOR && mode == KVQ_ASYM_MINMAX;
  const bool sym = !r.asym;
  r.xw = (sym && bits == 8) ? 0x80808080u : 0u;
  const int sub = !sym ? 0 : bits == 8 ? 128 : (1 << (bits - 1));
  r.bias = 8388608.f + (float)sub;
  r.lg = __ffs(group > 0 ? group : 1) - 1;  // group: a power of two (it divides D)
  r.ng = ng;
  return r;
}

// Signed code value of code field u (of a word already XOR-ed with r.xw), as an
// exact float: the field in the mantissa of 2^23, minus 2^23 + sub.
__device__ __forceinline__ float code_value(uint32_t u, const DeqRule& r) {
  return __int_as_float(0x4B000000 | u) - r.bias;
}

// Entries i..i+3 (i a multiple of 4) of a scale/min array, fp32 or binary16.
__device__ __forceinline__ float4 load_meta4(const uint8_t* p, int i, int m16) {
  if (m16) {
    const uint2 h = *reinterpret_cast<const uint2*>(p + 2 * i);
    const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&h.x));
    const float2 b = __half22float2(*reinterpret_cast<const __half2*>(&h.y));
    return make_float4(a.x, a.y, b.x, b.y);
  }
  return *reinterpret_cast<const float4*>(p + 4 * i);
}

// Dequantize the 32/BITS codes of word w (channels c0..) into dst (fp32).
// meta: PER_CHANNEL: the key group's entries (D scales, then D minima);
// PER_TOKEN: the token's entries (ng scales, then ng minima).  ts: per-tensor /
// FP8 scale.  Every step is the rounding of include/kvq.h: c*s, then + min.
template <int BITS>
__device__ __forceinline__ void deq_word(uint32_t w, int c0, const DeqRule& r, const uint8_t* meta, int D, int m16,
                                         float ts, float* dst) {
  constexpr int N = 32 / BITS;
  constexpr uint32_t M = (1u << BITS) - 1u;
  float x[N];
  if (r.kind != kFp8) w ^= r.xw;
  if (r.kind == kFp8) {
#pragma unroll
    for (int e = 0; e < N; ++e) x[e] = __fmul_rn(fp8_to_float((w >> (e * BITS)) & M, r.fmt), ts);
  } else if (r.kind == kTensor) {
#pragma unroll
    for (int e = 0; e < N; ++e) x[e] = __fmul_rn(code_value((w >> (e * BITS)) & M, r), ts);
  } else if (r.kind == kChannel) {
#pragma unroll
    for (int e4 = 0; e4 < N; e4 += 4) {
      const float4 s = load_meta4(meta, c0 + e4, m16);
      const float4 mn = r.asym ? load_meta4(meta, D + c0 + e4, m16) : make_float4(0.f, 0.f, 0.f, 0.f);
      const float sv[4] = {s.x, s.y, s.z, s.w}, mv[4] = {mn.x, mn.y, mn.z, mn.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float y = __fmul_rn(code_value((w >> ((e4 + e) * BITS)) & M, r), sv[e]);
        x[e4 + e] = r.asym ? __fadd_rn(y, mv[e]) : y;
      }
    }
  } else {
    // a word's N codes lie in one channel group (groups are multiples of 16
    // channels, N <= 16 divides them): one scale and one minimum per word
    const int g = c0 >> r.lg;
    const float sc = load_meta(meta, g, m16);
    const float mn = r.asym ? load_meta(meta, r.ng + g, m16) : 0.f;
#pragma unroll
    for (int e = 0; e < N; ++e) {
      const float y = __fmul_rn(code_value((w >> (e * BITS)) & M, r), sc);
      x[e] = r.asym ? __fadd_rn(y, mn) : y;
    }
  }
#pragma unroll
  for (int e = 0; e < N; e += 4) *reinterpret_cast<float4*>(dst + e) = make_float4(x[e], x[e + 1], x[e + 2], x[e + 3]);
}

// One window row (source dtype) -> dst[0..D), lanes over channel quads.
__device__ __forceinline__ void copy_src_row(const void* base, long long row_elem, int D, int bf16, float* dst,
                                             int lane) {
  for (int i = lane; i < D / 4; i += 32) {
    float4 x;
    if (bf16) {
      const uint2 h = reinterpret_cast<const uint2*>(static_cast<const uint16_t*>(base) + row_elem)[i];
      x = make_float4(__uint_as_float(h.x << 16), __uint_as_float(h.x & 0xFFFF0000u), __uint_as_float(h.y << 16),
                      __uint_as_float(h.y & 0xFFFF0000u));
    } else {
      x = reinterpret_cast<const float4*>(static_cast<const float*>(base) + row_elem)[i];
    }
    reinterpret_cast<float4*>(dst)[i] = x;
  }
}

// Lane src's pointer, to every lane.
__device__ __forceinline__ const uint8_t* shfl_ptr(const uint8_t* p, int src) {
  const unsigned long long x = reinterpret_cast<unsigned long long>(p);
  const unsigned lo = __shfl_sync(0xffffffffu, static_cast<unsigned>(x), src);
  const unsigned hi = __shfl_sync(0xffffffffu, static_cast<unsigned>(x >> 32), src);
  return reinterpret_cast<const uint8_t*>((static_cast<unsigned long long>(hi) << 32) | lo);
}

// 4- and 16-byte asynchronous copies global -> shared (both sides aligned to the
// size), and their groups.
__device__ __forceinline__ void cp_async4(void* dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;\n" ::"r"(ptx::smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(ptx::smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}

// Staged row pitch in bytes: a row plus 16, so that the 8 rows' words at one
// offset fall in 8 different 4-bank groups.
template <int D>
constexpr int stage_pitch() { return D + 16; }

// n <= 8 staged rows (row tt at stage + tt * pitch) -> buf rows (stride DP
// floats) in one pass: lane = (token lane/4, part lane%4), part p taking words
// p, p + 4, p + 8, ... of the row's NW (so a quarter-warp's four parts read and
// write adjacent words: no bank conflicts).  meta_of(tt) gives row tt's
// scale/min entries (every lane calls it: it may shuffle); rows marked in `bad`
// are written as zeros.  The word loop stays rolled: the kernel's code size
// decides the latency-bound calls, whose code is fetched cold from DRAM.
template <int BITS, int D, typename MetaOf>
__device__ __forceinline__ void deq_staged_t(const uint8_t* stage, int DP, int n, unsigned bad, const DeqRule& r,
                                             MetaOf meta_of, int m16, float ts, float* buf, int lane) {
  constexpr int N = 32 / BITS, NW = D * BITS / 32, CW = NW / 4;  // CW: 1..16 words per lane
  static_assert(kST == 8 && NW % 4 == 0, "one pass covers 8 rows in quarters");
  const int tt = lane >> 2, part = lane & 3;
  const uint8_t* meta = meta_of(tt);
  if (tt < n) {
    float* dst = buf + tt * DP + part * N;
    const uint32_t* row = reinterpret_cast<const uint32_t*>(stage + tt * stage_pitch<D>()) + part;
    if ((bad >> tt) & 1u) {
#pragma unroll 1
      for (int i = 0; i < CW; ++i) {
#pragma unroll
        for (int e = 0; e < N; e += 4)
          *reinterpret_cast<float4*>(dst + 4 * i * N + e) = make_float4(0.f, 0.f, 0.f, 0.f);
      }
    } else {
#pragma unroll 1
      for (int i = 0; i < CW; ++i) deq_word<BITS>(row[4 * i], (part + 4 * i) * N, r, meta, D, m16, ts, dst + 4 * i * N);
    }
  }
}
template <int D, typename MetaOf>
__device__ __forceinline__ void deq_staged(const uint8_t* stage, int DP, int n, unsigned bad, const DeqRule& r,
                                           MetaOf meta_of, int m16, float ts, float* buf, int lane) {
  if (r.bits == 8) deq_staged_t<8, D>(stage, DP, n, bad, r, meta_of, m16, ts, buf, lane);
  else if (r.bits == 4) deq_staged_t<4, D>(stage, DP, n, bad, r, meta_of, m16, ts, buf, lane);
  else deq_staged_t<2, D>(stage, DP, n, bad, r, meta_of, m16, ts, buf, lane);
}

// Asynchronous copy of the n <= 8 rows of `bytes` bytes (a power of two, a
// multiple of CHUNK) that lane tt's `src` points at, to dst + tt * pitch, in
// CHUNK-byte copies (16 for code rows: the pool is 16-byte aligned and every row
// a multiple of 16 bytes; 4 for per-token entries): lanes over (row, chunk).
// Rows marked in `bad` are skipped.  Every lane takes part (shuffles).
template <int CHUNK>
__device__ __forceinline__ void stage_rows(uint8_t* dst, int pitch, const uint8_t* src, int bytes, int n, unsigned bad,
                                           int lane) {
  constexpr int LG = CHUNK == 16 ? 4 : 2;
  const int per = bytes >> LG, lper = __ffs(per) - 1;  // chunks per row, a power of two
  for (int k0 = 0; k0 < n * per; k0 += 32) {
    const int k = k0 + lane, tt = min(k >> lper, kST - 1), c = (k & (per - 1)) << LG;
    const uint8_t* p = shfl_ptr(src, tt);
    if (k < n * per && !((bad >> tt) & 1u)) {
      if constexpr (CHUNK == 16) cp_async16(dst + tt * pitch + c, p + c);
      else cp_async4(dst + tt * pitch + c, p + c);
    }
  }
}

// Max and sum over the 8 lanes of a lane's group of 8 (lanes 8g .. 8g+7).
__device__ __forceinline__ float max8(float x) {
  for (int o = 1; o < 8; o <<= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
  return x;
}
__device__ __forceinline__ float sum8(float x) {
  for (int o = 1; o < 8; o <<= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

// What a staged sub-tile's dequantization reads besides the staging: lane tt's
// K and V entry pointers (used where they are not staged), the missing-page mask,
// and whether the key group's per-channel entries were staged.
struct TileRefs {
  const uint8_t* km;
  const uint8_t* vm;
  unsigned bad;
  bool kc;
};

// Partial record of one (item, query head of the block): running max, sum, two
// pad words, then D outputs (16-byte aligned).
__host__ __device__ inline int generic_rec(int D) { return D + 4; }

struct GenericSmem {
  float qs[kHB][kMaxHeadDim];  // q * scale * log2(e) of the head block
  float wm[kWarps][kHB];
  float wl[kWarps][kHB];
  float rope_hi[kMaxHeadDim / 2];
  float rope_lo[kMaxHeadDim / 2];
};

// Dynamic shared memory: GenericSmem, pref[B+1], then (16-byte aligned) per warp a
// sub-tile buffer [kST][D+4] and its probabilities [kHB][kST], then the warps'
// outputs [kWarps][kHB][D] for the CTA merge, then per warp the packed staging of
// a sub-tile: K rows [kST][D + 16 bytes], K entries [kST][kMetaStage], the same
// for V, and one key group's per-channel entries [8 D bytes].
__host__ __device__ inline size_t generic_tiles_offset(int batch) {
  return (sizeof(GenericSmem) + sizeof(int) * (batch + 1) + 15) / 16 * 16;
}
__host__ __device__ inline size_t generic_smem_bytes(int batch, int D) {
  return generic_tiles_offset(batch) +
         sizeof(float) * ((size_t)kWarps * kST * (D + 4) + (size_t)kWarps * kHB * kST + (size_t)kWarps * kHB * D) +
         (size_t)kWarps * (2 * kST * (D + 16 + kMetaStage) + 8 * D);
}

// NH: query heads per item at most (a power of two <= kHB); NJ = D / 32.
template <int NH, int NJ>
__global__ void __launch_bounds__(kThreads) split_generic_kernel(KvqView v, const void* q, float scale, float* ws) {
  extern __shared__ __align__(16) unsigned char dyn[];
  GenericSmem& sm = *reinterpret_cast<GenericSmem*>(dyn);
  int* pref = reinterpret_cast<int*>(dyn + sizeof(GenericSmem));
  constexpr int D = 32 * NJ, DP = D + 4, REC = D + 4;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  float* buf = reinterpret_cast<float*>(dyn + generic_tiles_offset(v.batch)) + warp * kST * DP;
  float* ps = reinterpret_cast<float*>(dyn + generic_tiles_offset(v.batch)) + kWarps * kST * DP + warp * kHB * kST;
  float* wo = reinterpret_cast<float*>(dyn + generic_tiles_offset(v.batch)) + kWarps * kST * DP + kWarps * kHB * kST;
  constexpr int SP = stage_pitch<D>();
  uint8_t* sk = reinterpret_cast<uint8_t*>(wo + kWarps * kHB * D) + warp * (2 * kST * (SP + kMetaStage) + 8 * D);
  uint8_t* skm = sk + kST * SP;
  uint8_t* sv = skm + kST * kMetaStage;
  uint8_t* svm = sv + kST * SP;
  uint8_t* skc = svm + kST * kMetaStage;
  const int HB = (v.n_rep + kHB - 1) / kHB;
  __shared__ int s_C, s_items;
  plan_items(v, HB, pref, &s_C, &s_items);
  if (blockIdx.x == 0) store_plan(v, ws, pref, s_C, s_items);
  ptx::grid_dep_launch();  // the combine's CTAs may be scheduled; they wait for this grid
  const int C = s_C, n_items = s_items;
  if (v.rope_pre) {
    for (int i = threadIdx.x; i < D / 2; i += kThreads) rope_split(v, i, &sm.rope_hi[i], &sm.rope_lo[i]);
  }
  const DeqRule kr = make_rule(v.kfmt, v.kmode, v.kaxis, v.kgroup, v.kbits, v.k_ng);
  const DeqRule vr = make_rule(v.vfmt, v.vmode, v.vaxis, v.vgroup, v.vbits, v.v_ng);
  const int kmeta_tok = v.k_ng * v.k_nmeta * v.mb, vmeta_tok = v.v_ng * v.v_nmeta * v.mb;
  // per-token entries that are staged with the rows (whole 4-byte words that fit)
  const bool stage_km = kr.kind == kToken && kmeta_tok <= kMetaStage && (kmeta_tok & 3) == 0;
  const bool stage_vm = vr.kind == kToken && vmeta_tok <= kMetaStage && (vmeta_tok & 3) == 0;
  const int kmeta_ch = D * v.k_nmeta * v.mb;  // one key group's per-channel entries (<= 8 D bytes)
  const int src = v.src_bf16 ? 2 : 4;
  float* part = plan_partials(ws, v.batch);
  for (int item = blockIdx.x; item < n_items; item += gridDim.x) {
    ItemInfo it = decode_item(v, pref, C, HB, item);
    const int nh = min(kHB, v.n_rep - it.hb * kHB);
    const float kts = (kr.kind == kFp8 || kr.kind == kTensor) ? v.k_scale[it.kvh] : 0.f;
    const float vts = (vr.kind == kFp8 || vr.kind == kTensor) ? v.v_scale[it.kvh] : 0.f;
    const long long wbase = ((long long)it.b * v.R - it.t0) * v.Hkv + it.kvh;  // window row of token t: wbase + t*Hkv
    // Sub-tile at token `tile` (warp-uniform): lane tt < n looks up token tile +
    // tt's rows; the packed rows go to the warp's staging, K (copy group 1) then V
    // (group 2).  Returns what the dequantization needs besides the staging.
    auto stage_tile = [&](int tile) -> TileRefs {
      const int n = min(kST, it.t1 - tile);
      const uint8_t *a_k = nullptr, *a_km = nullptr, *a_v = nullptr, *a_vm = nullptr;
      bool ok = true;
      if (lane < n) {
        const int t = tile + lane;
        if (it.window) {
          const long long wrow = (wbase + (long long)t * v.Hkv) * D;
          ptx::prefetch_l1_range(static_cast<const char*>(v.k_win) + wrow * src, D * src);
          ptx::prefetch_l1_range(static_cast<const char*>(v.v_win) + wrow * src, D * src);
        } else {
          const uint8_t* page = page_of(v, it.b, t);
          ok = page != nullptr;
          if (ok) {
            const uint8_t* hb = page + (long long)it.kvh * v.head_bytes;
            const int slot = t % v.P;
            a_k = hb + slot * v.krow;
            a_v = hb + v.off_vc + slot * v.vrow;
            a_vm = hb + v.off_vm + slot * vmeta_tok;
            if (kr.kind == kToken) {
              a_km = hb + v.off_km + slot * kmeta_tok;
              if (!stage_km) ptx::prefetch_l1_range(a_km, kmeta_tok);
            } else if (kr.kind == kChannel) {  // the key group's entries live in the page of its first token
              const int g0 = (t / v.kgroup) * v.kgroup;
              const uint8_t* gp = page_of(v, it.b, g0);
              ok = gp != nullptr;
              if (ok)
                a_km = gp + (long long)it.kvh * v.head_bytes + v.off_km +
                       (long long)((g0 % v.P) / v.kgroup) * D * v.k_nmeta * v.mb;
            }
            if (vr.kind == kToken && !stage_vm) ptx::prefetch_l1_range(a_vm, vmeta_tok);
          }
        }
      }
      TileRefs r;
      r.km = a_km;
      r.vm = a_vm;
      // tokens whose page (or key group's page) is missing: logits -inf, V rows zero
      r.bad = __ballot_sync(0xffffffffu, lane < n && !ok);
      r.kc = false;
      if (!it.window) {
        stage_rows<16>(sk, SP, a_k, v.krow, n, r.bad, lane);
        if (stage_km) stage_rows<4>(skm, kMetaStage, a_km, kmeta_tok, n, r.bad, lane);
        r.kc = kr.kind == kChannel && !(r.bad & 1u) && tile / v.kgroup == (tile + n - 1) / v.kgroup;
        if (r.kc) {
          const uint8_t* pm = shfl_ptr(a_km, 0);
          for (int c = 16 * lane; c < kmeta_ch; c += 512) cp_async16(skc + c, pm + c);
        }
        cp_async_commit();
        stage_rows<16>(sv, SP, a_v, v.vrow, n, r.bad, lane);
        if (stage_vm) stage_rows<4>(svm, kMetaStage, a_vm, vmeta_tok, n, r.bad, lane);
        cp_async_commit();
      }
      return r;
    };
    // the query's loads go out first, then the first sub-tile's lookups and copies
    constexpr int QPT = (NH * D + kThreads - 1) / kThreads;
    float qv[QPT];
#pragma unroll
    for (int i = 0; i < QPT; ++i) {
      const int e = threadIdx.x + i * kThreads, hh = e / D, c = e % D;
      qv[i] = 0.f;
      if (e < NH * D && hh < nh) {
        const int hq = it.kvh * v.n_rep + it.hb * kHB + hh;
        qv[i] = load_src(q, ((long long)it.b * v.Hq + hq) * D + c, v.src_bf16) * scale * kLog2e;
      }
    }
    __syncthreads();  // smem of the previous item is free
    int tile = it.t0 + warp * kST;
    TileRefs tr{nullptr, nullptr, 0u, false};
    if (tile < it.t1) tr = stage_tile(tile);
#pragma unroll
    for (int i = 0; i < QPT; ++i) {
      const int e = threadIdx.x + i * kThreads;
      if (e < NH * D) sm.qs[e / D][e % D] = qv[i];
    }
    __syncthreads();
    float m_run[NH], l_run[NH], o[NH][NJ];
#pragma unroll
    for (int hh = 0; hh < NH; ++hh) {
      m_run[hh] = -INFINITY;
      l_run[hh] = 0.f;
#pragma unroll
      for (int j = 0; j < NJ; ++j) o[hh][j] = 0.f;
    }
    for (; tile < it.t1; tile += kWarps * kST) {
      const int n = min(kST, it.t1 - tile);
      const unsigned bad = tr.bad;
      if (!it.window) {
        cp_async_wait<1>();
        __syncwarp();
      }
      // ---- K rows -> buf
      if (it.window) {
        for (int tt = 0; tt < n; ++tt)
          copy_src_row(v.k_win, (wbase + (long long)(tile + tt) * v.Hkv) * D, D, v.src_bf16, buf + tt * DP, lane);
      } else {
        const TileRefs& rf = tr;
        auto km_of = [&](int tt) -> const uint8_t* {
          return rf.kc ? skc : stage_km ? skm + tt * kMetaStage : shfl_ptr(rf.km, tt);
        };
        deq_staged<D>(sk, DP, n, bad, kr, km_of, v.meta16, kts, buf, lane);
      }
      __syncwarp();
      if (v.rope_pre) {  // rotate the pairs in place: lanes over (token, pair)
        for (int e = lane; e < n * (D / 2); e += 32) {
          const int tt = e / (D / 2), i = e % (D / 2);
          float2* pr = reinterpret_cast<float2*>(buf + tt * DP) + i;
          const float2 k = *pr;
          float sn, cs;
          sincospif(2.f * rope_turns(tile + tt, sm.rope_hi[i], sm.rope_lo[i]), &sn, &cs);
          *pr = make_float2(k.x * cs - k.y * sn, k.x * sn + k.y * cs);
        }
        __syncwarp();
      }
      // ---- logits: lane = token tt + 8 g.  With 4 or more heads, lane group g
      // takes heads g*HPG .. g*HPG+HPG-1 over all channels; with 1 or 2 heads,
      // CPG groups share a head, each over D/CPG channels, and add their parts.
      constexpr int HPG = NH >= 4 ? NH / 4 : 1, CPG = NH >= 4 ? 1 : 4 / NH;
      const int tt = lane & 7, g = lane >> 3;
      const int h0 = NH >= 4 ? g * HPG : g / CPG, cb = NH >= 4 ? 0 : (g % CPG) * (D / CPG);
      const bool valid = tt < n && !((bad >> tt) & 1u);
      float acc[HPG];
#pragma unroll
      for (int j = 0; j < HPG; ++j) acc[j] = 0.f;
      if (valid) {
        const float* krow = buf + tt * DP + cb;
#pragma unroll 4
        for (int c = 0; c < D / CPG; c += 4) {
          const float4 k4 = *reinterpret_cast<const float4*>(krow + c);
#pragma unroll
          for (int j = 0; j < HPG; ++j) {
            const float4 q4 = *reinterpret_cast<const float4*>(&sm.qs[h0 + j][cb + c]);
            acc[j] += q4.x * k4.x + q4.y * k4.y + q4.z * k4.z + q4.w * k4.w;
          }
        }
      }
      if (CPG >= 2) acc[0] += __shfl_xor_sync(0xffffffffu, acc[0], 8);
      if (CPG >= 4) acc[0] += __shfl_xor_sync(0xffffffffu, acc[0], 16);
      float lg[HPG], mx[HPG];
#pragma unroll
      for (int j = 0; j < HPG; ++j) {
        lg[j] = valid && h0 + j < nh ? acc[j] : -INFINITY;
        mx[j] = max8(lg[j]);
      }
      // every lane updates every head's running max, sum and output; the group
      // holding head hh supplies its max and probability sum
      float mine[HPG];
#pragma unroll
      for (int j = 0; j < HPG; ++j) mine[j] = -INFINITY;
      float alpha[NH];
#pragma unroll
      for (int hh = 0; hh < NH; ++hh) {
        const int src_lane = (NH >= 4 ? hh / HPG : hh * CPG) * 8;
        const float m_new = fmaxf(m_run[hh], __shfl_sync(0xffffffffu, mx[hh % HPG], src_lane));
        alpha[hh] = m_new == -INFINITY ? 1.f : exp2f(m_run[hh] - m_new);
        m_run[hh] = m_new;
        if (h0 + hh % HPG == hh) mine[hh % HPG] = m_new;
      }
      float psum[HPG];
#pragma unroll
      for (int j = 0; j < HPG; ++j) {
        const float p = valid && h0 + j < nh ? exp2f(lg[j] - mine[j]) : 0.f;
        if (cb == 0 && h0 + j < nh) ps[(h0 + j) * kST + tt] = p;
        psum[j] = sum8(p);
      }
#pragma unroll
      for (int hh = 0; hh < NH; ++hh) {
        const int src_lane = (NH >= 4 ? hh / HPG : hh * CPG) * 8;
        const float ls = __shfl_sync(0xffffffffu, psum[hh % HPG], src_lane);
        if (hh < nh) {
          l_run[hh] = l_run[hh] * alpha[hh] + ls;
#pragma unroll
          for (int j = 0; j < NJ; ++j) o[hh][j] *= alpha[hh];
        }
      }
      __syncwarp();
      // ---- V rows -> buf (marked tokens: zeros; their p is 0)
      if (!it.window) {
        cp_async_wait<0>();
        __syncwarp();
      }
      if (it.window) {
        for (int tt = 0; tt < n; ++tt)
          copy_src_row(v.v_win, (wbase + (long long)(tile + tt) * v.Hkv) * D, D, v.src_bf16, buf + tt * DP, lane);
      } else {
        const TileRefs& rf = tr;
        auto vm_of = [&](int tt) -> const uint8_t* {
          return stage_vm ? svm + tt * kMetaStage : shfl_ptr(rf.vm, tt);
        };
        deq_staged<D>(sv, DP, n, bad, vr, vm_of, v.meta16, vts, buf, lane);
      }
      __syncwarp();
      if (tile + kWarps * kST < it.t1) tr = stage_tile(tile + kWarps * kST);  // the staging is free again
      // ---- P V: lanes over channels
      for (int tt = 0; tt < n; ++tt) {
        float pv[NH];
#pragma unroll
        for (int hh = 0; hh < NH; ++hh) pv[hh] = hh < nh ? ps[hh * kST + tt] : 0.f;
#pragma unroll
        for (int j = 0; j < NJ; ++j) {
          const float vx = buf[tt * DP + lane + 32 * j];
#pragma unroll
          for (int hh = 0; hh < NH; ++hh) o[hh][j] = fmaf(pv[hh], vx, o[hh][j]);
        }
      }
      __syncwarp();
    }
    // merge the warps of this CTA
#pragma unroll
    for (int hh = 0; hh < NH; ++hh) {
      if (hh < nh) {
        if (lane == 0) {
          sm.wm[warp][hh] = m_run[hh];
          sm.wl[warp][hh] = l_run[hh];
        }
#pragma unroll
        for (int j = 0; j < NJ; ++j) wo[(warp * kHB + hh) * D + lane + 32 * j] = o[hh][j];
      }
    }
    __syncthreads();
    float* dst = part + (long long)item * kHB * REC;
    for (int e = threadIdx.x; e < nh * D; e += kThreads) {
      const int hh = e / D, c = e % D;
      float M = -INFINITY;
      for (int w = 0; w < kWarps; ++w) M = fmaxf(M, sm.wm[w][hh]);
      float L = 0.f, O = 0.f;
      for (int w = 0; w < kWarps; ++w) {
        const float f = sm.wm[w][hh] == -INFINITY ? 0.f : exp2f(sm.wm[w][hh] - M);
        L += sm.wl[w][hh] * f;
        O += wo[(w * kHB + hh) * D + c] * f;
      }
      if (c == 0) {
        dst[hh * REC + 0] = M;
        dst[hh * REC + 1] = L;
      }
      dst[hh * REC + 4 + c] = O;
    }
  }
}

}  // namespace

// Partials -> out: one CTA of 4 warps per (query head, sequence).  Each warp
// loads up to 16 of the head's records at once (lanes over channel quads) and
// merges them online; the warps then merge through shared memory.  Launched as a
// programmatic dependent of the split kernel: it waits for that grid to complete
// before reading the workspace.
__global__ void __launch_bounds__(128) combine_kernel(KvqView v, float* ws, float* out) {
  constexpr int kCW = 4, kBatch = 16, kQ = kMaxHeadDim / 128;  // channel quads per lane
  __shared__ float4 o_s[kCW][kMaxHeadDim / 4];
  __shared__ float m_s[kCW], l_s[kCW];
  ptx::grid_dep_wait();
  const int hq = blockIdx.x, b = blockIdx.y;
  const int D = v.D, REC = generic_rec(D), nqd = D / 4;
  const int HB = (v.n_rep + kHB - 1) / kHB;
  const int* pref = plan_prefix(ws);
  const float* part = plan_partials(ws, v.batch);
  const int kvh = hq / v.n_rep, hr = hq % v.n_rep, hb = hr / kHB, hh = hr % kHB;
  const int nc = (pref[b + 1] - pref[b]) / (v.Hkv * HB);
  const float* base = part + ((long long)pref[b] + (long long)(kvh * HB + hb) * nc) * kHB * REC + hh * REC;
  const long long stride = (long long)kHB * REC;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  float m = -INFINITY, l = 0.f;
  float4 o[kQ];
#pragma unroll
  for (int k = 0; k < kQ; ++k) o[k] = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int i0 = warp; i0 < nc; i0 += kCW * kBatch) {
    float rm[kBatch], rl[kBatch];
    float4 x[kBatch][kQ];
#pragma unroll
    for (int j = 0; j < kBatch; ++j) {
      const int i = i0 + j * kCW;
      rm[j] = -INFINITY;
      rl[j] = 0.f;
#pragma unroll
      for (int k = 0; k < kQ; ++k) x[j][k] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (i < nc) {
        const float* r = base + (long long)i * stride;
        rm[j] = r[0];
        rl[j] = r[1];
#pragma unroll
        for (int k = 0; k < kQ; ++k)
          if (lane + 32 * k < nqd) x[j][k] = reinterpret_cast<const float4*>(r + 4)[lane + 32 * k];
      }
    }
    float mn = m;
#pragma unroll
    for (int j = 0; j < kBatch; ++j) mn = fmaxf(mn, rm[j]);
    if (mn != -INFINITY) {
      const float a = exp2f(m - mn);
      l *= a;
#pragma unroll
      for (int k = 0; k < kQ; ++k) {
        o[k].x *= a; o[k].y *= a; o[k].z *= a; o[k].w *= a;
      }
#pragma unroll
      for (int j = 0; j < kBatch; ++j) {
        const float w = rm[j] == -INFINITY ? 0.f : exp2f(rm[j] - mn);
        l = fmaf(rl[j], w, l);
#pragma unroll
        for (int k = 0; k < kQ; ++k) {
          o[k].x = fmaf(x[j][k].x, w, o[k].x); o[k].y = fmaf(x[j][k].y, w, o[k].y);
          o[k].z = fmaf(x[j][k].z, w, o[k].z); o[k].w = fmaf(x[j][k].w, w, o[k].w);
        }
      }
      m = mn;
    }
  }
  if (lane == 0) {
    m_s[warp] = m;
    l_s[warp] = l;
  }
#pragma unroll
  for (int k = 0; k < kQ; ++k)
    if (lane + 32 * k < nqd) o_s[warp][lane + 32 * k] = o[k];
  __syncthreads();
  if (warp == 0) {
    float M = m_s[0];
#pragma unroll
    for (int w = 1; w < kCW; ++w) M = fmaxf(M, m_s[w]);
    float L = 0.f;
#pragma unroll
    for (int w = 0; w < kCW; ++w) L = fmaf(l_s[w], m_s[w] == -INFINITY ? 0.f : exp2f(m_s[w] - M), L);
    const float invL = L > 0.f ? 1.f / L : 0.f;
#pragma unroll
    for (int k = 0; k < kQ; ++k) {
      if (lane + 32 * k < nqd) {
        float4 r = make_float4(0.f, 0.f, 0.f, 0.f);
        if (M != -INFINITY) {
#pragma unroll
          for (int w = 0; w < kCW; ++w) {
            const float a = m_s[w] == -INFINITY ? 0.f : exp2f(m_s[w] - M);
            const float4 x = o_s[w][lane + 32 * k];
            r.x = fmaf(x.x, a, r.x); r.y = fmaf(x.y, a, r.y); r.z = fmaf(x.z, a, r.z); r.w = fmaf(x.w, a, r.w);
          }
        }
        r.x *= invL; r.y *= invL; r.z *= invL; r.w *= invL;
        reinterpret_cast<float4*>(out + ((long long)b * v.Hq + hq) * D)[lane + 32 * k] = r;
      }
    }
  }
}

size_t attention_workspace_bytes(const KvqView& v, int batch) {
  const int HB = (v.n_rep + kHB - 1) / kHB;
  const long long items = kTargetItems + 2LL * batch * v.Hkv * HB;
  const size_t generic = plan_header_bytes(batch) + (size_t)items * kHB * generic_rec(v.D) * sizeof(float);
  KvqView b = v;
  b.batch = batch;
  const size_t split = fast_workspace_bytes(v, batch);  // layout of the tensor-core kernels
  return (fast_eligible(b) || fp8_shape_eligible(b) || int2_shape_eligible(b)) && split > generic ? split : generic;
}

int pick_decode_kernel(const KvqView& v) {
  if (fast_eligible(v)) return KVQ_KERNEL_ROPE_I8I4;
  if (fp8_eligible(v)) return KVQ_KERNEL_FP8;
  if (int2_eligible(v)) return KVQ_KERNEL_INT2;
  return KVQ_KERNEL_GENERIC;
}

kvq_status launch_attention(const KvqView& v, const void* q, float* out, float scale, void* ws,
                            size_t ws_bytes, cudaStream_t st) {
  (void)ws_bytes;
  switch (pick_decode_kernel(v)) {
    case KVQ_KERNEL_ROPE_I8I4: return launch_fast(v, q, out, scale, ws, st);
    case KVQ_KERNEL_FP8: return launch_fp8(v, q, out, scale, ws, st);
    case KVQ_KERNEL_INT2: return launch_int2(v, q, out, scale, ws, st);
    default: break;
  }
  // dynamic shared memory grows with the batch (the plan prefix) and D: raise the
  // kernel's limit to what this call needs; beyond the device's limit the call
  // does not fit
  const int nh = v.n_rep < kHB ? v.n_rep : kHB;
  const int ih = nh <= 1 ? 0 : nh <= 2 ? 1 : nh <= 4 ? 2 : 3;
  const int id = v.D == 64 ? 0 : v.D == 128 ? 1 : 2;
  using Kern = void (*)(KvqView, const void*, float, float*);
  static const Kern kerns[4][3] = {
      {split_generic_kernel<1, 2>, split_generic_kernel<1, 4>, split_generic_kernel<1, 8>},
      {split_generic_kernel<2, 2>, split_generic_kernel<2, 4>, split_generic_kernel<2, 8>},
      {split_generic_kernel<4, 2>, split_generic_kernel<4, 4>, split_generic_kernel<4, 8>},
      {split_generic_kernel<8, 2>, split_generic_kernel<8, 4>, split_generic_kernel<8, 8>}};
  const Kern kern = kerns[ih][id];
  const size_t smem = generic_smem_bytes(v.batch, v.D);
  const kvq_status ss = ensure_dynamic_smem(kSlotGeneric + 3 * ih + id, kern, smem);
  if (ss != KVQ_OK) return ss;
  // as many CTAs as fit on the SMs at once (registers and shared memory): the
  // warps' dependent chains need company on each scheduler
  int occ = 0;
  const kvq_status so = occupancy_at(kSlotGenericOcc + 3 * ih + id, kern, kThreads, smem, &occ);
  if (so != KVQ_OK) return so;
  const int grid = num_sms() * occ;
  kern<<<grid, kThreads, smem, st>>>(v, q, scale, static_cast<float*>(ws));
  if (cudaGetLastError() != cudaSuccess) return KVQ_ERR_CUDA;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(v.Hq, v.batch);
  cfg.blockDim = dim3(128);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, combine_kernel, v, static_cast<float*>(ws), out) == cudaSuccess ? KVQ_OK
                                                                                                 : KVQ_ERR_CUDA;
}

}  // namespace kvq
