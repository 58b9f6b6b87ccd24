// Tensor-core split-K decode attention for 2-bit asymmetric keys quantized
// per channel over token groups and 2-bit asymmetric values quantized per token
// in 32-channel groups, head_dim 128, 4 query heads per kv-head, plus the bf16
// residual window: the KIVI-style layer ("Why Keys Are More Sensitive Than Values
// in INT8 KV Cache Quantization", section "Computational Paths for Key and
// Value", and "KV Cache Quantization: Why It's Different from Weight
// Quantization", section "Why Key and Value Tensors Have Different
// Distributions": 2-bit keys per channel, values per token, recent tokens kept in
// full precision).
//
// Work: a unit is (sequence, chunk of C tokens, kv-head); every warp takes units
// from a global counter and streams its 16-token tiles through a private 3-stage
// ring.  One 5-D TMA tensor copy brings a tile's K codes, V codes and V scale/min
// rows (three page sections with 32-byte rows); a tile that starts a key group
// also brings the group's scales and minima with a 2-D tensor copy in 128-byte
// swizzle, so the per-group reads meet no bank conflict.
//
// QK: with k = c * s + m per (group, channel), written as k = (c - 3/2) s + (m + 3/2 s),
//     q.k = sum_c (q_c s_c)(c - 3/2) + sum_c q_c (m_c + 3/2 s_c).  A = the centred
//     codes c - 3/2 in f16 (exact, built from the packed bytes: see centred_code);
//     B = q * s split hi/lo, rebuilt once per key group; the second sum is a
//     per-group, per-head bias.  Centring keeps the tensor-core sum of the order
//     of the logit: with the codes 0..3 as they are, the code sum and the bias
//     are each several times larger than the logit and cancel, and on the 8B
//     layer the logits lost enough to put heads at 4.5e-4 relative L2 (2-bit
//     values centred, keys not) instead of 4.5e-6 (both centred).
// PV: with v = c * s_t + m_t per (token, 32-channel group), written as
//     v = (c - 3/2) s_t + (m_t + 3/2 s_t), p.v = sum_t (p_t s_t)(c - 3/2)
//     + sum_t p_t (m_t + 3/2 s_t).  Lane row g holds byte 8G + g of every token
//     (channels 32G + 4g .. 32G + 4g + 3), so each 16-row MMA block stays inside
//     one value group G and B = p * s_t(G) split hi/lo; A = the centred codes
//     c - 3/2 in f16 (exact), and the group midpoints enter through running sums
//     of p * (m_t + 3/2 s_t).  Centring matters: the value groups of N(0,1) data
//     have m ~ -2 and c s in [0, 4], so the uncentred sums sum_t p s c and
//     sum_t p m are each ~2 sum_t p while a head that spreads its attention has an
//     output ~50x smaller; every relative error of the tensor-core sum (its
//     truncating fp32 accumulation, the hi/lo split of B) was magnified by that
//     ratio.  Centred, both sums are of the order of the output.
// Scales and minima stored as binary16 (meta_dtype F16) take a second instance:
// the codes come with one 2-section tensor copy, the value rows and a group's key
// scales and minima (256 and 512 bytes) with plain bulk copies, and the readers
// widen the halves to fp32.
#include <math.h>

#include "kvq_ptx.cuh"
#include "kvq_split_common.cuh"
#include "kvq_tmap.h"

namespace kvq {
namespace {

using namespace ptx;

constexpr int kTI = 32;  // tokens per tile of a quantized chunk: two 16-token halves (one MMA row block each)
constexpr int kHT = 16;  // tokens per half tile, and per tile of a residual window
constexpr int kWarpsI = 4;
constexpr int kThreadsI = kWarpsI * 32;
constexpr int kStagesI = 3;
constexpr int kRepI = 4;
constexpr int kRow2 = 32;                         // bytes of one token's 2-bit codes
constexpr int kVMetaRow = 32;                     // (scale x 4, min x 4) fp32 per token
constexpr int kKMeta2 = 2 * kD * 4;               // scales then minima of one key group (in the page)
// stage layout (1024-byte aligned): a key group's scales/minima (fp32: 8 swizzled
// rows of 128 bytes; binary16: 512 linear bytes), then the two half tiles, each
// K codes [16][32], V codes [16][32] and the value meta rows [16][32 or 16] bytes
constexpr int kVMetaRow16 = 16;                   // (scale x 4, min x 4) binary16 per token
constexpr int kKMeta16 = 2 * kD * 2;              // a key group's scales then minima, binary16
constexpr int kOffKM = 0;
constexpr int kOffH = kKMeta2;                    // first half tile
constexpr int kOffV = kHT * kRow2;                // V codes within a half tile
constexpr int kOffVM32 = 2 * kHT * kRow2;         // value meta rows within a half tile
constexpr int kOffVM16 = 2 * kHT * kRow2;
constexpr int kHalf32 = 3 * kHT * kRow2;          // fp32 meta: 1536 bytes per half tile
constexpr int kHalf16 = 2 * kHT * kRow2 + kHT * kVMetaRow16;  // binary16 meta: 1280
constexpr int kStageI = 4096;
constexpr uint32_t kSpinI = ptx::kWaitPolls;  // polls per bounded mbarrier wait
constexpr float kLog2eI = 1.4426950408889634f;
constexpr float kRescaleI = 8.f;
constexpr float kMinitI = -1e30f;

struct __align__(1024) SmemI2 {
  uint8_t stage[kWarpsI][kStagesI][kStageI];
  float4 qp[kWarpsI][8][32];  // per warp, step s, lane: q * scale * log2(e) at the lane's 4 channels of step s
  float pex[kWarpsI][5][32];  // p exchange (quantized tiles: per half 80 floats, window tiles: 64)
  float4 vmw[kWarpsI][2][kHT][2];  // binary16 metadata: the tile's value rows widened to fp32 (scales, minima)
  uint64_t bar[kWarpsI][kStagesI];
  int valid[kWarpsI][kStagesI];
};
static_assert(kStageI % 1024 == 0 && kOffH + 2 * kHalf32 <= kStageI && kOffH + 2 * kHalf16 <= kStageI &&
                  kHalf32 % 128 == 0 && kHalf16 % 128 == 0,
              "stages stay 1024-byte aligned and half tiles 128-byte aligned");

// Lane (g, t), step s: its four channels c0..c3 in k-slot order 2t, 2t+1, 2t+8,
// 2t+9 are 32t + 16(s/4) + {j, 8+j, 4+j, 12+j} with j = s % 4: the code bit
// fields (2j) of bytes 0/2 and 1/3 of the lane's word s/4.
__device__ __forceinline__ int step_channel(int t, int s, int e) {
  const int j = s & 3, base = 32 * t + 16 * (s >> 2);
  return base + j + (e == 0 ? 0 : e == 1 ? 8 : e == 2 ? 4 : 12);
}

// 4 consecutive source-dtype values at element index i (16-byte aligned for fp32,
// 8-byte aligned for bf16)
__device__ __forceinline__ float4 load4_src(const void* base, long long i, int bf16) {
  if (bf16) {
    const uint2 u = *reinterpret_cast<const uint2*>(reinterpret_cast<const unsigned short*>(base) + i);
    return make_float4(__uint_as_float(u.x << 16), __uint_as_float(u.x & 0xFFFF0000u), __uint_as_float(u.y << 16),
                       __uint_as_float(u.y & 0xFFFF0000u));
  }
  return *reinterpret_cast<const float4*>(reinterpret_cast<const float*>(base) + i);
}

// Per CTA: prefW[b] = number of sequences before b whose residual window is not
// empty, *s_NW their total.  NT threads; scratch holds NT ints.
template <int NT>
__device__ inline void window_prefix(const KvqView& v, int* prefW, int* s_NW, int* scratch) {
  const int B = v.batch;
  const int seg = (B + NT - 1) / NT;
  const int b0 = threadIdx.x * seg, b1 = min(B, b0 + seg);
  int cnt = 0;
  for (int b = b0; b < b1; ++b) {
    const int T = seq_tokens(v, b);
    cnt += T > n_quantized(T, v.R) ? 1 : 0;
  }
  scratch[threadIdx.x] = cnt;
  __syncthreads();
  if (threadIdx.x == 0) {
    int r = 0;
    for (int k = 0; k < NT; ++k) {
      const int x = scratch[k];
      scratch[k] = r;
      r += x;
    }
    *s_NW = r;
  }
  __syncthreads();
  int r = scratch[threadIdx.x];
  for (int b = b0; b < b1; ++b) {
    prefW[b] = r;
    const int T = seq_tokens(v, b);
    r += T > n_quantized(T, v.R) ? 1 : 0;
  }
  if (threadIdx.x == 0) prefW[B] = *s_NW;
  __syncthreads();
}

// f16x2 hi part of (x0, x1), or (hi - x) for lanes that carry the residual
// columns: a column pair then sums to hi - (hi - x) = x.
__device__ __forceinline__ void split_sel(float x0, float x1, bool lo, uint32_t& out) {
  uint32_t hi, nl;
  split_hi_neglo(x0, x1, hi, nl);
  out = lo ? nl : hi;
}

// PV k-slot -> tile token: within each group of four slots the tokens are
// rotated by (slot / 4) % 4, so the four lanes t of a quad, which read slots 2t
// (or 2t+1, 2t+8, 2t+9) from 32-byte rows, hit four different 128-byte bank
// offsets; tsig_inv is its inverse.  The p exchange stores each token's p at its
// slot, so B and the value rows agree.
__device__ __forceinline__ int tsig(int k) { return (k & ~3) | ((k + (k >> 2)) & 3); }
__device__ __forceinline__ int tsig_inv(int r) { return (r & ~3) | ((r - (r >> 2)) & 3); }

// The 2-bit code fields k (bits 2k, 2k+1 of each 16-bit half) of a packed word,
// centred: f16x2 (c - 3/2), exact.  OR-ing a field into the mantissa of 1024
// gives the half 1024 + c * 4^k (the mantissa step at 1024 is 1); for k > 0 one
// fused multiply-add by 4^-k and -(1024 / 4^k + 3/2) leaves c - 3/2; for k = 0,
// where 1025.5 is not a half, 1024 and then 3/2 are subtracted in turn.
template <int K>
__device__ __forceinline__ uint32_t centred_code(uint32_t w) {
  const uint32_t x = and_or(w, 0x00030003u << (2 * K), 0x64006400u);
  if constexpr (K == 0) {
    return hsub2(hsub2(x, 0x64006400u), 0x3E003E00u);  // - 1024, - 1.5
  } else if constexpr (K == 1) {
    return hfma2(x, 0x34003400u, 0xDC06DC06u);  // * 1/4, - 257.5
  } else if constexpr (K == 2) {
    return hfma2(x, 0x2C002C00u, 0xD418D418u);  // * 1/16, - 65.5
  } else {
    return hfma2(x, 0x24002400u, 0xCC60CC60u);  // * 1/64, - 17.5
  }
}

// The 2-bit code fields k + 1 (bits 2k + 2, 2k + 3 of each 16-bit half, k = 0..3),
// centred: OR-ing the field into the mantissa of 1024 gives 1024 + c * 4^(k+1), and
// one fused multiply-add by 4^-(k+1) and -(1024 / 4^(k+1) + 3/2) leaves c - 3/2
// exactly (for the top field, 4 + c - 5.5).
template <int K>
__device__ __forceinline__ uint32_t centred_code_up(uint32_t w) {
  const uint32_t x = and_or(w, 0x000C000Cu << (2 * K), 0x64006400u);
  if constexpr (K == 0) {
    return hfma2(x, 0x34003400u, 0xDC06DC06u);  // * 1/4, - 257.5
  } else if constexpr (K == 1) {
    return hfma2(x, 0x2C002C00u, 0xD418D418u);  // * 1/16, - 65.5
  } else if constexpr (K == 2) {
    return hfma2(x, 0x24002400u, 0xCC60CC60u);  // * 1/64, - 17.5
  } else {
    return hfma2(x, 0x1C001C00u, 0xC580C580u);  // * 1/256, - 5.5
  }
}
__device__ __forceinline__ uint32_t centred_field_up(uint32_t w, int k) {
  return k == 0 ? centred_code_up<0>(w) : k == 1 ? centred_code_up<1>(w) : k == 2 ? centred_code_up<2>(w)
                                                                                 : centred_code_up<3>(w);
}

// four binary16 values (two words) widened to fp32
__device__ __forceinline__ float4 halves4(uint2 w) {
  const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&w.x));
  const float2 b = __half22float2(*reinterpret_cast<const __half2*>(&w.y));
  return make_float4(a.x, a.y, b.x, b.y);
}

template <bool M16>
__global__ void __launch_bounds__(kThreadsI, 3)
    split_int2_kernel(KvqView v, const void* q, float scale, float* ws, const __grid_constant__ CUtensorMap tmc,
                      const __grid_constant__ CUtensorMap tmk) {
  extern __shared__ unsigned char dyn_raw[];
  unsigned char* dyn = dyn_raw + ((1024 - (smem_u32(dyn_raw) & 1023)) & 1023);  // 1024-byte aligned
  SmemI2& sm = *reinterpret_cast<SmemI2*>(dyn);
  int* prefA = reinterpret_cast<int*>(dyn + sizeof(SmemI2));
  int* prefB = prefA + v.batch + 1;
  int* prefW = prefB + v.batch + 1;
  __shared__ int s_C, s_NA, s_NB, s_NS, s_NW;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;
  const bool odd = (g & 1) != 0;  // this lane's B columns carry lo halves
  // PV: this lane's k-slots 2t, 2t+1, 2t+8, 2t+9 hold tile tokens T0, T1, T8, T9;
  // its logits (tokens g, g+8) go to slots X0, X1 + 8
  const int T0 = tsig(2 * t), T1 = tsig(2 * t + 1), T8 = tsig(2 * t + 8), T9 = tsig(2 * t + 9);
  const int X0 = tsig_inv(g), X1 = tsig_inv(g + 8) - 8;
  constexpr int kHalf = M16 ? kHalf16 : kHalf32;
  const uint64_t pol = l2_evict_first();  // the packed stream is read once: evict it first from L2
  const int G = v.kgroup;  // powers of two (checked on the host)
  const int lgP = __ffs(v.P) - 1, lgG = __ffs(G) - 1;
  // a warp takes one kv-head of an item: Hkv units per item, one worker per warp; no cuts
  fast_plan<kThreadsI>(v, G, v.Hkv, (int)gridDim.x * kWarpsI, false, prefA, prefB, &s_C, &s_NA, &s_NB, &s_NS,
                       reinterpret_cast<int*>(&sm.stage[0][0][0]));
  window_prefix<kThreadsI>(v, prefW, &s_NW, reinterpret_cast<int*>(&sm.stage[0][0][0]));
  if (blockIdx.x == 0) store_fast_plan(v, ws, prefA, prefB, s_C, s_NA, s_NB, s_NS);
  grid_dep_launch();  // the combine kernel may be scheduled; it waits for this grid to complete
  unsigned long long* counter =
      reinterpret_cast<unsigned long long*>(reinterpret_cast<char*>(ws) + fast_counter_offset(v.batch));
  if (lane == 0) {
    for (int s = 0; s < kStagesI; ++s) mbar_init(&sm.bar[warp][s], 1);
    fence_mbar_init();
  }
  __syncthreads();

  const int C = s_C, NA = s_NA, NS = s_NS, NW = s_NW;
  // execution order: the residual-window units first (the slowest per token),
  // then every unit of the plan in its long-first order, skipping the windows
  const int n_units = (NW + s_NA + s_NB) * v.Hkv;
  float* part = reinterpret_cast<float*>(reinterpret_cast<char*>(ws) + fast_header_bytes(v.batch));
  int lstage = 0, cstage = 0;
  uint32_t cphase = 0, n_loaded = 0, n_consumed = 0;
  bool stalled = false;
  const float qscale = scale * kLog2eI;

  int unit = blockIdx.x * kWarpsI + warp;
  const int unit_stride0 = gridDim.x * kWarpsI;
  while (unit < n_units) {
    unsigned long long nxt = 0;
    if (lane == 0) nxt = atomicAdd(counter, 1ull);
    int pair, h;
    if (unit < NW * v.Hkv) {
      const int w = unit / v.Hkv;
      h = unit - w * v.Hkv;
      const int b = seq_of(prefW, v.batch, w);
      pair = NA + prefB[b + 1] - 1;  // the window is the sequence's last short item
    } else {
      const int u = unit - NW * v.Hkv;
      pair = u / v.Hkv;
      h = u - pair * v.Hkv;
    }
    const FastItem it = decode_fast_item(v, prefA, prefB, C, NA, NS, G, false, pair);
    if (it.window && unit >= NW * v.Hkv) {  // done in the first phase
      unit = unit_stride0 + (int)__shfl_sync(0xffffffffu, (unsigned)nxt, 0);
      continue;
    }

    // q * scale * log2(e) of this lane's query head 4h + g/2 at its step channels
    {
      const long long qb = ((long long)it.b * v.Hq + h * kRepI + (g >> 1)) * kD;
      __syncwarp();
#pragma unroll
      for (int s = 0; s < 8; ++s) {
        float x[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) x[e] = load_src(q, qb + step_channel(t, s, e), v.src_bf16) * qscale;
        sm.qp[warp][s][lane] = make_float4(x[0], x[1], x[2], x[3]);
      }
      __syncwarp();
    }
    const float4* qps = &sm.qp[warp][0][lane];  // step s at qps[32 * s]

    // O[m]: rows g / g+8, columns 2t / 2t+1 = query head t hi / (hi - x)
    float O[8][4];
#pragma unroll
    for (int m = 0; m < 8; ++m) O[m][0] = O[m][1] = O[m][2] = O[m][3] = 0.f;
    float m_run = kMinitI, l_loc = 0.f;
    float mb[4] = {0.f, 0.f, 0.f, 0.f};  // sum of p * (v_min + 3/2 v_scale) per value group (head t)
    float* pe = &sm.pex[warp][0][0];

    // softmax step for logits of tokens g, g+8 (head t); returns p
    auto softmax = [&](float lg0, float lg1, float& p0, float& p1) {
      if (__any_sync(0xffffffffu, fmaxf(lg0, lg1) > m_run + kRescaleI)) {
        float mx = fmaxf(lg0, lg1);
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
        const float mn = fmaxf(m_run, mx);
        const float alpha = ex2(m_run - mn);
#pragma unroll
        for (int m = 0; m < 8; ++m) {
          O[m][0] *= alpha; O[m][1] *= alpha; O[m][2] *= alpha; O[m][3] *= alpha;
        }
        l_loc *= alpha;
#pragma unroll
        for (int G4 = 0; G4 < 4; ++G4) mb[G4] *= alpha;
        m_run = mn;
      }
      p0 = ex2(lg0 - m_run);
      p1 = ex2(lg1 - m_run);
      l_loc += p0 + p1;
    };
    // softmax step for the logits of tokens g, g+8 of both half tiles (head t)
    auto softmax4 = [&](const float (&lg)[4], float (&p)[4]) {
      float mx = fmaxf(fmaxf(lg[0], lg[1]), fmaxf(lg[2], lg[3]));
      if (__any_sync(0xffffffffu, mx > m_run + kRescaleI)) {
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
        const float mn = fmaxf(m_run, mx);
        const float alpha = ex2(m_run - mn);
#pragma unroll
        for (int m = 0; m < 8; ++m) {
          O[m][0] *= alpha; O[m][1] *= alpha; O[m][2] *= alpha; O[m][3] *= alpha;
        }
        l_loc *= alpha;
#pragma unroll
        for (int G4 = 0; G4 < 4; ++G4) mb[G4] *= alpha;
        m_run = mn;
      }
#pragma unroll
      for (int e = 0; e < 4; ++e) p[e] = ex2(lg[e] - m_run);
      l_loc += (p[0] + p[1]) + (p[2] + p[3]);
    };
    // p of head g/2 at k-slots 2t, 2t+1 (x01) and 2t+8, 2t+9 (x89)
    auto exchange = [&](float p0, float p1, float2& x01, float2& x89) {
      __syncwarp();
      pe[t * 8 + X0] = p0;
      pe[32 + t * 8 + X1] = p1;
      __syncwarp();
      x01 = *reinterpret_cast<const float2*>(pe + (g >> 1) * 8 + 2 * t);
      x89 = *reinterpret_cast<const float2*>(pe + 32 + (g >> 1) * 8 + 2 * t);
    };

    if (!it.window) {
      // ======================= quantized chunk: 32-token tiles (two 16-token halves)
      const int32_t* bt = v.block_table + (long long)it.b * v.max_pages;
      const int ntiles = (it.t1 - it.t0 + kTI - 1) / kTI;
      const uint8_t* pages_h = v.pages + (long long)h * v.head_bytes;
      // lane 0: the page ids of the next tile to load (the second half's page when P is 16)
      int pf0 = 0, pf1 = 0;
      auto page_pair = [&](int i, int& p0, int& p1) {
        const int tok = it.t0 + i * kTI;
        p0 = bt[tok >> lgP];
        // 16-token pages: the second half sits in the next page, unless it lies past the item's end
        // (its rows are then masked, and the table entry there need not be a page)
        p1 = (v.P >= kTI || tok + kHT >= it.t1) ? p0 : bt[(tok + kHT) >> lgP];
      };
      auto issue = [&](int i, int pid0, int pid1) {
        const int stage = lstage;
        if (++lstage == kStagesI) lstage = 0;
        ++n_loaded;
        const int tok = it.t0 + i * kTI;
        uint64_t* bar = &sm.bar[warp][stage];
        const bool ok = pid0 >= 0 && pid0 < v.n_pages && pid1 >= 0 && pid1 < v.n_pages;
        sm.valid[warp][stage] = ok;
        if (!ok) {
          atomicOr(v.status, KVQ_DEV_BAD_PAGE);
          mbar_arrive(bar);
          return;
        }
        const int slot0 = tok & (v.P - 1), slot1 = (tok + kHT) & (v.P - 1);
        const bool gstart = (tok & (G - 1)) == 0;
        uint8_t* dst = sm.stage[warp][stage];
        if constexpr (M16) {
          // codes of each half by one 2-section tensor copy, its value rows and the key meta by bulk copies
          mbar_arrive_expect_tx(bar, 2 * kHalf16 + (gstart ? kKMeta16 : 0));
          tma_load_5d_hint(dst + kOffH, &tmc, 0, slot0, 0, h, pid0, bar, pol);
          tma_load_5d_hint(dst + kOffH + kHalf16, &tmc, 0, slot1, 0, h, pid1, bar, pol);
          bulk_g2s_hint(dst + kOffH + kOffVM16, pages_h + (long long)pid0 * v.page_bytes + v.off_vm +
                        slot0 * kVMetaRow16, kHT * kVMetaRow16, bar, pol);
          bulk_g2s_hint(dst + kOffH + kHalf16 + kOffVM16, pages_h + (long long)pid1 * v.page_bytes + v.off_vm +
                        slot1 * kVMetaRow16, kHT * kVMetaRow16, bar, pol);
          if (gstart)
            bulk_g2s_hint(dst + kOffKM, pages_h + (long long)pid0 * v.page_bytes + v.off_km +
                          (v.P >= G ? slot0 >> lgG : 0) * kKMeta16, kKMeta16, bar, pol);
        } else {
          mbar_arrive_expect_tx(bar, 2 * kHalf32 + (gstart ? kKMeta2 : 0));
          tma_load_5d_hint(dst + kOffH, &tmc, 0, slot0, 0, h, pid0, bar, pol);
          tma_load_5d_hint(dst + kOffH + kHalf32, &tmc, 0, slot1, 0, h, pid1, bar, pol);
          if (gstart) {
            const long long byte0 = (long long)pid0 * v.page_bytes + (long long)h * v.head_bytes + v.off_km +
                                    (long long)(v.P >= G ? slot0 >> lgG : 0) * kKMeta2;
            tma_load_2d_hint(dst + kOffKM, &tmk, 0, (int)(byte0 >> 7), bar, pol);
          }
        }
      };
      if (lane == 0 && !stalled) {
        fence_proxy_async();
        for (int i = 0; i < min(kStagesI, ntiles); ++i) {
          int p0, p1;
          page_pair(i, p0, p1);
          issue(i, p0, p1);
        }
        if (kStagesI < ntiles) page_pair(kStagesI, pf0, pf1);
      }
      __syncwarp();

      uint32_t bk[8][2] = {};  // QK B: q * s of the current key group, hi (even g) / lo (odd g)
      float bias = 0.f;   // sum_c q_c (m_c + 3/2 s_c) of the current key group for query head t
      for (int i = 0; i < ntiles; ++i) {
        const int stage = cstage;
        bool valid = false;
        if (!stalled) {
          if (!mbar_wait_bounded(&sm.bar[warp][stage], cphase, kSpinI)) {
            atomicOr(v.status, KVQ_DEV_TIMEOUT);
            stalled = true;
          } else {
            valid = sm.valid[warp][stage] != 0;
          }
        }
        if (++cstage == kStagesI) {
          cstage = 0;
          cphase ^= 1u;
        }
        ++n_consumed;
        const uint8_t* buf = sm.stage[warp][stage];
        const int tok0 = it.t0 + i * kTI;
        if constexpr (M16) {
          // the tile's 32 value rows (4 scales, 4 minima in binary16) widened once to fp32: lane = (half, token)
          const int hf = lane >> 4, tk = lane & 15;
          const uint4 r = *reinterpret_cast<const uint4*>(buf + kOffH + hf * kHalf16 + kOffVM16 + tk * kVMetaRow16);
          sm.vmw[warp][hf][tk][0] = halves4(make_uint2(r.x, r.y));
          sm.vmw[warp][hf][tk][1] = halves4(make_uint2(r.z, r.w));
          __syncwarp();
        }

        if ((tok0 & (G - 1)) == 0) {
          // ---- new key group: B = q * s and the bias sum_c q_c (m_c + 3/2 s_c).  Lanes g and g ^ 1
          // (lane ^ 4) hold the same channels for the hi and the (hi - x) column of one query head:
          // the even lane splits steps 0..3 (channels 32t .. 32t + 15), the odd lane steps 4..7
          // (32t + 16 .. 32t + 31), and each hands the partner the half of the split it lacks.
          const uint8_t* ks = buf + kOffKM;
          const int hm = odd ? 1 : 0;
          float sc[16], mn[16];
#pragma unroll
          for (int k4 = 0; k4 < 4; ++k4) {
            float4 a, b;
            if constexpr (M16) {
              // linear halves: scales of channels 32t + 16 hm + 4 k4 .. at byte 2 * channel, minima after
              const int off = 64 * t + 32 * hm + 8 * k4;
              a = halves4(*reinterpret_cast<const uint2*>(ks + off));
              b = halves4(*reinterpret_cast<const uint2*>(ks + 2 * kD + off));
            } else {
              // rows r < 4: scales of channels 32r .., rows 4 + r: minima; 16-byte chunk c of row r at c ^ r
              const int c = 4 * hm + k4;
              a = *reinterpret_cast<const float4*>(ks + t * 128 + ((c ^ t) << 4));
              b = *reinterpret_cast<const float4*>(ks + (4 + t) * 128 + ((c ^ (4 + t)) << 4));
            }
            sc[4 * k4] = a.x; sc[4 * k4 + 1] = a.y; sc[4 * k4 + 2] = a.z; sc[4 * k4 + 3] = a.w;
            mn[4 * k4] = b.x; mn[4 * k4 + 1] = b.y; mn[4 * k4 + 2] = b.z; mn[4 * k4 + 3] = b.w;
          }
          float bl = 0.f;
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            // q at channels j, 8+j, 4+j, 12+j of this lane's half (step 4 hm + j)
            const float4 x = qps[32 * (4 * hm + j)];
            const float2 pa = __fmul2_rn(make_float2(x.x, x.y), make_float2(sc[j], sc[8 + j]));
            const float2 pb = __fmul2_rn(make_float2(x.z, x.w), make_float2(sc[4 + j], sc[12 + j]));
            uint32_t ha, na, hb2, nb;
            split_hi_neglo(pa.x, pa.y, ha, na);
            split_hi_neglo(pb.x, pb.y, hb2, nb);
            // the even lane keeps hi and sends (hi - x); the odd lane the other way round
            const uint32_t ra = __shfl_xor_sync(0xffffffffu, odd ? ha : na, 4);
            const uint32_t rb = __shfl_xor_sync(0xffffffffu, odd ? hb2 : nb, 4);
            bk[j][0] = odd ? ra : ha;
            bk[j][1] = odd ? rb : hb2;
            bk[4 + j][0] = odd ? na : ra;
            bk[4 + j][1] = odd ? nb : rb;
            bl = fmaf(x.x, fmaf(1.5f, sc[j], mn[j]), bl);
            bl = fmaf(x.y, fmaf(1.5f, sc[8 + j], mn[8 + j]), bl);
            bl = fmaf(x.z, fmaf(1.5f, sc[4 + j], mn[4 + j]), bl);
            bl = fmaf(x.w, fmaf(1.5f, sc[12 + j], mn[12 + j]), bl);
          }
          // the head's 128 channels: this lane's 16, its partner's 16 (lane ^ 4), the other t (^1, ^2);
          // the logit lanes (head t) take it from lane 8t
          bl += __shfl_xor_sync(0xffffffffu, bl, 4);
          bl += __shfl_xor_sync(0xffffffffu, bl, 1);
          bl += __shfl_xor_sync(0xffffffffu, bl, 2);
          bias = __shfl_sync(0xffffffffu, bl, 8 * t);
        }

        // ---- QK per half: rows g / g+8 = tokens 16 hf + g / + 8; centred codes
        const int nvalid = valid ? min(kTI, it.t1 - tok0) : 0;
        float lg[4];
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
          const uint8_t* hb = buf + kOffH + hf * kHalf;
          const uint2 w0 = *reinterpret_cast<const uint2*>(hb + g * kRow2 + 8 * t);
          const uint2 w1 = *reinterpret_cast<const uint2*>(hb + (g + 8) * kRow2 + 8 * t);
          // fields 0..3 of each half moved up to 1..4 (w << 2), fields 4..7 down to 1..4 (w >> 6):
          // every field then takes one mask and one fused multiply-add (centred_code_up)
          const uint32_t u0[2] = {w0.x << 2, w0.y << 2}, u1[2] = {w1.x << 2, w1.y << 2};
          const uint32_t s0[2] = {w0.x >> 6, w0.y >> 6}, s1[2] = {w1.x >> 6, w1.y >> 6};
          float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
          for (int s = 0; s < 8; ++s) {
            const int wd = s >> 2, j = s & 3;
            mma_16816(acc, centred_field_up(u0[wd], j), centred_field_up(u1[wd], j), centred_field_up(s0[wd], j),
                      centred_field_up(s1[wd], j), bk[s][0], bk[s][1]);
          }
          lg[2 * hf] = kHT * hf + g < nvalid ? (acc[0] - acc[1]) + bias : -INFINITY;
          lg[2 * hf + 1] = kHT * hf + g + 8 < nvalid ? (acc[2] - acc[3]) + bias : -INFINITY;
        }
        float p[4];
        softmax4(lg, p);

        // ---- value rows: per token 4 scales then 4 minima (fp32, or binary16 in M16)
        auto vrow = [&](int hf, int tok, int part) -> float4 {
          if constexpr (M16) {
            return sm.vmw[warp][hf][tok][part];
          } else {
            return reinterpret_cast<const float4*>(buf + kOffH + hf * kHalf32 + kOffVM32 + tok * kVMetaRow)[part];
          }
        };
        if (valid) {
          // group midpoints m + 3/2 s of tokens g, g+8 of both halves
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float4 n = vrow(e >> 1, g + 8 * (e & 1), 1), z = vrow(e >> 1, g + 8 * (e & 1), 0);
            const float2 pp = make_float2(p[e], p[e]), h15 = make_float2(1.5f, 1.5f);
            const float2 m01 = __ffma2_rn(pp, __ffma2_rn(h15, make_float2(z.x, z.y), make_float2(n.x, n.y)),
                                          make_float2(mb[0], mb[1]));
            const float2 m23 = __ffma2_rn(pp, __ffma2_rn(h15, make_float2(z.z, z.w), make_float2(n.z, n.w)),
                                          make_float2(mb[2], mb[3]));
            mb[0] = m01.x; mb[1] = m01.y; mb[2] = m23.x; mb[3] = m23.y;
          }
        }
        // p of head g/2 at the k-slots of both halves
        __syncwarp();
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
          pe[80 * hf + t * 8 + X0] = p[2 * hf];
          pe[80 * hf + 48 + t * 8 + X1] = p[2 * hf + 1];
        }
        __syncwarp();

        // ---- PV per half (k block of 16 tokens), value group G: byte 8G + g of tokens T0, T1 (ya), T8, T9 (yc)
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
          // B = p * s_t(G) of head g/2: the even lane of a pair (lane, lane ^ 4) forms the products of
          // k-slots 2t, 2t+1 (tokens T0, T1), the odd lane those of 2t+8, 2t+9 (T8, T9); each splits its
          // pair and hands the partner the half it needs (hi to the even lane, hi - x to the odd lane).
          // Within a half the slots 8.. sit 48 floats after the slots 0.., so the loads of the two lanes
          // of a pair fall in different banks.
          const float2 xo = *reinterpret_cast<const float2*>(pe + 80 * hf + (odd ? 48 : 0) + (g >> 1) * 8 + 2 * t);
          const float4 sp = vrow(hf, odd ? T8 : T0, 0), sq = vrow(hf, odd ? T9 : T1, 0);
          const float sP[4] = {sp.x, sp.y, sp.z, sp.w}, sQ[4] = {sq.x, sq.y, sq.z, sq.w};
          const uint8_t* vc = buf + kOffH + hf * kHalf + kOffV;
          const int gb = g & 3;
          const uint32_t sel = gb * 0x0011u + (4 + gb) * 0x1100u;
          const int woff = 4 * (g >> 2);
#pragma unroll
          for (int G4 = 0; G4 < 4; ++G4) {
            uint32_t hi, nl;
            split_hi_neglo(xo.x * sP[G4], xo.y * sQ[G4], hi, nl);
            const uint32_t r = __shfl_xor_sync(0xffffffffu, odd ? hi : nl, 4);
            const uint32_t b01 = odd ? r : hi, b89 = odd ? nl : r;
            const int off = 8 * G4 + woff;
            const uint32_t wa = *reinterpret_cast<const uint32_t*>(vc + T0 * kRow2 + off);
            const uint32_t wb = *reinterpret_cast<const uint32_t*>(vc + T1 * kRow2 + off);
            const uint32_t wc = *reinterpret_cast<const uint32_t*>(vc + T8 * kRow2 + off);
            const uint32_t wd = *reinterpret_cast<const uint32_t*>(vc + T9 * kRow2 + off);
            // each half of ya / yc holds the selected byte twice (as its low and its high byte)
            const uint32_t ya = prmt(wa, wb, sel), yc = prmt(wc, wd, sel);
            // m-block 2G4: rows g / g+8 = channels 32G4 + 4g + 0 / + 1 (code fields 0, 1; field 0 read from
            // the high copy, where it is field 4 of the half and takes one multiply-add)
            mma_16816(O[2 * G4], centred_code_up<3>(ya), centred_code<1>(ya), centred_code_up<3>(yc),
                      centred_code<1>(yc), b01, b89);
            // m-block 2G4+1: channels 32G4 + 4g + 2 / + 3 (code fields 2, 3)
            mma_16816(O[2 * G4 + 1], centred_code<2>(ya), centred_code<3>(ya), centred_code<2>(yc),
                      centred_code<3>(yc), b01, b89);
          }
        }

        // ---- release the stage and refill it
        __syncwarp();
        if (lane == 0 && i + kStagesI < ntiles && !stalled) {
          fence_proxy_async();
          issue(i + kStagesI, pf0, pf1);
          if (i + kStagesI + 1 < ntiles) page_pair(i + kStagesI + 1, pf0, pf1);
        }
        __syncwarp();
      }
    } else {
      // ======================= residual window: source-dtype rows from k_win / v_win
      uint32_t bw[8][2];  // B = q (no group scale), hi / lo
#pragma unroll
      for (int s = 0; s < 8; ++s) {
        const float4 x = qps[32 * s];
        split_sel(x.x, x.y, odd, bw[s][0]);
        split_sel(x.z, x.w, odd, bw[s][1]);
      }
      const int T = it.t1;
      const long long wrow = ((long long)it.b * v.R) * v.Hkv + h;
      const int ntiles = (it.t1 - it.t0 + kHT - 1) / kHT;
      for (int i = 0; i < ntiles; ++i) {
        const int tok0 = it.t0 + i * kHT;
        float acc[4] = {0.f, 0.f, 0.f, 0.f}, accn[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          // key rows of tokens g, g+8: channels 32t + 16 half .. + 15 (zero past the end)
          float kw[2][16];
#pragma unroll
          for (int r = 0; r < 2; ++r) {
            const int tok = tok0 + g + 8 * r;
            const long long wi = (wrow + (long long)(tok - it.t0) * v.Hkv) * kD + 32 * t + 16 * half;
#pragma unroll
            for (int c4 = 0; c4 < 4; ++c4) {
              const float4 x =
                  tok < T ? load4_src(v.k_win, wi + 4 * c4, v.src_bf16) : make_float4(0.f, 0.f, 0.f, 0.f);
              kw[r][4 * c4] = x.x; kw[r][4 * c4 + 1] = x.y; kw[r][4 * c4 + 2] = x.z; kw[r][4 * c4 + 3] = x.w;
            }
          }
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const int s = 4 * half + j;
            uint32_t ahi[2][2], anl[2][2];
#pragma unroll
            for (int r = 0; r < 2; ++r) {  // channels j, 8+j | 4+j, 12+j of the half
              split_hi_neglo(kw[r][j], kw[r][8 + j], ahi[r][0], anl[r][0]);
              split_hi_neglo(kw[r][4 + j], kw[r][12 + j], ahi[r][1], anl[r][1]);
            }
            mma_16816(acc, ahi[0][0], ahi[1][0], ahi[0][1], ahi[1][1], bw[s][0], bw[s][1]);
            mma_16816(accn, anl[0][0], anl[1][0], anl[0][1], anl[1][1], bw[s][0], bw[s][1]);
          }
        }
        const float lg0 = tok0 + g < T ? (acc[0] - acc[1]) - (accn[0] - accn[1]) : -INFINITY;
        const float lg1 = tok0 + g + 8 < T ? (acc[2] - acc[3]) - (accn[2] - accn[3]) : -INFINITY;
        float p0, p1;
        softmax(lg0, lg1, p0, p1);
        float2 x01, x89;
        exchange(p0, p1, x01, x89);
        uint32_t b01, b89;
        split_sel(x01.x, x01.y, odd, b01);
        split_sel(x89.x, x89.y, odd, b89);
        // values as f16, same row -> channel map as the quantized path (32G + 4g + k)
        const int slots[4] = {T0, T1, T8, T9};
#pragma unroll
        for (int G4 = 0; G4 < 4; ++G4) {
          float vv[4][4];
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const int tok = tok0 + slots[u];
            const long long wi = (wrow + (long long)(tok - it.t0) * v.Hkv) * kD + 32 * G4 + 4 * g;
            const float4 x = tok < T ? load4_src(v.v_win, wi, v.src_bf16) : make_float4(0.f, 0.f, 0.f, 0.f);
            vv[u][0] = x.x; vv[u][1] = x.y; vv[u][2] = x.z; vv[u][3] = x.w;
          }
#pragma unroll
          for (int hb = 0; hb < 2; ++hb) {
            const int k0 = 2 * hb;
            mma_16816(O[2 * G4 + hb], pack_f16x2(vv[0][k0], vv[1][k0]), pack_f16x2(vv[0][k0 + 1], vv[1][k0 + 1]),
                      pack_f16x2(vv[2][k0], vv[3][k0]), pack_f16x2(vv[2][k0 + 1], vv[3][k0 + 1]), b01, b89);
          }
        }
      }
    }

    // ---- epilogue: partial record of query head 4h + t
#pragma unroll
    for (int o = 4; o < 32; o <<= 1) {
      l_loc += __shfl_xor_sync(0xffffffffu, l_loc, o);
#pragma unroll
      for (int G4 = 0; G4 < 4; ++G4) mb[G4] += __shfl_xor_sync(0xffffffffu, mb[G4], o);
    }
    float* rec = part + ((long long)pair * v.Hq + h * kRepI + t) * (kD + 4);
    if (g == 0) {
      rec[0] = m_run;
      rec[1] = l_loc;
    }
    // quantized codes entered centred (c - 3/2), window values as they are; the
    // midpoint sums are zero for window units
#pragma unroll
    for (int G4 = 0; G4 < 4; ++G4) {
      const float4 o4 = make_float4((O[2 * G4][0] - O[2 * G4][1]) + mb[G4], (O[2 * G4][2] - O[2 * G4][3]) + mb[G4],
                                    (O[2 * G4 + 1][0] - O[2 * G4 + 1][1]) + mb[G4],
                                    (O[2 * G4 + 1][2] - O[2 * G4 + 1][3]) + mb[G4]);
      *reinterpret_cast<float4*>(rec + 4 + 32 * G4 + 4 * g) = o4;
    }
    unit = unit_stride0 + (int)__shfl_sync(0xffffffffu, (unsigned)nxt, 0);
  }

  if (lane == 0) {
    while (n_consumed < n_loaded) {
      mbar_wait_bounded(&sm.bar[warp][cstage], cphase, kSpinI);
      if (++cstage == kStagesI) {
        cstage = 0;
        cphase ^= 1u;
      }
      ++n_consumed;
    }
  }
}

}  // namespace

long long int2_pool_rows(const KvqView& v) { return (long long)v.n_pages * v.page_bytes / 128; }

bool int2_shape_eligible(const KvqView& v) {
  const bool pow2_g = v.kgroup > 0 && (v.kgroup & (v.kgroup - 1)) == 0;
  // the three per-token sections (K codes, V codes, V meta) share 32-byte rows at a
  // uniform section stride, and every offset is a multiple of 128 bytes
  // (binary16 metadata: 16-byte value rows and 16-byte aligned key meta, read by bulk copies)
  const int vmeta_row = v.v_ng * v.v_nmeta * v.mb;
  const bool meta_ok = v.meta16 ? (vmeta_row == kVMetaRow16 && v.off_km % 16 == 0)
                                : (vmeta_row == kVMetaRow && v.off_km % 128 == 0);
  return meta_ok && v.krow == kRow2 && v.vrow == kRow2 && v.off_vc == v.P * kRow2 &&
         v.off_vm == 2 * v.P * kRow2 && v.head_bytes % 128 == 0 && v.page_bytes % 128 == 0 &&
         v.D == kD && v.n_rep == kRepI && v.kfmt == KVQ_INT2 && v.kmode == KVQ_ASYM_MINMAX &&
         v.kaxis == KVQ_PER_CHANNEL && v.vfmt == KVQ_INT2 && v.vmode == KVQ_ASYM_MINMAX &&
         v.vaxis == KVQ_PER_TOKEN && v.vgroup == 32 && v.rope_pre == 0 && pow2_g && v.kgroup >= kTI &&
         v.P >= kHT && (v.P & (v.P - 1)) == 0 && v.batch <= 4096;
}

bool int2_eligible(const KvqView& v) {
  return int2_shape_eligible(v) && (reinterpret_cast<uintptr_t>(v.pages) & 15) == 0 && int2_pool_rows(v) > 0 &&
         int2_pool_rows(v) < (1LL << 31) && v.n_pages < (1 << 30) && tensor_map_encoder() != nullptr;
}

kvq_status launch_int2(const KvqView& v, const void* q, float* out, float scale, void* ws, cudaStream_t st) {
  // the per-token sections as a 5-D tensor (row bytes, slot, section, head, page), one tile per box
  CUtensorMap tmc, tmk;
  {
    const cuuint32_t nsec = v.meta16 ? 2 : 3;  // binary16 metadata: codes only (value rows by bulk copies)
    const cuuint64_t dims[5] = {(cuuint64_t)kRow2, (cuuint64_t)v.P, nsec, (cuuint64_t)v.Hkv, (cuuint64_t)v.n_pages};
    const cuuint64_t strides[4] = {(cuuint64_t)kRow2, (cuuint64_t)v.P * kRow2, (cuuint64_t)v.head_bytes,
                                   (cuuint64_t)v.page_bytes};
    const cuuint32_t box[5] = {(cuuint32_t)kRow2, (cuuint32_t)kHT, nsec, 1, 1};
    const cuuint32_t estr[5] = {1, 1, 1, 1, 1};
    if (tensor_map_encoder()(&tmc, CU_TENSOR_MAP_DATA_TYPE_UINT8, 5, v.pages, dims, strides, box, estr,
                             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return KVQ_ERR_UNSUPPORTED;
  }
  {
    // the pool as rows of 128 bytes: a key group's scales and minima are 8 rows
    const cuuint64_t dims[2] = {128, (cuuint64_t)int2_pool_rows(v)};
    const cuuint64_t strides[1] = {128};
    const cuuint32_t box[2] = {128, 8};
    const cuuint32_t estr[2] = {1, 1};
    if (tensor_map_encoder()(&tmk, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, v.pages, dims, strides, box, estr,
                             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return KVQ_ERR_UNSUPPORTED;
  }
  const size_t smem = sizeof(SmemI2) + 1024 + sizeof(int) * 3 * (v.batch + 1);
  void (*kern)(KvqView, const void*, float, float*, const CUtensorMap, const CUtensorMap) =
      v.meta16 ? split_int2_kernel<true> : split_int2_kernel<false>;
  int occ = 0;
  const kvq_status so = occupancy_once(kSlotInt2 + (v.meta16 ? 1 : 0), kern, kThreadsI, smem,
                                       sizeof(SmemI2) + 1024 + sizeof(int) * 3 * 4097, &occ);
  if (so != KVQ_OK) return so;
  const int grid = num_sms() * occ;
  if (cudaMemsetAsync(static_cast<char*>(ws) + fast_counter_offset(v.batch), 0, 8, st) != cudaSuccess)
    return KVQ_ERR_CUDA;
  kern<<<grid, kThreadsI, smem, st>>>(v, q, scale, static_cast<float*>(ws), tmc, tmk);
  if (cudaGetLastError() != cudaSuccess) return KVQ_ERR_CUDA;
  return launch_split_combine(v, static_cast<float*>(ws), out, st) == cudaSuccess ? KVQ_OK : KVQ_ERR_CUDA;
}

}  // namespace kvq
