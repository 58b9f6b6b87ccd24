// Tensor-core split-K decode attention for pre-RoPE INT8 per-channel keys and
// INT4 asymmetric per-token values (head_dim 128, 8 kv-heads, 4 query heads per
// kv-head): the paged, ragged decode layer of the pre-RoPE scheme ("KV Cache
// Quantization: Why Keys and Values Need Different Axes", section "Where does
// RoPE break this?": dequantize -> rotate -> dot inside the attention kernel).
//
// Work: an item is (sequence, chunk of C tokens) for all 8 kv-heads; CTA = 8
// warps, warp w owns kv-head w.  Each warp streams its head's 16-token tiles
// through a private 3-stage shared-memory ring filled by TMA bulk copies
// (cp.async.bulk, completion on an mbarrier, every wait bounded).
//
// Per 16-token tile and warp:
//   QK: K codes -> fp32 (x per-channel scale) -> RoPE rotation by the token's
//       absolute position (cos/sin from a per-tile table shared by the 8 warps)
//       -> split into f16 hi + lo -> two mma.m16n8k16 per 16 channels with
//       A = keys (16 tokens x 16 channels) and B = q (16 channels x 8 columns:
//       4 query heads x {hi, lo} halves of q*scale*log2(e)).  The hi/lo split
//       of both operands keeps the logits to ~2^-21 relative.
//   softmax: online in base 2, one running max per head with lazy rescaling
//       (only when the max grows by more than 2^8).
//   PV: A = V^T codes (16 channels x 16 tokens) formed with PRMT/LOP3 and one
//       f16x2 fix-up as exact f16 integers, B = p * v_scale split hi/lo; the
//       per-token minimum enters through a running sum of p * v_min.
// Partials (max, sum, unnormalised output) per (item, query head) go to the
// workspace; the combine kernel merges them.
#include <math.h>

#include "kvq_attn_plan.cuh"
#include "kvq_ptx.cuh"

namespace kvq {
namespace {

using namespace ptx;

constexpr int kTile = 16;
constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
constexpr int kStages = 3;
constexpr uint32_t kSpin = 1u << 20;  // polls per bounded mbarrier wait
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kRescale = 8.f;  // lazy rescale threshold in log2 units
constexpr int kFastTarget = 1536;
constexpr int kFastMinChunk = 256;
constexpr int kD = 128;
constexpr int kNRep = 4;

// Bytes per 16-token tile of one head: K codes, V codes, V meta (scale, min).
constexpr int kKC = kTile * kD;          // 2048
constexpr int kVC = kTile * kD / 2;      // 1024
constexpr int kVM = kTile * 8;           // 128
constexpr int kStageBytes = kKC + kVC + kVM;
constexpr int kKMeta = kD * 4;           // per-channel scales of one key group

struct __align__(128) SmemRI {
  uint8_t stage[kWarps][kStages][kStageBytes];
  float kmeta[kWarps][2][kD];
  float4 trig[2][kTile][32];  // per (token, pair pair): cos0, sin0, cos1, sin1; swizzled
  uint64_t bar[kWarps][kStages];
  int valid[kWarps][kStages];
  float w_hi[kD / 2], w_lo[kD / 2];
  int abort;
};

struct FastItem {
  int b, t0, t1, window;
};

__device__ inline FastItem decode_fast_item(const KvqView& v, const int* pref, int C, int item) {
  int lo = 0, hi = v.batch - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (pref[mid] <= item) lo = mid; else hi = mid - 1;
  }
  FastItem it;
  it.b = lo;
  const int chunk = item - pref[lo];
  const int T = seq_tokens(v, lo);
  const int nq = n_quantized(T, v.R);
  const int nqc = (nq + C - 1) / C;
  if (chunk < nqc) {
    it.window = 0;
    it.t0 = chunk * C;
    it.t1 = min(nq, it.t0 + C);
  } else {
    it.window = 1;
    it.t0 = nq;
    it.t1 = T;
  }
  return it;
}

__device__ __forceinline__ float2 cmul(float2 a, float2 b) {
  return make_float2(a.x * b.x - a.y * b.y, a.x * b.y + a.y * b.x);
}

__device__ __forceinline__ float2 rope_cs(int p, float w_hi, float w_lo) {
  float s, c;
  sincospif(2.f * rope_turns(p, w_hi, w_lo), &s, &c);
  return make_float2(c, s);
}

// Signed INT8 code j of word w as an exact float.
__device__ __forceinline__ float i8_to_f32(uint32_t w_offset_binary, uint32_t j) {
  const uint32_t x = prmt(w_offset_binary, 0x4B000000u, 0x7540u | j);
  return __uint_as_float(x) - 8388736.f;  // 2^23 + 128
}

__global__ void __launch_bounds__(kThreads, 2)
    split_rope_i8i4_kernel(KvqView v, const void* q, float scale, float* ws) {
  extern __shared__ __align__(128) unsigned char dyn[];
  SmemRI& sm = *reinterpret_cast<SmemRI*>(dyn);
  int* pref = reinterpret_cast<int*>(dyn + sizeof(SmemRI));
  __shared__ int s_C, s_items;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;
  const int G = v.kgroup;
  plan_items_ex(v, 1, G, kFastTarget, kFastMinChunk, pref, &s_C, &s_items);
  if (blockIdx.x == 0) store_plan(v, ws, pref, s_C, s_items);
  if (lane == 0) {
    for (int s = 0; s < kStages; ++s) mbar_init(&sm.bar[warp][s], 1);
    fence_mbar_init();
  }
  if (threadIdx.x < kD / 2) rope_split(v, threadIdx.x, &sm.w_hi[threadIdx.x], &sm.w_lo[threadIdx.x]);
  if (threadIdx.x == 0) sm.abort = 0;
  __syncthreads();

  // RoPE table producer role: pair tp, token offsets td + 4j within a tile.
  const int tp = threadIdx.x & 63, td = threadIdx.x >> 6;
  float2 Td[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) Td[j] = rope_cs(td + 4 * j, sm.w_hi[tp], sm.w_lo[tp]);
  const float2 R16 = rope_cs(16, sm.w_hi[tp], sm.w_lo[tp]);
  float2 Bp = make_float2(1.f, 0.f);

  const int C = s_C, n_items = s_items;
  float* part = plan_partials(ws, v.batch);
  const float qscale = scale * kLog2e;
  uint32_t load_seq = 0, cons_seq = 0;
  uint32_t tc = 0;  // tiles processed by this CTA: selects the RoPE table buffer
  const int h = warp;

  for (int item = blockIdx.x; item < n_items; item += gridDim.x) {
    const FastItem it = decode_fast_item(v, pref, C, item);
    const int ntiles = (it.t1 - it.t0 + kTile - 1) / kTile;
    const int T = it.window ? it.t1 : 0;

    // B operand: q * scale * log2(e) for query head 4h + g/2, split hi (even g) / lo (odd g)
    uint32_t bq[8][2];
    {
      const int hq = h * kNRep + (g >> 1);
      const long long qb = ((long long)it.b * v.Hq + hq) * kD + 32 * t;
#pragma unroll
      for (int s = 0; s < 8; ++s) {
        float x[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) x[j] = load_src(q, qb + 4 * s + j, v.src_bf16) * qscale;
        uint32_t h01, l01, h23, l23;
        split_hi_lo(x[0], x[1], h01, l01);
        split_hi_lo(x[2], x[3], h23, l23);
        bq[s][0] = (g & 1) ? l01 : h01;
        bq[s][1] = (g & 1) ? l23 : h23;
      }
    }

    // prologue: this warp's first tile loads
    auto issue = [&](int i) {
      const int stage = load_seq % kStages;
      ++load_seq;
      const int tok = it.t0 + i * kTile;
      uint64_t* bar = &sm.bar[warp][stage];
      const int pid = v.block_table[(long long)it.b * v.max_pages + tok / v.P];
      const bool ok = pid >= 0 && pid < v.n_pages;
      sm.valid[warp][stage] = ok;
      if (!ok) {
        atomicOr(v.status, KVQ_DEV_BAD_PAGE);
        mbar_arrive(bar);
        return;
      }
      const uint8_t* hbk = v.pages + (long long)pid * v.page_bytes + (long long)h * v.head_bytes;
      const int slot = tok % v.P;
      const bool gstart = (tok % G) == 0;
      mbar_arrive_expect_tx(bar, kStageBytes + (gstart ? kKMeta : 0));
      uint8_t* dst = sm.stage[warp][stage];
      if (v.P == kTile) {
        bulk_g2s(dst, hbk, kStageBytes, bar);
      } else {
        bulk_g2s(dst, hbk + slot * kD, kKC, bar);
        bulk_g2s(dst + kKC, hbk + v.off_vc + slot * (kD / 2), kVC, bar);
        bulk_g2s(dst + kKC + kVC, hbk + v.off_vm + slot * 8, kVM, bar);
      }
      if (gstart) {
        const int gslot = v.P >= G ? slot / G : 0;
        bulk_g2s(sm.kmeta[warp][(tok / G) & 1], hbk + v.off_km + gslot * kKMeta, kKMeta, bar);
      }
    };
    if (!it.window && lane == 0 && !sm.abort) {
      for (int i = 0; i < min(kStages, ntiles); ++i) issue(i);
    }
    __syncwarp();

    float O[8][4];
#pragma unroll
    for (int m = 0; m < 8; ++m) O[m][0] = O[m][1] = O[m][2] = O[m][3] = 0.f;
    float m_run = -INFINITY, l_loc = 0.f, mb = 0.f;

    for (int i = 0; i < ntiles; ++i) {
      const int tok0 = it.t0 + i * kTile;
      // ---- RoPE table for this tile (all warps), then one CTA barrier
      {
        if ((i & 15) == 0) Bp = rope_cs(tok0, sm.w_hi[tp], sm.w_lo[tp]);
        else Bp = cmul(Bp, R16);
        float* tb = reinterpret_cast<float*>(&sm.trig[tc & 1][0][0]);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int d = td + 4 * j;
          const float2 e = cmul(Bp, Td[j]);
          const int unit = (tp >> 1) ^ (d & 7);
          float* p = tb + (d * 32 + unit) * 4 + (tp & 1) * 2;
          p[0] = e.x;
          p[1] = e.y;
        }
      }
      named_bar_sync(1, kThreads);

      // ---- wait for this warp's tile
      int stage = 0;
      bool valid = true;
      if (!it.window) {
        stage = cons_seq % kStages;
        const uint32_t parity = (cons_seq / kStages) & 1;
        ++cons_seq;
        if (!*reinterpret_cast<volatile int*>(&sm.abort)) {
          if (!mbar_wait_bounded(&sm.bar[warp][stage], parity, kSpin)) {
            atomicOr(v.status, KVQ_DEV_TIMEOUT);
            sm.abort = 1;
            valid = false;
          } else {
            valid = sm.valid[warp][stage] != 0;
          }
        } else {
          valid = false;
        }
      }
      const uint8_t* buf = sm.stage[warp][stage];
      // per-channel key scales of this tile's group (channels 32t .. 32t+31)
      const float4* km = reinterpret_cast<const float4*>(&sm.kmeta[warp][(tok0 / G) & 1][32 * t]);

      // ---- QK: rows g and g+8 of the tile, channels 32t .. 32t+31
      float acc[4] = {0.f, 0.f, 0.f, 0.f}, accn[4] = {0.f, 0.f, 0.f, 0.f};
      const float4* trow0 = &sm.trig[tc & 1][g][0];
      const float4* trow1 = &sm.trig[tc & 1][g + 8][0];
      if (!it.window) {
        uint32_t kw[2][8];
#pragma unroll
        for (int r = 0; r < 2; ++r) {
          const uint4* src = reinterpret_cast<const uint4*>(buf + (g + 8 * r) * kD + 32 * t);
          const int rot = g & 1;
          const uint4 a = src[rot], b = src[rot ^ 1];
          const uint4 lo = rot ? b : a, hi = rot ? a : b;
          kw[r][0] = lo.x ^ 0x80808080u; kw[r][1] = lo.y ^ 0x80808080u;
          kw[r][2] = lo.z ^ 0x80808080u; kw[r][3] = lo.w ^ 0x80808080u;
          kw[r][4] = hi.x ^ 0x80808080u; kw[r][5] = hi.y ^ 0x80808080u;
          kw[r][6] = hi.z ^ 0x80808080u; kw[r][7] = hi.w ^ 0x80808080u;
        }
#pragma unroll
        for (int s = 0; s < 8; ++s) {
          uint32_t ahi[2][2], anl[2][2];
          const float4 ks = km[s];
#pragma unroll
          for (int r = 0; r < 2; ++r) {
            const float4 cs = (r ? trow1 : trow0)[(8 * t + s) ^ (g & 7)];
            const float k0 = i8_to_f32(kw[r][s], 0) * ks.x;
            const float k1 = i8_to_f32(kw[r][s], 1) * ks.y;
            const float k2 = i8_to_f32(kw[r][s], 2) * ks.z;
            const float k3 = i8_to_f32(kw[r][s], 3) * ks.w;
            const float r0 = k0 * cs.x - k1 * cs.y, r1 = k0 * cs.y + k1 * cs.x;
            const float r2 = k2 * cs.z - k3 * cs.w, r3 = k2 * cs.w + k3 * cs.z;
            split_hi_neglo(r0, r1, ahi[r][0], anl[r][0]);
            split_hi_neglo(r2, r3, ahi[r][1], anl[r][1]);
          }
          mma_16816(acc, ahi[0][0], ahi[1][0], ahi[0][1], ahi[1][1], bq[s][0], bq[s][1]);
          mma_16816(accn, anl[0][0], anl[1][0], anl[0][1], anl[1][1], bq[s][0], bq[s][1]);
        }
      } else {
        // residual window: bf16/f32 keys straight from k_win
#pragma unroll
        for (int s = 0; s < 8; ++s) {
          uint32_t ahi[2][2], anl[2][2];
#pragma unroll
          for (int r = 0; r < 2; ++r) {
            const int tok = tok0 + g + 8 * r;
            float k[4] = {0.f, 0.f, 0.f, 0.f};
            if (tok < T) {
              const long long wi = (((long long)it.b * v.R + (tok - it.t0)) * v.Hkv + h) * kD + 32 * t + 4 * s;
#pragma unroll
              for (int j = 0; j < 4; ++j) k[j] = load_src(v.k_win, wi + j, v.src_bf16);
            }
            const float4 cs = (r ? trow1 : trow0)[(8 * t + s) ^ (g & 7)];
            const float r0 = k[0] * cs.x - k[1] * cs.y, r1 = k[0] * cs.y + k[1] * cs.x;
            const float r2 = k[2] * cs.z - k[3] * cs.w, r3 = k[2] * cs.w + k[3] * cs.z;
            split_hi_neglo(r0, r1, ahi[r][0], anl[r][0]);
            split_hi_neglo(r2, r3, ahi[r][1], anl[r][1]);
          }
          mma_16816(acc, ahi[0][0], ahi[1][0], ahi[0][1], ahi[1][1], bq[s][0], bq[s][1]);
          mma_16816(accn, anl[0][0], anl[1][0], anl[0][1], anl[1][1], bq[s][0], bq[s][1]);
        }
      }
      float lg0 = acc[0] + acc[1] - accn[0] - accn[1];
      float lg1 = acc[2] + acc[3] - accn[2] - accn[3];
      const int last = it.window ? T : it.t1;
      if (!valid || tok0 + g >= last) lg0 = -INFINITY;
      if (!valid || tok0 + g + 8 >= last) lg1 = -INFINITY;

      // ---- online softmax for head t (tokens g, g+8 in this lane)
      float mx = fmaxf(lg0, lg1);
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
      const bool need = mx > m_run + kRescale;
      if (__any_sync(0xffffffffu, need)) {
        const float mn = need ? mx : m_run;
        const float alpha = (m_run == -INFINITY) ? 0.f : ex2(m_run - mn);
#pragma unroll
        for (int m = 0; m < 8; ++m) {
          O[m][0] *= alpha; O[m][1] *= alpha; O[m][2] *= alpha; O[m][3] *= alpha;
        }
        l_loc *= alpha;
        mb *= alpha;
        m_run = mn;
      }
      float p0 = 0.f, p1 = 0.f;
      if (m_run != -INFINITY) {
        p0 = ex2(lg0 - m_run);
        p1 = ex2(lg1 - m_run);
      }
      l_loc += p0 + p1;
      float pv0 = p0, pv1 = p1;
      if (!it.window) {
        const float2 m0 = valid ? reinterpret_cast<const float2*>(buf + kKC + kVC)[g] : make_float2(0.f, 0.f);
        const float2 m1 = valid ? reinterpret_cast<const float2*>(buf + kKC + kVC)[g + 8] : make_float2(0.f, 0.f);
        pv0 = p0 * m0.x;
        pv1 = p1 * m1.x;
        mb += p0 * m0.y + p1 * m1.y;
      }

      // ---- P' to the PV B layout: tokens 2t, 2t+1 (b0b1) and 2t+8, 2t+9 (b2b3) of head g/2
      const int src0 = 4 * (2 * t) + (g >> 1), src1 = src0 + 4;
      const float x0 = __shfl_sync(0xffffffffu, pv0, src0);
      const float y0 = __shfl_sync(0xffffffffu, pv1, src0);
      const float x1 = __shfl_sync(0xffffffffu, pv0, src1);
      const float y1 = __shfl_sync(0xffffffffu, pv1, src1);
      uint32_t b01, b23;
      {
        uint32_t hA, lA, hB, lB;
        split_hi_lo(x0, x1, hA, lA);
        split_hi_lo(y0, y1, hB, lB);
        b01 = (g & 1) ? lA : hA;
        b23 = (g & 1) ? lB : hB;
      }

      // ---- PV: A = V^T (channel rows 16g + 2m (+1), tokens 2t, 2t+1, 2t+8, 2t+9)
      if (!it.window) {
        uint2 vw[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int tok = 2 * t + (u & 1) + 8 * (u >> 1);
          vw[u] = *reinterpret_cast<const uint2*>(buf + kKC + tok * (kD / 2) + 8 * g);
        }
#pragma unroll
        for (int w = 0; w < 2; ++w) {
          const uint32_t a01 = w ? vw[0].y : vw[0].x, a1 = w ? vw[1].y : vw[1].x;
          const uint32_t c01 = w ? vw[2].y : vw[2].x, c1 = w ? vw[3].y : vw[3].x;
          const uint32_t xa[2] = {prmt(a01, a1, 0x5410u), prmt(a01, a1, 0x7632u)};
          const uint32_t xc[2] = {prmt(c01, c1, 0x5410u), prmt(c01, c1, 0x7632u)};
#pragma unroll
          for (int hb = 0; hb < 2; ++hb) {
#pragma unroll
            for (int sh = 0; sh < 2; ++sh) {
              const int m = 4 * w + 2 * hb + sh;
              const uint32_t ya = xa[hb] >> (8 * sh), yc = xc[hb] >> (8 * sh);
              // 1024 + c -> c and 1024 + 16c -> c, both exact (tensor-core accumulation
              // loses bits when an accumulator carries a large constant offset)
              const uint32_t lo_a = hsub2(and_or(ya, 0x000F000Fu, 0x64006400u), 0x64006400u);
              const uint32_t hi_a = hfma2(and_or(ya, 0x00F000F0u, 0x64006400u), 0x2C002C00u, 0xD400D400u);
              const uint32_t lo_c = hsub2(and_or(yc, 0x000F000Fu, 0x64006400u), 0x64006400u);
              const uint32_t hi_c = hfma2(and_or(yc, 0x00F000F0u, 0x64006400u), 0x2C002C00u, 0xD400D400u);
              mma_16816(O[m], lo_a, hi_a, lo_c, hi_c, b01, b23);
            }
          }
        }
      } else {
        // window values: f16 pairs (token 2t+u, 2t+1+u) per channel 16g + 2m (+1)
        float vv[4][16];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int tok = tok0 + 2 * t + (u & 1) + 8 * (u >> 1);
          const long long wi = (((long long)it.b * v.R + (tok - it.t0)) * v.Hkv + h) * kD + 16 * g;
#pragma unroll
          for (int c = 0; c < 16; ++c) vv[u][c] = tok < T ? load_src(v.v_win, wi + c, v.src_bf16) : 0.f;
        }
#pragma unroll
        for (int m = 0; m < 8; ++m) {
          const uint32_t a0 = pack_f16x2(vv[0][2 * m], vv[1][2 * m]);
          const uint32_t a1 = pack_f16x2(vv[0][2 * m + 1], vv[1][2 * m + 1]);
          const uint32_t a2 = pack_f16x2(vv[2][2 * m], vv[3][2 * m]);
          const uint32_t a3 = pack_f16x2(vv[2][2 * m + 1], vv[3][2 * m + 1]);
          mma_16816(O[m], a0, a1, a2, a3, b01, b23);
        }
      }

      ++tc;
      // ---- release the stage and refill it with tile i + kStages
      if (!it.window) {
        __syncwarp();
        if (lane == 0 && i + kStages < ntiles && !sm.abort) {
          fence_proxy_async();
          issue(i + kStages);
        }
        __syncwarp();
      }
    }

    // ---- epilogue: this warp's partial for query heads 4h .. 4h+3
#pragma unroll
    for (int o = 4; o < 32; o <<= 1) {
      l_loc += __shfl_xor_sync(0xffffffffu, l_loc, o);
      mb += __shfl_xor_sync(0xffffffffu, mb, o);
    }
    const int hq = h * kNRep + t;
    float* dst = part + ((long long)item * v.Hq + hq) * (kD + 2);
    if (g == 0) {
      dst[0] = m_run;
      dst[1] = l_loc;
    }
#pragma unroll
    for (int m = 0; m < 8; ++m) {
      dst[2 + 16 * g + 2 * m] = (O[m][0] + O[m][1]) + mb;
      dst[2 + 16 * g + 2 * m + 1] = (O[m][2] + O[m][3]) + mb;
    }
  }

  // drain: wait (bounded) for loads that were issued but never consumed
  if (lane == 0) {
    while (cons_seq < load_seq) {
      const int stage = cons_seq % kStages;
      const uint32_t parity = (cons_seq / kStages) & 1;
      ++cons_seq;
      mbar_wait_bounded(&sm.bar[warp][stage], parity, kSpin);
    }
  }
}

__global__ void combine_fast_kernel(KvqView v, float* ws, float* out) {
  const int hq = blockIdx.x, b = blockIdx.y;
  const int D = v.D;
  const int* pref = plan_prefix(ws);
  const float* part = plan_partials(ws, v.batch);
  const int i0 = pref[b], i1 = pref[b + 1];
  float M = -INFINITY;
  for (int i = i0; i < i1; ++i) M = fmaxf(M, part[((long long)i * v.Hq + hq) * (D + 2)]);
  float L = 0.f;
  for (int i = i0; i < i1; ++i) {
    const float* p = part + ((long long)i * v.Hq + hq) * (D + 2);
    L += p[0] == -INFINITY ? 0.f : p[1] * exp2f(p[0] - M);
  }
  const float invL = L > 0.f ? 1.f / L : 0.f;
  for (int c = threadIdx.x; c < D; c += blockDim.x) {
    float O = 0.f;
    for (int i = i0; i < i1; ++i) {
      const float* p = part + ((long long)i * v.Hq + hq) * (D + 2);
      if (p[0] != -INFINITY) O += p[2 + c] * exp2f(p[0] - M);
    }
    out[((long long)b * v.Hq + hq) * D + c] = O * invL;
  }
}

}  // namespace

bool fast_eligible(const KvqView& v) {
  return v.D == kD && v.Hkv == kWarps && v.n_rep == kNRep && v.kfmt == KVQ_INT8 &&
         v.kmode == KVQ_SYM_ABSMAX && v.kaxis == KVQ_PER_CHANNEL && v.rope_pre == 1 &&
         v.vfmt == KVQ_INT4 && v.vmode == KVQ_ASYM_MINMAX && v.vaxis == KVQ_PER_TOKEN &&
         v.vgroup == kD && v.kgroup % kTile == 0 && v.kgroup >= kTile * kStages && v.P % kTile == 0 &&
         v.batch <= 4096;
}

size_t fast_workspace_bytes(const KvqView& v, int batch) {
  const long long items = kFastTarget + 2LL * batch;
  return plan_header_bytes(batch) + (size_t)items * v.Hq * (v.D + 2) * sizeof(float);
}

kvq_status launch_fast(const KvqView& v, const void* q, float* out, float scale, void* ws,
                       cudaStream_t st) {
  const size_t smem = sizeof(SmemRI) + sizeof(int) * (v.batch + 1);
  static int occ_cache[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) return KVQ_ERR_UNSUPPORTED;
  if (!occ_cache[dev]) {
    if (cudaFuncSetAttribute(split_rope_i8i4_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)(sizeof(SmemRI) + sizeof(int) * 4097)) != cudaSuccess)
      return KVQ_ERR_CUDA;
    int occ = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, split_rope_i8i4_kernel, kThreads, smem) !=
        cudaSuccess)
      return KVQ_ERR_CUDA;
    occ_cache[dev] = occ > 0 ? occ : 1;
  }
  const int grid = num_sms() * occ_cache[dev];
  split_rope_i8i4_kernel<<<grid, kThreads, smem, st>>>(v, q, scale, static_cast<float*>(ws));
  combine_fast_kernel<<<dim3(v.Hq, v.batch), 128, 0, st>>>(v, static_cast<float*>(ws), out);
  return cudaGetLastError() == cudaSuccess ? KVQ_OK : KVQ_ERR_CUDA;
}

}  // namespace kvq
