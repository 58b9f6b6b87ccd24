// Tensor-core split-K decode attention for FP8 E4M3 (or E5M2) keys and values with
// per-head static scales (k_scale, v_scale), head_dim 128, 8 query heads per
// kv-head, no residual window: the 70B-shaped decode layer of the FP8 scheme
// ("Quantized KV Cache" / vLLM documentation, section "FP8 E4M3 with
// k_scale/v_scale": the cache stores e4m3(x / scale) and attention multiplies
// the scale back in).
//
// Work: a unit is (sequence, chunk of C tokens, kv-head); every warp takes units
// from a global counter and streams its 16-token tiles through a private 3-stage
// ring filled by 2-D TMA tensor copies with 128-byte swizzle (K tile, V tile),
// so the warps never wait on one another.
//
// Per 16-token tile and warp:
//   QK: K bytes -> f16 with cvt.e4m3x2 / cvt.e5m2x2 (exact), A = keys (16 tokens x 16
//       channels), B = q * k_scale * softmax_scale * log2(e) split hi/lo, two
//       8-column blocks (4 query heads x {hi, lo} each).  K needs no split: its
//       f16 values are exact.
//   softmax: online in base 2, lazy running max per head.
//   PV: A = V^T (16 channels x 16 tokens) as exact f16 (PRMT + cvt.e4m3x2),
//       B = p for the 8 query heads (one column each), once with the f16 hi
//       part of p and once with the residual, into the same accumulators;
//       v_scale multiplies the output once at the end.
#include <math.h>

#include "kvq_ptx.cuh"
#include "kvq_split_common.cuh"
#include "kvq_tmap.h"

namespace kvq {
namespace {

using namespace ptx;

constexpr int kTileT = 16;
constexpr int kWarps8 = 4;
constexpr int kThreads8 = kWarps8 * 32;
constexpr int kStages8 = 3;
constexpr int kRep8 = 8;
constexpr int kRowB = 128;                // bytes of one token's K (or V) codes
constexpr int kTileB = kTileT * kRowB;    // one TMA box
constexpr uint32_t kSpin8 = ptx::kWaitPolls;  // polls per bounded mbarrier wait
constexpr float kLog2e8 = 1.4426950408889634f;
constexpr float kRescale8 = 8.f;
constexpr float kMinit8 = -1e30f;

// Shared memory of one CTA.  Tiles arrive 128-byte swizzled: 16-byte chunk c of
// row r sits at chunk c ^ (r % 8), so the fragment loads below meet no bank
// conflict (tile bases are 1024-byte aligned).
struct __align__(1024) SmemF8 {
  uint8_t kv[kWarps8][kStages8][2][kTileB];  // [warp][stage][K, V]
  uint4 bq[kWarps8][8][32];                   // QK B fragments (two column blocks) per step and lane
  float pex[kWarps8][2][64];                  // p exchange: [token / 8][head * 8 + token % 8]
  uint64_t bar[kWarps8][kStages8];
  int valid[kWarps8][kStages8];
};

__device__ __forceinline__ const uint4* swz_row(const uint8_t* tile, int row) {
  return reinterpret_cast<const uint4*>(tile + row * kRowB);
}

template <bool kE5M2>
__global__ void __launch_bounds__(kThreads8)
    split_fp8_kernel(KvqView v, const void* q, float scale, float* ws, const __grid_constant__ CUtensorMap tmap) {
  extern __shared__ unsigned char dyn_raw[];
  // 1024-byte aligned base for the swizzled tiles
  unsigned char* dyn = dyn_raw + ((1024 - (smem_u32(dyn_raw) & 1023)) & 1023);
  SmemF8& sm = *reinterpret_cast<SmemF8*>(dyn);
  int* prefA = reinterpret_cast<int*>(dyn + sizeof(SmemF8));
  int* prefB = prefA + v.batch + 1;
  __shared__ int s_C, s_NA, s_NB, s_NS;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;
  const int lgP = __ffs(v.P) - 1;  // a power of two (checked on the host)
  // a warp takes one kv-head of an item: Hkv units per item, one worker per warp; no cuts
  fast_plan<kThreads8>(v, kTileT, v.Hkv, (int)gridDim.x * kWarps8, false, prefA, prefB, &s_C, &s_NA, &s_NB, &s_NS,
                       reinterpret_cast<int*>(&sm.kv[0][0][0][0]));
  if (blockIdx.x == 0) store_fast_plan(v, ws, prefA, prefB, s_C, s_NA, s_NB, s_NS);
  grid_dep_launch();  // the combine kernel may be scheduled; it waits for this grid to complete
  unsigned long long* counter =
      reinterpret_cast<unsigned long long*>(reinterpret_cast<char*>(ws) + fast_counter_offset(v.batch));
  if (lane == 0) {
    for (int s = 0; s < kStages8; ++s) mbar_init(&sm.bar[warp][s], 1);
    fence_mbar_init();
  }
  __syncthreads();

  const int C = s_C, NA = s_NA, NS = s_NS;
  const int n_units = (s_NA + s_NB) * v.Hkv;
  float* part = reinterpret_cast<float*>(reinterpret_cast<char*>(ws) + fast_header_bytes(v.batch));
  uint8_t (*ring)[2][kTileB] = sm.kv[warp];
  int lstage = 0, cstage = 0;
  uint32_t cphase = 0, n_loaded = 0, n_consumed = 0;
  bool stalled = false;

  int unit = blockIdx.x * kWarps8 + warp;
  const int unit_stride0 = gridDim.x * kWarps8;
  while (unit < n_units) {
    // the warp's next unit, read after this one
    unsigned long long nxt = 0;
    if (lane == 0) nxt = atomicAdd(counter, 1ull);
    const int pair = unit / v.Hkv, h = unit - pair * v.Hkv;
    const FastItem it = decode_fast_item(v, prefA, prefB, C, NA, NS, kTileT, false, pair);
    const int ntiles = (it.t1 - it.t0 + kTileT - 1) / kTileT;

    // QK B operand, step s: column block nb holds query heads 4nb .. 4nb+3; column g
    // is head 4nb + g/2, hi (even g) or lo (odd g); k-slots 2t, 2t+1 <- channels
    // c, c+1 and 2t+8, 2t+9 <- c+2, c+3 (c = 32t + 4s).
    {
      const float qs = scale * kLog2e8 * v.k_scale[h];
      __syncwarp();
#pragma unroll
      for (int s = 0; s < 8; ++s) {
        uint32_t f[2][2];
#pragma unroll
        for (int nb = 0; nb < 2; ++nb) {
          const long long qb = ((long long)it.b * v.Hq + h * kRep8 + 4 * nb + (g >> 1)) * kD + 32 * t + 4 * s;
          float x[4];
#pragma unroll
          for (int j = 0; j < 4; ++j) x[j] = load_src(q, qb + j, v.src_bf16) * qs;
          uint32_t h01, l01, h23, l23;
          split_hi_lo(x[0], x[1], h01, l01);
          split_hi_lo(x[2], x[3], h23, l23);
          f[nb][0] = (g & 1) ? l01 : h01;
          f[nb][1] = (g & 1) ? l23 : h23;
        }
        sm.bq[warp][s][lane] = make_uint4(f[0][0], f[0][1], f[1][0], f[1][1]);
      }
      __syncwarp();
    }

    // accumulators: O[m] rows g / g+8 = channels 16g + 2m / 16g + 2m + 1, columns
    // 2t, 2t+1 = query heads 2t, 2t+1; running max and sum for the QK heads t, 4+t
    float O[8][4];
#pragma unroll
    for (int m = 0; m < 8; ++m) O[m][0] = O[m][1] = O[m][2] = O[m][3] = 0.f;
    float m_run[2] = {kMinit8, kMinit8}, l_loc[2] = {0.f, 0.f};

    const int32_t* bt = v.block_table + (long long)it.b * v.max_pages;
    const long long head_off = (long long)h * v.head_bytes;
    auto issue = [&](int i, int pid) {
      const int stage = lstage;
      if (++lstage == kStages8) lstage = 0;
      ++n_loaded;
      const int tok = it.t0 + i * kTileT;
      uint64_t* bar = &sm.bar[warp][stage];
      const bool ok = pid >= 0 && pid < v.n_pages;
      sm.valid[warp][stage] = ok;
      if (!ok) {
        atomicOr(v.status, KVQ_DEV_BAD_PAGE);
        mbar_arrive(bar);
        return;
      }
      const long long byte0 = (long long)pid * v.page_bytes + head_off + (long long)(tok & (v.P - 1)) * kRowB;
      const int yk = (int)(byte0 / kRowB), yv = yk + v.off_vc / kRowB;
      mbar_arrive_expect_tx(bar, 2 * kTileB);
      const uint64_t pol = l2_evict_first();
      tma_load_2d_hint(ring[stage][0], &tmap, 0, yk, bar, pol);
      tma_load_2d_hint(ring[stage][1], &tmap, 0, yv, bar, pol);
    };
    int pf = 0;  // lane 0: page id of the next tile to load, read one tile ahead
    if (lane == 0 && !stalled) {
      fence_proxy_async();  // the ring's bytes were last written through the generic proxy
      for (int i = 0; i < min(kStages8, ntiles); ++i) issue(i, bt[(it.t0 + i * kTileT) >> lgP]);
      if (kStages8 < ntiles) pf = bt[(it.t0 + kStages8 * kTileT) >> lgP];
    }
    __syncwarp();

    for (int i = 0; i < ntiles; ++i) {
      const int stage = cstage;
      bool valid = false;
      if (!stalled) {
        if (!mbar_wait_bounded(&sm.bar[warp][stage], cphase, kSpin8)) {
          atomicOr(v.status, KVQ_DEV_TIMEOUT);
          stalled = true;
        } else {
          valid = sm.valid[warp][stage] != 0;
        }
      }
      if (++cstage == kStages8) {
        cstage = 0;
        cphase ^= 1u;
      }
      ++n_consumed;
      const uint8_t* kt = ring[stage][0];
      const uint8_t* vt = ring[stage][1];

      // ---- QK: rows g / g+8 = tile tokens g / g+8, channels 32t .. 32t+31 (chunks 2t, 2t+1)
      float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        const uint4 k0 = swz_row(kt, g)[(2 * t + hh) ^ g];
        const uint4 k1 = swz_row(kt, g + 8)[(2 * t + hh) ^ g];
        const uint32_t w0[4] = {k0.x, k0.y, k0.z, k0.w}, w1[4] = {k1.x, k1.y, k1.z, k1.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int s = 4 * hh + j;
          const uint4 b = sm.bq[warp][s][lane];
          const uint32_t a0 = fp8x2_to_f16x2<kE5M2>(lo16(w0[j])), a2 = fp8x2_to_f16x2<kE5M2>(hi16(w0[j]));
          const uint32_t a1 = fp8x2_to_f16x2<kE5M2>(lo16(w1[j])), a3 = fp8x2_to_f16x2<kE5M2>(hi16(w1[j]));
          mma_16816(acc[0], a0, a1, a2, a3, b.x, b.y);
          mma_16816(acc[1], a0, a1, a2, a3, b.z, b.w);
        }
      }
      // tokens at or past the chunk end (last tile of a sequence) take no weight
      const int nvalid = valid ? min(kTileT, it.t1 - (it.t0 + i * kTileT)) : 0;
      float lg[2][2];
#pragma unroll
      for (int nb = 0; nb < 2; ++nb) {
        lg[nb][0] = g < nvalid ? acc[nb][0] + acc[nb][1] : -INFINITY;
        lg[nb][1] = g + 8 < nvalid ? acc[nb][2] + acc[nb][3] : -INFINITY;
      }

      // ---- softmax (QK heads t and 4+t), lazy max
      const bool need = fmaxf(lg[0][0], lg[0][1]) > m_run[0] + kRescale8 ||
                        fmaxf(lg[1][0], lg[1][1]) > m_run[1] + kRescale8;
      if (__any_sync(0xffffffffu, need)) {
        float alpha[2];
#pragma unroll
        for (int nb = 0; nb < 2; ++nb) {
          float mx = fmaxf(lg[nb][0], lg[nb][1]);
          mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
          mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
          mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
          const float mn = fmaxf(m_run[nb], mx);
          alpha[nb] = ex2(m_run[nb] - mn);
          l_loc[nb] *= alpha[nb];
          m_run[nb] = mn;
        }
        // the O columns of this lane are heads 2t, 2t+1: their factors live in the
        // lanes of QK head 2t (t' = 2t % 4, block 2t / 4) and 2t+1
        const int src = (2 * t) & 3;
        const float a00 = __shfl_sync(0xffffffffu, alpha[0], src), a01 = __shfl_sync(0xffffffffu, alpha[1], src);
        const float a10 = __shfl_sync(0xffffffffu, alpha[0], src + 1),
                    a11 = __shfl_sync(0xffffffffu, alpha[1], src + 1);
        const float f0 = t < 2 ? a00 : a01, f1 = t < 2 ? a10 : a11;
#pragma unroll
        for (int m = 0; m < 8; ++m) {
          O[m][0] *= f0; O[m][2] *= f0;
          O[m][1] *= f1; O[m][3] *= f1;
        }
      }
      float p[2][2];
#pragma unroll
      for (int nb = 0; nb < 2; ++nb) {
        p[nb][0] = ex2(lg[nb][0] - m_run[nb]);
        p[nb][1] = ex2(lg[nb][1] - m_run[nb]);
        l_loc[nb] += p[nb][0] + p[nb][1];
      }
      // ---- PV B operand: column g = query head g, k-slots 2t, 2t+1 (tokens 2t, 2t+1)
      //      and 2t+8, 2t+9, through a per-warp exchange buffer
      float* pe = &sm.pex[warp][0][0];
      __syncwarp();
#pragma unroll
      for (int nb = 0; nb < 2; ++nb) {
        pe[(4 * nb + t) * 8 + g] = p[nb][0];
        pe[64 + (4 * nb + t) * 8 + g] = p[nb][1];
      }
      __syncwarp();
      const float2 x01 = *reinterpret_cast<const float2*>(pe + g * 8 + 2 * t);
      const float2 x89 = *reinterpret_cast<const float2*>(pe + 64 + g * 8 + 2 * t);
      uint32_t b0h, b0l, b1h, b1l;
      split_hi_lo(x01.x, x01.y, b0h, b0l);
      split_hi_lo(x89.x, x89.y, b1h, b1l);

      // ---- PV: A = V^T, rows g / g+8 = channels 16g + 2m / +1 (chunk g of each token row),
      //      k-slots 2t, 2t+1, 2t+8, 2t+9 = tokens 2t, 2t+1, 2t+8, 2t+9
      const uint4 z4 = make_uint4(0u, 0u, 0u, 0u);  // rows past the end may hold any byte, even NaN
      const uint4 v0 = 2 * t < nvalid ? swz_row(vt, 2 * t)[g ^ (2 * t)] : z4;
      const uint4 v1 = 2 * t + 1 < nvalid ? swz_row(vt, 2 * t + 1)[g ^ (2 * t + 1)] : z4;
      const uint4 v2 = 2 * t + 8 < nvalid ? swz_row(vt, 2 * t + 8)[g ^ (2 * t)] : z4;
      const uint4 v3 = 2 * t + 9 < nvalid ? swz_row(vt, 2 * t + 9)[g ^ (2 * t + 1)] : z4;
      const uint32_t wa[4] = {v0.x, v0.y, v0.z, v0.w}, wb[4] = {v1.x, v1.y, v1.z, v1.w};
      const uint32_t wc[4] = {v2.x, v2.y, v2.z, v2.w}, wd[4] = {v3.x, v3.y, v3.z, v3.w};
#pragma unroll
      for (int m = 0; m < 8; ++m) {
        // bytes 2(m%2), 2(m%2)+1 of word m/2 of the two tokens: (ch even: tok A, tok B, ch odd: tok A, tok B)
        const uint32_t sel = (m & 1) ? 0x7362u : 0x5140u;
        const uint32_t ya = prmt(wa[m >> 1], wb[m >> 1], sel), yc = prmt(wc[m >> 1], wd[m >> 1], sel);
        const uint32_t a0 = fp8x2_to_f16x2<kE5M2>(lo16(ya)), a1 = fp8x2_to_f16x2<kE5M2>(hi16(ya));
        const uint32_t a2 = fp8x2_to_f16x2<kE5M2>(lo16(yc)), a3 = fp8x2_to_f16x2<kE5M2>(hi16(yc));
        mma_16816(O[m], a0, a1, a2, a3, b0h, b1h);
        mma_16816(O[m], a0, a1, a2, a3, b0l, b1l);
      }

      // ---- release the stage and refill it with tile i + kStages8
      __syncwarp();
      if (lane == 0 && i + kStages8 < ntiles && !stalled) {
        fence_proxy_async();
        issue(i + kStages8, pf);
        if (i + kStages8 + 1 < ntiles) pf = bt[(it.t0 + (i + kStages8 + 1) * kTileT) >> lgP];
      }
      __syncwarp();
    }

    // ---- epilogue: partial records of query heads 8h .. 8h+7
#pragma unroll
    for (int nb = 0; nb < 2; ++nb) {
#pragma unroll
      for (int o = 4; o < 32; o <<= 1) l_loc[nb] += __shfl_xor_sync(0xffffffffu, l_loc[nb], o);
    }
    float* rec = part + ((long long)pair * v.Hq + h * kRep8) * (kD + 4);
    if (g == 0) {
#pragma unroll
      for (int nb = 0; nb < 2; ++nb) {
        rec[(4 * nb + t) * (kD + 4) + 0] = m_run[nb];
        rec[(4 * nb + t) * (kD + 4) + 1] = l_loc[nb];
      }
    }
    const float vs = v.v_scale[h];
#pragma unroll
    for (int m = 0; m < 8; ++m) {
#pragma unroll
      for (int e = 0; e < 2; ++e) {  // query head 2t + e
        float* o = rec + (2 * t + e) * (kD + 4) + 4 + 16 * g + 2 * m;
        *reinterpret_cast<float2*>(o) = make_float2(O[m][e] * vs, O[m][2 + e] * vs);
      }
    }
    unit = unit_stride0 + (int)__shfl_sync(0xffffffffu, (unsigned)nxt, 0);
  }

  // drain: wait (bounded) for loads that were issued but never consumed
  if (lane == 0) {
    while (n_consumed < n_loaded) {
      mbar_wait_bounded(&sm.bar[warp][cstage], cphase, kSpin8);
      if (++cstage == kStages8) {
        cstage = 0;
        cphase ^= 1u;
      }
      ++n_consumed;
    }
  }
}

long long pool_rows(const KvqView& v) { return (long long)v.n_pages * v.page_bytes / kRowB; }

}  // namespace

bool fp8_shape_eligible(const KvqView& v) {
  return v.D == kD && v.n_rep == kRep8 && (v.kfmt == KVQ_FP8_E4M3 || v.kfmt == KVQ_FP8_E5M2) &&
         v.vfmt == v.kfmt && v.R == 0 &&
         v.P >= kTileT && (v.P & (v.P - 1)) == 0 && v.page_bytes % kRowB == 0 && v.head_bytes % kRowB == 0 && v.off_vc % kRowB == 0 &&
         v.batch <= 4096;
}

bool fp8_eligible(const KvqView& v) {
  return fp8_shape_eligible(v) && (reinterpret_cast<uintptr_t>(v.pages) & 15) == 0 && pool_rows(v) > 0 &&
         pool_rows(v) < (1LL << 31) && tensor_map_encoder() != nullptr;
}

kvq_status launch_fp8(const KvqView& v, const void* q, float* out, float scale, void* ws, cudaStream_t st) {
  // the page pool as rows of 128 bytes, read in 16-row boxes with 128-byte swizzle
  CUtensorMap tmap;
  const cuuint64_t dims[2] = {(cuuint64_t)kRowB, (cuuint64_t)pool_rows(v)};
  const cuuint64_t strides[1] = {(cuuint64_t)kRowB};
  const cuuint32_t box[2] = {(cuuint32_t)kRowB, (cuuint32_t)kTileT};
  const cuuint32_t estr[2] = {1, 1};
  if (tensor_map_encoder()(&tmap, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, v.pages, dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return KVQ_ERR_UNSUPPORTED;
  const size_t smem = sizeof(SmemF8) + 1024 + sizeof(int) * 2 * (v.batch + 1);
  const bool e5m2 = v.kfmt == KVQ_FP8_E5M2;
  void (*kern)(KvqView, const void*, float, float*, const CUtensorMap) =
      e5m2 ? split_fp8_kernel<true> : split_fp8_kernel<false>;
  int occ = 0;
  const kvq_status so = occupancy_once(kSlotFp8 + (e5m2 ? 1 : 0), kern, kThreads8, smem,
                                       sizeof(SmemF8) + 1024 + sizeof(int) * 2 * 4097, &occ);
  if (so != KVQ_OK) return so;
  const int grid = num_sms() * occ;
  if (cudaMemsetAsync(static_cast<char*>(ws) + fast_counter_offset(v.batch), 0, 8, st) != cudaSuccess)
    return KVQ_ERR_CUDA;
  kern<<<grid, kThreads8, smem, st>>>(v, q, scale, static_cast<float*>(ws), tmap);
  if (cudaGetLastError() != cudaSuccess) return KVQ_ERR_CUDA;
  return launch_split_combine(v, static_cast<float*>(ws), out, st) == cudaSuccess ? KVQ_OK : KVQ_ERR_CUDA;
}

}  // namespace kvq
