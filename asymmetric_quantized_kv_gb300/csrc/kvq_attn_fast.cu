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
//   QK: K codes -> fp32 (PRMT into the mantissa of 2^23, minus 2^23 + 128)
//       -> x per-channel scale -> RoPE rotation by the token's
//       absolute position -> split into f16 hi + (hi - x) -> two mma.m16n8k16
//       per 16 channels with A = keys (16 tokens x 16 channels) and B = q (16
//       channels x 8 columns: 4 query heads x {hi, lo} halves of
//       q*scale*log2(e)).  The hi/lo split of both operands keeps the logits to
//       ~2^-21 relative.  Scaling and rotation run as packed f32x2 arithmetic on
//       the even channels (x0, x2) and odd channels (x1, x3) of two RoPE pairs.
//   RoPE table: cos/sin of every (token, pair) of two tiles, in one of two
//       shared buffers handed between the 8 warps through full/empty mbarriers,
//       so warps may drift by up to two tiles instead of meeting at a CTA
//       barrier every tile.  With the caller's table (kvq_cache.rope_table,
//       covering every position the pages hold, rounded up to a whole table) a
//       second instance fills the buffer with one bulk copy of its 32 rows,
//       requested one table ahead; otherwise the CTA computes it.
//   softmax: online in base 2, one running max per head, raised lazily (only
//       when a logit exceeds it by more than 2^8; the common tile needs no
//       cross-lane reduction).
//   PV: with v = c * s + m per token (asymmetric INT4, c in 0..15), written as
//       v = (c - 8) s + (m + 8 s): A = V^T codes (16 channels x 16 tokens) as the
//       centred f16 values c - 8 (exact: each nibble OR-ed into the mantissa of
//       1024, then one f16 subtract or fused multiply-add), B = p * v_scale split
//       hi/lo, and the per-token midpoints m + 8 s enter through a running sum of
//       p * (m + 8 s).  Centring keeps the tensor-core sum of the order of the
//       output: with the codes 0..15 as they are, the code sum and the minimum sum
//       are each many times larger than the output and cancel (the paged layer's
//       worst head was at 4.1e-4 relative L2 that way, 1.6e-5 centred).
// Residual-window items use the same steps on the source-dtype rows.
// Partials (max, sum, unnormalised output) per (item, query head) go to the
// workspace; the combine kernel merges them.
// Scales and minima stored as binary16 take a second instance (M16): the tile's
// value (scale, min) rows and a group's key scales arrive in half the bytes and
// are widened to fp32 where they are read.
#include <math.h>

#include "kvq_ptx.cuh"
#include "kvq_split_common.cuh"

namespace kvq {
namespace {

using namespace ptx;

constexpr int kTile = 16;
constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
constexpr int kStages = 2;
constexpr uint32_t kSpin = ptx::kWaitPolls;  // polls per bounded mbarrier wait
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kRescale = 8.f;  // lazy rescale threshold in log2 units
constexpr float kMinit = -1e30f;  // running max before the first logit (finite: no inf - inf)
constexpr int kSuper = 2;    // tiles per RoPE table (one handoff between the warps per table)
constexpr int kReseed = 16;  // RoPE table entries are recomputed exactly every kReseed tables
constexpr int kNRep = 4;
constexpr uint32_t kTableBytes = kSuper * kTile * 32 * 16;  // one shared RoPE table: 32 rows of 32 float4

// Bytes per 16-token tile of one head: K codes, V codes, V meta (scale, min);
// a tile that starts a key group also carries the group's 128 key scales.  With
// binary16 scales and minima (M16) the metadata halves.
constexpr int kKC = kTile * kD;          // 2048
constexpr int kVC = kTile * kD / 2;      // 1024
template <bool M16> constexpr int vm_bytes() { return kTile * (M16 ? 4 : 8); }    // 64 / 128
template <bool M16> constexpr int stage_bytes() { return kKC + kVC + vm_bytes<M16>(); }
template <bool M16> constexpr int kmeta_bytes() { return kD * (M16 ? 2 : 4); }   // 256 / 512
constexpr int kStageAlloc = stage_bytes<false>() + kmeta_bytes<false>();

// two binary16 values (low half first) widened to fp32
__device__ __forceinline__ float2 half2_to_float2(uint32_t w) {
  return __half22float2(*reinterpret_cast<const __half2*>(&w));
}

// Shared-memory layouts are chosen so that every 64/128-bit load of a warp
// meets no bank conflict within the quarter- or half-warp that the hardware
// serves in one wavefront:
//   trig: per (token row, unit of two RoPE pairs A = 2u, B = 2u + 1) the float4
//         (cos A, cos B, sin A, sin B); units are XOR-swizzled by
//         (2 * (u / 8) + row % 2) % 8;
//   kmeta: the 128 key scales of the current group as 4 rows of 32, each row
//         padded to 36 floats, one row per lane quarter t; each quad of
//         channels c..c+3 is stored as (s_c, s_c+2, s_c+1, s_c+3) so that the
//         even and odd channels of two pairs are adjacent register pairs;
//   tokens: MMA row r holds tile token sig(r) = r ^ ((r >> 1) & 1), which
//         spreads the value rows a half-warp reads over two bank offsets.
struct __align__(128) SmemRI {
  uint8_t stage[kWarps][kStages][kStageAlloc];
  float4 trig[2][kSuper * kTile][32];
  uint2 bq[kWarps][8][32];  // q B fragments of the current item, per warp, step and lane
  float4 rstep[32];         // (cos A, cos B, sin A, sin B) of kSuper * 16 theta per unit
  float kmeta[kWarps][4][36];
  uint64_t bar[kWarps][kStages];
  uint64_t tfull[2], tempty[2];
  int valid[kWarps][kStages];
  float w_hi[kD / 2], w_lo[kD / 2];
};
static_assert(kStageAlloc % 16 == 0, "bulk-copy destinations must stay 16-byte aligned");
static_assert(sizeof(SmemRI::stage) >= 2 * kThreads * sizeof(int), "plan scratch lives in the stage ring");
static_assert(stage_bytes<true>() % 16 == 0 && vm_bytes<true>() % 16 == 0 && kmeta_bytes<true>() % 16 == 0 &&
                  stage_bytes<true>() + kmeta_bytes<true>() <= kStageAlloc,
              "binary16 tiles: 16-byte bulk-copy sizes that fit the stage");

__device__ __forceinline__ float2 rope_cs(int p, float w_hi, float w_lo) {
  float s, c;
  sincospif(2.f * rope_turns(p, w_hi, w_lo), &s, &c);
  return make_float2(c, s);
}

// byte j of w placed in the low mantissa bits of 2^23: the float 2^23 + byte
__device__ __forceinline__ float magic_f32(uint32_t w, int j) {
  return __uint_as_float(prmt(w, 0x4B000000u, 0x7540u | j));
}
// (2^23 + 128, 2^23 + 128): 2^23 + u minus this is the signed code u - 128
__device__ __forceinline__ float2 magic_bias() { return make_float2(8388736.f, 8388736.f); }

__device__ __forceinline__ int sig(int x) { return x ^ ((x >> 1) & 1); }

// The 4-bit code in the low / high nibble of the low byte of each f16 half of w,
// centred: f16x2 (c - 8), exact.  OR-ing the nibble into the mantissa of 1024
// gives 1024 + c (low) or 1024 + 16c (high); subtracting 1032, or multiplying by
// 1/16 and subtracting 72, leaves c - 8.
__device__ __forceinline__ uint32_t centred_lo(uint32_t w) {
  return hsub2(and_or(w, 0x000F000Fu, 0x64006400u), 0x64086408u);
}
__device__ __forceinline__ uint32_t centred_hi(uint32_t w) {
  return hfma2(and_or(w, 0x00F000F0u, 0x64006400u), 0x2C002C00u, 0xD480D480u);
}

// Bounded wait on an mbarrier phase by every lane; a timeout raises the status
// flag and this thread's `stalled` flag, after which it attempts no further wait
// (the kernel then runs to completion on whatever the buffers hold).
__device__ __forceinline__ void bounded_wait(uint64_t* bar, uint32_t parity, bool& stalled, int* status) {
  if (stalled) return;
  if (!mbar_wait_bounded(bar, parity, kSpin)) {
    atomicOr(status, KVQ_DEV_TIMEOUT);
    stalled = true;
  }
}

// One arrival per warp, after every lane's shared-memory accesses are ordered
// before it by the warp barrier.
__device__ __forceinline__ void warp_arrive(uint64_t* bar) {
  __syncwarp();
  if ((threadIdx.x & 31) == 0) mbar_arrive(bar);
}

// Per-warp attention state of one item: PV accumulators (16-channel MMA tiles m,
// rows g / g+8 = channels 16g + 2m / 16g + 2m + 1, columns head t hi / (hi - x)),
// running max (log2 units), this lane's share of the softmax sum and of the
// p * v_min sum.
struct Acc {
  float O[8][4];
  float m_run, l_loc, mb;
};

// RoPE table producer: thread (unit u = tid % 32, rows d0 + 8j, j < 2 * kSuper)
// owns 2 * kSuper float4 entries per table, e^{i (tok0 + d) theta} for pairs 2u,
// 2u + 1.  Entries are advanced table to table by e^{i 32 theta} (read back from
// the thread's own slots of the previous table's buffer) and recomputed exactly
// at an item's first table and every kReseed tables.

// (cos A, cos B, sin A, sin B) of pairs A = 2u, B = 2u + 1 at position pos
__device__ __forceinline__ float4 trig_entry(const float* w_hi, const float* w_lo, int pos, int u) {
  const float2 a = rope_cs(pos, w_hi[2 * u], w_lo[2 * u]);
  const float2 b = rope_cs(pos, w_hi[2 * u + 1], w_lo[2 * u + 1]);
  return make_float4(a.x, b.x, a.y, b.y);
}
__device__ __forceinline__ float4 trig_entry(const SmemRI& sm, int pos, int u) {
  return trig_entry(sm.w_hi, sm.w_lo, pos, u);
}

// Slot of unit u in a table row of token parity `odd`: the bank swizzle of the
// shared table, also used by the caller's table (whose row p is stored as the
// shared row of parity p & 1, so a bulk copy of rows from an even position
// lands in the shared layout).
__device__ __forceinline__ int trig_slot(int u, int odd) { return u ^ ((((u >> 3) << 1) | odd) & 7); }

__device__ __forceinline__ void trig_produce(SmemRI& sm, uint32_t buf, int ip, int tok0) {
  const int u = threadIdx.x & 31, d0 = threadIdx.x >> 5;
  const float4 r = sm.rstep[u];
  const float2 rc = make_float2(r.x, r.y), rs = make_float2(r.z, r.w);
#pragma unroll
  for (int j = 0; j < 2 * kSuper; ++j) {
    const int d = d0 + 8 * j;
    const int slot = trig_slot(u, d & 1);
    float4 e;
    if (ip % kReseed == 0) {
      e = trig_entry(sm, tok0 + d, u);
    } else {
      const float4 p = sm.trig[buf ^ 1][d][slot];
      const float2 c = make_float2(p.x, p.y), s = make_float2(p.z, p.w);
      const float2 c2 = sub2(mul2(c, rc), mul2(s, rs));
      const float2 s2 = fma2(c, rs, mul2(s, rc));
      e = make_float4(c2.x, c2.y, s2.x, s2.y);
    }
    sm.trig[buf][d][slot] = e;
  }
}

// Rotate two RoPE pairs held as even channels X = (x0, x2) and odd channels
// Y = (x1, x3) by the table's float4 (cos A, cos B, sin A, sin B), then split
// each rotated half into f16x2 hi and (hi - x): *0 = channels (0, 2), *1 = (1, 3).
__device__ __forceinline__ void rot_split(float2 X, float2 Y, float4 cs, uint32_t& hi0, uint32_t& nl0,
                                          uint32_t& hi1, uint32_t& nl1) {
  const float2 C = make_float2(cs.x, cs.y), S = make_float2(cs.z, cs.w);
  const float2 RA = sub2(mul2(X, C), mul2(Y, S));
  const float2 RB = fma2(X, S, mul2(Y, C));
  split_hi_neglo(RA.x, RA.y, hi0, nl0);
  split_hi_neglo(RB.x, RB.y, hi1, nl1);
}

// Online-softmax step for the two logits of this lane (tokens of MMA rows g and
// g+8, head t), then the PV B operand: P' = p * pscale for k-slots 2t, 2t+1 and
// 2t+8, 2t+9 of column g (head g/2, hi half for even g, (hi - x) for odd g).
// m0, m1 = (scale, minimum) of the two tokens; the midpoint m + 8 s goes to A.mb.
__device__ __forceinline__ void softmax_step(Acc& A, float lg0, float lg1, float2 m0, float2 m1, int g, int t,
                                             uint32_t& b01, uint32_t& b23) {
  if (__any_sync(0xffffffffu, fmaxf(lg0, lg1) > A.m_run + kRescale)) {
    float mx = fmaxf(lg0, lg1);
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
    const float mn = fmaxf(A.m_run, mx);
    const float alpha = ex2(A.m_run - mn);
#pragma unroll
    for (int m = 0; m < 8; ++m) {
      A.O[m][0] *= alpha; A.O[m][1] *= alpha; A.O[m][2] *= alpha; A.O[m][3] *= alpha;
    }
    A.l_loc *= alpha;
    A.mb *= alpha;
    A.m_run = mn;
  }
  const float p0 = ex2(lg0 - A.m_run), p1 = ex2(lg1 - A.m_run);
  A.l_loc += p0 + p1;
  A.mb = fmaf(p1, fmaf(8.f, m1.x, m1.y), fmaf(p0, fmaf(8.f, m0.x, m0.y), A.mb));
  const float pv0 = p0 * m0.x, pv1 = p1 * m1.x;
  const int src0 = 4 * (2 * t) + (g >> 1), src1 = src0 + 4;
  const float x0 = __shfl_sync(0xffffffffu, pv0, src0);
  const float y0 = __shfl_sync(0xffffffffu, pv1, src0);
  const float x1 = __shfl_sync(0xffffffffu, pv0, src1);
  const float y1 = __shfl_sync(0xffffffffu, pv1, src1);
  uint32_t hA, nA, hB, nB;
  split_hi_neglo(x0, x1, hA, nA);
  split_hi_neglo(y0, y1, hB, nB);
  b01 = (g & 1) ? nA : hA;
  b23 = (g & 1) ? nB : hB;
}

// TAB: the RoPE tables come from the caller's table (which covers every position
// the cache can hold); otherwise the CTA computes them.
template <bool M16, bool TAB>
__global__ void __launch_bounds__(kThreads, 2)
    split_rope_i8i4_kernel(KvqView v, const void* q, float scale, float* ws) {
  constexpr int kStageBytes = stage_bytes<M16>(), kKMeta = kmeta_bytes<M16>(), kVM = vm_bytes<M16>();
  extern __shared__ __align__(128) unsigned char dyn[];
  SmemRI& sm = *reinterpret_cast<SmemRI*>(dyn);
  int* prefA = reinterpret_cast<int*>(dyn + sizeof(SmemRI));
  int* prefB = prefA + v.batch + 1;
  __shared__ int s_C, s_NA, s_NB, s_NS, s_next[2];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;
  const int G = v.kgroup;  // powers of two (checked on the host)
  const int lgG = __ffs(G) - 1, lgP = __ffs(v.P) - 1;
  // one CTA takes all kv-heads of an item: one unit per item, gridDim.x workers
  fast_plan<kThreads>(v, G, 1, (int)gridDim.x, true, prefA, prefB, &s_C, &s_NA, &s_NB, &s_NS,
                      reinterpret_cast<int*>(&sm.stage[0][0][0]));
  if (blockIdx.x == 0) store_fast_plan(v, ws, prefA, prefB, s_C, s_NA, s_NB, s_NS);
  grid_dep_launch();  // the combine kernel may be scheduled; it waits for this grid to complete
  unsigned long long* counter =
      reinterpret_cast<unsigned long long*>(reinterpret_cast<char*>(ws) + fast_counter_offset(v.batch));
  if (lane == 0) {
    for (int s = 0; s < kStages; ++s) mbar_init(&sm.bar[warp][s], 1);
  }
  if (threadIdx.x == 0) {
    for (int b = 0; b < 2; ++b) {
      mbar_init(&sm.tfull[b], kWarps);
      mbar_init(&sm.tempty[b], kWarps);
    }
  }
  if (lane == 0) fence_mbar_init();
  if constexpr (!TAB) {
    if (threadIdx.x < kD / 2) rope_split(v, threadIdx.x, &sm.w_hi[threadIdx.x], &sm.w_lo[threadIdx.x]);
    __syncthreads();
    if (threadIdx.x < 32) sm.rstep[threadIdx.x] = trig_entry(sm, kSuper * kTile, threadIdx.x);
  }
  __syncthreads();


  const int C = s_C, NA = s_NA, NS = s_NS, n_items = s_NA + s_NB;
  float* part = reinterpret_cast<float*>(reinterpret_cast<char*>(ws) + fast_header_bytes(v.batch));
  const float qscale = scale * kLog2e;
  const int h = warp;
  const int sg = sig(g);  // tile token of MMA row g (row g + 8: token sg + 8)
  const int tkey = ((t << 1) | (sg & 1)) & 7;
  const long long head_off = (long long)h * v.head_bytes;
  // this warp's ring: lane 0 loads at lstage, everyone consumes at cstage / cphase
  int lstage = 0, cstage = 0;
  uint32_t cphase = 0, n_loaded = 0, n_consumed = 0;
  bool stalled = false;  // set by a timed-out wait: no further waits
  uint32_t tc = 0;  // RoPE tables used by this CTA: table tc in buffer tc & 1, its use tc >> 1

  const float4* rope_tab = static_cast<const float4*>(v.rope_table);
  // thread 0: copy CTA table tcp (first token tok0) into its buffer once the
  // warps are done with the buffer's previous use; this arrival carries the
  // byte count (a timed-out wait leaves the buffer as it is).  tok0 is a
  // multiple of 32 (items start on key-group boundaries, G >= 32), so the rows
  // have the shared table's parity, and tok0 + 32 <= rope_positions (the host
  // takes this instance only then)
  auto issue_copy = [&](uint32_t tcp, int tok0) {
    const uint32_t b = tcp & 1;
    if (tcp >= 2) bounded_wait(&sm.tempty[b], ((tcp >> 1) - 1) & 1, stalled, v.status);
    if (!stalled) {
      fence_proxy_async();  // the buffer may last have been written through the generic proxy
      mbar_arrive_expect_tx(&sm.tfull[b], kTableBytes);
      bulk_g2s_hint(&sm.trig[b][0][0], rope_tab + (long long)tok0 * 32, kTableBytes, &sm.tfull[b],
                    l2_evict_last());
    } else {
      mbar_arrive(&sm.tfull[b]);
    }
  };
  // every warp: make CTA table tcp (item table ip, first token tok0) ready.  A
  // copied table's bytes were requested by thread 0 (at the item's start for its
  // first table, else one table ahead), whose arrival that was; the other warps
  // arrive.  A computed table: wait for the buffer, compute this thread's
  // entries, arrive.
  auto produce = [&](uint32_t tcp, int ip, int tok0, bool first) {
    const uint32_t b = tcp & 1;
    if constexpr (TAB) {
      if (warp != 0) {
        warp_arrive(&sm.tfull[b]);
      } else if (first) {
        __syncwarp();
        if (lane == 0) issue_copy(tcp, tok0);
      }
    } else {
      if (tcp >= 2) bounded_wait(&sm.tempty[b], ((tcp >> 1) - 1) & 1, stalled, v.status);
      trig_produce(sm, b, ip, tok0);
      warp_arrive(&sm.tfull[b]);
    }
  };
  // before the K loop of item tile i (item from token t0, ntiles tiles): at a
  // table's first tile, thread 0 requests the next table's copy (TAB), then
  // every warp waits for this table; returns this thread's rows
  auto table_rows = [&](int i, int ntiles, int t0) {
    if ((i & (kSuper - 1)) == 0) {
      if constexpr (TAB) {
        if (warp == 0 && i + kSuper < ntiles) {
          __syncwarp();
          if (lane == 0) issue_copy(tc + 1, t0 + (i + kSuper) * kTile);
        }
      }
      bounded_wait(&sm.tfull[tc & 1], (tc >> 1) & 1, stalled, v.status);
    }
    return &sm.trig[tc & 1][kTile * (i & (kSuper - 1)) + sg][0];
  };
  // after the K loop of item tile i: release the table after its last tile and
  // make the next one ready
  auto table_done = [&](int i, int ntiles, int tok0) {
    if ((i & (kSuper - 1)) == kSuper - 1 || i + 1 == ntiles) {
      warp_arrive(&sm.tempty[tc & 1]);
      if (i + 1 < ntiles) produce(tc + 1, (i + 1) / kSuper, tok0 + kTile, false);
      ++tc;
    }
  };

  int item = blockIdx.x, npar = 0;
  while (item < n_items) {
    // the CTA's next item, fetched now and read after this item's closing barrier
    if (threadIdx.x == 0) s_next[npar] = (int)gridDim.x + (int)atomicAdd(counter, 1ull);
    const FastItem it = decode_fast_item(v, prefA, prefB, C, NA, NS, G, true, item);
    const int ntiles = (it.t1 - it.t0 + kTile - 1) / kTile;

    // B operand: q * scale * log2(e) for query head 4h + g/2, split hi (even g) / lo (odd g);
    // k-slots 2t, 2t+1 <- channels c, c+2 and 2t+8, 2t+9 <- c+1, c+3 (c = 32t + 4s)
    {
      const int hq = h * kNRep + (g >> 1);
      const long long qb = ((long long)it.b * v.Hq + hq) * kD + 32 * t;
#pragma unroll
      for (int s = 0; s < 8; ++s) {
        float x[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) x[j] = load_src(q, qb + 4 * s + j, v.src_bf16) * qscale;
        uint32_t h02, l02, h13, l13;
        split_hi_lo(x[0], x[2], h02, l02);
        split_hi_lo(x[1], x[3], h13, l13);
        sm.bq[warp][s][lane] = make_uint2((g & 1) ? l02 : h02, (g & 1) ? l13 : h13);
      }
    }
    __syncwarp();
    const uint2* bqs = &sm.bq[warp][0][lane];  // step s at bqs[32 * s]

    Acc A;
#pragma unroll
    for (int m = 0; m < 8; ++m) A.O[m][0] = A.O[m][1] = A.O[m][2] = A.O[m][3] = 0.f;
    A.m_run = kMinit;
    A.l_loc = 0.f;
    A.mb = 0.f;

    produce(tc, 0, it.t0, true);
    const float4* trow0 = &sm.trig[0][sg][0];  // re-pointed per tile
    if (!it.window) {
      // ======================= quantized chunk: tiles through the TMA ring
      const int32_t* bt = v.block_table + (long long)it.b * v.max_pages;
      auto issue = [&](int i, int pid) {
        const int stage = lstage;
        if (++lstage == kStages) lstage = 0;
        ++n_loaded;
        const int tok = it.t0 + i * kTile;
        uint64_t* bar = &sm.bar[warp][stage];
        const bool ok = pid >= 0 && pid < v.n_pages;
        sm.valid[warp][stage] = ok;
        if (!ok) {
          atomicOr(v.status, KVQ_DEV_BAD_PAGE);
          mbar_arrive(bar);
          return;
        }
        const uint8_t* hbk = v.pages + (long long)pid * v.page_bytes + head_off;
        const bool gstart = (tok & (G - 1)) == 0;
        const uint32_t bytes = kStageBytes + (gstart ? kKMeta : 0);
        mbar_arrive_expect_tx(bar, bytes);
        uint8_t* dst = sm.stage[warp][stage];
        const uint64_t pol = l2_evict_first();
        if (v.P == kTile) {
          // the head's whole page section: codes, value meta, then the key scales
          bulk_g2s_hint(dst, hbk, bytes, bar, pol);
        } else {
          const int slot = tok & (v.P - 1);
          bulk_g2s_hint(dst, hbk + slot * kD, kKC, bar, pol);
          bulk_g2s_hint(dst + kKC, hbk + v.off_vc + slot * (kD / 2), kVC, bar, pol);
          bulk_g2s_hint(dst + kKC + kVC, hbk + v.off_vm + slot * (kVM / kTile), kVM, bar, pol);
          if (gstart) {
            const int gslot = v.P >= G ? (slot >> lgG) : 0;
            bulk_g2s_hint(dst + kStageBytes, hbk + v.off_km + gslot * kKMeta, kKMeta, bar, pol);
          }
        }
      };
      int pf = 0;  // lane 0: page id of the next tile to load, read one tile ahead
      if (lane == 0 && !stalled) {
        fence_proxy_async();  // the ring's bytes were last written through the generic proxy
        for (int i = 0; i < min(kStages, ntiles); ++i) issue(i, bt[(it.t0 + i * kTile) >> lgP]);
        if (kStages < ntiles) pf = bt[(it.t0 + kStages * kTile) >> lgP];
      }
      __syncwarp();

      for (int i = 0; i < ntiles; ++i) {
        const int tok0 = it.t0 + i * kTile;
        const int stage = cstage;
        bool valid = false;
        if (!stalled) {
          if (!mbar_wait_bounded(&sm.bar[warp][stage], cphase, kSpin)) {
            atomicOr(v.status, KVQ_DEV_TIMEOUT);
            stalled = true;
          } else {
            valid = sm.valid[warp][stage] != 0;
          }
        }
        if (++cstage == kStages) {
          cstage = 0;
          cphase ^= 1u;
        }
        ++n_consumed;
        const uint8_t* buf = sm.stage[warp][stage];
        if (valid && (tok0 & (G - 1)) == 0) {
          // new key group: its scales, quad (c, c+1, c+2, c+3) stored as (c, c+2, c+1, c+3)
          float4 raw;
          if constexpr (M16) {
            const uint2 h = reinterpret_cast<const uint2*>(buf + kStageBytes)[lane];
            const float2 a = half2_to_float2(h.x), b = half2_to_float2(h.y);
            raw = make_float4(a.x, a.y, b.x, b.y);
          } else {
            raw = reinterpret_cast<const float4*>(buf + kStageBytes)[lane];
          }
          *reinterpret_cast<float4*>(&sm.kmeta[warp][lane >> 3][4 * (lane & 7)]) =
              make_float4(raw.x, raw.z, raw.y, raw.w);
          __syncwarp();
        }
        trow0 = table_rows(i, ntiles, it.t0);
        const float4* trow1 = trow0 + 8 * 32;

        // ---- QK: MMA rows g / g+8 = tile tokens sg / sg+8, channels 32t .. 32t+31
        const float4* km = reinterpret_cast<const float4*>(&sm.kmeta[warp][t][0]);
        float acc[4] = {0.f, 0.f, 0.f, 0.f}, accn[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          uint32_t kw[2][4];
#pragma unroll
          for (int r = 0; r < 2; ++r) {
            const uint4 x = reinterpret_cast<const uint4*>(buf + (sg + 8 * r) * kD + 32 * t)[half];
            kw[r][0] = x.x ^ 0x80808080u; kw[r][1] = x.y ^ 0x80808080u;
            kw[r][2] = x.z ^ 0x80808080u; kw[r][3] = x.w ^ 0x80808080u;
          }
#pragma unroll
          for (int sq = 0; sq < 4; ++sq) {
            const int s = 4 * half + sq;
            uint32_t ahi[2][2], anl[2][2];
            const float4 ks = km[s];
#pragma unroll
            for (int r = 0; r < 2; ++r) {
              const float4 cs = (r ? trow1 : trow0)[(8 * t + s) ^ tkey];
              const uint32_t w = kw[r][sq];
              // offset-binary byte u = code + 128 -> fp32 2^23 + u -> code -> code * scale
              const float2 X = mul2(sub2(make_float2(magic_f32(w, 0), magic_f32(w, 2)), magic_bias()),
                                    make_float2(ks.x, ks.y));
              const float2 Y = mul2(sub2(make_float2(magic_f32(w, 1), magic_f32(w, 3)), magic_bias()),
                                    make_float2(ks.z, ks.w));
              rot_split(X, Y, cs, ahi[r][0], anl[r][0], ahi[r][1], anl[r][1]);
            }
            const uint2 bq = bqs[32 * s];
            mma_16816(acc, ahi[0][0], ahi[1][0], ahi[0][1], ahi[1][1], bq.x, bq.y);
            mma_16816(accn, anl[0][0], anl[1][0], anl[0][1], anl[1][1], bq.x, bq.y);
          }
        }
        table_done(i, ntiles, tok0);
        const float2 d01 = sub2(make_float2(acc[0], acc[1]), make_float2(accn[0], accn[1]));
        const float2 d23 = sub2(make_float2(acc[2], acc[3]), make_float2(accn[2], accn[3]));
        float lg0 = d01.x + d01.y, lg1 = d23.x + d23.y;
        if (!valid) lg0 = lg1 = -INFINITY;

        // ---- softmax and the PV B operand (P' = p * v_scale, v_min into A.mb)
        float2 m0 = make_float2(0.f, 0.f), m1 = m0;  // (scale, min) of tokens sg and sg + 8
        if (valid) {
          if constexpr (M16) {
            const uint32_t* vm = reinterpret_cast<const uint32_t*>(buf + kKC + kVC);
            m0 = half2_to_float2(vm[sg]);
            m1 = half2_to_float2(vm[sg + 8]);
          } else {
            const float2* vm = reinterpret_cast<const float2*>(buf + kKC + kVC);
            m0 = vm[sg];
            m1 = vm[sg + 8];
          }
        }
        uint32_t b01, b23;
        softmax_step(A, lg0, lg1, m0, m1, g, t, b01, b23);

        // ---- PV: A = V^T (channel rows 16g + 2m (+1); k-slots 2t, 2t+1, 2t+8, 2t+9 =
        //      tokens sig(2t), sig(2t+1), +8) as centred codes c - 8: low nibbles (rows g),
        //      high nibbles (rows g+8)
        uint2 vw[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int tok = sig(2 * t + (u & 1)) + 8 * (u >> 1);
          vw[u] = *reinterpret_cast<const uint2*>(buf + kKC + tok * (kD / 2) + 8 * g);
        }
#pragma unroll
        for (int w = 0; w < 2; ++w) {
          const uint32_t a0 = w ? vw[0].y : vw[0].x, a1 = w ? vw[1].y : vw[1].x;
          const uint32_t c0 = w ? vw[2].y : vw[2].x, c1 = w ? vw[3].y : vw[3].x;
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            // byte j of the two tokens' words into the low bytes of the two f16 halves
            const uint32_t sel = 0x4400u + 0x1111u * j;
            const uint32_t ya = prmt(a0, a1, sel), yc = prmt(c0, c1, sel);
            mma_16816(A.O[4 * w + j], centred_lo(ya), centred_hi(ya), centred_lo(yc), centred_hi(yc), b01, b23);
          }
        }

        // ---- release the stage and refill it with tile i + kStages
        __syncwarp();
        if (lane == 0 && i + kStages < ntiles && !stalled) {
          fence_proxy_async();
          issue(i + kStages, pf);
          if (i + kStages + 1 < ntiles) pf = bt[(it.t0 + (i + kStages + 1) * kTile) >> lgP];
        }
        __syncwarp();
      }
    } else {
      // ======================= residual window: source-dtype rows from k_win / v_win
      const int T = it.t1;
      const long long wrow = ((long long)it.b * v.R) * v.Hkv + h;  // (b, slot 0, h) row index
      for (int i = 0; i < ntiles; ++i) {
        const int tok0 = it.t0 + i * kTile;
        trow0 = table_rows(i, ntiles, it.t0);
        const float4* trow1 = trow0 + 8 * 32;
        float acc[4] = {0.f, 0.f, 0.f, 0.f}, accn[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int s = 0; s < 8; ++s) {
          uint32_t ahi[2][2], anl[2][2];
#pragma unroll
          for (int r = 0; r < 2; ++r) {
            const int tok = tok0 + sg + 8 * r;
            float k[4] = {0.f, 0.f, 0.f, 0.f};
            if (tok < T) {
              const long long wi = (wrow + (long long)(tok - it.t0) * v.Hkv) * kD + 32 * t + 4 * s;
#pragma unroll
              for (int j = 0; j < 4; ++j) k[j] = load_src(v.k_win, wi + j, v.src_bf16);
            }
            const float4 cs = (r ? trow1 : trow0)[(8 * t + s) ^ tkey];
            rot_split(make_float2(k[0], k[2]), make_float2(k[1], k[3]), cs, ahi[r][0], anl[r][0], ahi[r][1],
                      anl[r][1]);
          }
          const uint2 bq = bqs[32 * s];
          mma_16816(acc, ahi[0][0], ahi[1][0], ahi[0][1], ahi[1][1], bq.x, bq.y);
          mma_16816(accn, anl[0][0], anl[1][0], anl[0][1], anl[1][1], bq.x, bq.y);
        }
        table_done(i, ntiles, tok0);
        float lg0 = acc[0] + acc[1] - accn[0] - accn[1];
        float lg1 = acc[2] + acc[3] - accn[2] - accn[3];
        if (tok0 + sg >= T) lg0 = -INFINITY;
        if (tok0 + sg + 8 >= T) lg1 = -INFINITY;
        uint32_t b01, b23;
        // window values enter as they are: scale 1 and a minimum of -8 make the midpoint term 0
        softmax_step(A, lg0, lg1, make_float2(1.f, -8.f), make_float2(1.f, -8.f), g, t, b01, b23);
        // values as f16 pairs (k-slots 2t+u, 2t+1+u) per channel 16g + 2m (+1)
        long long vi[4];
        bool vok[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int tok = tok0 + sig(2 * t + (u & 1)) + 8 * (u >> 1);
          vok[u] = tok < T;
          vi[u] = (wrow + (long long)(tok - it.t0) * v.Hkv) * kD + 16 * g;
        }
#pragma unroll
        for (int m = 0; m < 8; ++m) {
          float x[4][2];
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            x[u][0] = vok[u] ? load_src(v.v_win, vi[u] + 2 * m, v.src_bf16) : 0.f;
            x[u][1] = vok[u] ? load_src(v.v_win, vi[u] + 2 * m + 1, v.src_bf16) : 0.f;
          }
          mma_16816(A.O[m], pack_f16x2(x[0][0], x[1][0]), pack_f16x2(x[0][1], x[1][1]),
                    pack_f16x2(x[2][0], x[3][0]), pack_f16x2(x[2][1], x[3][1]), b01, b23);
        }
      }
    }

    // ---- epilogue: this warp's partial for query heads 4h .. 4h+3
#pragma unroll
    for (int o = 4; o < 32; o <<= 1) {
      A.l_loc += __shfl_xor_sync(0xffffffffu, A.l_loc, o);
      A.mb += __shfl_xor_sync(0xffffffffu, A.mb, o);
    }
    // values entered as they are (window) or centred (c - 8) with the midpoints in A.mb
    const int hq = h * kNRep + t;
    float* dst = part + ((long long)item * v.Hq + hq) * (kD + 4);
    if (g == 0) {
      dst[0] = A.m_run;
      dst[1] = A.l_loc;
    }
#pragma unroll
    for (int m = 0; m < 8; ++m) {
      const float2 o2 = make_float2((A.O[m][0] - A.O[m][1]) + A.mb, (A.O[m][2] - A.O[m][3]) + A.mb);
      reinterpret_cast<float2*>(dst + 4 + 16 * g)[m] = o2;  // channels 16g + 2m, 16g + 2m + 1
    }
    named_bar_sync(1, kThreads);
    item = s_next[npar];
    npar ^= 1;
  }

  // drain: wait (bounded) for loads that were issued but never consumed
  if (lane == 0) {
    while (n_consumed < n_loaded) {
      mbar_wait_bounded(&sm.bar[warp][cstage], cphase, kSpin);
      if (++cstage == kStages) {
        cstage = 0;
        cphase ^= 1u;
      }
      ++n_consumed;
    }
  }
}


// Caller's RoPE table: row p (D/4 float4) holds trig_entry(p, u) at trig_slot(u, p & 1).
__global__ void __launch_bounds__(256) rope_table_kernel(KvqView v, int positions, float4* table) {
  __shared__ float w_hi[kMaxHeadDim / 2], w_lo[kMaxHeadDim / 2];
  for (int i = threadIdx.x; i < v.D / 2; i += blockDim.x) rope_split(v, i, &w_hi[i], &w_lo[i]);
  __syncthreads();
  const int U = v.D / 4;
  const long long n = (long long)positions * U;
  for (long long e = blockIdx.x * (long long)blockDim.x + threadIdx.x; e < n; e += (long long)gridDim.x * blockDim.x) {
    const int p = (int)(e / U), u = (int)(e - (long long)p * U);
    table[(long long)p * U + trig_slot(u, p & 1)] = trig_entry(w_hi, w_lo, p, u);
  }
}

}  // namespace

kvq_status launch_rope_table(const KvqView& v, int positions, void* table, cudaStream_t st) {
  const long long n = (long long)positions * (v.D / 4);
  const long long blocks = (n + 255) / 256, cap = (long long)num_sms() * 8;
  const int grid = (int)(blocks < cap ? blocks : cap);
  rope_table_kernel<<<grid, 256, 0, st>>>(v, positions, static_cast<float4*>(table));
  return cudaGetLastError() == cudaSuccess ? KVQ_OK : KVQ_ERR_CUDA;
}

bool fast_eligible(const KvqView& v) {
  const bool pow2_g = v.kgroup > 0 && (v.kgroup & (v.kgroup - 1)) == 0;
  const bool pow2_p = (v.P & (v.P - 1)) == 0;
  const int whole_page = v.meta16 ? stage_bytes<true>() : stage_bytes<false>();
  return v.D == kD && v.Hkv == kWarps && v.n_rep == kNRep && v.kfmt == KVQ_INT8 &&
         v.kmode == KVQ_SYM_ABSMAX && v.kaxis == KVQ_PER_CHANNEL && v.rope_pre == 1 &&
         v.vfmt == KVQ_INT4 && v.vmode == KVQ_ASYM_MINMAX && v.vaxis == KVQ_PER_TOKEN &&
         v.vgroup == kD && pow2_g && pow2_p && v.kgroup >= kTile * kStages && v.P >= kTile &&
         (v.P != kTile || v.off_km == whole_page) && v.batch <= 4096;
}

size_t fast_workspace_bytes(const KvqView& v, int batch) { return split_workspace_bytes(v, batch); }

kvq_status launch_fast(const KvqView& v, const void* q, float* out, float scale, void* ws,
                       cudaStream_t st) {
  const size_t smem = sizeof(SmemRI) + sizeof(int) * 2 * (v.batch + 1);
  // the caller's RoPE table when it covers every position the cache can hold,
  // rounded up to a whole table (the last table's copy reads all 32 rows)
  const long long span = ((long long)v.max_pages * v.P + kSuper * kTile - 1) / (kSuper * kTile) * (kSuper * kTile);
  const bool tab = v.rope_table != nullptr && (long long)v.rope_positions >= span;
  const int m = (v.meta16 ? 1 : 0) + (tab ? 2 : 0);
  auto kern = m == 3   ? split_rope_i8i4_kernel<true, true>
              : m == 2 ? split_rope_i8i4_kernel<false, true>
              : m == 1 ? split_rope_i8i4_kernel<true, false>
                       : split_rope_i8i4_kernel<false, false>;
  int occ = 0;
  const kvq_status so =
      occupancy_once(kSlotFast + m, kern, kThreads, smem, sizeof(SmemRI) + sizeof(int) * 2 * 4097, &occ);
  if (so != KVQ_OK) return so;
  const int grid = num_sms() * occ;
  // the dynamic item counter starts at zero on every call
  if (cudaMemsetAsync(static_cast<char*>(ws) + fast_counter_offset(v.batch), 0, 8, st) != cudaSuccess)
    return KVQ_ERR_CUDA;
  kern<<<grid, kThreads, smem, st>>>(v, q, scale, static_cast<float*>(ws));
  if (cudaGetLastError() != cudaSuccess) return KVQ_ERR_CUDA;
  return launch_split_combine(v, static_cast<float*>(ws), out, st) == cudaSuccess ? KVQ_OK : KVQ_ERR_CUDA;
}

}  // namespace kvq
