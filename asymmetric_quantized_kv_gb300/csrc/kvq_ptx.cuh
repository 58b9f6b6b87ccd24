// Inline-PTX helpers for the sm_103a decode kernels: warp-level tensor-core MMA
// (m16n8k16, f16 inputs, f32 accumulate), mbarriers with bounded waits, TMA bulk
// copies global -> shared, and packed conversions.
#pragma once

#include <stdint.h>

namespace kvq {
namespace ptx {

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// D += A * B, A 16x16 row-major f16 (4 regs), B 16x8 col-major f16 (2 regs), D 16x8 f32.
__device__ __forceinline__ void mma_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                          uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(smem_u32(bar)), "r"(count));
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async() {
  asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, "
      "0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Polls of every bounded pipeline wait in the decode kernels (and in their
// self-test): each poll may suspend the thread briefly, so a wait on a phase that
// never completes gives up after well under a few seconds.
constexpr uint32_t kWaitPolls = 1u << 20;

// Bounded wait on an mbarrier phase: gives up after `limit` polls (each poll may
// itself suspend the warp briefly) and reports false.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity, uint32_t limit) {
  for (uint32_t i = 0; i < limit; ++i)
    if (mbar_try_wait(bar, parity)) return true;
  return false;
}

// TMA bulk copy global -> shared::cta (the CTA is its own one-CTA cluster),
// completion counted in bytes on `bar`.  dst, src 16-byte aligned, bytes % 16 == 0.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// Start bringing the 128-byte lines of [p, p + n) into L1 (no data returned, no
// wait); every address issued lies inside the range.
__device__ __forceinline__ void prefetch_l1_range(const void* p, int n) {
  const char* c = static_cast<const char*>(p);
  for (int o = 0; o < n; o += 128) asm volatile("prefetch.global.L1 [%0];\n" ::"l"(c + o));
  if (n > 0 && ((reinterpret_cast<uintptr_t>(c) & 127) + (n - 1)) / 128 > (n - 1) / 128)
    asm volatile("prefetch.global.L1 [%0];\n" ::"l"(c + n - 1));
}

// L2 policy for data read once per call (the packed KV stream): evict first, so
// the stream does not push small reused data (code, window rows, block tables,
// partial records) out of L2.
__device__ __forceinline__ uint64_t l2_evict_first() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;\n" : "=l"(pol));
  return pol;
}

// L2 policy for small data that many CTAs read (a RoPE table): evict last.
__device__ __forceinline__ uint64_t l2_evict_last() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;\n" : "=l"(pol));
  return pol;
}

// bulk_g2s with an L2 cache policy
__device__ __forceinline__ void bulk_g2s_hint(void* dst, const void* src, uint32_t bytes, uint64_t* bar,
                                              uint64_t pol) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], "
      "%4;\n" ::"r"(smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(pol)
      : "memory");
}

// TMA tensor copy global -> shared::cta of one box of a 2-D tensor map at
// element coordinates (x, y); completion counted in bytes on `bar`.  x must keep
// the copy 16-byte aligned (x = 0 here); the destination is aligned to the
// map's swizzle span.
__device__ __forceinline__ void tma_load_2d(void* dst, const void* tmap, int x, int y, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], "
      "[%4];\n" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}

// tma_load_2d with an L2 cache policy
__device__ __forceinline__ void tma_load_2d_hint(void* dst, const void* tmap, int x, int y, uint64_t* bar,
                                                 uint64_t pol) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1, "
      "{%2, %3}], [%4], %5;\n" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(x), "r"(y), "r"(smem_u32(bar)), "l"(pol)
      : "memory");
}

// TMA tensor copy of one box of a 5-D tensor map at coordinates (c0 .. c4), with an L2 cache policy.
__device__ __forceinline__ void tma_load_5d_hint(void* dst, const void* tmap, int c0, int c1, int c2, int c3,
                                                 int c4, uint64_t* bar, uint64_t pol) {
  asm volatile(
      "cp.async.bulk.tensor.5d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1, "
      "{%2, %3, %4, %5, %6}], [%7], %8;\n" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(c4), "r"(smem_u32(bar)),
      "l"(pol)
      : "memory");
}

// TMA tensor copy of one box of a 5-D tensor map at coordinates (c0 .. c4).
__device__ __forceinline__ void tma_load_5d(void* dst, const void* tmap, int c0, int c1, int c2, int c3, int c4,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.5d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4, "
      "%5, %6}], [%7];\n" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(c4), "r"(smem_u32(bar))
      : "memory");
}

// Two OCP E4M3 bytes (low byte -> low half) to f16x2; every E4M3 value is exact in f16.
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(unsigned short x) {
  uint32_t r;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;\n" : "=r"(r) : "h"(x));
  return r;
}
// Two E5M2 bytes (low byte -> low half) to f16x2; E5M2 is a subset of f16, so
// the conversion is exact.
__device__ __forceinline__ uint32_t e5m2x2_to_f16x2(unsigned short x) {
  uint32_t r;
  asm("cvt.rn.f16x2.e5m2x2 %0, %1;\n" : "=r"(r) : "h"(x));
  return r;
}
template <bool E5M2>
__device__ __forceinline__ uint32_t fp8x2_to_f16x2(unsigned short x) {
  return E5M2 ? e5m2x2_to_f16x2(x) : e4m3x2_to_f16x2(x);
}
__device__ __forceinline__ unsigned short lo16(uint32_t x) { return static_cast<unsigned short>(x & 0xFFFFu); }
__device__ __forceinline__ unsigned short hi16(uint32_t x) { return static_cast<unsigned short>(x >> 16); }

// Programmatic dependent launch (sm_90+).  grid_dep_wait blocks until the grids
// this one depends on have completed and their writes are visible (it returns at
// once when the kernel was launched without the attribute); grid_dep_launch lets
// the dependent grid's CTAs be scheduled before this grid completes.
__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;\n" ::: "memory"); }
__device__ __forceinline__ void grid_dep_launch() { asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory"); }

__device__ __forceinline__ void named_bar_sync(uint32_t id, uint32_t threads) {
  asm volatile("bar.sync %0, %1;\n" ::"r"(id), "r"(threads) : "memory");
}

// Pack two floats to f16x2 (round to nearest): low half = lo, high half = hi.
__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;\n" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// Split (x0, x1) into an f16x2 "hi" part and an f16x2 holding (hi - x) per
// element, so that x = hi - neg_lo up to ~2^-22 relative.
__device__ __forceinline__ void split_hi_neglo(float x0, float x1, uint32_t& hi, uint32_t& neglo) {
  hi = pack_f16x2(x0, x1);
  unsigned short h0, h1;
  asm("mov.b32 {%0, %1}, %2;\n" : "=h"(h0), "=h"(h1) : "r"(hi));
  float d0, d1;
  asm("sub.rn.f32.f16 %0, %1, %2;\n" : "=f"(d0) : "h"(h0), "f"(x0));
  asm("sub.rn.f32.f16 %0, %1, %2;\n" : "=f"(d1) : "h"(h1), "f"(x1));
  neglo = pack_f16x2(d0, d1);
}

// Split x into f16 hi and lo parts (x ~= hi + lo), both as floats' f16 bits.
__device__ __forceinline__ void split_hi_lo(float x0, float x1, uint32_t& hi, uint32_t& lo) {
  uint32_t nl;
  split_hi_neglo(x0, x1, hi, nl);
  lo = nl ^ 0x80008000u;
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t r;
  asm("prmt.b32 %0, %1, %2, %3;\n" : "=r"(r) : "r"(a), "r"(b), "r"(sel));
  return r;
}

template <uint32_t LUT>
__device__ __forceinline__ uint32_t lop3(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t r;
  asm("lop3.b32 %0, %1, %2, %3, %4;\n" : "=r"(r) : "r"(a), "r"(b), "r"(c), "n"(LUT));
  return r;
}

// (a & b) | c
__device__ __forceinline__ uint32_t and_or(uint32_t a, uint32_t b, uint32_t c) {
  return lop3<(0xF0 & 0xCC) | 0xAA>(a, b, c);
}

// f16x2 arithmetic on raw registers
__device__ __forceinline__ uint32_t hsub2(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("sub.rn.f16x2 %0, %1, %2;\n" : "=r"(r) : "r"(a), "r"(b));
  return r;
}
__device__ __forceinline__ uint32_t hfma2(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t r;
  asm("fma.rn.f16x2 %0, %1, %2, %3;\n" : "=r"(r) : "r"(a), "r"(b), "r"(c));
  return r;
}

// Packed fp32x2 arithmetic (one instruction for two lanes of work on sm_100+).
__device__ __forceinline__ float2 add2(float2 a, float2 b) {
  float2 r;
  asm("{\n .reg .b64 ra, rb, rd;\n mov.b64 ra, {%2, %3};\n mov.b64 rb, {%4, %5};\n"
      " add.rn.f32x2 rd, ra, rb;\n mov.b64 {%0, %1}, rd;\n}\n"
      : "=f"(r.x), "=f"(r.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return r;
}
__device__ __forceinline__ float2 mul2(float2 a, float2 b) {
  float2 r;
  asm("{\n .reg .b64 ra, rb, rd;\n mov.b64 ra, {%2, %3};\n mov.b64 rb, {%4, %5};\n"
      " mul.rn.f32x2 rd, ra, rb;\n mov.b64 {%0, %1}, rd;\n}\n"
      : "=f"(r.x), "=f"(r.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return r;
}

__device__ __forceinline__ float2 sub2(float2 a, float2 b) {
  float2 r;
  asm("{\n .reg .b64 ra, rb, rd;\n mov.b64 ra, {%2, %3};\n mov.b64 rb, {%4, %5};\n"
      " sub.rn.f32x2 rd, ra, rb;\n mov.b64 {%0, %1}, rd;\n}\n"
      : "=f"(r.x), "=f"(r.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return r;
}
// a * b + c, one rounding per lane
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) {
  float2 r;
  asm("{\n .reg .b64 ra, rb, rc, rd;\n mov.b64 ra, {%2, %3};\n mov.b64 rb, {%4, %5};\n"
      " mov.b64 rc, {%6, %7};\n fma.rn.f32x2 rd, ra, rb, rc;\n mov.b64 {%0, %1}, rd;\n}\n"
      : "=f"(r.x), "=f"(r.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
  return r;
}

__device__ __forceinline__ float ex2(float x) {
  float r;
  asm("ex2.approx.ftz.f32 %0, %1;\n" : "=f"(r) : "f"(x));
  return r;
}

}  // namespace ptx
}  // namespace kvq
