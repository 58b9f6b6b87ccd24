// Work plan shared by the split-K decode kernels and the combine.
//
// Every CTA derives the same plan from the device-side sequence lengths, so no
// host synchronisation is needed: a chunk size C, and for each sequence b the
// item range [pref[b], pref[b+1]) = (quantized chunks + 1 window item if the
// window is not empty) x items per chunk.  The generic kernel's items are
// (sequence, kv-head, head block, chunk); the tensor-core kernels' items are
// (sequence, chunk) with all kv-heads.  The first CTA stores the plan at the
// head of the workspace for the combine kernel.
#pragma once

#include "kvq_host.h"
#include "kvq_internal.cuh"

namespace kvq {

constexpr int kHB = 8;              // query heads per work item (head block)
constexpr int kMaxHeadDim = 256;
constexpr int kTargetItems = 4096;  // upper bound on quantized chunks per call
constexpr int kMinChunk = 32;      // generic kernel: one 8-token sub-tile for each of its 4 warps

struct ItemInfo {
  int b, kvh, hb, t0, t1, window;
};

__host__ __device__ inline size_t plan_header_bytes(int batch) {
  return ((size_t)(batch + 3) * sizeof(int) + 255) / 256 * 256;
}

__device__ inline const int* plan_prefix(const float* ws) {
  return reinterpret_cast<const int*>(ws) + 2;
}

__host__ __device__ inline float* plan_partials(float* ws, int batch) {
  return reinterpret_cast<float*>(reinterpret_cast<char*>(ws) + plan_header_bytes(batch));
}
__host__ __device__ inline const float* plan_partials(const float* ws, int batch) {
  return reinterpret_cast<const float*>(reinterpret_cast<const char*>(ws) + plan_header_bytes(batch));
}

__device__ inline int seq_tokens(const KvqView& v, int b) {
  const int T = v.seq_lens[b];
  if (T < 0 || (long long)T > (long long)v.max_pages * v.P) {
    atomicOr(v.status, KVQ_DEV_BAD_LENGTH);
    return 0;
  }
  return T;
}

__device__ inline int seq_chunks(const KvqView& v, int T, int C) {
  const int nq = n_quantized(T, v.R);
  return (nq + C - 1) / C + (T > nq ? 1 : 0);
}

// Block-wide: pref[0..B] (shared, B+1 ints), *s_C, *s_items.  All threads call it.
// Each chunk of a sequence counts `mult` items; C is a multiple of `align`, at
// least `cmin`, and large enough that the quantized chunks number at most about
// `target`.
__device__ inline void plan_items_ex(const KvqView& v, int mult, int align, int target, int cmin,
                                     int* pref, int* s_C, int* s_items) {
  __shared__ unsigned long long s_total;
  __shared__ int s_part[1024];
  const int B = v.batch;
  if (threadIdx.x == 0) s_total = 0ull;
  __syncthreads();
  unsigned long long sum = 0;
  for (int b = threadIdx.x; b < B; b += blockDim.x) sum += (unsigned long long)seq_tokens(v, b);
  atomicAdd(&s_total, sum);
  __syncthreads();
  const unsigned long long work = s_total * (unsigned long long)mult;
  long long C = (long long)((work + target - 1) / target);
  if (C < cmin) C = cmin;
  C = (C + align - 1) / align * align;
  const int nt = blockDim.x;
  const int seg = (B + nt - 1) / nt;
  const int b0 = threadIdx.x * seg, b1 = min(B, b0 + seg);
  int local = 0;
  for (int b = b0; b < b1; ++b) local += seq_chunks(v, seq_tokens(v, b), (int)C) * mult;
  s_part[threadIdx.x] = local;
  __syncthreads();
  if (threadIdx.x < 32) {  // exclusive scan of s_part[0..nt): lanes over segments, then a shuffle scan
    const int lane = threadIdx.x, per = (nt + 31) / 32;
    const int i0 = min(nt, lane * per), i1 = min(nt, i0 + per);
    int seg = 0;
    for (int i = i0; i < i1; ++i) seg += s_part[i];
    int incl = seg;
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    int run = incl - seg;
    for (int i = i0; i < i1; ++i) {
      const int x = s_part[i];
      s_part[i] = run;
      run += x;
    }
    if (lane == 31) {
      *s_items = incl;
      *s_C = (int)C;
    }
  }
  __syncthreads();
  int run = s_part[threadIdx.x];
  for (int b = b0; b < b1; ++b) {
    pref[b] = run;
    run += seq_chunks(v, seq_tokens(v, b), (int)C) * mult;
  }
  if (threadIdx.x == 0) pref[B] = *s_items;
  __syncthreads();
}

// The generic kernel's plan: items are (sequence, kv-head, head block, chunk).
__device__ inline void plan_items(const KvqView& v, int HB, int* pref, int* s_C, int* s_items) {
  plan_items_ex(v, v.Hkv * HB, 16, kTargetItems, kMinChunk, pref, s_C, s_items);
}

__device__ inline void store_plan(const KvqView& v, float* ws, const int* pref, int C, int items) {
  int* h = reinterpret_cast<int*>(ws);
  if (threadIdx.x == 0) {
    h[0] = C;
    h[1] = items;
  }
  for (int b = threadIdx.x; b <= v.batch; b += blockDim.x) h[2 + b] = pref[b];
}

__device__ inline ItemInfo decode_item(const KvqView& v, const int* pref, int C, int HB, int item) {
  int lo = 0, hi = v.batch - 1;  // largest b with pref[b] <= item
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (pref[mid] <= item) lo = mid; else hi = mid - 1;
  }
  ItemInfo it;
  it.b = lo;
  const int nc = (pref[lo + 1] - pref[lo]) / (v.Hkv * HB);
  const int local = item - pref[lo];
  const int kh = local / nc, chunk = local % nc;
  it.kvh = kh / HB;
  it.hb = kh % HB;
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

// omega_i = theta^(-2i/D) / (2 pi) as a two-float hi + lo (computed in fp64 once per CTA).
__device__ inline void rope_split(const KvqView& v, int i, float* hi, float* lo) {
  const double th = exp2(-(2.0 * i / v.D) * log2((double)v.rope_theta));
  const double w = th / (2.0 * 3.14159265358979323846);
  const float h = (float)w;
  *hi = h;
  *lo = (float)(w - (double)h);
}

}  // namespace kvq
