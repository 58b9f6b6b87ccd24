// Split-K work plan, workspace layout and partial combine shared by the
// tensor-core decode kernels (head_dim 128).  An item is (sequence, chunk of
// C tokens); a kernel processes it for every kv-head, and writes one partial
// record (running max, softmax sum, unnormalised output) per (item, query head).
#pragma once

#include "kvq_attn_plan.cuh"

namespace kvq {
namespace {

constexpr int kD = 128;
constexpr int kFastTarget = 1024;
constexpr int kFastMinChunk = 256;

struct FastItem {
  int b, t0, t1, window;
};

// Work plan of the tensor-core kernels, at the head of the workspace:
//   int C, NA, NB, pad; int prefA[B+1]; int prefB[B+1]; u64 counter
// Items d < NA are the full C-token chunks of every sequence (prefA: per-sequence
// prefix of counts); items d >= NA are the short ones (each sequence's last,
// partial chunk and its residual window; prefB).  Long items come first, and
// CTAs take items dynamically from the counter (zeroed by the host before each
// call), so the last wave holds only short items.
__host__ __device__ inline size_t fast_header_ints(int B) { return (size_t)2 * (B + 1) + 4; }
__host__ __device__ inline size_t fast_counter_offset(int B) { return (fast_header_ints(B) * 4 + 7) & ~(size_t)7; }
__host__ __device__ inline size_t fast_header_bytes(int B) { return (fast_counter_offset(B) + 8 + 255) / 256 * 256; }

// NT threads per block; scratch: 2 * NT ints of shared memory that are free
// until the caller's main loop
template <int NT>
__device__ inline void fast_plan(const KvqView& v, int align, int* sA, int* sB, int* s_C, int* s_NA, int* s_NB,
                                 int* scratch) {
  __shared__ unsigned long long s_total;
  int* s_pa = scratch;
  int* s_pb = scratch + NT;
  const int B = v.batch;
  if (threadIdx.x == 0) s_total = 0ull;
  __syncthreads();
  unsigned long long sum = 0;
  for (int b = threadIdx.x; b < B; b += blockDim.x) sum += (unsigned long long)seq_tokens(v, b);
  atomicAdd(&s_total, sum);
  __syncthreads();
  long long C = (long long)((s_total + kFastTarget - 1) / kFastTarget);
  if (C < kFastMinChunk) C = kFastMinChunk;
  C = (C + align - 1) / align * align;
  const int seg = (B + NT - 1) / NT;
  const int b0 = threadIdx.x * seg, b1 = min(B, b0 + seg);
  int la = 0, lb = 0;
  for (int b = b0; b < b1; ++b) {
    const int T = seq_tokens(v, b), nq = n_quantized(T, v.R);
    la += nq / (int)C;
    lb += (nq % (int)C ? 1 : 0) + (T > nq ? 1 : 0);
  }
  s_pa[threadIdx.x] = la;
  s_pb[threadIdx.x] = lb;
  __syncthreads();
  if (threadIdx.x == 0) {
    int ra = 0, rb = 0;
    for (int k = 0; k < NT; ++k) {
      const int xa = s_pa[k], xb = s_pb[k];
      s_pa[k] = ra;
      s_pb[k] = rb;
      ra += xa;
      rb += xb;
    }
    *s_NA = ra;
    *s_NB = rb;
    *s_C = (int)C;
  }
  __syncthreads();
  int ra = s_pa[threadIdx.x], rb = s_pb[threadIdx.x];
  for (int b = b0; b < b1; ++b) {
    const int T = seq_tokens(v, b), nq = n_quantized(T, v.R);
    sA[b] = ra;
    sB[b] = rb;
    ra += nq / (int)C;
    rb += (nq % (int)C ? 1 : 0) + (T > nq ? 1 : 0);
  }
  if (threadIdx.x == 0) {
    sA[B] = *s_NA;
    sB[B] = *s_NB;
  }
  __syncthreads();
}

__device__ inline void store_fast_plan(const KvqView& v, float* ws, const int* sA, const int* sB, int C, int NA,
                                       int NB) {
  int* h = reinterpret_cast<int*>(ws);
  if (threadIdx.x == 0) {
    h[0] = C;
    h[1] = NA;
    h[2] = NB;
  }
  for (int b = threadIdx.x; b <= v.batch; b += blockDim.x) {
    h[4 + b] = sA[b];
    h[4 + v.batch + 1 + b] = sB[b];
  }
}

// largest b with pref[b] <= x (pref[0] = 0, x < pref[B])
__device__ inline int seq_of(const int* pref, int B, int x) {
  int lo = 0, hi = B - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (pref[mid] <= x) lo = mid; else hi = mid - 1;
  }
  return lo;
}

__device__ inline FastItem decode_fast_item(const KvqView& v, const int* sA, const int* sB, int C, int NA,
                                            int d) {
  FastItem it;
  if (d < NA) {
    it.b = seq_of(sA, v.batch, d);
    it.window = 0;
    it.t0 = (d - sA[it.b]) * C;
    it.t1 = it.t0 + C;
    return it;
  }
  const int e = d - NA;
  it.b = seq_of(sB, v.batch, e);
  const int T = seq_tokens(v, it.b), nq = n_quantized(T, v.R);
  if (e == sB[it.b] && nq % C) {
    it.window = 0;
    it.t0 = (nq / C) * C;
    it.t1 = nq;
  } else {
    it.window = 1;
    it.t0 = nq;
    it.t1 = T;
  }
  return it;
}


// Merge the chunk partials of one (sequence, query head).  Records are
// kRec = D + 4 floats (max, sum, 2 pad, output) so outputs are 16-byte aligned.
// Weights 2^(m_i - M) are computed once into shared memory; then 8 chunk lanes x
// 32 channel quads read the outputs with float4 loads and reduce through smem.
constexpr int kRec = kD + 4;
constexpr int kCombineThreads = 256;
constexpr int kCombineCache = 2048;

__global__ void __launch_bounds__(kCombineThreads) combine_fast_kernel(KvqView v, float* ws, float* out) {
  __shared__ float wts[kCombineCache];
  __shared__ float red[kCombineThreads / 32];
  __shared__ float4 acc_s[8][kD / 4];
  const int hq = blockIdx.x, b = blockIdx.y;
  const int* hdr = reinterpret_cast<const int*>(ws);
  const int NA = hdr[1];
  const int* pA = hdr + 4;
  const int* pB = pA + v.batch + 1;
  const float* part = reinterpret_cast<const float*>(reinterpret_cast<const char*>(ws) + fast_header_bytes(v.batch));
  // this sequence's items: nA full chunks at pA[b].., then nB short items at NA + pB[b]..
  const int nA = pA[b + 1] - pA[b], nB = pB[b + 1] - pB[b];
  const int n = nA + nB;
  const long long stride = (long long)v.Hq * kRec;
  const float* baseA = part + ((long long)pA[b] * v.Hq + hq) * kRec;
  const float* baseB = part + ((long long)(NA + pB[b]) * v.Hq + hq) * kRec;
#define KVQ_REC(i) ((i) < nA ? baseA + (long long)(i) * stride : baseB + (long long)((i) - nA) * stride)
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  float M = -INFINITY;
  for (int i = threadIdx.x; i < n; i += kCombineThreads) M = fmaxf(M, KVQ_REC(i)[0]);
  for (int o = 16; o; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  if (lane == 0) red[warp] = M;
  __syncthreads();
  M = red[0];
  for (int w = 1; w < kCombineThreads / 32; ++w) M = fmaxf(M, red[w]);
  __syncthreads();
  float L = 0.f;
  for (int i = threadIdx.x; i < n; i += kCombineThreads) {
    const float* r = KVQ_REC(i);
    const float w = r[0] == -INFINITY ? 0.f : exp2f(r[0] - M);
    if (i < kCombineCache) wts[i] = w;
    L += r[1] * w;
  }
  for (int o = 16; o; o >>= 1) L += __shfl_xor_sync(0xffffffffu, L, o);
  if (lane == 0) red[warp] = L;
  __syncthreads();
  L = 0.f;
  for (int w = 0; w < kCombineThreads / 32; ++w) L += red[w];
  const float invL = L > 0.f ? 1.f / L : 0.f;
  // chunk lane j = warp (0..7), channel quad = lane (channels 4 lane .. 4 lane + 3)
  float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int i = warp; i < n; i += 8) {
    const float* r = KVQ_REC(i);
    float w;
    if (i < kCombineCache) {
      w = wts[i];
    } else {
      w = r[0] == -INFINITY ? 0.f : exp2f(r[0] - M);
    }
    const float4 x = reinterpret_cast<const float4*>(r + 4)[lane];
    o.x += x.x * w;
    o.y += x.y * w;
    o.z += x.z * w;
    o.w += x.w * w;
  }
  acc_s[warp][lane] = o;
  __syncthreads();
  if (threadIdx.x < kD / 4) {
    float4 r = acc_s[0][threadIdx.x];
#pragma unroll
    for (int j = 1; j < 8; ++j) {
      const float4 x = acc_s[j][threadIdx.x];
      r.x += x.x; r.y += x.y; r.z += x.z; r.w += x.w;
    }
    r.x *= invL; r.y *= invL; r.z *= invL; r.w *= invL;
    reinterpret_cast<float4*>(out + ((long long)b * v.Hq + hq) * kD)[threadIdx.x] = r;
  }
}
#undef KVQ_REC

inline size_t split_workspace_bytes(const KvqView& v, int batch) {
  const long long items = kFastTarget + 2LL * batch;
  return fast_header_bytes(batch) + (size_t)items * v.Hq * (v.D + 4) * sizeof(float);
}

// Partials -> out: one CTA per (query head, sequence).
inline cudaError_t launch_split_combine(const KvqView& v, float* ws, float* out, cudaStream_t st) {
  combine_fast_kernel<<<dim3(v.Hq, v.batch), kCombineThreads, 0, st>>>(v, ws, out);
  return cudaGetLastError();
}

}  // namespace
}  // namespace kvq
