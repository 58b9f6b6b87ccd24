// Split-K work plan, workspace layout and partial combine shared by the
// tensor-core decode kernels (head_dim 128).  An item is (sequence, chunk of
// C tokens); a kernel processes it for every kv-head, and writes one partial
// record (running max, softmax sum, unnormalised output) per (item, query head).
#pragma once

#include "kvq_attn_plan.cuh"
#include "kvq_ptx.cuh"

namespace kvq {
namespace {

constexpr int kD = 128;
constexpr int kFastTarget = 1024;     // chunks per call (about): C = total tokens / target
constexpr int kFastTargetCut = 768;   // the same for kernels that cut the final round (measured best)
constexpr int kMinPiece = 256;        // cut only when a piece keeps at least this many tokens
constexpr int kFastMinChunk = 256;
constexpr int kTailPieces = 4;   // pieces per chunk of the final round, and per partial chunk at most
constexpr int kTailMax = 320;    // chunks of the final round that are cut (one round of work at most)

struct FastItem {
  int b, t0, t1, window;
};

// Work plan of the tensor-core kernels, at the head of the workspace:
//   int C, NA, NB, NS; int prefA[B+1]; int prefB[B+1]; u64 counter
// Workers take items dynamically from the counter (zeroed by the host before each
// call), in this order:
//   - whole C-token chunks of every sequence (prefA: per-sequence prefix of chunk
//     counts), all but the last NS;
//   - those last NS chunks (about one round of work), each cut into kTailPieces
//     group-aligned pieces: items up to NA;
//   - per sequence (prefB: prefix of its short items): its last, partial chunk cut
//     into pieces of at most piece_tokens(C) tokens, then its residual window.
// Everything fetched in the final round is then at most a quarter chunk, so the
// workers, which do not all run at one speed, finish close together.  The cuts
// are made for kernels whose worker is a whole CTA (two CTAs share an SM and one
// of them runs markedly slower); kernels whose workers are warps pass cut = false
// and keep whole chunks and whole partial chunks (NS = 0, one piece per partial).
__host__ __device__ inline size_t fast_header_ints(int B) { return (size_t)2 * (B + 1) + 4; }
__host__ __device__ inline size_t fast_counter_offset(int B) { return (fast_header_ints(B) * 4 + 7) & ~(size_t)7; }
__host__ __device__ inline size_t fast_header_bytes(int B) { return (fast_counter_offset(B) + 8 + 255) / 256 * 256; }

// Whether a plan with chunk size C cuts (the kernel asks for cuts and the pieces
// keep at least kMinPiece tokens; the plan and the item decoder both apply this).
__host__ __device__ inline bool cuts(int C, bool cut) { return cut && C / kTailPieces >= kMinPiece; }

// Tokens of one piece of a partial chunk: a quarter chunk, group-aligned (the
// whole chunk when the plan does not cut).
__host__ __device__ inline int piece_tokens(int C, int align, bool cut) {
  return cuts(C, cut) ? ((C / kTailPieces + align - 1) / align) * align : C;
}
__host__ __device__ inline int partial_pieces(int p, int S) { return p ? (p + S - 1) / S : 0; }

// NT threads per block; scratch: 2 * NT ints of shared memory that are free
// until the caller's main loop.  units: work units per item (kv-heads when a
// worker takes one head of an item, else 1); workers: how many take units at once.
template <int NT>
__device__ inline void fast_plan(const KvqView& v, int align, int units, int workers, bool cut, int* sA, int* sB,
                                 int* s_C, int* s_NA, int* s_NB, int* s_NS, int* scratch) {
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
  // cutting kernels: chunks for about kFastTargetCut items, cut at the end -- unless
  // the pieces would fall below kMinPiece tokens (small calls), where the per-item
  // setup outweighs the balance and the plain plan of kFastTarget chunks is used
  auto chunk_of = [&](int target) {
    long long c = (long long)((s_total + target - 1) / target);
    if (c < kFastMinChunk) c = kFastMinChunk;
    return (c + align - 1) / align * align;
  };
  long long C = chunk_of(cut ? kFastTargetCut : kFastTarget);
  if (!cuts((int)C, cut)) {
    cut = false;
    C = chunk_of(kFastTarget);  // below kMinPiece * kTailPieces as well, so cuts() stays false
  }
  const int S = piece_tokens((int)C, align, cut);
  const int seg = (B + NT - 1) / NT;
  const int b0 = threadIdx.x * seg, b1 = min(B, b0 + seg);
  int la = 0, lb = 0;
  for (int b = b0; b < b1; ++b) {
    const int T = seq_tokens(v, b), nq = n_quantized(T, v.R);
    la += nq / (int)C;
    lb += partial_pieces(nq % (int)C, S) + (T > nq ? 1 : 0);
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
    // about one round of work units is cut into pieces
    int NS = (cut && C / align >= kTailPieces) ? min(min(ra, (workers + units - 1) / units), kTailMax) : 0;
    *s_NA = ra - NS + NS * kTailPieces;
    *s_NB = rb;
    *s_C = (int)C;
    *s_NS = NS;
  }
  __syncthreads();
  int ra = s_pa[threadIdx.x], rb = s_pb[threadIdx.x];
  for (int b = b0; b < b1; ++b) {
    const int T = seq_tokens(v, b), nq = n_quantized(T, v.R);
    sA[b] = ra;
    sB[b] = rb;
    ra += nq / (int)C;
    rb += partial_pieces(nq % (int)C, S) + (T > nq ? 1 : 0);
  }
  if (threadIdx.x == 0) {
    sA[B] = *s_NA - *s_NS * (kTailPieces - 1);  // total full chunks
    sB[B] = *s_NB;
  }
  __syncthreads();
}

__device__ inline void store_fast_plan(const KvqView& v, float* ws, const int* sA, const int* sB, int C, int NA,
                                       int NB, int NS) {
  int* h = reinterpret_cast<int*>(ws);
  if (threadIdx.x == 0) {
    h[0] = C;
    h[1] = NA;
    h[2] = NB;
    h[3] = NS;
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

// Item d of the plan (NA: chunk items including the pieces, NS: chunks cut).
__device__ inline FastItem decode_fast_item(const KvqView& v, const int* sA, const int* sB, int C, int NA,
                                            int NS, int align, bool cut, int d) {
  FastItem it;
  const int NU = NA - NS * kTailPieces;  // chunks kept whole
  if (d < NA) {
    int c = d, k = -1;
    if (d >= NU) {  // piece k of chunk c
      c = NU + (d - NU) / kTailPieces;
      k = (d - NU) % kTailPieces;
    }
    it.b = seq_of(sA, v.batch, c);
    it.window = 0;
    it.t0 = (c - sA[it.b]) * C;
    it.t1 = it.t0 + C;
    if (k >= 0) {
      const int groups = C / align, base = it.t0;
      it.t0 = base + (k * groups / kTailPieces) * align;
      it.t1 = base + ((k + 1) * groups / kTailPieces) * align;
    }
    return it;
  }
  const int e = d - NA;
  it.b = seq_of(sB, v.batch, e);
  const int T = seq_tokens(v, it.b), nq = n_quantized(T, v.R);
  const int S = piece_tokens(C, align, cut), j = e - sB[it.b];
  if (j < partial_pieces(nq % C, S)) {  // piece j of the partial chunk
    it.window = 0;
    it.t0 = (nq / C) * C + j * S;
    it.t1 = min(nq, it.t0 + S);
  } else {
    it.window = 1;
    it.t0 = nq;
    it.t1 = T;
  }
  return it;
}


// Merge the chunk partials of one (sequence, query head).  Records are
// kRec = D + 4 floats (max, sum, 2 pad, output) so outputs are 16-byte aligned.
// Four warps take every fourth record; a warp loads a batch of up to
// kCombineBatch records at once (lane = channel quad, float4 loads) and merges
// them online into its running max, sum and output, so one round of loads covers
// a typical sequence.  The warps then merge through shared memory.  Launched as a
// programmatic dependent of the split kernel: it waits for that grid to complete
// before reading the workspace.
constexpr int kRec = kD + 4;
constexpr int kCombineWarps = 4;
constexpr int kCombineThreads = kCombineWarps * 32;
constexpr int kCombineBatch = 8;

__global__ void __launch_bounds__(kCombineThreads) combine_fast_kernel(KvqView v, float* ws, float* out) {
  __shared__ float4 o_s[kCombineWarps][kD / 4];
  __shared__ float m_s[kCombineWarps], l_s[kCombineWarps];
  ptx::grid_dep_wait();
  const int hq = blockIdx.x, b = blockIdx.y;
  const int* hdr = reinterpret_cast<const int*>(ws);
  const int NA = hdr[1], NS = hdr[3];
  const int NU = NA - NS * kTailPieces;
  const int* pA = hdr + 4;
  const int* pB = pA + v.batch + 1;
  const float* part = reinterpret_cast<const float*>(reinterpret_cast<const char*>(ws) + fast_header_bytes(v.batch));
  // this sequence's records: its whole chunks at item pA[b].., the pieces of its
  // cut chunks (chunks >= NU), then its nB short items at NA + pB[b]..
  const int a0 = pA[b], nC = pA[b + 1] - pA[b], nB = pB[b + 1] - pB[b];
  const int nWhole = max(0, min(nC, NU - a0));
  const int nA = nWhole + (nC - nWhole) * kTailPieces;
  const int n = nA + nB;
  const long long stride = (long long)v.Hq * kRec;
  const long long firstPiece = NU + (long long)(a0 + nWhole - NU) * kTailPieces;  // item of its first piece
  const float* baseA = part + ((long long)a0 * v.Hq + hq) * kRec;
  const float* baseP = part + (firstPiece * v.Hq + hq) * kRec;
  const float* baseB = part + ((long long)(NA + pB[b]) * v.Hq + hq) * kRec;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  float m = -INFINITY, l = 0.f;
  float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int i0 = warp; i0 < n; i0 += kCombineWarps * kCombineBatch) {
    float rm[kCombineBatch], rl[kCombineBatch];
    float4 x[kCombineBatch];
#pragma unroll
    for (int j = 0; j < kCombineBatch; ++j) {
      const int i = i0 + j * kCombineWarps;
      rm[j] = -INFINITY;
      rl[j] = 0.f;
      x[j] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (i < n) {
        const float* r = i < nWhole ? baseA + (long long)i * stride
                          : i < nA   ? baseP + (long long)(i - nWhole) * stride
                                     : baseB + (long long)(i - nA) * stride;
        rm[j] = r[0];
        rl[j] = r[1];
        x[j] = reinterpret_cast<const float4*>(r + 4)[lane];
      }
    }
    float mn = m;
#pragma unroll
    for (int j = 0; j < kCombineBatch; ++j) mn = fmaxf(mn, rm[j]);
    if (mn != -INFINITY) {  // warp-uniform: every lane read the same records
      const float a = exp2f(m - mn);  // 0 while nothing has been merged
      l *= a;
      o.x *= a; o.y *= a; o.z *= a; o.w *= a;
#pragma unroll
      for (int j = 0; j < kCombineBatch; ++j) {
        const float w = rm[j] == -INFINITY ? 0.f : exp2f(rm[j] - mn);
        l = fmaf(rl[j], w, l);
        o.x = fmaf(x[j].x, w, o.x); o.y = fmaf(x[j].y, w, o.y);
        o.z = fmaf(x[j].z, w, o.z); o.w = fmaf(x[j].w, w, o.w);
      }
      m = mn;
    }
  }
  if (lane == 0) {
    m_s[warp] = m;
    l_s[warp] = l;
  }
  o_s[warp][lane] = o;
  __syncthreads();
  if (warp == 0) {
    float M = m_s[0];
#pragma unroll
    for (int w = 1; w < kCombineWarps; ++w) M = fmaxf(M, m_s[w]);
    float L = 0.f;
    float4 r = make_float4(0.f, 0.f, 0.f, 0.f);
    if (M != -INFINITY) {
#pragma unroll
      for (int w = 0; w < kCombineWarps; ++w) {
        const float a = m_s[w] == -INFINITY ? 0.f : exp2f(m_s[w] - M);
        const float4 x = o_s[w][lane];
        L = fmaf(l_s[w], a, L);
        r.x = fmaf(x.x, a, r.x); r.y = fmaf(x.y, a, r.y); r.z = fmaf(x.z, a, r.z); r.w = fmaf(x.w, a, r.w);
      }
    }
    const float invL = L > 0.f ? 1.f / L : 0.f;
    r.x *= invL; r.y *= invL; r.z *= invL; r.w *= invL;
    reinterpret_cast<float4*>(out + ((long long)b * v.Hq + hq) * kD)[lane] = r;
  }
}

inline size_t split_workspace_bytes(const KvqView& v, int batch) {
  // whole chunks + the pieces of at most kTailMax cut chunks + per sequence up
  // to kTailPieces + 1 partial-chunk pieces and one window
  const long long items = kFastTarget + (long long)(kTailPieces - 1) * kTailMax + (kTailPieces + 2LL) * batch;
  return fast_header_bytes(batch) + (size_t)items * v.Hq * (v.D + 4) * sizeof(float);
}

// Partials -> out: one CTA per (query head, sequence), launched as a programmatic
// dependent of the split kernel just before it in the stream, so its CTAs are
// scheduled as the split kernel's CTAs retire.
inline cudaError_t launch_split_combine(const KvqView& v, float* ws, float* out, cudaStream_t st) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(v.Hq, v.batch);
  cfg.blockDim = dim3(kCombineThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, combine_fast_kernel, v, ws, out);
}

}  // namespace
}  // namespace kvq
