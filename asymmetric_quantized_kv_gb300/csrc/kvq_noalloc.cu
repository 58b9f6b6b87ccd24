// kvq_decode_attention_noalloc: decode attention whose split-K workspace is a
// fixed array that lives inside this library, for callers that cannot allocate
// device memory themselves.
//
// Who needs it: a plugin running inside a serving process whose memory pool has
// already claimed the GPU's memory (a cudaMalloc behind the pool's back can fail
// or break its accounting), or code on a latency-critical path that must not
// call cudaMalloc (which can synchronise the device).  Such callers still pass
// q and out; the scratch comes from here.
//
// The array below is a file-scope __device__ variable: every GPU on which this
// library's module is loaded holds KVQ_NOALLOC_SCRATCH_BYTES of it until the
// process exits.  Host code cannot use the name g_scratch as a device address
// (on the host it is only a stand-in), so the device address is looked up once
// per device with cudaGetSymbolAddress, with that device current, and cached.
// All calls on a device share the array and it keeps the last call's contents;
// the attention kernels write every workspace byte before they read it, so
// nothing has to be cleared between calls.  The cached address belongs to the
// device's primary context: after a cudaDeviceReset() the library (like its
// other per-device launch settings) has to be reloaded; a reset is not supported.
#include <mutex>

#include "kvq_host.h"
#include "kvq_internal.cuh"

namespace {

static __device__ __align__(256) unsigned char g_scratch[KVQ_NOALLOC_SCRATCH_BYTES];

std::mutex g_mutex;
void* g_scratch_addr[64] = {nullptr};

// Device address of g_scratch on the calling thread's current device.
kvq_status scratch_address(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return KVQ_ERR_CUDA;
  }
  if (dev < 0 || dev >= 64) return KVQ_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_mutex);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_scratch);
    if (e != cudaSuccess || p == nullptr) {
      cudaGetLastError();
      return KVQ_ERR_CUDA;
    }
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return KVQ_OK;
}

}  // namespace

extern "C" kvq_status kvq_decode_attention_noalloc(const kvq_config* cfg, const kvq_cache* cache,
                                                   const void* q, float* out, float softmax_scale,
                                                   void* stream) {
  const kvq::NvtxRange range("kvq_decode_attention_noalloc");
  if (!cfg || !cache) return KVQ_ERR_INVALID_ARG;
  const kvq_status valid = kvq_validate(cfg);
  if (valid != KVQ_OK) return valid;
  if (cache->batch < 1 || cache->max_pages_per_seq < 1) return KVQ_ERR_INVALID_ARG;
  // the longest sequence the block table can address, in 64-bit arithmetic
  const long long max_len = (long long)cache->max_pages_per_seq * cfg->page_size;
  if (max_len > 0x7fffffffLL) return KVQ_ERR_INVALID_ARG;
  const size_t need = kvq_workspace_bytes(cfg, cache->batch, (int)max_len);
  if (need == 0) return KVQ_ERR_INVALID_ARG;
  if (need > (size_t)KVQ_NOALLOC_SCRATCH_BYTES) return KVQ_ERR_CAPACITY;
  void* scratch = nullptr;
  const kvq_status s = scratch_address(&scratch);
  if (s != KVQ_OK) return s;
  return kvq_decode_attention(cfg, cache, q, out, softmax_scale, scratch,
                              (size_t)KVQ_NOALLOC_SCRATCH_BYTES, stream);
}
