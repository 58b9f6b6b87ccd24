// Host-side launch bookkeeping shared by the translation units: settings that a
// launcher computes once per device (a kernel's dynamic shared-memory limit,
// its occupancy, the SM count), kept per (device, slot) behind one lock so
// that host threads calling the library at the same time, or one thread that
// moves between devices, never skip a setting or read a half-written one.
//
// The cached values belong to the process's primary context of each device; a
// cudaDeviceReset() drops the kernel attributes they stand for, so the library
// does not support being used across a device reset.
#pragma once

#include <cuda_runtime.h>
#include <nvtx3/nvToolsExt.h>

#include <mutex>

#include "../../include/kvq.h"

namespace kvq {
// Internal linkage: every translation unit (and every copy of the library loaded
// into one process) keeps its own table.  Function-local statics of ordinary
// inline functions would become process-wide unique symbols, shared between two
// builds of the library loaded side by side, and one build would then skip a
// kernel attribute that only its own kernels carry.
namespace {

constexpr int kMaxDevices = 64;

enum SetupSlot {
  kSlotSms = 0,        // multiprocessor count
  kSlotAppend,         // append kernel: dynamic shared-memory limit raised
  kSlotGeneric,        // generic decode kernels (12 instances): shared-memory limit set so far
  kSlotGenericOcc = kSlotGeneric + 12,  // the same instances: last (shared memory, CTAs per SM)
  kSlotFast = kSlotGenericOcc + 12,     // pre-RoPE tensor-core kernel, 4 instances: CTAs per SM
  kSlotFp8 = kSlotFast + 4,       // FP8 tensor-core kernel, 2 instances
  kSlotInt2 = kSlotFp8 + 2,       // 2-bit tensor-core kernel, 2 instances
  kSlotCount = kSlotInt2 + 2
};

inline std::mutex& setup_mutex() {
  static std::mutex m;
  return m;
}

inline long long& setup_value(int dev, int slot) {
  static long long table[kMaxDevices][kSlotCount] = {};
  return table[dev][slot];
}

// The calling thread's current device, or -1 (the CUDA error is cleared).
inline int current_device() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    (void)cudaGetLastError();
    return -1;
  }
  return dev;
}

// Value of `slot` on the current device: computed by setup(&value) on the first
// call (setup returns KVQ_OK and a value > 0), cached afterwards.
template <class F>
kvq_status per_device_once(int slot, F&& setup, long long* value) {
  const int dev = current_device();
  if (dev < 0) return KVQ_ERR_CUDA;
  if (dev >= kMaxDevices) return KVQ_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(setup_mutex());
  long long& v = setup_value(dev, slot);
  if (v <= 0) {
    long long r = 0;
    const kvq_status s = setup(&r);
    if (s != KVQ_OK) return s;
    if (r <= 0) return KVQ_ERR_CUDA;
    v = r;
  }
  *value = v;
  return KVQ_OK;
}

// Raise a kernel's dynamic shared-memory limit on the current device to at
// least `bytes` (remembered per device in `slot`, so the attribute is set again
// only when a call needs more).
template <class Kern>
kvq_status ensure_dynamic_smem(int slot, Kern kern, size_t bytes) {
  const int dev = current_device();
  if (dev < 0) return KVQ_ERR_CUDA;
  if (dev >= kMaxDevices) return KVQ_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(setup_mutex());
  long long& v = setup_value(dev, slot);
  if ((long long)bytes > v) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes) != cudaSuccess) {
      (void)cudaGetLastError();
      return KVQ_ERR_CAPACITY;
    }
    v = (long long)bytes;
  }
  return KVQ_OK;
}

// Multiprocessor count of the current device (148 when it cannot be read).
inline int num_sms() {
  long long n = 0;
  const kvq_status s = per_device_once(
      kSlotSms,
      [](long long* out) {
        int c = 0;
        if (cudaDeviceGetAttribute(&c, cudaDevAttrMultiProcessorCount, current_device()) != cudaSuccess) {
          (void)cudaGetLastError();
          return KVQ_ERR_CUDA;
        }
        *out = c;
        return KVQ_OK;
      },
      &n);
  return s == KVQ_OK ? (int)n : 148;
}

// CTAs per SM of a kernel at a block size and dynamic shared memory, after its
// dynamic shared-memory limit is raised to `smem_limit`; cached per device in `slot`.
template <class Kern>
kvq_status occupancy_once(int slot, Kern kern, int threads, size_t smem, size_t smem_limit, int* ctas) {
  long long occ = 0;
  const kvq_status s = per_device_once(
      slot,
      [&](long long* out) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_limit) !=
            cudaSuccess) {
          (void)cudaGetLastError();
          return KVQ_ERR_CUDA;
        }
        int o = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&o, kern, threads, smem) != cudaSuccess) {
          (void)cudaGetLastError();
          return KVQ_ERR_CUDA;
        }
        *out = o > 0 ? o : 1;
        return KVQ_OK;
      },
      &occ);
  *ctas = (int)occ;
  return s;
}

// CTAs per SM of `kern` at `threads` threads and `smem` dynamic bytes (its
// shared-memory limit already raised that far).  The last answer per device is
// kept in `slot` with its byte count: consecutive calls of one workload ask for
// the same bytes and skip the query.
template <class Kern>
kvq_status occupancy_at(int slot, Kern kern, int threads, size_t smem, int* ctas) {
  const int dev = current_device();
  if (dev < 0) return KVQ_ERR_CUDA;
  if (dev >= kMaxDevices) return KVQ_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(setup_mutex());
  long long& v = setup_value(dev, slot);
  if (v > 0 && (v >> 16) == (long long)smem) {
    *ctas = (int)(v & 0xFFFF);
    return KVQ_OK;
  }
  int o = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&o, kern, threads, smem) != cudaSuccess) {
    (void)cudaGetLastError();
    return KVQ_ERR_CUDA;
  }
  if (o < 1) o = 1;
  if (o > 0xFFFF) o = 0xFFFF;
  v = ((long long)smem << 16) | o;
  *ctas = o;
  return KVQ_OK;
}

// NVTX range around one public call, in the "libkvq" domain: profilers show the
// host time of each call and can attribute the kernels it launches to it (ncu:
// --nvtx --nvtx-include "libkvq@kvq_decode_attention/").  With no tool attached
// a push or pop is a test of one function pointer.
inline nvtxDomainHandle_t nvtx_domain() {
  static const nvtxDomainHandle_t d = nvtxDomainCreateA("libkvq");
  return d;
}

struct NvtxRange {
  explicit NvtxRange(const char* name) {
    nvtxEventAttributes_t a = {};
    a.version = NVTX_VERSION;
    a.size = NVTX_EVENT_ATTRIB_STRUCT_SIZE;
    a.messageType = NVTX_MESSAGE_TYPE_ASCII;
    a.message.ascii = name;
    nvtxDomainRangePushEx(nvtx_domain(), &a);
  }
  ~NvtxRange() { nvtxDomainRangePop(nvtx_domain()); }
  NvtxRange(const NvtxRange&) = delete;
  NvtxRange& operator=(const NvtxRange&) = delete;
};

}  // namespace
}  // namespace kvq
