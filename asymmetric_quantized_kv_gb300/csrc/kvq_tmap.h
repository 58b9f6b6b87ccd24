// Host helper: the driver's cuTensorMapEncodeTiled, looked up through the
// runtime (no link against the driver library), or nullptr when unavailable.
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

namespace kvq {
namespace {  // internal linkage: one lookup per translation unit, never shared across libraries

inline PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  // looked up once per process (a function-local static initialises once, even
  // when several threads arrive together)
  static const PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult res;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &res) ==
            cudaSuccess &&
        res == cudaDriverEntryPointSuccess)
      return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    (void)cudaGetLastError();
    return static_cast<PFN_cuTensorMapEncodeTiled_v12000>(nullptr);
  }();
  return fn;
}

}  // namespace
}  // namespace kvq
