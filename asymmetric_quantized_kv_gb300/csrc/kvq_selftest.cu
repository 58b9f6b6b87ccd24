// Self-test of the decode kernels' failure detection: every pipeline wait in
// them is bounded (ptx::kWaitPolls polls), and a wait that gives up sets
// KVQ_DEV_TIMEOUT in the caller's status word and lets the kernel finish, so the
// context stays usable.  Here one warp waits, with that same bounded wait, on an
// mbarrier phase that nothing completes; no copy is in flight, nothing faults.
#include "kvq_host.h"
#include "kvq_internal.cuh"
#include "kvq_ptx.cuh"

namespace {

__global__ void bounded_wait_selftest_kernel(int32_t* status) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    kvq::ptx::mbar_init(&bar, 1);  // one arrival would complete phase 0; none comes
    kvq::ptx::fence_mbar_init();
  }
  __syncwarp();
  if (threadIdx.x == 0 && !kvq::ptx::mbar_wait_bounded(&bar, 0, kvq::ptx::kWaitPolls))
    atomicOr(status, KVQ_DEV_TIMEOUT);
}

}  // namespace

extern "C" kvq_status kvq_selftest_bounded_wait(int32_t* status, void* stream) {
  const kvq::NvtxRange range("kvq_selftest_bounded_wait");
  if (!status) return KVQ_ERR_INVALID_ARG;
  bounded_wait_selftest_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(status);
  return cudaGetLastError() == cudaSuccess ? KVQ_OK : KVQ_ERR_CUDA;
}
