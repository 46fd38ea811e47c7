// Diagnostic of the bounded pipeline waits (moe_selftest_wait_timeout in moe.h).
//
// Every mbarrier wait in the GEMM pipelines goes through mbar_wait_bounded.  This
// kernel runs that routine on a barrier phase that nothing will ever complete, with
// a short limit, so a test can check -- without faulting or hanging anything -- that
// a wait which cannot finish ends with MOE_DEVERR_TIMEOUT in the flag word and a
// kernel that returns normally.

#include <cuda_runtime.h>

#include "../../include/moe.h"
#include "common.cuh"

namespace {

__global__ void wait_timeout_kernel(int* flags, uint64_t limit_ns) {
  __shared__ uint64_t bar;
  __shared__ int abort;
  if (threadIdx.x == 0) {
    moe::mbar_init(moe::smem_u32(&bar), 1);
    abort = 0;
    moe::fence_mbar_init();
  }
  __syncthreads();
  // Phase 0 needs one arrival that no thread makes.
  if (threadIdx.x == 0) moe::mbar_wait_bounded(moe::smem_u32(&bar), 0, &abort, flags, limit_ns);
}

}  // namespace

extern "C" __attribute__((visibility("default"))) moe_status moe_selftest_wait_timeout(
    int32_t* device_flags, uint64_t limit_ns, moe_stream_t stream) {
  if (!device_flags || (reinterpret_cast<uintptr_t>(device_flags) & 3u) != 0)
    return MOE_ERR_INVALID_ARGUMENT;
  if (limit_ns == 0 || limit_ns > moe::kWaitLimitNs) return MOE_ERR_INVALID_ARGUMENT;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(device_flags, 0, sizeof(int32_t), st) != cudaSuccess) return MOE_ERR_CUDA;
  wait_timeout_kernel<<<1, 32, 0, st>>>(device_flags, limit_ns);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
