// Diagnostics of the library's own error paths, runnable on any device
// without faulting it.
#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"
#include "internal.cuh"

namespace moe {

namespace {

// One warp: lane 0 initialises a shared-memory mbarrier that expects one
// arrival, and nobody ever arrives.  Lane 0 then waits on its first phase with
// the same bounded wait the pipelines use; when the limit runs out it records
// MOE_DEVERR_TIMEOUT.  No copy, MMA or other asynchronous work is in flight,
// so the kernel simply returns.
__global__ void bounded_wait_check_kernel(long long limit, uint32_t* dev_err) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_barrier_init();
  }
  __syncwarp();
  if (threadIdx.x == 0 && !mbar_wait(&bar, 0, limit)) set_err(dev_err, MOE_DEVERR_TIMEOUT);
}

}  // namespace

cudaError_t launch_bounded_wait_check(long long cycles, uint32_t* dev_err, cudaStream_t s) {
  bounded_wait_check_kernel<<<1, 32, 0, s>>>(cycles, dev_err);
  return cudaGetLastError();
}

}  // namespace moe
