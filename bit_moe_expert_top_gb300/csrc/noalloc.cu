// Scratch of the 2-bit decode GEMV held by the library itself, for callers
// that cannot hand it a workspace.
//
// The table GEMV needs a few MB of device scratch per call (the per-slice
// row sums that its second kernel adds up).  moe_w2_mm takes it from the caller.  Some callers
// cannot provide it: plain C host code that drives the library with nothing
// but the model's own buffers and has no device allocator of its own, or a
// serving engine that has already handed all of its spare device memory to
// its KV cache and may not allocate on the decode path.  For them the scratch
// below is a fixed array in the library's own module: it exists from the
// moment the module is loaded, so a call here allocates and frees nothing.
//
// Set-up: the first call on a device (with that device current) looks up the
// array's device address with cudaGetSymbolAddress.  That lookup may load the
// module on the device, so that first call should come before any stream
// capture.  One array serves every call on a device: calls that overlap on the
// GPU (different streams, or other threads) race on it.
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "../../include/moe.h"
#include "internal.cuh"

namespace moe {

namespace {

static __device__ __align__(256) uint8_t g_w2_scratch[MOE_W2_NOALLOC_SCRATCH_BYTES];

std::mutex g_scratch_mu;
void* g_scratch_ptr[64] = {nullptr};

}  // namespace

cudaError_t noalloc_scratch(void** ptr) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_w2_scratch);
    if (e != cudaSuccess) return e;
    if (!p) return cudaErrorInvalidSymbol;
    g_scratch_ptr[dev] = p;
  }
  *ptr = g_scratch_ptr[dev];
  return cudaSuccess;
}

cudaError_t launch_lut_gemv_noalloc(MMArgs a, int rows, cudaStream_t s) {
  void* ws = nullptr;
  cudaError_t e = noalloc_scratch(&ws);
  if (e != cudaSuccess) return e;
  a.ws = ws;
  a.ws_rows = rows;
  a.ws_bytes = lut_workspace_bytes(a.stage, rows, a.N, a.K);
  // nothing in the scratch needs to start at zero: every slice sum is
  // written before it is read
  return launch_lut_gemv(a, ws, s);
}

}  // namespace moe
