// Management of the FP4 delta cache on the device: which experts hold an
// MXFP4 slot, updated from the routing between steps with no host sync, and
// the copies that fill the slots of newly promoted experts.
//
// The pages keep the hottest experts at FP4 precision over the 2-bit base
// (blog "这个项目我们能学到什么?" on vLLM-Moet, FP4 delta-cache paragraph) and
// use the GPU as a cache of hot experts (same blog, "GPU作为专家缓存").  The
// policy (readings, the pages fix neither part):
//   * hotness: per expert an integer moving average of routed assignments,
//     c <- c - (c >> d) + n_e each step (d >= 31: cumulative), saturating;
//   * the cached set: the S largest counts, ties to the lowest expert id;
//   * slots are stable: a retained expert keeps its slot, leaving experts
//     free theirs, entering experts take the free slots in ascending order,
//     hottest first.
// One CTA does the selection (E <= 1024); the fill is a grid of 16-byte
// copies per (slot, chunk) that reads the expert store through any
// device-accessible pointer: device memory, or pinned host memory mapped into
// the device's address space (read over the CPU-GPU link).
#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"
#include "internal.cuh"

namespace moe {

namespace {

constexpr int kSelThreads = 1024;

__global__ void __launch_bounds__(kSelThreads) cache_select_kernel(const int32_t* __restrict__ offsets, int E,
                                                                   uint32_t* __restrict__ counts, int decay_shift,
                                                                   int S, int32_t* __restrict__ expert_slot,
                                                                   int32_t* __restrict__ slot_expert,
                                                                   int32_t* __restrict__ promoted, uint32_t* dev_err) {
  __shared__ uint32_t sc[1024];   // updated counts
  __shared__ int in_slot[1024];   // slot of each expert before the update, -1 if none
  __shared__ int by_rank[1024];   // expert of rank r (r < S)
  __shared__ int new_se[1024];    // slot -> expert after eviction, then after promotion
  __shared__ int bad;
  pdl_wait();
  pdl_trigger();
  const int tid = threadIdx.x;
  if (tid == 0) bad = 0;
  if (tid < S) new_se[tid] = -1;
  if (tid < E) {
    const int n = offsets[tid + 1] - offsets[tid];
    uint64_t c = counts[tid];
    if (decay_shift < 31) c -= c >> decay_shift;
    c += static_cast<uint64_t>(n < 0 ? 0 : n);
    const uint32_t c32 = c > 0xFFFFFFFFull ? 0xFFFFFFFFu : static_cast<uint32_t>(c);
    sc[tid] = c32;
    counts[tid] = c32;
    in_slot[tid] = -1;
  }
  __syncthreads();
  // residency comes from the slot -> expert map (the source of truth)
  if (tid < S) {
    const int e = slot_expert[tid];
    if (e >= E) atomicOr(&bad, 1);
    if (e >= 0 && e < E) in_slot[e] = tid;
  }
  __syncthreads();
  // rank of each expert in (count desc, id asc); a cached expert that stays
  // in the top S keeps its slot, the other slots are free
  if (tid < E) {
    const uint32_t mine = sc[tid];
    int r = 0;
    for (int f = 0; f < E; ++f) {
      const uint32_t o = sc[f];
      r += (o > mine || (o == mine && f < tid)) ? 1 : 0;
    }
    if (r < S) by_rank[r] = tid;
    const int s = in_slot[tid];
    if (s >= 0 && r < S) new_se[s] = tid;
  }
  __syncthreads();
  // promotion: the top-S experts without a slot, in rank order, take the free
  // slots in ascending order (serial over S <= 1024 slots)
  if (tid == 0) {
    int fs = 0;
    const int top = S < E ? S : E;
    for (int r = 0; r < top; ++r) {
      const int e = by_rank[r];
      if (in_slot[e] >= 0) continue;
      while (fs < S && new_se[fs] >= 0) ++fs;
      if (fs >= S) break;  // cannot happen: at most S - retained experts enter
      new_se[fs] = e;
      promoted[fs] = e;
      in_slot[e] = -2 - fs;  // marks "promoted into fs"
    }
    if (bad) set_err(dev_err, MOE_DEVERR_BAD_ID);
  }
  __syncthreads();
  if (tid < S) {
    const int e = new_se[tid];
    const int old = slot_expert[tid];
    if (!(e >= 0 && old != e)) promoted[tid] = -1;
    slot_expert[tid] = e;
  }
  if (tid < E) {
    // after the scan: in_slot = s (retained or evicted), -2 - s (promoted), -1
    const int s = in_slot[tid];
    int ns = -1;
    if (s <= -2) ns = -2 - s;
    else if (s >= 0 && new_se[s] == tid) ns = s;
    expert_slot[tid] = ns;
  }
}

// Host-resident experts staged per step: every expert routed in this step
// that has no resident slot gets a staging slot (R + j, j in ascending
// expert order); its weights are then copied in (cache_fill_kernel) while the
// resident experts' matmuls run.
__global__ void __launch_bounds__(kSelThreads) stage_select_kernel(const int32_t* __restrict__ offsets, int E,
                                                                   const int32_t* __restrict__ res_slot, int R,
                                                                   int S, int32_t* __restrict__ weight_slot,
                                                                   int32_t* __restrict__ staged, uint32_t* dev_err) {
  __shared__ int warp_tot[32];
  pdl_wait();
  pdl_trigger();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  int cold = 0, rs = -1;
  if (tid < E) {
    rs = res_slot[tid];
    if (rs >= R) {
      set_err(dev_err, MOE_DEVERR_BAD_ID);
      rs = -1;
    }
    cold = (offsets[tid + 1] > offsets[tid] && rs < 0) ? 1 : 0;
  }
  // exclusive prefix of the cold flags over the block (ascending expert id)
  int incl = cold;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) warp_tot[warp] = incl;
  __syncthreads();
  int before = 0;
  for (int w = 0; w < warp; ++w) before += warp_tot[w];
  const int j = before + incl - cold;
  if (tid < S) staged[tid] = -1;
  __syncthreads();
  if (tid < E) {
    int ws = rs;
    if (cold) {
      if (j < S) {
        ws = R + j;
        staged[j] = tid;
      } else {
        set_err(dev_err, MOE_DEVERR_OVERFLOW);  // more routed cold experts than staging slots: skipped
        ws = -1;
      }
    }
    weight_slot[tid] = ws;
  }
}

struct FillArgs {
  const uint8_t* src[4];
  uint8_t* dst[4];
  size_t bytes[4];  // per expert (src) and per slot (dst)
  int n;
};

__global__ void __launch_bounds__(256) cache_fill_kernel(const int32_t* __restrict__ promoted, const FillArgs F) {
  pdl_wait();
  pdl_trigger();
  const int s = blockIdx.y;
  const int e = promoted[s];
  if (e < 0) return;
  // four independent 16-byte loads in flight per thread: the source may be
  // host memory behind the CPU-GPU link, where latency is long
  const size_t stride = static_cast<size_t>(gridDim.x) * blockDim.x;
  for (int a = 0; a < F.n; ++a) {
    const size_t n16 = F.bytes[a] / 16;
    const uint4* src = reinterpret_cast<const uint4*>(F.src[a] + static_cast<size_t>(e) * F.bytes[a]);
    uint4* dst = reinterpret_cast<uint4*>(F.dst[a] + static_cast<size_t>(s) * F.bytes[a]);
    size_t i = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    for (; i + 3 * stride < n16; i += 4 * stride) {
      uint4 v[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) v[u] = __ldcs(src + i + u * stride);
#pragma unroll
      for (int u = 0; u < 4; ++u) dst[i + u * stride] = v[u];
    }
    for (; i < n16; i += stride) dst[i] = __ldcs(src + i);
  }
}

// The same copy on the side SMs (moe_set_side_sms): one CTA of 1024
// threads per side SM (its unused shared-memory request is over half an
// SM's, so no second CTA fits beside it); the CTAs walk every slot's bytes
// together, four 16-byte loads in flight per thread, which keeps a few SMs
// enough to fill the CPU-GPU link.
constexpr int kFillThreads = 1024;
constexpr int kFillPinSmem = 120 * 1024;

__global__ void __launch_bounds__(kFillThreads, 1) cache_fill_sm_kernel(const int32_t* __restrict__ promoted, int S,
                                                                        const FillArgs F) {
  pdl_wait();
  pdl_trigger();
  const size_t stride = static_cast<size_t>(gridDim.x) * blockDim.x;
  for (int s = 0; s < S; ++s) {
    const int e = promoted[s];
    if (e < 0) continue;
    for (int a = 0; a < F.n; ++a) {
      const size_t n16 = F.bytes[a] / 16;
      const uint4* src = reinterpret_cast<const uint4*>(F.src[a] + static_cast<size_t>(e) * F.bytes[a]);
      uint4* dst = reinterpret_cast<uint4*>(F.dst[a] + static_cast<size_t>(s) * F.bytes[a]);
      size_t i = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x;
      for (; i + 3 * stride < n16; i += 4 * stride) {
        uint4 v[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) v[u] = __ldcs(src + i + u * stride);
#pragma unroll
        for (int u = 0; u < 4; ++u) dst[i + u * stride] = v[u];
      }
      for (; i < n16; i += stride) dst[i] = __ldcs(src + i);
    }
  }
}

}  // namespace

cudaError_t launch_cache_select(const int32_t* offsets, int E, uint32_t* counts, int decay_shift, int S,
                                int32_t* expert_slot, int32_t* slot_expert, int32_t* promoted, uint32_t* dev_err,
                                cudaStream_t s) {
  return launch_pdl(cache_select_kernel, dim3(1), dim3(kSelThreads), 0, s, offsets, E, counts, decay_shift, S,
                    expert_slot, slot_expert, promoted, dev_err);
}

cudaError_t launch_stage_select(const int32_t* offsets, int E, const int32_t* res_slot, int R, int S,
                                int32_t* weight_slot, int32_t* staged, uint32_t* dev_err, cudaStream_t s) {
  return launch_pdl(stage_select_kernel, dim3(1), dim3(kSelThreads), 0, s, offsets, E, res_slot, R, S, weight_slot,
                    staged, dev_err);
}

cudaError_t launch_cache_fill(const int32_t* promoted, int S, int n, const void* const* src, void* const* dst,
                              const size_t* bytes, cudaStream_t s) {
  FillArgs F{};
  F.n = n;
  size_t most = 0;
  for (int a = 0; a < n; ++a) {
    F.src[a] = static_cast<const uint8_t*>(src[a]);
    F.dst[a] = static_cast<uint8_t*>(dst[a]);
    F.bytes[a] = bytes[a];
    if (bytes[a] > most) most = bytes[a];
  }
  if (const int nside = side_sms()) {  // the side SMs only, beside a persistent matmul
    const cudaError_t e = set_smem_limit(cache_fill_sm_kernel, kFillPinSmem);
    if (e != cudaSuccess) return e;
    return launch_pdl(cache_fill_sm_kernel, dim3(static_cast<unsigned>(nside)), dim3(kFillThreads), kFillPinSmem, s,
                      promoted, S, F);
  }
  // enough blocks per slot that one slot's copy spreads over the GPU when few
  // slots change (the usual case between decode steps)
  unsigned bx = static_cast<unsigned>((most / 16 + 255) / 256);
  const unsigned cap = static_cast<unsigned>(4 * device_info().sms);
  if (bx > cap) bx = cap;
  if (bx < 1) bx = 1;
  return launch_pdl(cache_fill_kernel, dim3(bx, static_cast<unsigned>(S)), dim3(256), 0, s, promoted, F);
}

}  // namespace moe
