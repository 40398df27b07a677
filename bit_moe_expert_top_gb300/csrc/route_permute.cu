// Routing, grouping, activation gather (bf16 / MXFP8) and the weighted
// combine.  All HBM-bound or latency-bound; deterministic, no global atomics
// on data (only the error word).
#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"
#include "internal.cuh"
#include "route_common.cuh"

namespace moe {

// ------------------------------------------------------------------ routing
// One warp per token (route_token).
template <int NPL>
__global__ void __launch_bounds__(256) route_kernel(const float* __restrict__ logits, int T, int E, int k,
                                                    int32_t* __restrict__ ids, float* __restrict__ w,
                                                    uint32_t* dev_err) {
  pdl_wait();
  pdl_trigger();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = blockIdx.x * 8 + warp;
  if (t >= T) return;
  int id;
  float wt;
  if (route_token<NPL>(logits + static_cast<size_t>(t) * E, E, k, lane, id, wt) && lane == 0)
    set_err(dev_err, MOE_DEVERR_NAN_LOGIT);
  if (lane < k) {
    ids[static_cast<size_t>(t) * k + lane] = id;
    w[static_cast<size_t>(t) * k + lane] = wt;
  }
}

cudaError_t launch_route(const float* logits, int T, int E, int k, int32_t* ids, float* w, uint32_t* dev_err,
                         cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  const dim3 grid((T + 7) / 8), block(256);
  if (E <= 128) return launch_pdl(route_kernel<4>, grid, block, 0, s, logits, T, E, k, ids, w, dev_err);
  if (E <= 256) return launch_pdl(route_kernel<8>, grid, block, 0, s, logits, T, E, k, ids, w, dev_err);
  if (E <= 512) return launch_pdl(route_kernel<16>, grid, block, 0, s, logits, T, E, k, ids, w, dev_err);
  return launch_pdl(route_kernel<32>, grid, block, 0, s, logits, T, E, k, ids, w, dev_err);
}

// ------------------------------------------------------------------ grouping
// Single CTA of 32 warps.  Warp w owns a contiguous chunk of assignments and
// keeps its own per-expert count (hist[w][e]); a warp-level match_any turns a
// tile of 32 ids into groups whose leader updates the count, so each count
// has one writer.  Exclusive scans over warps and experts give every warp the
// first output row of each of its groups; the second walk writes perm/inv in
// increasing assignment order within each expert (stable).
constexpr int kPermWarps = 32;
constexpr int kPermU = 8;  // 32-id tiles whose loads a warp keeps in flight

__global__ void __launch_bounds__(1024) permute_kernel(const int32_t* __restrict__ ids, int A, int E,
                                                       int32_t* __restrict__ offsets, int32_t* __restrict__ perm,
                                                       int32_t* __restrict__ inv, uint32_t* dev_err) {
  extern __shared__ int s_perm[];
  int* hist = s_perm;                    // [32][E]
  int* tot = s_perm + kPermWarps * E;    // [E]
  __shared__ int warp_sums[32];
  pdl_wait();
  pdl_trigger();
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const unsigned lt_mask = (1u << lane) - 1u;
  int chunk = (A + kPermWarps - 1) / kPermWarps;
  chunk = (chunk + 31) & ~31;
  const int nw = chunk > 0 ? (A + chunk - 1) / chunk : 0;  // warps with a non-empty chunk
  const int beg = warp * chunk;
  const int end = min(A, beg + chunk);

  for (int i = tid; i < nw * E; i += blockDim.x) hist[i] = 0;
  __syncthreads();

  // the warp walks its chunk in tiles of 32 ids, kPermU tiles' loads in flight at once
  bool bad = false;
  for (int base0 = beg; base0 < end; base0 += 32 * kPermU) {
    int ev[kPermU];
#pragma unroll
    for (int u = 0; u < kPermU; ++u) {
      const int a = base0 + 32 * u + lane;
      ev[u] = (a < end) ? ids[a] : -1;
    }
#pragma unroll
    for (int u = 0; u < kPermU; ++u) {
      if (base0 + 32 * u >= end) break;  // warp-uniform: past the chunk
      const int a = base0 + 32 * u + lane;
      int e = ev[u];
      if (a < end && (e < 0 || e >= E)) {
        bad = true;
        e = -1;
      }
      const int key = (e >= 0) ? e : (E + lane);  // invalid lanes form singleton groups
      const unsigned m = __match_any_sync(0xffffffffu, key);
      if (e >= 0 && (m & lt_mask) == 0) hist[warp * E + e] += __popc(m);
      __syncwarp();
    }
  }
  if (bad) set_err(dev_err, MOE_DEVERR_BAD_ID);
  __syncthreads();

  // per-expert exclusive scan over warps; totals
  for (int e = tid; e < E; e += blockDim.x) {
    int run = 0;
    for (int w = 0; w < nw; ++w) {
      const int c = hist[w * E + e];
      hist[w * E + e] = run;
      run += c;
    }
    tot[e] = run;
  }
  __syncthreads();

  // exclusive scan of tot over experts (E <= 1024: one element per thread)
  int v = (tid < E) ? tot[tid] : 0;
  int incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int n = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += n;
  }
  if (lane == 31) warp_sums[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int ws = warp_sums[lane];
    int wi = ws;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int n = __shfl_up_sync(0xffffffffu, wi, o);
      if (lane >= o) wi += n;
    }
    warp_sums[lane] = wi - ws;  // exclusive
  }
  __syncthreads();
  const int excl = incl - v + warp_sums[warp];
  if (tid < E) {
    offsets[tid] = excl;
    tot[tid] = excl;
    if (tid == E - 1) offsets[E] = excl + v;
  }
  __syncthreads();
  for (int i = tid; i < nw * E; i += blockDim.x) hist[i] += tot[i % E];
  __syncthreads();

  for (int base0 = beg; base0 < end; base0 += 32 * kPermU) {
    int ev[kPermU];
#pragma unroll
    for (int u = 0; u < kPermU; ++u) {
      const int a = base0 + 32 * u + lane;
      ev[u] = (a < end) ? ids[a] : -1;
    }
#pragma unroll
    for (int u = 0; u < kPermU; ++u) {
      if (base0 + 32 * u >= end) break;  // warp-uniform: past the chunk
      const int a = base0 + 32 * u + lane;
      int e = ev[u];
      if (a < end && (e < 0 || e >= E)) e = -1;
      const int key = (e >= 0) ? e : (E + lane);
      const unsigned m = __match_any_sync(0xffffffffu, key);
      int pos = -1;
      if (e >= 0) pos = hist[warp * E + e] + __popc(m & lt_mask);
      __syncwarp();
      if (e >= 0 && (m & lt_mask) == 0) hist[warp * E + e] += __popc(m);
      __syncwarp();
      if (a < end) {
        inv[a] = pos;
        if (pos >= 0) perm[pos] = a;
      }
    }
  }
}

// Multi-CTA grouping for large A (prefill): block b owns the contiguous
// assignments [b*CB, (b+1)*CB).  permute_count: per-block expert counts
// (each warp counts its 32-id tiles as above, the block adds its warps);
// permute_scan (one CTA): per expert, the exclusive prefix over blocks plus
// the expert's group start; permute_place: each block recounts per warp,
// takes its warps' exclusive prefix on top of the block's base and writes
// perm/inv in increasing assignment order within each expert (stable, the
// same result as the single-CTA kernel).
constexpr int kPermCB = 4096;  // assignments per block

// per-warp counts of the warp's slice [beg, end) into h (this warp's row)
MOE_D bool perm_count_warp(const int32_t* __restrict__ ids, int beg, int end, int E, int* h, int lane) {
  const unsigned lt_mask = (1u << lane) - 1u;
  bool bad = false;
  for (int base0 = beg; base0 < end; base0 += 32 * kPermU) {
    int ev[kPermU];
#pragma unroll
    for (int u = 0; u < kPermU; ++u) {
      const int a = base0 + 32 * u + lane;
      ev[u] = (a < end) ? ids[a] : -1;
    }
#pragma unroll
    for (int u = 0; u < kPermU; ++u) {
      if (base0 + 32 * u >= end) break;  // warp-uniform
      const int a = base0 + 32 * u + lane;
      int e = ev[u];
      if (a < end && (e < 0 || e >= E)) {
        bad = true;
        e = -1;
      }
      const int key = (e >= 0) ? e : (E + lane);
      const unsigned m = __match_any_sync(0xffffffffu, key);
      if (e >= 0 && (m & lt_mask) == 0) h[e] += __popc(m);
      __syncwarp();
    }
  }
  return bad;
}

// positions of the warp's slice from the running bases in h (this warp's row)
MOE_D void perm_place_warp(const int32_t* __restrict__ ids, int beg, int end, int E, int* h, int lane,
                           int32_t* __restrict__ perm, int32_t* __restrict__ inv) {
  const unsigned lt_mask = (1u << lane) - 1u;
  for (int base0 = beg; base0 < end; base0 += 32 * kPermU) {
    int ev[kPermU];
#pragma unroll
    for (int u = 0; u < kPermU; ++u) {
      const int a = base0 + 32 * u + lane;
      ev[u] = (a < end) ? ids[a] : -1;
    }
#pragma unroll
    for (int u = 0; u < kPermU; ++u) {
      if (base0 + 32 * u >= end) break;
      const int a = base0 + 32 * u + lane;
      int e = ev[u];
      if (a < end && (e < 0 || e >= E)) e = -1;
      const int key = (e >= 0) ? e : (E + lane);
      const unsigned m = __match_any_sync(0xffffffffu, key);
      int pos = -1;
      if (e >= 0) pos = h[e] + __popc(m & lt_mask);
      __syncwarp();
      if (e >= 0 && (m & lt_mask) == 0) h[e] += __popc(m);
      __syncwarp();
      if (a < end) {
        inv[a] = pos;
        if (pos >= 0) perm[pos] = a;
      }
    }
  }
}

__global__ void __launch_bounds__(1024) permute_count_kernel(const int32_t* __restrict__ ids, int A, int E,
                                                             int32_t* __restrict__ blk, uint32_t* dev_err) {
  extern __shared__ int s_perm[];  // [32][E]
  pdl_wait();
  pdl_trigger();
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int b0 = blockIdx.x * kPermCB, b1 = min(A, b0 + kPermCB);
  const int wc = kPermCB / kPermWarps;
  for (int i = tid; i < kPermWarps * E; i += blockDim.x) s_perm[i] = 0;
  __syncthreads();
  const bool bad = perm_count_warp(ids, b0 + warp * wc, min(b1, b0 + (warp + 1) * wc), E, s_perm + warp * E, lane);
  if (bad) set_err(dev_err, MOE_DEVERR_BAD_ID);
  __syncthreads();
  for (int e = tid; e < E; e += blockDim.x) {
    int c = 0;
    for (int w = 0; w < kPermWarps; ++w) c += s_perm[w * E + e];
    blk[static_cast<size_t>(blockIdx.x) * E + e] = c;
  }
}

__global__ void __launch_bounds__(1024) permute_scan_kernel(int32_t* __restrict__ blk, int nb, int E,
                                                            int32_t* __restrict__ offsets) {
  __shared__ int warp_sums[32];
  pdl_wait();
  pdl_trigger();
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  int run = 0;
  if (tid < E)
    for (int b = 0; b < nb; ++b) {
      const int c = blk[static_cast<size_t>(b) * E + tid];
      blk[static_cast<size_t>(b) * E + tid] = run;
      run += c;
    }
  const int v = tid < E ? run : 0;
  int incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int n = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += n;
  }
  if (lane == 31) warp_sums[warp] = incl;
  __syncthreads();
  int before = 0;
  for (int w = 0; w < warp; ++w) before += warp_sums[w];
  const int excl = before + incl - v;
  if (tid < E) {
    offsets[tid] = excl;
    if (tid == E - 1) offsets[E] = excl + v;
    for (int b = 0; b < nb; ++b) blk[static_cast<size_t>(b) * E + tid] += excl;
  }
}

__global__ void __launch_bounds__(1024) permute_place_kernel(const int32_t* __restrict__ ids, int A, int E,
                                                             const int32_t* __restrict__ blk,
                                                             int32_t* __restrict__ perm, int32_t* __restrict__ inv) {
  extern __shared__ int s_perm[];  // [32][E]
  pdl_wait();
  pdl_trigger();
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int b0 = blockIdx.x * kPermCB, b1 = min(A, b0 + kPermCB);
  const int wc = kPermCB / kPermWarps;
  const int beg = b0 + warp * wc, end = min(b1, b0 + (warp + 1) * wc);
  for (int i = tid; i < kPermWarps * E; i += blockDim.x) s_perm[i] = 0;
  __syncthreads();
  perm_count_warp(ids, beg, end, E, s_perm + warp * E, lane);
  __syncthreads();
  // per expert: exclusive prefix over the block's warps on top of the block's base
  for (int e = tid; e < E; e += blockDim.x) {
    int run = blk[static_cast<size_t>(blockIdx.x) * E + e];
    for (int w = 0; w < kPermWarps; ++w) {
      const int c = s_perm[w * E + e];
      s_perm[w * E + e] = run;
      run += c;
    }
  }
  __syncthreads();
  perm_place_warp(ids, beg, end, E, s_perm + warp * E, lane, perm, inv);
}

size_t permute_workspace_bytes(int A, int E) {
  if (A < 2 * kPermCB) return 0;  // one CTA does it
  const size_t nb = (static_cast<size_t>(A) + kPermCB - 1) / kPermCB;
  return nb * static_cast<size_t>(E) * sizeof(int32_t);
}

cudaError_t launch_permute(const int32_t* ids, int T, int k, int E, int32_t* offsets, int32_t* perm, int32_t* inv,
                           void* ws, size_t ws_bytes, uint32_t* dev_err, cudaStream_t s) {
  const int A = T * k;
  const size_t need = permute_workspace_bytes(A, E);
  if (need > 0 && ws != nullptr && ws_bytes >= need) {
    const int nb = (A + kPermCB - 1) / kPermCB;
    const size_t smem = static_cast<size_t>(kPermWarps) * E * sizeof(int);
    int32_t* blk = static_cast<int32_t*>(ws);
    cudaError_t e = set_smem_limit(permute_count_kernel, static_cast<int>(kPermWarps * 1024 * sizeof(int)));
    if (e == cudaSuccess) e = set_smem_limit(permute_place_kernel, static_cast<int>(kPermWarps * 1024 * sizeof(int)));
    if (e == cudaSuccess) e = launch_pdl(permute_count_kernel, dim3(nb), dim3(1024), smem, s, ids, A, E, blk, dev_err);
    if (e == cudaSuccess) e = launch_pdl(permute_scan_kernel, dim3(1), dim3(1024), 0, s, blk, nb, E, offsets);
    if (e == cudaSuccess)
      e = launch_pdl(permute_place_kernel, dim3(nb), dim3(1024), smem, s, ids, A, E,
                     static_cast<const int32_t*>(blk), perm, inv);
    return e;
  }
  const size_t smem = static_cast<size_t>(kPermWarps + 1) * E * sizeof(int);
  cudaError_t e = set_smem_limit(permute_kernel, static_cast<int>((kPermWarps + 1) * 1024 * sizeof(int)));
  if (e != cudaSuccess) return e;
  return launch_pdl(permute_kernel, dim3(1), dim3(1024), smem, s, ids, A, E, offsets, perm, inv, dev_err);
}

// ------------------------------------------------------------------ gather
// Token-major: a warp takes one (token, 1024-element chunk) unit, reads the
// token's activations once and writes them to the k permuted rows of that
// token (inv of its k assignments), so each token row is read from HBM once
// and, for MXFP8, quantised once.
__global__ void scatter_bf16_kernel(const uint16_t* __restrict__ x, const int32_t* __restrict__ inv, int T, int k,
                                    int H, uint16_t* __restrict__ xp) {
  pdl_wait();
  pdl_trigger();
  const int lane = threadIdx.x & 31;
  const int nch = (H + 1023) / 1024;
  const int64_t units = static_cast<int64_t>(T) * nch;
  for (int64_t u0 = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5); u0 < units;
       u0 += static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5)) {
    const int t = static_cast<int>(u0 / nch), base0 = static_cast<int>(u0 - static_cast<int64_t>(t) * nch) * 1024;
    const uint16_t* src = x + static_cast<size_t>(t) * H;
    uint4 raw[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int e0 = base0 + 256 * u + lane * 8;
      if (e0 < H) raw[u] = __ldg(reinterpret_cast<const uint4*>(src + e0));
    }
    for (int j = 0; j < k; ++j) {
      const int p = inv[static_cast<size_t>(t) * k + j];
      if (p < 0) continue;
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int e0 = base0 + 256 * u + lane * 8;
        if (e0 < H) *reinterpret_cast<uint4*>(xp + static_cast<size_t>(p) * H + e0) = raw[u];
      }
    }
  }
}

// MXFP8 quantisation fused into the gather: each lane takes 8 consecutive
// elements, 4 lanes form one block of 32 (block max by two shuffles).
// AS_BF16: write each element's MXFP8 value q * 2^X as bf16 instead of q + X.
template <bool AS_BF16>
__global__ void scatter_mxfp8_kernel(const uint16_t* __restrict__ x, const int32_t* __restrict__ inv, int T, int k,
                                     int H, uint8_t* __restrict__ q, uint8_t* __restrict__ sc) {
  pdl_wait();
  pdl_trigger();
  const int lane = threadIdx.x & 31;
  const int nch = (H + 1023) / 1024;
  const int64_t units = static_cast<int64_t>(T) * nch;
  for (int64_t u0 = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5); u0 < units;
       u0 += static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5)) {
    const int t = static_cast<int>(u0 / nch), base0 = static_cast<int>(u0 - static_cast<int64_t>(t) * nch) * 1024;
    const uint16_t* src = x + static_cast<size_t>(t) * H;
    uint4 raw[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int e0 = base0 + 256 * u + lane * 8;
      if (e0 < H) raw[u] = __ldg(reinterpret_cast<const uint4*>(src + e0));
    }
    // quantise the chunk once: per lane 4 x 8 elements -> 4 x (8 codes, or 8 bf16 values) + the block scales
    uint2 codes[4];
    uint4 vals[4];
    uint32_t xs[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int e0 = base0 + 256 * u + lane * 8;
      const bool ok = e0 < H;
      float f[8];
      float amax = 0.f;
      const uint32_t wv[4] = {raw[u].x, raw[u].y, raw[u].z, raw[u].w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        f[2 * i] = ok ? __uint_as_float(wv[i] << 16) : 0.f;
        f[2 * i + 1] = ok ? __uint_as_float(wv[i] & 0xffff0000u) : 0.f;
        amax = fmaxf(amax, fmaxf(fabsf(f[2 * i]), fabsf(f[2 * i + 1])));
      }
      amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
      amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
      const int X = mx_scale_exp(amax);
      const float iv = exp2i(-X);
      uint32_t packed[2];
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        uint32_t lo = f32x2_to_e4m3x2(f[4 * i] * iv, f[4 * i + 1] * iv);
        uint32_t hi = f32x2_to_e4m3x2(f[4 * i + 2] * iv, f[4 * i + 3] * iv);
        packed[i] = lo | (hi << 16);
      }
      codes[u] = make_uint2(packed[0], packed[1]);
      xs[u] = static_cast<uint32_t>(X + 127);
      if (AS_BF16) {
        const float sc2 = exp2i(X);
        uint32_t o[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float2 v = e4m3x2_to_f32x2(static_cast<uint16_t>(packed[i >> 1] >> (16 * (i & 1))));
          asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(o[i]) : "f"(v.y * sc2), "f"(v.x * sc2));
        }
        vals[u] = make_uint4(o[0], o[1], o[2], o[3]);
      }
    }
    for (int j = 0; j < k; ++j) {
      const int p = inv[static_cast<size_t>(t) * k + j];
      if (p < 0) continue;
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int e0 = base0 + 256 * u + lane * 8;
        if (e0 >= H) continue;
        if (AS_BF16) {
          *reinterpret_cast<uint4*>(reinterpret_cast<uint16_t*>(q) + static_cast<size_t>(p) * H + e0) = vals[u];
        } else {
          *reinterpret_cast<uint2*>(q + static_cast<size_t>(p) * H + e0) = codes[u];
          if ((lane & 3) == 0) sc[static_cast<size_t>(p) * (H / 32) + e0 / 32] = static_cast<uint8_t>(xs[u]);
        }
      }
    }
  }
}

cudaError_t launch_gather(const uint16_t* x, const int32_t* inv, int T, int k, int H, int act_fmt, void* x_perm,
                          uint8_t* x_perm_scale, cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  const int64_t units = static_cast<int64_t>(T) * ((H + 1023) / 1024);
  const int64_t cap = static_cast<int64_t>(device_info().sms) * 8;
  const int blocks = static_cast<int>((units + 7) / 8 < cap ? (units + 7) / 8 : cap);
  if (act_fmt == MOE_FMT_BF16)
    return launch_pdl(scatter_bf16_kernel, dim3(blocks), dim3(256), 0, s, x, inv, T, k, H,
                      static_cast<uint16_t*>(x_perm));
  if (act_fmt == MOE_FMT_MXFP8_BF16)
    return launch_pdl(scatter_mxfp8_kernel<true>, dim3(blocks), dim3(256), 0, s, x, inv, T, k, H,
                      static_cast<uint8_t*>(x_perm), static_cast<uint8_t*>(nullptr));
  return launch_pdl(scatter_mxfp8_kernel<false>, dim3(blocks), dim3(256), 0, s, x, inv, T, k, H,
                    static_cast<uint8_t*>(x_perm), x_perm_scale);
}

__global__ void unpermute_kernel(const uint8_t* __restrict__ src, const int32_t* __restrict__ inv, int A,
                                 int row_bytes, uint8_t* __restrict__ dst) {
  const int lane = threadIdx.x & 31;
  for (int a = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); a < A; a += gridDim.x * (blockDim.x >> 5)) {
    const int p = inv[a];
    if (p < 0) continue;
    const uint4* s4 = reinterpret_cast<const uint4*>(src + static_cast<size_t>(p) * row_bytes);
    uint4* d4 = reinterpret_cast<uint4*>(dst + static_cast<size_t>(a) * row_bytes);
    for (int i = lane; i < row_bytes / 16; i += 32) d4[i] = s4[i];
  }
}

cudaError_t launch_unpermute(const void* rows_perm, int fmt, const int32_t* inv, int A, int cols, void* rows,
                             cudaStream_t s) {
  if (A == 0) return cudaSuccess;
  const int row_bytes = cols * (fmt == MOE_FMT_F32 ? 4 : 2);
  const int blocks = min((A + 7) / 8, device_info().sms * 8);
  unpermute_kernel<<<blocks, 256, 0, s>>>(static_cast<const uint8_t*>(rows_perm), inv, A, row_bytes,
                                          static_cast<uint8_t*>(rows));
  return cudaGetLastError();
}

// ------------------------------------------------------------------ combine
// Grid (column blocks of 2048, tokens): thread i of block (cb, t) owns
// columns cb*2048 + 8i .. +7 of token t and accumulates the k rows of its
// token in ascending slot order; loads of four slots are issued together.
template <bool kYF32>
MOE_D void load8(const void* y, size_t off, float (&v)[8]) {
  if (kYF32) {
    const float4* src = reinterpret_cast<const float4*>(static_cast<const float*>(y) + off);
    const float4 a = __ldg(src), b = __ldg(src + 1);
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
    v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
  } else {
    const uint4 a = __ldg(reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(y) + off));
    const uint32_t wv[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      v[2 * i] = __uint_as_float(wv[i] << 16);
      v[2 * i + 1] = __uint_as_float(wv[i] & 0xffff0000u);
    }
  }
}

template <bool kYF32, bool kOutF32>
__global__ void __launch_bounds__(128) combine_kernel(const void* __restrict__ y, const float* __restrict__ w,
                                                      const int32_t* __restrict__ inv, int T, int k, int H,
                                                      void* __restrict__ out) {
  pdl_wait();
  pdl_trigger();
  const int t = blockIdx.y;
  const int c0 = blockIdx.x * 1024 + threadIdx.x * 8;
  if (t >= T || c0 >= H) return;
  float acc[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) acc[i] = 0.f;
  const int32_t* iv = inv + static_cast<size_t>(t) * k;
  const float* wt = w + static_cast<size_t>(t) * k;
  int j = 0;
  for (; j + 8 <= k; j += 8) {  // all eight slots' rows in flight at once, summed in slot order
    int p[8];
    float wj[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      p[u] = iv[j + u];
      wj[u] = wt[j + u];
    }
    if (!kYF32) {  // bf16 rows stay packed until used: 4 registers per row in flight instead of 8
      uint4 raw[8];
#pragma unroll
      for (int u = 0; u < 8; ++u)
        if (p[u] >= 0)
          raw[u] = __ldg(reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(y) +
                                                        static_cast<size_t>(p[u]) * H + c0));
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        if (p[u] < 0) continue;
        const uint32_t wv[4] = {raw[u].x, raw[u].y, raw[u].z, raw[u].w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          acc[2 * i] = fmaf(wj[u], __uint_as_float(wv[i] << 16), acc[2 * i]);
          acc[2 * i + 1] = fmaf(wj[u], __uint_as_float(wv[i] & 0xffff0000u), acc[2 * i + 1]);
        }
      }
    } else {
      float v[8][8];
#pragma unroll
      for (int u = 0; u < 8; ++u)
        if (p[u] >= 0) load8<kYF32>(y, static_cast<size_t>(p[u]) * H + c0, v[u]);
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        if (p[u] < 0) continue;
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[i] = fmaf(wj[u], v[u][i], acc[i]);
      }
    }
  }
  for (; j + 4 <= k; j += 4) {
    float v[4][8];
    int p[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      p[u] = iv[j + u];
      if (p[u] >= 0) load8<kYF32>(y, static_cast<size_t>(p[u]) * H + c0, v[u]);
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      if (p[u] < 0) continue;
      const float wj = wt[j + u];
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[i] = fmaf(wj, v[u][i], acc[i]);
    }
  }
  for (; j < k; ++j) {
    const int p = iv[j];
    if (p < 0) continue;
    float v[8];
    load8<kYF32>(y, static_cast<size_t>(p) * H + c0, v);
    const float wj = wt[j];
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] = fmaf(wj, v[i], acc[i]);
  }
  if (kOutF32) {
    float4* dst = reinterpret_cast<float4*>(static_cast<float*>(out) + static_cast<size_t>(t) * H + c0);
    dst[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
    dst[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
  } else {
    uint32_t o[4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
      o[i] = static_cast<uint32_t>(f32_to_bf16_rne(acc[2 * i])) |
             (static_cast<uint32_t>(f32_to_bf16_rne(acc[2 * i + 1])) << 16);
    *reinterpret_cast<uint4*>(static_cast<uint16_t*>(out) + static_cast<size_t>(t) * H + c0) =
        make_uint4(o[0], o[1], o[2], o[3]);
  }
}

cudaError_t launch_combine(const void* y, int y_fmt, const float* w, const int32_t* inv, int T, int k, int H,
                           void* out, int out_fmt, cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  const dim3 grid((H + 1023) / 1024, T);  // 128 threads x 8 outputs per block
  const bool yf = y_fmt == MOE_FMT_F32, of = out_fmt == MOE_FMT_F32;
  if (yf && of) return launch_pdl(combine_kernel<true, true>, grid, dim3(128), 0, s, y, w, inv, T, k, H, out);
  if (yf) return launch_pdl(combine_kernel<true, false>, grid, dim3(128), 0, s, y, w, inv, T, k, H, out);
  if (of) return launch_pdl(combine_kernel<false, true>, grid, dim3(128), 0, s, y, w, inv, T, k, H, out);
  return launch_pdl(combine_kernel<false, false>, grid, dim3(128), 0, s, y, w, inv, T, k, H, out);
}

}  // namespace moe
