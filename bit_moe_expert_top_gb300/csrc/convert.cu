// Weight-format kernels: the one-time 2-bit repack into the kernel layout,
// exact dequantisation exports, and the MXFP4 -> FP8 workspace conversion
// ("国产GPU完成MoE大模型Day-0适配" §四).  All elementwise and HBM-bound:
// consecutive threads own consecutive 32-element groups, so every load and
// store is a contiguous vector access.
#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"
#include "internal.cuh"

namespace moe {

namespace {

__global__ void w2_repack_kernel(const uint32_t* __restrict__ codes, const __half* __restrict__ scales,
                                 int64_t mats, int64_t R, int K, uint32_t* __restrict__ codes_k,
                                 uint16_t* __restrict__ scales_k) {
  const int64_t wpr = K / 16, gpr = K / 32;
  const int64_t nwords = mats * R * wpr, nsc = mats * R * gpr;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < nwords; i += stride) {
    const int64_t m = i / (R * wpr), rem = i % (R * wpr), row = rem / wpr, kw = rem % wpr;
    codes_k[m * R * wpr + w2l_word(row, R, K, kw)] = codes[i];
  }
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < nsc; i += stride) {
    const int64_t m = i / (R * gpr), rem = i % (R * gpr), row = rem / gpr, g = rem % gpr;
    scales_k[m * R * gpr + w2l_scale(row, R, K, g)] = f32_to_bf16_rne(__half2float(scales[i]));
  }
}

// Exact dequantised value entry * scale as bf16 bits, element j (0..15) of a
// canonical code word.
MOE_D uint16_t w2_value_bf16(uint32_t w, int j, uint32_t sb) {
  const uint32_t c = (w >> (2 * j)) & 3u;
  const float entry = (c == 0u) ? -4.f : (c == 1u) ? -1.f : (c == 2u) ? 1.f : 4.f;
  return f32_to_bf16_rne(entry * bf16_bits_to_f32(sb));
}

__global__ void dequant_w2_kernel(const uint32_t* __restrict__ codes_k, const uint16_t* __restrict__ scales_k,
                                  int64_t mats, int64_t R, int K, uint16_t* __restrict__ out) {
  const int64_t wpr = K / 16;
  const int64_t nwords = mats * R * wpr;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < nwords; i += stride) {
    const int64_t m = i / (R * wpr), rem = i % (R * wpr), row = rem / wpr, kw = rem % wpr;
    const uint32_t w = codes_k[m * R * wpr + w2l_word(row, R, K, kw)];
    const uint32_t sb = scales_k[m * R * (K / 32) + w2l_scale(row, R, K, kw / 2)];
    uint16_t* o = out + i * 16;
#pragma unroll
    for (int j = 0; j < 16; ++j) o[j] = w2_value_bf16(w, j, sb);
  }
}

__global__ void dequant_mxfp4_kernel(const uint8_t* __restrict__ e2m1, const uint8_t* __restrict__ e8m0,
                                     int64_t ngroups, float* __restrict__ out) {
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t gi = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; gi < ngroups; gi += stride) {
    const uint32_t b = e8m0[gi];
    const float sc = (b == 255u) ? __uint_as_float(0x7fc00000u) : exp2i(static_cast<int>(b) - 127);
    const uint4 v = reinterpret_cast<const uint4*>(e2m1)[gi];
    const uint32_t ws[4] = {v.x, v.y, v.z, v.w};
    float* o = out + gi * 32;
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float2 f = e2m1x2_to_f32x2((ws[i] >> (8 * j)) & 0xffu);
        o[i * 8 + j * 2] = f.x * sc;
        o[i * 8 + j * 2 + 1] = f.y * sc;
      }
  }
}

// One 32-element block: 16 bytes of E2M1 codes and their E8M0 scale byte b
// to 32 E4M3 bytes (scale folded in, RNE, saturating); a NaN scale (255)
// gives 0x7F bytes.  Returns whether the scale was NaN.
MOE_D bool e2m1_block_to_e4m3(uint4 v, uint32_t b, uint32_t* o) {
  if (b == 255u) {
#pragma unroll
    for (int k = 0; k < 8; ++k) o[k] = 0x7f7f7f7fu;
    return true;
  }
  const float sc = exp2i(static_cast<int>(b) - 127);
  const uint32_t wsw[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const float2 f0 = e2m1x2_to_f32x2(wsw[k] & 0xffu);
    const float2 f1 = e2m1x2_to_f32x2((wsw[k] >> 8) & 0xffu);
    const float2 f2 = e2m1x2_to_f32x2((wsw[k] >> 16) & 0xffu);
    const float2 f3 = e2m1x2_to_f32x2(wsw[k] >> 24);
    const uint32_t a0 = f32x2_to_e4m3x2(f0.x * sc, f0.y * sc);
    const uint32_t a1 = f32x2_to_e4m3x2(f1.x * sc, f1.y * sc);
    const uint32_t a2 = f32x2_to_e4m3x2(f2.x * sc, f2.y * sc);
    const uint32_t a3 = f32x2_to_e4m3x2(f3.x * sc, f3.y * sc);
    o[2 * k] = a0 | (a1 << 16);
    o[2 * k + 1] = a2 | (a3 << 16);
  }
  return false;
}

// Block i of the batch (expert experts[i / groups_per_mat]) -> its source
// block index and its workspace byte offset; false if the expert or its slot
// is out of range (the caller flags OVERFLOW and skips it).
MOE_D bool block_place(int64_t i, const int32_t* experts, const int32_t* ws_slots, int64_t groups_per_mat,
                       uint64_t ws_bytes, int64_t& sg, int64_t& dst) {
  const int xi = static_cast<int>(i / groups_per_mat);
  const int64_t gi = i - static_cast<int64_t>(xi) * groups_per_mat;
  const int64_t src = experts[xi];
  const int64_t slot = ws_slots[xi];
  const uint64_t end = static_cast<uint64_t>(slot + 1) * static_cast<uint64_t>(groups_per_mat) * 32u;
  if (slot < 0 || src < 0 || end > ws_bytes) return false;
  sg = src * groups_per_mat + gi;
  dst = (slot * groups_per_mat + gi) * 32;
  return true;
}

// One thread per 32-element block: 16 bytes of E2M1 + one E8M0 byte in,
// 32 E4M3 bytes out.
__global__ void mxfp4_to_fp8_kernel(const uint8_t* __restrict__ e2m1, const uint8_t* __restrict__ e8m0,
                                    const int32_t* __restrict__ experts, int n_experts, int64_t groups_per_mat,
                                    uint8_t* __restrict__ ws, uint64_t ws_bytes, const int32_t* __restrict__ ws_slots,
                                    uint32_t* dev_err) {
  const int64_t total = groups_per_mat * n_experts;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  bool nan_seen = false, overflow = false;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total; i += stride) {
    int64_t sg, dst;
    if (!block_place(i, experts, ws_slots, groups_per_mat, ws_bytes, sg, dst)) {
      overflow = true;
      continue;
    }
    uint32_t o[8];
    nan_seen |= e2m1_block_to_e4m3(reinterpret_cast<const uint4*>(e2m1)[sg], e8m0[sg], o);
    uint4* d = reinterpret_cast<uint4*>(ws + dst);
    d[0] = make_uint4(o[0], o[1], o[2], o[3]);
    d[1] = make_uint4(o[4], o[5], o[6], o[7]);
  }
  if (nan_seen) set_err(dev_err, MOE_DEVERR_NAN_SCALE);
  if (overflow) set_err(dev_err, MOE_DEVERR_OVERFLOW);
}

// The same conversion on the side SMs (moe_set_side_sms): one
// CTA of 1024 threads per reserved SM (its unused shared-memory request is
// over half an SM's, so no second CTA fits beside it), every thread with
// kConvU blocks' loads in flight, enough for one SM to pull its share of HBM
// while the persistent matmul holds the other SMs.
constexpr int kConvU = 4;
constexpr int kConvThreads = 1024;
constexpr int kConvPinSmem = 120 * 1024;

__global__ void __launch_bounds__(kConvThreads, 1)
    mxfp4_to_fp8_sm_kernel(const uint8_t* __restrict__ e2m1, const uint8_t* __restrict__ e8m0,
                           const int32_t* __restrict__ experts, int n_experts, int64_t groups_per_mat,
                           uint8_t* __restrict__ ws, uint64_t ws_bytes, const int32_t* __restrict__ ws_slots,
                           uint32_t* dev_err) {
  const int64_t total = groups_per_mat * n_experts;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  bool nan_seen = false, overflow = false;
  for (int64_t i0 = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i0 < total; i0 += kConvU * stride) {
    uint4 v[kConvU];
    uint32_t b[kConvU];
    int64_t dst[kConvU];
    bool ok[kConvU];
#pragma unroll
    for (int u = 0; u < kConvU; ++u) {
      const int64_t i = i0 + u * stride;
      int64_t sg = 0;
      ok[u] = i < total && block_place(i, experts, ws_slots, groups_per_mat, ws_bytes, sg, dst[u]);
      if (i < total && !ok[u]) overflow = true;
      if (ok[u]) {
        v[u] = __ldcs(reinterpret_cast<const uint4*>(e2m1) + sg);
        b[u] = e8m0[sg];
      }
    }
#pragma unroll
    for (int u = 0; u < kConvU; ++u) {
      if (!ok[u]) continue;
      uint32_t o[8];
      nan_seen |= e2m1_block_to_e4m3(v[u], b[u], o);
      uint4* d = reinterpret_cast<uint4*>(ws + dst[u]);
      d[0] = make_uint4(o[0], o[1], o[2], o[3]);
      d[1] = make_uint4(o[4], o[5], o[6], o[7]);
    }
  }
  if (nan_seen) set_err(dev_err, MOE_DEVERR_NAN_SCALE);
  if (overflow) set_err(dev_err, MOE_DEVERR_OVERFLOW);
}

int grid_for(int64_t work, int threads) {
  const int64_t want = (work + threads - 1) / threads;
  const int64_t cap = static_cast<int64_t>(device_info().sms) * 16;
  return static_cast<int>(want < 1 ? 1 : (want > cap ? cap : want));
}

}  // namespace

cudaError_t launch_w2_repack(const uint8_t* codes, const uint16_t* scales, int64_t mats, int64_t R, int K,
                             uint8_t* codes_k, uint16_t* scales_k, cudaStream_t s) {
  const int64_t nwords = mats * R * (K / 16);
  if (nwords == 0) return cudaSuccess;
  w2_repack_kernel<<<grid_for(nwords, 256), 256, 0, s>>>(reinterpret_cast<const uint32_t*>(codes),
                                                         reinterpret_cast<const __half*>(scales), mats, R, K,
                                                         reinterpret_cast<uint32_t*>(codes_k), scales_k);
  return cudaGetLastError();
}

cudaError_t launch_dequant_w2(const uint8_t* codes_k, const uint16_t* scales_k, int64_t mats, int64_t R, int K,
                              uint16_t* out, cudaStream_t s) {
  const int64_t nw = mats * R * (K / 16);
  if (nw == 0) return cudaSuccess;
  dequant_w2_kernel<<<grid_for(nw, 256), 256, 0, s>>>(reinterpret_cast<const uint32_t*>(codes_k), scales_k, mats,
                                                      R, K, out);
  return cudaGetLastError();
}

cudaError_t launch_dequant_mxfp4(const uint8_t* e2m1, const uint8_t* e8m0, int64_t rows, int K, float* out,
                                 cudaStream_t s) {
  const int64_t ng = rows * (K / 32);
  if (ng == 0) return cudaSuccess;
  dequant_mxfp4_kernel<<<grid_for(ng, 256), 256, 0, s>>>(e2m1, e8m0, ng, out);
  return cudaGetLastError();
}

cudaError_t launch_mxfp4_to_fp8(const uint8_t* e2m1, const uint8_t* e8m0, const int32_t* experts, int n_experts,
                                int rows, int K, uint8_t* ws, size_t ws_bytes, const int32_t* ws_slots,
                                uint32_t* dev_err, cudaStream_t s) {
  const int64_t gpm = static_cast<int64_t>(rows) * (K / 32);
  const int64_t work = gpm * n_experts;
  if (work == 0) return cudaSuccess;
  if (const int n = side_sms()) {  // the reserved SMs only, beside a persistent matmul
    const cudaError_t e = set_smem_limit(mxfp4_to_fp8_sm_kernel, kConvPinSmem);
    if (e != cudaSuccess) return e;
    mxfp4_to_fp8_sm_kernel<<<n, kConvThreads, kConvPinSmem, s>>>(e2m1, e8m0, experts, n_experts, gpm, ws,
                                                                 static_cast<uint64_t>(ws_bytes), ws_slots, dev_err);
    return cudaGetLastError();
  }
  mxfp4_to_fp8_kernel<<<grid_for(work, 256), 256, 0, s>>>(e2m1, e8m0, experts, n_experts, gpm, ws,
                                                          static_cast<uint64_t>(ws_bytes), ws_slots, dev_err);
  return cudaGetLastError();
}

}  // namespace moe
