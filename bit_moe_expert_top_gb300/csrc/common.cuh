// Shared device helpers for libmoe (sm_103a).  Hand-written PTX for the
// mbarrier / bulk-copy plumbing; no third-party headers.
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/moe.h"

#define MOE_HD __host__ __device__ __forceinline__
#define MOE_D __device__ __forceinline__

namespace moe {

// A bounded wait gives up after a limit of SM clock cycles and the waiter
// then reports MOE_DEVERR_TIMEOUT instead of hanging the GPU.  The limit is a
// kernel parameter (moe_set_wait_limit); this is its default (~1.5 s).
constexpr long long kWaitCycles = 3000000000LL;

MOE_D uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

MOE_D void set_err(uint32_t* dev_err, uint32_t bits) {
  if (dev_err) atomicOr(dev_err, bits);
}

// ---------------------------------------------------------------- mbarrier
MOE_D void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}
MOE_D void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
MOE_D void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}
MOE_D void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
MOE_D bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// Bounded wait for the phase with the given parity to complete.  Returns
// false if it did not complete within `limit` SM clock cycles.
MOE_D bool mbar_wait(uint64_t* bar, uint32_t parity, long long limit) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity)) {
    if (clock64() - t0 > limit) return false;
  }
  return true;
}

// ---------------------------------------------------------------- bulk copy
// 1-D bulk async copy global -> shared, completion counted on `bar` in bytes.
// dst/src 16-byte aligned, bytes a multiple of 16.
MOE_D void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// Bulk prefetch of [src, src + bytes) into L2 (16-byte aligned address and
// size); no completion to wait for and no scoreboard held.
MOE_D void prefetch_l2(const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

// Programmatic dependent launch: wait until the preceding grid in the stream
// has completed and its memory is visible (a no-op when the kernel was not
// launched as a dependent), then let the next grid be scheduled.  Kernels call
// pdl_wait() before their first global-memory access.
MOE_D void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
MOE_D void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

MOE_D void named_bar_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// Named barrier over `nthreads` threads that also ORs a flag across them, so
// every participant takes the same decision (e.g. to abort after a timeout).
MOE_D bool named_bar_or(int id, int nthreads, bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 q, %1, 0;\n\t"
      "barrier.cta.red.or.pred p, %2, %3, q;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(r)
      : "r"(static_cast<uint32_t>(v)), "r"(id), "r"(nthreads)
      : "memory");
  return r != 0;
}

// ---------------------------------------------------------------- numerics
MOE_D float bf16_bits_to_f32(uint32_t b16) { return __uint_as_float(b16 << 16); }

// Round-to-nearest-even of an fp32 value to bf16 (NaN kept quiet).
MOE_D uint16_t f32_to_bf16_rne(float f) {
  uint32_t u = __float_as_uint(f);
  if ((u & 0x7fffffffu) > 0x7f800000u) return static_cast<uint16_t>((u >> 16) | 0x40u);
  u += 0x7fffu + ((u >> 16) & 1u);
  return static_cast<uint16_t>(u >> 16);
}

MOE_D float silu_f32(float g) { return g / (1.0f + expf(-g)); }

// Packed fp32x2 FMA (one instruction on sm_100-family): d = a*b + c per lane.
MOE_D float2 ffma2(float2 a, float2 b, float2 c) {
  unsigned long long ra = *reinterpret_cast<unsigned long long*>(&a);
  unsigned long long rb = *reinterpret_cast<unsigned long long*>(&b);
  unsigned long long rc = *reinterpret_cast<unsigned long long*>(&c);
  unsigned long long rd;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(rd) : "l"(ra), "l"(rb), "l"(rc));
  return *reinterpret_cast<float2*>(&rd);
}

// Two E4M3 bytes (lo = element 0) -> two exact fp32 values.
MOE_D float2 e4m3x2_to_f32x2(uint16_t v) {
  uint32_t h2;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(v));
  __half2 h = *reinterpret_cast<__half2*>(&h2);
  return __half22float2(h);
}

// One byte of two E2M1 nibbles (lo nibble = element 0) -> two exact fp32 values.
MOE_D float2 e2m1x2_to_f32x2(uint32_t byte) {
  uint32_t h2;
  asm("{\n\t.reg .b8 t;\n\tcvt.u8.u32 t, %1;\n\tcvt.rn.f16x2.e2m1x2 %0, t;\n\t}" : "=r"(h2) : "r"(byte));
  __half2 h = *reinterpret_cast<__half2*>(&h2);
  return __half22float2(h);
}

// fp32 pair -> two E4M3 bytes (RNE, saturating to +-448; NaN -> 0x7F), lo byte = a.
MOE_D uint16_t f32x2_to_e4m3x2(float a, float b) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(b), "f"(a));
  return r;
}

// 2^e for e in [-126, 127] exactly, and for e = -127 the subnormal 2^-127.
MOE_D float exp2i(int e) {
  if (e >= -126) return __uint_as_float(static_cast<uint32_t>(e + 127) << 23);
  return __uint_as_float(0x00400000u);  // 2^-127
}

// OCP MX block scale exponent for a block maximum (floor(log2 amax) - 8,
// clamped to [-127, 127]; amax == 0 -> -127), read from the exponent bits.
MOE_D int mx_scale_exp(float amax) {
  uint32_t u = __float_as_uint(amax);
  int be = static_cast<int>((u >> 23) & 0xff);
  int fl;
  if (amax == 0.0f) return -127;
  if (be == 0) {  // subnormal: floor(log2) from the leading mantissa bit
    fl = -127 - (__clz(u & 0x7fffff) - 9);
  } else {
    fl = be - 127;
  }
  int X = fl - 8;
  return X < -127 ? -127 : (X > 127 ? 127 : X);
}

// ---------------------------------------------------------------- w2l layout
// The 2-bit kernel layout keeps the canonical code bytes (4 codes per byte,
// element i at bits 2(i%4)) but moves whole 32-bit words: a row's K is cut
// into slices of SW elements (w2l_sw); inside a slice, lane l (of SW/16)
// owns the word of elements 16l..16l+15, and the words of 4 consecutive rows
// of one lane sit together.  Word (row, slice s, lane l) lands at
//   s*(R*SW/16) + (row/4)*(4*SW/16) + l*4 + row%4          (in words, per matrix)
// and bf16 scale (row, slice s, group g of the slice) at
//   s*(R*SW/32) + (row/4)*(4*SW/32) + g*4 + row%4.
// A block of 4*n rows of one slice is contiguous (one bulk copy), and a lane
// reads its 4 rows' words with one 16-byte load.
// Slice width: K itself up to 512, else the largest of 512/256/128 dividing K.
MOE_HD int w2l_sw(int K) { return K <= 512 ? K : (K % 512 == 0 ? 512 : (K % 256 == 0 ? 256 : 128)); }

MOE_HD int64_t w2l_word(int64_t row, int64_t R, int K, int64_t kw) {
  // kw = canonical word index within the row (16 elements per word)
  const int SW = w2l_sw(K);
  const int64_t s = (kw * 16) / SW, l = ((kw * 16) % SW) / 16;
  return s * (R * SW / 16) + (row / 4) * (4 * (SW / 16)) + l * 4 + row % 4;
}
MOE_HD int64_t w2l_scale(int64_t row, int64_t R, int K, int64_t g) {
  const int SW = w2l_sw(K);
  const int64_t s = (g * 32) / SW, gs = ((g * 32) % SW) / 32;
  return s * (R * SW / 32) + (row / 4) * (4 * (SW / 32)) + gs * 4 + row % 4;
}

}  // namespace moe
