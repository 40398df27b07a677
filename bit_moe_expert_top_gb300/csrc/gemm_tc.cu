// Prefill expert matmul on the 5th-generation tensor cores (tcgen05 / TMEM).
//
// For each expert group (permuted rows offsets[e]..offsets[e+1]) and each
// block of weight rows, the CTA computes D[128 rows x BN] = A[128 x K] . B^T
// with A = the group's bf16 activation rows and B = BN weight rows of the
// expert, dequantised from the 2-bit codebook into bf16 in shared memory:
//
//   warp 0      TMA: A tiles [128 rows x 64 K] (128-byte swizzle) per k-block
//   warps 1-4   decode: the 2-bit codes + bf16 scales of BN rows x 64 K into
//               bf16 (codebook entry x scale, exact) in the same swizzled
//               K-major layout the MMA reads; fence.proxy.async, arrive
//   warp 5      MMA: one thread issues tcgen05.mma kind::f16 (M=128, N=BN,
//               K=16) x 4 per k-block into a TMEM accumulator; tcgen05.commit
//               frees the stage / publishes the accumulator
//   warps 6-9   epilogue: tcgen05.ld the accumulator (each warp its 32 TMEM
//               lanes = 32 rows), SwiGLU for FC1 (gate columns 0..BN/2-1, up
//               columns BN/2..BN-1), RNE to bf16, store the group's rows
//
// Two TMEM accumulators (2 x BN columns) let the epilogue of one tile overlap
// the main loop of the next.  Tiles are (expert, row block, m block) with the
// m blocks of one weight block adjacent; a persistent grid walks them
// round-robin.  Rows of a 128-row tile past the group end are computed but not
// stored.  Every mbarrier wait is bounded (MOE_DEVERR_TIMEOUT).
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"
#include "internal.cuh"

namespace moe {

namespace {

constexpr int kGemmThreads = 320;
constexpr int kBM = 128;      // rows per tile (TMEM lanes)
constexpr int kBK = 64;       // K per stage: 64 bf16 = one 128-byte swizzle row
constexpr int kStagesTC = 4;
constexpr int kATile = kBM * kBK * 2;  // 16 KB

struct TcParams {
  const uint8_t* codes;    // w2l
  const uint16_t* scales;  // w2l bf16
  const int32_t* select_map;
  int select;
  const int32_t* offsets;
  int E, N, K, R;
  int fc1;
  void* out;
  int out_fmt;
  uint32_t* dev_err;
  long long wait;  // bounded-wait limit (SM clock cycles)
};

// ------------------------------------------------------------------ PTX
MOE_D void tmem_alloc(uint32_t* dst, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst)), "r"(ncols)
               : "memory");
}
MOE_D void tmem_relinquish() { asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory"); }
MOE_D void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
MOE_D void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
MOE_D void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
MOE_D void fence_proxy_async() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

MOE_D void umma_f16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc, uint32_t accum) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accum)
      : "memory");
}
MOE_D void umma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}
// 32 consecutive TMEM columns of this thread's lane (warp-collective).
MOE_D void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}
MOE_D void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

MOE_D void tma_load_2d(void* dst, const CUtensorMap* map, int x, int y, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
          smem_u32(dst)),
      "l"(map), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}

// Shared-memory matrix descriptor: K-major operand in the 128-byte swizzle
// layout (8-row atoms of 1024 bytes stacked along M/N).
MOE_D uint64_t sdesc_sw128(uint32_t saddr) {
  uint64_t d = static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>(16u >> 4) << 16;    // leading byte offset (unused for this layout)
  d |= static_cast<uint64_t>(1024u >> 4) << 32;  // stride byte offset: next 8-row atom
  d |= static_cast<uint64_t>(1) << 46;           // descriptor version
  d |= static_cast<uint64_t>(2) << 61;           // 128-byte swizzle
  return d;
}

// Instruction descriptor: BF16 x BF16 -> FP32, both operands K-major.
MOE_HD uint32_t idesc_bf16(int M, int N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(N >> 3) << 17) |
         (static_cast<uint32_t>(M >> 4) << 24);
}

template <int BN>
__global__ void __launch_bounds__(kGemmThreads, 1) w2_gemm_kernel(const __grid_constant__ CUtensorMap tmap_a,
                                                                  const TcParams P) {
  constexpr int kBTile = BN * kBK * 2;
  constexpr int kStageBytes = kATile + kBTile;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // 1024-byte alignment of the tiles (swizzle atoms)
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* tiles = smem;                                           // [stages][A | B]
  uint64_t* full_a = reinterpret_cast<uint64_t*>(smem + kStagesTC * kStageBytes);
  uint64_t* full_b = full_a + kStagesTC;
  uint64_t* empty = full_b + kStagesTC;
  uint64_t* acc_full = empty + kStagesTC;                          // [2]
  uint64_t* acc_empty = acc_full + 2;                              // [2]
  uint32_t* tmem_base_s = reinterpret_cast<uint32_t*>(acc_empty + 2);
  int* flags = reinterpret_cast<int*>(tmem_base_s + 4);
  uint2* lut = reinterpret_cast<uint2*>(flags + 4);                // [256] byte -> 4 bf16 codebook entries
  int* tile_start = reinterpret_cast<int*>(lut + 256);             // [E+1]

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const bool fc1 = P.fc1 != 0;
  const int NBLK = fc1 ? P.N / (BN / 2) : P.N / BN;  // weight-row blocks
  const int KB = P.K / kBK;

  // ---- setup: tile table, codebook LUT, barriers, TMEM
  if (warp == 0) {
    int run = 0;
    for (int b0 = 0; b0 <= P.E; b0 += 32) {
      const int e = b0 + lane;
      int n = 0;
      if (e < P.E) {
        const int c = P.offsets[e + 1] - P.offsets[e];
        bool sel = c > 0;
        if (sel && P.select == 1) sel = P.select_map[e] < 0;
        if (sel && P.select == 2) sel = P.select_map[e] >= 0;
        if (sel) n = ((c + kBM - 1) / kBM) * NBLK;
      }
      int incl = n;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      if (e <= P.E) tile_start[e] = run + incl - n;
      run += __shfl_sync(0xffffffffu, incl, 31);
    }
  }
  if (tid < 256) {  // entry bits of {-4,-1,1,4} as bf16: 0xC080, 0xBF80, 0x3F80, 0x4080
    const uint32_t ent[4] = {0xC080u, 0xBF80u, 0x3F80u, 0x4080u};
    const uint32_t b = tid;
    lut[b] = make_uint2(ent[b & 3] | (ent[(b >> 2) & 3] << 16), ent[(b >> 4) & 3] | (ent[b >> 6] << 16));
  }
  if (tid == 0) {
    for (int s = 0; s < kStagesTC; ++s) {
      mbar_init(&full_a[s], 1);
      mbar_init(&full_b[s], 4);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&acc_full[a], 1);
      mbar_init(&acc_empty[a], 4);
    }
    flags[0] = 0;
    fence_barrier_init();
  }
  if (warp == 5) {
    tmem_alloc(tmem_base_s, 2 * BN);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_base_s;
  const int total = tile_start[P.E];

  auto decode_tile = [&](int i, int& e, int& blk, int& mt) {
    int lo = 0, hi = P.E;
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (tile_start[mid] <= i) lo = mid; else hi = mid;
    }
    e = lo;
    const int loc = i - tile_start[e];
    const int nm = (P.offsets[e + 1] - P.offsets[e] + kBM - 1) / kBM;
    blk = loc / nm;
    mt = loc - blk * nm;
  };
  auto aborted = [&]() { return *reinterpret_cast<volatile int*>(&flags[0]) != 0; };
  auto abort_all = [&]() {
    flags[0] = 1;
    set_err(P.dev_err, MOE_DEVERR_TIMEOUT);
  };

  if (warp == 0) {
    // ================= A tiles by TMA =================
    if (lane == 0) {
      uint32_t L = 0;
      for (int i = blockIdx.x; i < total && !aborted(); i += gridDim.x) {
        int e, blk, mt;
        decode_tile(i, e, blk, mt);
        const int row0 = P.offsets[e] + mt * kBM;
        for (int kb = 0; kb < KB; ++kb, ++L) {
          const int s = L % kStagesTC;
          if (L >= kStagesTC && !mbar_wait(&empty[s], ((L / kStagesTC) - 1) & 1, P.wait)) {
            abort_all();
            break;
          }
          mbar_arrive_expect_tx(&full_a[s], kATile);
          tma_load_2d(tiles + s * kStageBytes, &tmap_a, kb * kBK, row0, &full_a[s]);
        }
      }
    }
  } else if (warp >= 1 && warp <= 4) {
    // ================= B tiles: 2-bit codes -> bf16, swizzled K-major =================
    const int dt = tid - 32;  // 0..127
    const int SW = w2l_sw(P.K), NLn = SW / 16, Gs = SW / 32;
    const int64_t mat_words = static_cast<int64_t>(P.R) * (P.K / 16);
    const int64_t mat_scales = static_cast<int64_t>(P.R) * (P.K / 32);
    const uint32_t* codes32 = reinterpret_cast<const uint32_t*>(P.codes);
    uint32_t L = 0;
    for (int i = blockIdx.x; i < total && !aborted(); i += gridDim.x) {
      int e, blk, mt;
      decode_tile(i, e, blk, mt);
      for (int kb = 0; kb < KB; ++kb, ++L) {
        const int s = L % kStagesTC;
        if (L >= kStagesTC && !mbar_wait(&empty[s], ((L / kStagesTC) - 1) & 1, P.wait)) {
          abort_all();
          break;
        }
        uint8_t* btile = tiles + s * kStageBytes + kATile;
        const int k0 = kb * kBK;
        const int sl = k0 / SW, lb = (k0 % SW) / 16;  // slice, first lane of this k-block
        // tasks: (row quad q, lane-in-block lk): 4 rows x 16 elements
        for (int task = dt; task < (BN / 4) * 4; task += 128) {
          const int q = task >> 2, lk = task & 3;
          const int nrow = q * 4;  // tile row of the quad
          int wrow;                // weight row of the quad
          if (fc1) wrow = (nrow < BN / 2) ? blk * (BN / 2) + nrow : P.N + blk * (BN / 2) + (nrow - BN / 2);
          else wrow = blk * BN + nrow;
          const int64_t wbase = e * mat_words + static_cast<int64_t>(sl) * (P.R * (SW / 16)) +
                                static_cast<int64_t>(wrow / 4) * (4 * NLn) + (lb + lk) * 4;
          const uint4 w4 = __ldg(reinterpret_cast<const uint4*>(codes32 + wbase));
          const int g = (k0 % SW) / 32 + (lk >> 1);
          const int64_t sbase = e * mat_scales + static_cast<int64_t>(sl) * (P.R * Gs) +
                                static_cast<int64_t>(wrow / 4) * (4 * Gs) + g * 4;
          const uint2 s4 = __ldg(reinterpret_cast<const uint2*>(P.scales + sbase));
          const uint32_t ws[4] = {w4.x, w4.y, w4.z, w4.w};
          const uint32_t sc[4] = {s4.x & 0xffffu, s4.x >> 16, s4.y & 0xffffu, s4.y >> 16};
#pragma unroll
          for (int r = 0; r < 4; ++r) {
            const uint32_t sc2 = sc[r] | (sc[r] << 16);
            const __nv_bfloat162 scb = *reinterpret_cast<const __nv_bfloat162*>(&sc2);
            uint32_t o[8];
#pragma unroll
            for (int by = 0; by < 4; ++by) {
              const uint2 ent = lut[(ws[r] >> (8 * by)) & 0xffu];
              __nv_bfloat162 e0 = *reinterpret_cast<const __nv_bfloat162*>(&ent.x);
              __nv_bfloat162 e1 = *reinterpret_cast<const __nv_bfloat162*>(&ent.y);
              e0 = __hmul2(e0, scb);
              e1 = __hmul2(e1, scb);
              o[2 * by] = *reinterpret_cast<uint32_t*>(&e0);
              o[2 * by + 1] = *reinterpret_cast<uint32_t*>(&e1);
            }
            const int n = nrow + r;
            uint8_t* rowp = btile + n * 128;
            const int c0 = 2 * lk, c1 = 2 * lk + 1;  // 16-byte chunks of this row's 64 K
            *reinterpret_cast<uint4*>(rowp + ((c0 ^ (n & 7)) << 4)) = make_uint4(o[0], o[1], o[2], o[3]);
            *reinterpret_cast<uint4*>(rowp + ((c1 ^ (n & 7)) << 4)) = make_uint4(o[4], o[5], o[6], o[7]);
          }
        }
        fence_proxy_async();  // generic-proxy stores -> visible to the tensor core
        __syncwarp();
        if (lane == 0) mbar_arrive(&full_b[s]);
      }
    }
  } else if (warp == 5) {
    // ================= MMA issue =================
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16(kBM, BN);
      uint32_t L = 0;
      int t = 0;
      for (int i = blockIdx.x; i < total && !aborted(); i += gridDim.x, ++t) {
        const int a = t & 1;
        if (t >= 2 && !mbar_wait(&acc_empty[a], ((t >> 1) - 1) & 1, P.wait)) {
          abort_all();
          break;
        }
        tc_fence_after();
        const uint32_t dt = tmem_base + static_cast<uint32_t>(a * BN);
        bool ok = true;
        for (int kb = 0; kb < KB; ++kb, ++L) {
          const int s = L % kStagesTC;
          const uint32_t par = (L / kStagesTC) & 1;
          if (!mbar_wait(&full_a[s], par, P.wait) || !mbar_wait(&full_b[s], par, P.wait)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sa = smem_u32(tiles + s * kStageBytes);
          const uint32_t sb = sa + kATile;
#pragma unroll
          for (int ks = 0; ks < kBK / 16; ++ks)
            umma_f16(dt, sdesc_sw128(sa + ks * 32), sdesc_sw128(sb + ks * 32), idesc, (kb | ks) != 0);
          umma_commit(&empty[s]);  // stage s is free once these MMAs have read it
        }
        if (!ok) {
          abort_all();
          break;
        }
        umma_commit(&acc_full[a]);  // accumulator a complete
      }
    }
  } else {
    // ================= epilogue: TMEM -> registers -> global =================
    const int q = warp & 3;  // TMEM lane quarter this warp may access
    int t = 0;
    for (int i = blockIdx.x; i < total && !aborted(); i += gridDim.x, ++t) {
      int e, blk, mt;
      decode_tile(i, e, blk, mt);
      const int a = t & 1;
      if (!mbar_wait(&acc_full[a], (t >> 1) & 1, P.wait)) {
        abort_all();
        break;
      }
      tc_fence_after();
      const int gstart = P.offsets[e], gend = P.offsets[e + 1];
      const int m = q * 32 + lane;
      const int p = gstart + mt * kBM + m;
      const bool valid = p < gend;
      const uint32_t tbase = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(a * BN);
      if (fc1) {
#pragma unroll 1
        for (int c = 0; c < BN / 2; c += 32) {
          uint32_t gr[32], ur[32];
          tmem_ld32(tbase + c, gr);
          tmem_ld32(tbase + BN / 2 + c, ur);
          tmem_ld_wait();
          if (valid) {
            const int n0 = blk * (BN / 2) + c;
            if (P.out_fmt == MOE_FMT_F32) {
              float* o = static_cast<float*>(P.out) + static_cast<size_t>(p) * P.N + n0;
#pragma unroll
              for (int j = 0; j < 32; j += 4)
                *reinterpret_cast<float4*>(o + j) = make_float4(
                    silu_f32(__uint_as_float(gr[j])) * __uint_as_float(ur[j]),
                    silu_f32(__uint_as_float(gr[j + 1])) * __uint_as_float(ur[j + 1]),
                    silu_f32(__uint_as_float(gr[j + 2])) * __uint_as_float(ur[j + 2]),
                    silu_f32(__uint_as_float(gr[j + 3])) * __uint_as_float(ur[j + 3]));
            } else {
              uint16_t* o = static_cast<uint16_t*>(P.out) + static_cast<size_t>(p) * P.N + n0;
#pragma unroll
              for (int j = 0; j < 32; j += 8) {
                uint32_t w[4];
#pragma unroll
                for (int h = 0; h < 4; ++h) {
                  const float v0 = silu_f32(__uint_as_float(gr[j + 2 * h])) * __uint_as_float(ur[j + 2 * h]);
                  const float v1 = silu_f32(__uint_as_float(gr[j + 2 * h + 1])) * __uint_as_float(ur[j + 2 * h + 1]);
                  w[h] = static_cast<uint32_t>(f32_to_bf16_rne(v0)) | (static_cast<uint32_t>(f32_to_bf16_rne(v1)) << 16);
                }
                *reinterpret_cast<uint4*>(o + j) = make_uint4(w[0], w[1], w[2], w[3]);
              }
            }
          }
        }
      } else {
#pragma unroll 1
        for (int c = 0; c < BN; c += 32) {
          uint32_t yr[32];
          tmem_ld32(tbase + c, yr);
          tmem_ld_wait();
          if (valid) {
            const int n0 = blk * BN + c;
            if (P.out_fmt == MOE_FMT_F32) {
              float* o = static_cast<float*>(P.out) + static_cast<size_t>(p) * P.N + n0;
#pragma unroll
              for (int j = 0; j < 32; j += 4)
                *reinterpret_cast<float4*>(o + j) = make_float4(__uint_as_float(yr[j]), __uint_as_float(yr[j + 1]),
                                                                __uint_as_float(yr[j + 2]), __uint_as_float(yr[j + 3]));
            } else {
              uint16_t* o = static_cast<uint16_t*>(P.out) + static_cast<size_t>(p) * P.N + n0;
#pragma unroll
              for (int j = 0; j < 32; j += 8) {
                uint32_t w[4];
#pragma unroll
                for (int h = 0; h < 4; ++h)
                  w[h] = static_cast<uint32_t>(f32_to_bf16_rne(__uint_as_float(yr[j + 2 * h]))) |
                         (static_cast<uint32_t>(f32_to_bf16_rne(__uint_as_float(yr[j + 2 * h + 1]))) << 16);
                *reinterpret_cast<uint4*>(o + j) = make_uint4(w[0], w[1], w[2], w[3]);
              }
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acc_empty[a]);
    }
  }

  // ---- teardown: every role is done (or gave up); free TMEM
  tc_fence_before();
  __syncthreads();
  if (warp == 5) {
    tc_fence_after();
    tmem_dealloc(tmem_base, 2 * BN);
  }
}

// ------------------------------------------------------------------ host side
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn get_encode() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPoint("cuTensorMapEncodeTiled", &p, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  return fn;
}

size_t gemm_smem_bytes(int BN, int E) {
  const size_t stage = kATile + static_cast<size_t>(BN) * kBK * 2;
  return 1024 + kStagesTC * stage + 256 + 2048 + 4 * (E + 1) + 64;
}

}  // namespace

bool gemm_supported(const MMArgs& a) {
  if (a.wkind != kW2 || a.act_fmt != MOE_FMT_BF16 || a.act_row != nullptr) return false;
  if (a.out_fmt != MOE_FMT_BF16 && a.out_fmt != MOE_FMT_F32) return false;
  if (a.expert_begin != 0 || a.expert_end != a.E) return false;
  if (a.K % kBK) return false;
  const int SW = w2l_sw(a.K);
  if (a.K % SW) return false;
  if (a.stage == MOE_STAGE_FC1_SWIGLU) return a.N % 128 == 0;
  return a.N % 128 == 0;
}

cudaError_t launch_gemm_tc(const MMArgs& a, int rows_total, cudaStream_t s) {
  EncodeTiledFn enc = get_encode();
  if (!enc) return cudaErrorNotSupported;
  TcParams P;
  P.codes = a.wq;
  P.scales = static_cast<const uint16_t*>(a.wscale);
  P.select_map = a.select_map;
  P.select = a.select;
  P.offsets = a.offsets;
  P.E = a.E;
  P.N = a.N;
  P.K = a.K;
  P.fc1 = a.stage == MOE_STAGE_FC1_SWIGLU;
  P.R = P.fc1 ? 2 * a.N : a.N;
  P.out = a.out;
  P.out_fmt = a.out_fmt;
  P.dev_err = a.dev_err;
  P.wait = a.wait;
  // A: [rows_total][K] bf16, box 64 x 128 with the 128-byte swizzle
  CUtensorMap map;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(a.K), static_cast<cuuint64_t>(rows_total > 0 ? rows_total : 1)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(a.K) * 2};
  const cuuint32_t box[2] = {kBK, kBM};
  const cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(&map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(a.act), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
  const bool bn256 = P.fc1 || a.N % 256 == 0;
  const size_t smem = gemm_smem_bytes(bn256 ? 256 : 128, a.E);
  const DeviceInfo& di = device_info();
  cudaError_t e;
  if (bn256) {
    e = set_smem_limit(w2_gemm_kernel<256>, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    w2_gemm_kernel<256><<<di.sms, kGemmThreads, smem, s>>>(map, P);
  } else {
    e = set_smem_limit(w2_gemm_kernel<128>, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    w2_gemm_kernel<128><<<di.sms, kGemmThreads, smem, s>>>(map, P);
  }
  return cudaGetLastError();
}

}  // namespace moe
