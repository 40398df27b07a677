// Grouped expert matmul on the tensor cores with the dequantised WEIGHTS as
// the A operand in tensor memory (tcgen05 "A from TMEM" form).
//
// For each expert group (permuted rows offsets[e]..offsets[e+1]) the CTA
// computes, per tile of NT tokens and a pair of 128-row weight blocks,
//     D0[128 x NT] = W_block0 . X^T,   D1[128 x NT] = W_block1 . X^T
// (FC1: block 0 = 128 gate rows, block 1 = the matching 128 up rows, so a
// thread of the epilogue holds g and u of the same output; FC2: two
// consecutive 128-row blocks).  TMEM lane = weight row, column = token.
//
//   warp 0      TMA: token tiles [NT rows x 64 K] bf16 (128-byte swizzle),
//               one per A stage
//   warps 1, 15 MMA issue, one weight block each (warp 1 also allocates
//               TMEM): tcgen05.mma kind::f16, A from TMEM, B = token tile in
//               shared memory, M=128, N = the tile's tokens rounded up to 16,
//               K=16; tcgen05.commit frees the block's A stage.  One
//               thread's MMAs run back to back (~100-120 cycles each at N <=
//               128, measured), so two issuers keep the tensor pipe fed.
//   warp 14     TMA: the weight ring, both blocks' share of each 64-K stage
//               six stages ahead (2-bit codes + bf16 scales, E4M3 bytes, or
//               E2M1 nibbles; 64- / 32-byte swizzles so the decode warps'
//               shared loads are conflict-free)
//   warps 2-9   weight decode: each thread owns one weight row of one block
//               (its TMEM lane) and per 64-K stage turns the row's codes into
//               64 bf16 values in registers and writes them to its lane of
//               the stage's A columns with tcgen05.st, then hands the ring
//               slot back (only after that store: it consumed every word read
//               from the slot).  The decoded weights never touch shared
//               memory, so the tensor core keeps the shared-memory bandwidth
//               for the token tiles.
//   warps 10-13 epilogue: tcgen05.ld of D0/D1 (a warp reads its 32 lanes),
//               releases each block's accumulator after its last column
//               chunk is read, SwiGLU for FC1 / MXFP8 rounding, rounding,
//               then a shared staging tile and 16-byte row stores
//
// MXFP4 decode (delta-cache experts): a per-lane 256-entry byte -> 2 bf16
// E2M1 table (same window, lane l's copy in bank l: a 4-byte lookup per lane
// is one wavefront; at an 8-byte stride lanes l and l + 16 collided and the
// decode took 1.8x the MMA issue time per stage), scaled by 2^(E8M0-127) as
// bf16 (exact).
// 2-bit decode: a per-lane copy of the 256-entry byte -> 4 bf16 codebook
// table (64 KB at a 64 KB-aligned shared address, lane l's copy in banks
// 2l, 2l+1) is read with one PRMT-formed address per code byte, then scaled
// by the group's bf16 scale (exact: the entries are powers of two).
//
// Tiles (expert, weight-block pair, token tile) with the token tiles of one
// weight block adjacent (the blocks' weights are read from HBM once and then
// from L2); a persistent grid walks them round-robin.  Tokens of a tile past
// the group end are computed but not stored.  Every mbarrier wait is bounded
// (MOE_DEVERR_TIMEOUT).
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"
#include "internal.cuh"
#include "tc_common.cuh"

namespace moe {

namespace {

constexpr int kTmWarps = 16;  // TMA, MMA (block 0), 8 decode, 4 epilogue, code TMA, MMA (block 1)
constexpr int kTmThreads = kTmWarps * 32;
constexpr int kKB = 64;    // K per stage (one 128-byte swizzle row of bf16)
constexpr int kTS = 4;     // pipeline stages (TMEM: 2 x 128 accumulator + 4 x 64 A columns = 512)
constexpr int kTab = 12288;             // barriers and tile tables (E <= 1024)
constexpr int kStg = 128 * 128 * 2;     // epilogue staging: [NT tokens][128 outputs] bf16
constexpr int kCodeStage = 4096 + 1024; // 2-bit: codes [2 blocks][32 quads][64 B] + scales [2][32][16 B]
constexpr int kCS = 6;                  // 2-bit: code ring stages (runs ahead of the TMEM stages)
constexpr int kCodes = kCS * kCodeStage; // after the token tiles
constexpr int kWStage = 2 * 128 * kKB;  // E4M3: both blocks' rows x 64 K bytes per ring stage
constexpr int kQStage = 2 * 128 * kKB / 2;  // MXFP4: both blocks' rows x 64 K nibbles per ring stage
constexpr int kPre = kTab + kStg;           // shared bytes before the LUT window

enum { kFmtW2 = 0, kFmtE4M3 = 1, kFmtMX4 = 2 };
// TMA-fed weight ring after the token tiles: 2-bit codes + scales, E4M3
// bytes or E2M1 nibbles; stages in flight (MXFP4 with 128-token tiles: 4, as
// its LUT window leaves less room)
template <int WF, int NT>
__host__ __device__ constexpr int ring_depth() { return (WF == kFmtMX4 && NT == 128) ? 4 : kCS; }
template <int WF, int NT>
__host__ __device__ constexpr int ring_bytes() {
  return ring_depth<WF, NT>() * (WF == kFmtW2 ? kCodeStage : (WF == kFmtE4M3 ? kWStage : kQStage));
}

struct TmParams {
  const uint8_t* wq;        // W2: w2l codes; E4M3: workspace bytes [slots][R][K]; MX4: E2M1 [slots][R][K/2]
  const uint16_t* wscale;   // W2: w2l bf16 scales; MX4: E8M0 bytes [slots][R][K/32]
  const int32_t* wslot_of;  // E4M3: expert -> workspace slot (< 0: skipped)
  const int32_t* select_map;
  int select;
  int split;                 // 2: only groups of kSplitRows rows or more
  const int32_t* offsets;
  int ebeg, eend;           // experts processed: [ebeg, eend)
  int E, N, K, R;
  int fc1;
  void* out;
  int out_fmt;
  uint32_t* dev_err;
  long long wait;           // bounded-wait limit (SM clock cycles)
};

MOE_D uint32_t bf16x2_mul(uint32_t a, uint32_t b) {
  __nv_bfloat162 x = *reinterpret_cast<__nv_bfloat162*>(&a);
  const __nv_bfloat162 y = *reinterpret_cast<__nv_bfloat162*>(&b);
  x = __hmul2(x, y);
  return *reinterpret_cast<uint32_t*>(&x);
}

// One code word's four LUT entries (4 bf16 each) for this lane, scaled.
MOE_D void w2_decode_word(uint32_t w, uint32_t lanebase, uint32_t sc2, uint32_t* o) {
  uint32_t a0, a1, a2, a3;
  asm("prmt.b32 %0, %1, %2, 0x7604;" : "=r"(a0) : "r"(w), "r"(lanebase));
  asm("prmt.b32 %0, %1, %2, 0x7614;" : "=r"(a1) : "r"(w), "r"(lanebase));
  asm("prmt.b32 %0, %1, %2, 0x7624;" : "=r"(a2) : "r"(w), "r"(lanebase));
  asm("prmt.b32 %0, %1, %2, 0x7634;" : "=r"(a3) : "r"(w), "r"(lanebase));
  uint2 e0, e1, e2, e3;
  asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(e0.x), "=r"(e0.y) : "r"(a0));
  asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(e1.x), "=r"(e1.y) : "r"(a1));
  asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(e2.x), "=r"(e2.y) : "r"(a2));
  asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(e3.x), "=r"(e3.y) : "r"(a3));
  o[0] = bf16x2_mul(e0.x, sc2);
  o[1] = bf16x2_mul(e0.y, sc2);
  o[2] = bf16x2_mul(e1.x, sc2);
  o[3] = bf16x2_mul(e1.y, sc2);
  o[4] = bf16x2_mul(e2.x, sc2);
  o[5] = bf16x2_mul(e2.y, sc2);
  o[6] = bf16x2_mul(e3.x, sc2);
  o[7] = bf16x2_mul(e3.y, sc2);
}

// Two E4M3 bytes -> bf16x2 (exact: every E4M3 value is a bf16 value).
MOE_D uint32_t e4m3x2_to_bf16x2(uint32_t two) {
  const float2 f = e4m3x2_to_f32x2(static_cast<uint16_t>(two));
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(f.y), "f"(f.x));
  return r;
}

template <int WF, int NT>
__global__ void __launch_bounds__(kTmThreads, 1) tmem_mm_kernel(const __grid_constant__ CUtensorMap tmap_b,
                                                                const __grid_constant__ CUtensorMap tmap_c,
                                                                const __grid_constant__ CUtensorMap tmap_s,
                                                                const TmParams P) {
  constexpr int kBTile = NT * kKB * 2;  // token tile bytes per stage
  constexpr uint32_t kColA = 2 * NT;   // first A column (after D0, D1)
  constexpr uint32_t kCols = (2 * NT + kTS * 64 <= 256) ? 256 : 512;  // TMEM columns allocated
  constexpr bool kLut = WF == kFmtW2 || WF == kFmtMX4;
  extern __shared__ __align__(1024) uint8_t smem[];
  const uint32_t base = smem_u32(smem);
  // [barriers, tile table][LUT window (W2), 64 KB aligned][token tiles, 1024 aligned]
  const uint32_t win = (base + kPre + 65535u) & ~65535u;
  const uint32_t tiles_off =
      kLut ? (win - base + 65536u) : (((base + static_cast<uint32_t>(kPre) + 1023u) & ~1023u) - base);
  uint8_t* tiles = smem + tiles_off;
  uint8_t* codes_s = tiles + kTS * kBTile;  // per-stage weight tiles (TMA): 2-bit codes / scales, E4M3 bytes
  uint64_t* full_a = reinterpret_cast<uint64_t*>(smem);  // [2][kTS] A stage of weight block b decoded
  uint64_t* full_b = full_a + 2 * kTS;                     // [kTS] token tile landed
  uint64_t* empty = full_b + kTS;                          // [2][kTS] block b's MMAs of the stage done
  uint64_t* acc_full = empty + 2 * kTS;
  uint64_t* acc_empty = acc_full + 1;    // [2] weight block b's accumulator read
  uint64_t* code_full = acc_empty + 2;    // [kCS] 2-bit code ring
  uint64_t* code_empty = code_full + kCS; // [kCS]
  uint32_t* tmem_base_s = reinterpret_cast<uint32_t*>(code_empty + kCS);
  int* flags = reinterpret_cast<int*>(tmem_base_s + 2);
  int* tile_start = flags + 8;  // [E+1]
  int* wslot = tile_start + (P.E + 1);  // [E] weight slot of each expert (-1: skipped)

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  {
    uint32_t dyn;
    asm("mov.u32 %0, %%dynamic_smem_size;" : "=r"(dyn));
    if (tiles_off + static_cast<uint32_t>(kTS * kBTile + ring_bytes<WF, NT>()) > dyn) {  // refuse
      if (tid == 0) set_err(P.dev_err, MOE_DEVERR_LAUNCH);
      return;
    }
  }
  const bool fc1 = P.fc1 != 0;
  const int NBLK = fc1 ? P.N / 128 : P.N / 256;  // weight-block pairs
  const int KB = P.K / kKB;

  // ---- setup (shared memory only until pdl_wait: it overlaps the previous kernel)
  if (WF == kFmtMX4) {  // per-lane E2M1 pair LUT: byte b -> bf16x2 (lo nibble first) at win + 256 b + 4 l
    const uint32_t mag[8] = {0x0000u, 0x3F00u, 0x3F80u, 0x3FC0u, 0x4000u, 0x4040u, 0x4080u, 0x40C0u};
    for (int i = tid; i < 256 * 32; i += kTmThreads) {
      const uint32_t b = static_cast<uint32_t>(i >> 5);
      const uint32_t lo = mag[b & 7] | ((b & 8u) << 12), hi = mag[(b >> 4) & 7] | ((b & 0x80u) << 8);
      *reinterpret_cast<uint32_t*>(smem + (win - base) + b * 256u + (i & 31) * 4u) = lo | (hi << 16);
    }
  }
  if (WF == kFmtW2) {  // per-lane codebook LUT: entry b of lane l at win + 256 b + 8 l
    const uint32_t ent[4] = {0xC080u, 0xBF80u, 0x3F80u, 0x4080u};  // -4, -1, 1, 4 as bf16
    for (int i = tid; i < 256 * 32; i += kTmThreads) {
      const uint32_t b = static_cast<uint32_t>(i >> 5);
      const uint2 v =
          make_uint2(ent[b & 3] | (ent[(b >> 2) & 3] << 16), ent[(b >> 4) & 3] | (ent[b >> 6] << 16));
      *reinterpret_cast<uint2*>(smem + (win - base) + b * 256u + (i & 31) * 8u) = v;
    }
  }
  pdl_wait();
  pdl_trigger();
  for (int e = tid; e < P.E; e += kTmThreads) {
    int sl = -1;
    if (e >= P.ebeg && e < P.eend && P.offsets[e + 1] > P.offsets[e]) {
      if (WF == kFmtW2) {
        sl = e;
        if (P.select == 1 && P.select_map[e] >= 0) sl = -1;
        if (P.split == 2 && P.offsets[e + 1] - P.offsets[e] < kSplitRows) sl = -1;
      } else {
        sl = P.wslot_of ? P.wslot_of[e] : e;  // E4M3: workspace slot; MX4: cache slot (< 0: skipped)
        if (sl >= P.E) {                      // beyond the E slots the weight tensor map spans
          set_err(P.dev_err, MOE_DEVERR_BAD_ID);
          sl = -1;
        }
      }
    }
    wslot[e] = sl;
  }
  __syncthreads();
  if (warp == 0) {
    int run = 0;
    for (int b0 = 0; b0 <= P.E; b0 += 32) {
      const int e = b0 + lane;
      int n = 0;
      if (e < P.E && wslot[e] >= 0) n = ((P.offsets[e + 1] - P.offsets[e] + NT - 1) / NT) * NBLK;
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
  if (tid == 0) {
    for (int s = 0; s < kTS; ++s) {
      mbar_init(&full_a[s], 4);
      mbar_init(&full_a[kTS + s], 4);
      mbar_init(&full_b[s], 1);
      mbar_init(&empty[s], 1);
      mbar_init(&empty[kTS + s], 1);
    }
    mbar_init(acc_full, 2);
    mbar_init(&acc_empty[0], 4);
    mbar_init(&acc_empty[1], 4);
    for (int c = 0; c < kCS; ++c) {
      mbar_init(&code_full[c], 1);
      mbar_init(&code_empty[c], 8);
    }
    flags[0] = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tm_alloc(tmem_base_s, kCols);
    tm_relinquish();
  }
  tm_fence_before();
  __syncthreads();
  tm_fence_after();
  const uint32_t tmem = *tmem_base_s;
  const int total = tile_start[P.E];

  auto decode_tile = [&](int i, int& e, int& blk, int& mt) {
    int lo = 0, hi = P.E;
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (tile_start[mid] <= i) lo = mid; else hi = mid;
    }
    e = lo;
    const int loc = i - tile_start[e];
    const int nm = (P.offsets[e + 1] - P.offsets[e] + NT - 1) / NT;
    blk = loc / nm;
    mt = loc - blk * nm;
  };
  auto aborted = [&]() { return *reinterpret_cast<volatile int*>(&flags[0]) != 0; };
  auto abort_all = [&]() {
    flags[0] = 1;
    set_err(P.dev_err, MOE_DEVERR_TIMEOUT);
  };

  const int SWc = w2l_sw(P.K);        // 2-bit: w2l slice width
  const int kbs = SWc / kKB;           // k-blocks per slice
  const int NSL = P.K / SWc;
  if (warp == 0) {
    // ================= token tiles (lane 0) and 2-bit codes (lane 1) by TMA =================
    if (lane == 0) {
      uint32_t L = 0;
      for (int i = blockIdx.x; i < total && !aborted(); i += gridDim.x) {
        int e, blk, mt;
        decode_tile(i, e, blk, mt);
        const int row0 = P.offsets[e] + mt * NT;
        bool ok = true;
        for (int kb = 0; kb < KB; ++kb, ++L) {
          const int s = L % kTS;
          if (L >= kTS && (!mbar_wait(&empty[s], ((L / kTS) - 1) & 1, P.wait) ||
                           !mbar_wait(&empty[kTS + s], ((L / kTS) - 1) & 1, P.wait))) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&full_b[s], kBTile);
          tma_load_tile(tiles + s * kBTile, &tmap_b, kb * kKB, row0, &full_b[s]);
        }
        if (!ok) {
          abort_all();
          break;
        }
      }
    }
  } else if (warp == 14) {
    if (lane == 0 && WF == kFmtE4M3) {
      // the stage's E4M3 bytes of both weight blocks (128 rows x 64 K each), up to kCS stages ahead
      uint32_t L = 0;
      for (int i = blockIdx.x; i < total && !aborted(); i += gridDim.x) {
        int e, blk, mt;
        decode_tile(i, e, blk, mt);
        const int rbase = wslot[e] * P.R;
        bool ok = true;
        for (int kb = 0; kb < KB; ++kb, ++L) {
          const int c = L % kCS;
          if (L >= kCS && !mbar_wait(&code_empty[c], ((L / kCS) - 1) & 1, P.wait)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&code_full[c], kWStage);
#pragma unroll
          for (int bs = 0; bs < 2; ++bs) {
            const int r0 = rbase + (fc1 ? (bs ? P.N : 0) + blk * 128 : blk * 256 + bs * 128);
            tma_load_tile(codes_s + c * kWStage + bs * (kWStage / 2), &tmap_c, kb * kKB, r0, &code_full[c]);
          }
        }
        if (!ok) {
          abort_all();
          break;
        }
      }
    }
    if (lane == 0 && WF == kFmtMX4) {
      // the stage's E2M1 nibbles of both weight blocks (128 rows x 32 bytes each)
      constexpr int RD = ring_depth<WF, NT>();
      uint32_t L = 0;
      for (int i = blockIdx.x; i < total && !aborted(); i += gridDim.x) {
        int e, blk, mt;
        decode_tile(i, e, blk, mt);
        const int rbase = wslot[e] * P.R;
        bool ok = true;
        for (int kb = 0; kb < KB; ++kb, ++L) {
          const int c = L % RD;
          if (L >= RD && !mbar_wait(&code_empty[c], ((L / RD) - 1) & 1, P.wait)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&code_full[c], kQStage);
#pragma unroll
          for (int bs = 0; bs < 2; ++bs) {
            const int r0 = rbase + (fc1 ? (bs ? P.N : 0) + blk * 128 : blk * 256 + bs * 128);
            tma_load_tile(codes_s + c * kQStage + bs * (kQStage / 2), &tmap_c, kb * (kKB / 2), r0, &code_full[c]);
          }
        }
        if (!ok) {
          abort_all();
          break;
        }
      }
    }
    if (lane == 0 && WF == kFmtW2) {
      // the stage's codes and scales of both weight blocks, up to kCS stages ahead
      uint32_t L = 0;
      for (int i = blockIdx.x; i < total && !aborted(); i += gridDim.x) {
        int e, blk, mt;
        decode_tile(i, e, blk, mt);
        bool ok = true;
        for (int kb = 0; kb < KB; ++kb, ++L) {
          const int c = L % kCS;
          if (L >= kCS && !mbar_wait(&code_empty[c], ((L / kCS) - 1) & 1, P.wait)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&code_full[c], kCodeStage);
          const int sl = kb / kbs, kin = kb - sl * kbs;
          const int qrow = (e * NSL + sl) * (P.R >> 2);
#pragma unroll
          for (int bs = 0; bs < 2; ++bs) {
            const int q0 = qrow + (fc1 ? (bs ? (P.N >> 2) : 0) + blk * 32 : blk * 64 + bs * 32);
            tma_load_tile(codes_s + c * kCodeStage + bs * 2048, &tmap_c, kin * 64, q0, &code_full[c]);
            tma_load_tile(codes_s + c * kCodeStage + 4096 + bs * 512, &tmap_s, kin * 16, q0, &code_full[c]);
          }
        }
        if (!ok) {
          abort_all();
          break;
        }
      }
    }
  } else if (warp == 1 || warp == 15) {
    // ================= MMA issue: weight block 0 from warp 1, block 1 from warp 15 =================
    // (one thread's MMAs run back to back; two issuers keep the tensor pipe fed)
    if (lane == 0) {
      const int bs = warp == 1 ? 0 : 1;
      uint32_t L = 0;
      int t = 0;
      for (int i = blockIdx.x; i < total && !aborted(); i += gridDim.x, ++t) {
        // N of this tile's MMAs: its tokens rounded up to 16 (a group's last
        // tile is usually partial; the tensor time scales with N)
        int e, blk, mt;
        decode_tile(i, e, blk, mt);
        const int nvalid = min(NT, P.offsets[e + 1] - P.offsets[e] - mt * NT);
        const uint32_t idesc = idesc_bf16_mn(128, min(NT, (nvalid + 15) & ~15));
        if (t >= 1 && !mbar_wait(&acc_empty[bs], (t - 1) & 1, P.wait)) {
          abort_all();
          break;
        }
        tm_fence_after();
        bool ok = true;
        for (int kb = 0; kb < KB; ++kb, ++L) {
          const int s = L % kTS;
          const uint32_t par = (L / kTS) & 1;
          if (!mbar_wait(&full_b[s], par, P.wait) || !mbar_wait(&full_a[bs * kTS + s], par, P.wait)) {
            ok = false;
            break;
          }
          tm_fence_after();
          const uint32_t sb = smem_u32(tiles + s * kBTile);
          const uint32_t a0 = tmem + kColA + static_cast<uint32_t>(s * 64 + bs * 32);
#pragma unroll
          for (int ks = 0; ks < kKB / 16; ++ks) {
            const uint64_t bd = desc_sw128(sb + ks * 32);
            const uint32_t acc = (kb | ks) != 0;
            umma_ts(tmem + static_cast<uint32_t>(bs * NT), a0 + ks * 8, bd, idesc, acc);
          }
          umma_commit_to(&empty[bs * kTS + s]);
        }
        if (!ok) {
          abort_all();
          break;
        }
        umma_commit_to(acc_full);
      }
    }
  } else if (warp < 10) {
    // ================= weight decode: one weight row per thread =================
    const int d = warp - 2;
    const int bsel = d >> 2;       // weight block 0 / 1
    const int q = warp & 3;        // TMEM lane quarter this warp may access
    const int m = 32 * q + lane;   // row within the 128-row block
    // lane l's table entries: 8 bytes at 8 l (2-bit: 4 bf16 per byte) or 4
    // bytes at 4 l (MXFP4: 2 bf16 per byte), so a warp's lookups take one
    // shared-memory wavefront per 128 bytes (lane l always in the same banks)
    const uint32_t lanebase = win + (WF == kFmtMX4 ? 4u : 8u) * static_cast<uint32_t>(lane);
    const uint32_t tlane = static_cast<uint32_t>(32 * q) << 16;
    // weight row (within the expert) of block bsel of pair blk
    auto wrow = [&](int blk) {
      return fc1 ? (bsel ? P.N : 0) + blk * 128 + m : blk * 256 + bsel * 128 + m;
    };
    // this CTA's tiles are blockIdx.x, +gridDim.x, ...; flat stage index L
    const int ntile = blockIdx.x < total ? (total - 1 - static_cast<int>(blockIdx.x)) / gridDim.x + 1 : 0;
    const uint32_t Ltot = static_cast<uint32_t>(ntile) * static_cast<uint32_t>(KB);
    // prefetch cursor: (tile pi, k-block pkb) of the next stage to load; the
    // formats keep running pointers (no divisions per stage) and re-base them
    // when the cursor moves to the next tile
    int pi = blockIdx.x, pkb = 0, pe = 0, pblk = 0, pmt = 0;
    if (pi < total) decode_tile(pi, pe, pblk, pmt);
    auto next_tile = [&]() -> bool {  // true when the cursor moved to a new tile
      if (++pkb < KB) return false;
      pkb = 0;
      pi += gridDim.x;
      if (pi < total) decode_tile(pi, pe, pblk, pmt);
      return true;
    };
    bool ok = true;
    if (WF == kFmtW2) {
      // codes and scales of this thread's row come from the TMA-filled stage
      // tiles: quad qd = block bsel's quad m/4, row rr = m % 4.  The code tile
      // is written with the 64-byte swizzle (16-byte chunk w of tile row qd at
      // chunk w ^ ((qd >> 1) & 3)), so the warp's 32 word reads hit 32 banks
      const uint32_t cbase = smem_u32(codes_s) + static_cast<uint32_t>(bsel * 2048 + (m >> 2) * 64 + (m & 3) * 4);
      const uint32_t cx = static_cast<uint32_t>((m >> 3) & 3);
      const uint32_t cw0 = (0u ^ cx) << 4, cw1 = (1u ^ cx) << 4, cw2 = (2u ^ cx) << 4, cw3 = (3u ^ cx) << 4;
      const uint32_t sbase = smem_u32(codes_s) + static_cast<uint32_t>(4096 + bsel * 512 + (m >> 2) * 16 + (m & 3) * 2);
      for (uint32_t L = 0; L < Ltot && ok && !aborted(); ++L) {
        const int s = L % kTS, c = L % kCS;
        if (!mbar_wait(&code_full[c], (L / kCS) & 1, P.wait)) {
          ok = false;
          break;
        }
        uint32_t w[4], sc0, sc1;
        const uint32_t co = cbase + static_cast<uint32_t>(c * kCodeStage);
        const uint32_t so = sbase + static_cast<uint32_t>(c * kCodeStage);
        asm volatile("ld.shared.u32 %0, [%1];" : "=r"(w[0]) : "r"(co + cw0) : "memory");
        asm volatile("ld.shared.u32 %0, [%1];" : "=r"(w[1]) : "r"(co + cw1) : "memory");
        asm volatile("ld.shared.u32 %0, [%1];" : "=r"(w[2]) : "r"(co + cw2) : "memory");
        asm volatile("ld.shared.u32 %0, [%1];" : "=r"(w[3]) : "r"(co + cw3) : "memory");
        asm volatile("ld.shared.u16 %0, [%1];" : "=r"(sc0) : "r"(so) : "memory");
        asm volatile("ld.shared.u16 %0, [%1+8];" : "=r"(sc1) : "r"(so) : "memory");
        if (L >= kTS && !mbar_wait(&empty[bsel * kTS + s], ((L / kTS) - 1) & 1, P.wait)) {
          ok = false;
          break;
        }
        tm_fence_after();  // the MMAs that read this A stage are complete
        uint32_t o[32];
        const uint32_t s_lo = sc0 | (sc0 << 16), s_hi = sc1 | (sc1 << 16);
        w2_decode_word(w[0], lanebase, s_lo, o);
        w2_decode_word(w[1], lanebase, s_lo, o + 8);
        w2_decode_word(w[2], lanebase, s_hi, o + 16);
        w2_decode_word(w[3], lanebase, s_hi, o + 24);
        tm_st32(tmem + tlane + kColA + static_cast<uint32_t>(s * 64 + bsel * 32), o);
        tm_st_wait();
        tm_fence_before();
        __syncwarp();
        // the ring slot is released only now: tcgen05.st consumed values
        // derived from every word read from it, so those reads are complete
        // before the TMA may refill the slot
        if (lane == 0) {
          mbar_arrive(&code_empty[c]);
          mbar_arrive(&full_a[bsel * kTS + s]);
        }
      }
    } else if (WF == kFmtMX4) {  // MXFP4: E2M1 [slot][R][K/2] fed by TMA, E8M0 [slot][R][K/32] loaded here
      constexpr int RD = ring_depth<WF, NT>();
      const int64_t mat_s = static_cast<int64_t>(P.R) * (P.K / 32);
      const uint8_t* e8 = reinterpret_cast<const uint8_t*>(P.wscale);
      const uint8_t* ep = e8;  // the load cursor's scale pair (this thread's row)
      auto rebase = [&]() { ep = e8 + wslot[pe] * mat_s + static_cast<int64_t>(wrow(pblk)) * (P.K / 32); };
      if (pi < total) rebase();
      // this thread's row: tile row m of block bsel, 32 bytes written with the
      // 32-byte swizzle (16-byte chunk h at chunk h ^ ((m >> 2) & 1)); a
      // quarter-warp's 8 rows then cover all 32 banks
      const uint32_t qrow = smem_u32(codes_s) + static_cast<uint32_t>(bsel * (kQStage / 2) + m * 32);
      const uint32_t qx = static_cast<uint32_t>((m >> 2) & 1);
      // 2^(x-127) as bf16x2 (x = 0: the subnormal 2^-127; x = 255: NaN, flagged)
      auto scale2 = [&](uint32_t x) -> uint32_t {
        const uint32_t b = x == 0 ? 0x0040u : (x == 255 ? 0x7FC0u : (x << 7));
        return b | (b << 16);
      };
      // one stage: the row's 64 E2M1 codes of the ring slot, scaled by the
      // stage's E8M0 pair sc (group 0 low byte), into this lane's A columns
      auto stage = [&](uint32_t L, uint32_t sc) -> bool {
        const int s = L % kTS, c = L % RD;
        if (!mbar_wait(&code_full[c], (L / RD) & 1, P.wait)) return false;
        uint4 q[2];
        const uint32_t qo = qrow + static_cast<uint32_t>(c * kQStage);
#pragma unroll
        for (int h = 0; h < 2; ++h)
          asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                       : "=r"(q[h].x), "=r"(q[h].y), "=r"(q[h].z), "=r"(q[h].w)
                       : "r"(qo + ((static_cast<uint32_t>(h) ^ qx) << 4))
                       : "memory");
        if (L >= kTS && !mbar_wait(&empty[bsel * kTS + s], ((L / kTS) - 1) & 1, P.wait)) return false;
        tm_fence_after();
        if ((sc & 0xffu) == 255u || (sc >> 8) == 255u) set_err(P.dev_err, MOE_DEVERR_NAN_SCALE);
        const uint32_t s0 = scale2(sc & 0xffu), s1 = scale2(sc >> 8);
        uint32_t o[32];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const uint32_t ww[4] = {q[h].x, q[h].y, q[h].z, q[h].w};
          const uint32_t sh = h ? s1 : s0;  // bytes 0..15: group 0, 16..31: group 1
#pragma unroll
          for (int wi = 0; wi < 4; ++wi) {
            uint32_t a[4];
            asm("prmt.b32 %0, %1, %2, 0x7604;" : "=r"(a[0]) : "r"(ww[wi]), "r"(lanebase));
            asm("prmt.b32 %0, %1, %2, 0x7614;" : "=r"(a[1]) : "r"(ww[wi]), "r"(lanebase));
            asm("prmt.b32 %0, %1, %2, 0x7624;" : "=r"(a[2]) : "r"(ww[wi]), "r"(lanebase));
            asm("prmt.b32 %0, %1, %2, 0x7634;" : "=r"(a[3]) : "r"(ww[wi]), "r"(lanebase));
#pragma unroll
            for (int bb = 0; bb < 4; ++bb) {
              uint32_t ent;
              asm volatile("ld.shared.u32 %0, [%1];" : "=r"(ent) : "r"(a[bb]));
              o[16 * h + 4 * wi + bb] = bf16x2_mul(ent, sh);
            }
          }
        }
        tm_st32(tmem + tlane + kColA + static_cast<uint32_t>(s * 64 + bsel * 32), o);
        tm_st_wait();
        tm_fence_before();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(&code_empty[c]);  // after tcgen05.st consumed values from every word read
          mbar_arrive(&full_a[bsel * kTS + s]);
        }
        return true;
      };
      if (P.K % 512 == 0 && (reinterpret_cast<uintptr_t>(e8) & 15) == 0) {
        // 16-byte scale loads, one per 8 stages (a warp's 2-byte loads from 32
        // rows cost 32 L1 wavefronts each, as many as its table lookups), one
        // group of 8 ahead; a tile's K-blocks are a multiple of 8, so a group
        // never straddles two tiles
        auto load8 = [&](uint4& v) {
          if (pi >= total) return;
          v = __ldg(reinterpret_cast<const uint4*>(ep));
          pkb += 7;
          if (next_tile()) {
            if (pi < total) rebase();
          } else {
            ep += 16;
          }
        };
        uint4 nxt = make_uint4(0, 0, 0, 0);
        load8(nxt);
        for (uint32_t L0 = 0; L0 < Ltot && ok && !aborted(); L0 += 8) {
          const uint4 cur = nxt;
          load8(nxt);
          const uint32_t w4[4] = {cur.x, cur.y, cur.z, cur.w};
#pragma unroll
          for (int j = 0; j < 8; ++j)
            if (ok) ok = stage(L0 + j, (w4[j >> 1] >> (16 * (j & 1))) & 0xffffu);
        }
      } else {
        constexpr int D = 6;  // 2-byte scale loads in flight
        uint32_t sb[D];
        auto load = [&](uint32_t& sc) {
          if (pi >= total) return;
          sc = __ldg(reinterpret_cast<const uint16_t*>(ep));
          if (next_tile()) {
            if (pi < total) rebase();
          } else {
            ep += 2;
          }
        };
#pragma unroll
        for (int d0 = 0; d0 < D; ++d0) load(sb[d0]);
        for (uint32_t L0 = 0; L0 < Ltot && ok && !aborted(); L0 += D) {
#pragma unroll
          for (int d0 = 0; d0 < D; ++d0) {
            const uint32_t L = L0 + d0;
            if (L < Ltot && ok) {
              ok = stage(L, sb[d0]);
              load(sb[d0]);
            }
          }
        }
      }
    } else {  // E4M3 workspace: [slot][R][K] bytes, scale folded in, fed by TMA
      // this thread's row: tile row m of block bsel, 64 bytes written with the
      // 64-byte swizzle (16-byte chunk j at chunk j ^ ((m >> 1) & 3)); a
      // quarter-warp's 8 rows then cover all 32 banks
      const uint32_t rb = smem_u32(codes_s) + static_cast<uint32_t>(bsel * (kWStage / 2) + m * 64);
      const uint32_t rx = static_cast<uint32_t>((m >> 1) & 3);
      for (uint32_t L = 0; L < Ltot && ok && !aborted(); ++L) {
        const int s = L % kTS, c = L % kCS;
        if (!mbar_wait(&code_full[c], (L / kCS) & 1, P.wait)) {
          ok = false;
          break;
        }
        uint4 vb[4];
        const uint32_t ro = rb + static_cast<uint32_t>(c * kWStage);
#pragma unroll
        for (int j = 0; j < 4; ++j)
          asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                       : "=r"(vb[j].x), "=r"(vb[j].y), "=r"(vb[j].z), "=r"(vb[j].w)
                       : "r"(ro + ((static_cast<uint32_t>(j) ^ rx) << 4))
                       : "memory");
        if (L >= kTS && !mbar_wait(&empty[bsel * kTS + s], ((L / kTS) - 1) & 1, P.wait)) {
          ok = false;
          break;
        }
        tm_fence_after();  // the MMAs that read this A stage are complete
        uint32_t o[32];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const uint32_t ww[4] = {vb[j].x, vb[j].y, vb[j].z, vb[j].w};
#pragma unroll
          for (int h = 0; h < 4; ++h) {
            o[8 * j + 2 * h] = e4m3x2_to_bf16x2(ww[h] & 0xffffu);
            o[8 * j + 2 * h + 1] = e4m3x2_to_bf16x2(ww[h] >> 16);
          }
        }
        tm_st32(tmem + tlane + kColA + static_cast<uint32_t>(s * 64 + bsel * 32), o);
        tm_st_wait();
        tm_fence_before();
        __syncwarp();
        // the ring slot is released only now: tcgen05.st consumed values
        // derived from every word read from it, so those reads are complete
        // before the TMA may refill the slot
        if (lane == 0) {
          mbar_arrive(&code_empty[c]);
          mbar_arrive(&full_a[bsel * kTS + s]);
        }
      }
    }
    if (!ok) abort_all();
  } else {
    // ================= epilogue =================
    // bf16 outputs: each warp stages a chunk (32 tokens x its 32 outputs) in
    // a private shared tile and writes it out itself as 16-byte row pieces
    // (storing 2 bytes per lane straight from registers measured slower; a
    // tile shared by the four warps needs a barrier per flush)
    const int q = warp & 3;
    const uint32_t tlane = static_cast<uint32_t>(32 * q) << 16;
    uint16_t* wst = reinterpret_cast<uint16_t*>(smem + kTab) + q * 1024;  // [32 tokens][32 outputs]
    const int nl = 32 * q + lane;  // output within the 128-row block
    int t = 0;
    for (int i = blockIdx.x; i < total && !aborted(); i += gridDim.x, ++t) {
      int e, blk, mt;
      decode_tile(i, e, blk, mt);
      if (!mbar_wait(acc_full, t & 1, P.wait)) {
        abort_all();
        break;
      }
      tm_fence_after();
      const int p0 = P.offsets[e] + mt * NT;
      const int nvalid = min(NT, P.offsets[e + 1] - p0);
      const bool bf16_out = P.out_fmt != MOE_FMT_F32;
      const bool mx_out = P.out_fmt == MOE_FMT_MXFP8_BF16;
      // a weight block's accumulator is free once its last column chunk is
      // read (FC1: gate and up together), before that chunk's math
      auto release = [&](int which) {  // 0 / 1: that block, 2: both
        tm_fence_before();
        __syncwarp();
        if (lane == 0) {
          if (which != 1) mbar_arrive(&acc_empty[0]);
          if (which != 0) mbar_arrive(&acc_empty[1]);
        }
      };
      if (bf16_out) {
        const int nb0 = fc1 ? blk * 128 : blk * 256;
        for (int half = 0; half < (fc1 ? 1 : 2); ++half) {
          const int nw = nb0 + half * 128 + 32 * q;  // first output of this warp
#pragma unroll 1
          for (int c = 0; c < nvalid; c += 32) {
            uint32_t r0[32], r1[32];
            if (fc1) {
              tm_ld32(tmem + tlane + static_cast<uint32_t>(c), r0);
              tm_ld32(tmem + tlane + static_cast<uint32_t>(NT + c), r1);
            } else {
              tm_ld32(tmem + tlane + static_cast<uint32_t>(half * NT + c), r0);
            }
            tm_ld_wait();
            if (c + 32 >= nvalid) release(fc1 ? 2 : half);
            if (mx_out) {
              // MXFP8 rounding: token j's block of 32 outputs is this warp's 32 lanes
#pragma unroll
              for (int j = 0; j < 32; j += 2) {
                const float v0 = silu_fast(__uint_as_float(r0[j])) * __uint_as_float(r1[j]);
                const float v1 = silu_fast(__uint_as_float(r0[j + 1])) * __uint_as_float(r1[j + 1]);
                float m0 = fabsf(v0), m1 = fabsf(v1);
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) {
                  m0 = fmaxf(m0, __shfl_xor_sync(0xffffffffu, m0, o));
                  m1 = fmaxf(m1, __shfl_xor_sync(0xffffffffu, m1, o));
                }
                const int X0 = mx_scale_exp(m0), X1 = mx_scale_exp(m1);
                const uint16_t qq = f32x2_to_e4m3x2(v0 * exp2i(-X0), v1 * exp2i(-X1));
                const float2 d = e4m3x2_to_f32x2(qq);
                uint32_t b2;
                asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(b2) : "f"(d.y * exp2i(X1)), "f"(d.x * exp2i(X0)));
                wst[j * 32 + lane] = static_cast<uint16_t>(b2 & 0xffffu);
                wst[(j + 1) * 32 + lane] = static_cast<uint16_t>(b2 >> 16);
              }
            } else {
#pragma unroll
              for (int j = 0; j < 32; j += 2) {  // hardware RNE, two tokens per conversion
                const float v0 =
                    fc1 ? silu_fast(__uint_as_float(r0[j])) * __uint_as_float(r1[j]) : __uint_as_float(r0[j]);
                const float v1 = fc1 ? silu_fast(__uint_as_float(r0[j + 1])) * __uint_as_float(r1[j + 1])
                                     : __uint_as_float(r0[j + 1]);
                uint32_t b2;
                asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(b2) : "f"(v1), "f"(v0));
                wst[j * 32 + lane] = static_cast<uint16_t>(b2 & 0xffffu);
                wst[(j + 1) * 32 + lane] = static_cast<uint16_t>(b2 >> 16);
              }
            }
            __syncwarp();
#pragma unroll 1
            for (int k2 = 0; k2 < 4; ++k2) {  // 32 rows x 64 bytes as 16-byte pieces
              const int row = (lane >> 2) + 8 * k2, pc = lane & 3;
              if (c + row < nvalid)
                *reinterpret_cast<uint4*>(static_cast<uint16_t*>(P.out) + static_cast<size_t>(p0 + c + row) * P.N +
                                          nw + pc * 8) = *reinterpret_cast<const uint4*>(wst + row * 32 + pc * 8);
            }
            __syncwarp();  // the tile is free for the next chunk
          }
        }
      } else {
        const int n0 = fc1 ? blk * 128 + nl : blk * 256 + nl;
#pragma unroll 1
        for (int c = 0; c < nvalid; c += 32) {
          uint32_t r0[32], r1[32];
          tm_ld32(tmem + tlane + static_cast<uint32_t>(c), r0);
          tm_ld32(tmem + tlane + static_cast<uint32_t>(NT + c), r1);
          tm_ld_wait();
          if (c + 32 >= nvalid) release(2);
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            if (c + j < nvalid) {
              float* o = static_cast<float*>(P.out) + static_cast<size_t>(p0 + c + j) * P.N;
              if (fc1) {
                o[n0] = silu_fast(__uint_as_float(r0[j])) * __uint_as_float(r1[j]);
              } else {
                o[n0] = __uint_as_float(r0[j]);
                o[n0 + 128] = __uint_as_float(r1[j]);
              }
            }
          }
        }
      }
    }
  }

  // ---- teardown: every role is done (or gave up); free TMEM
  tm_fence_before();
  __syncthreads();
  if (warp == 1) {
    tm_fence_after();
    tm_dealloc(tmem, kCols);
  }
}

// ------------------------------------------------------------------ host side
template <int WF, int NT>
cudaError_t launch_tm(const MMArgs& a, const CUtensorMap& map, const CUtensorMap& cmap, const CUtensorMap& smap,
                      const TmParams& P, cudaStream_t s) {
  (void)a;
  const bool lut = WF == kFmtW2 || WF == kFmtMX4;
  // the shared window starts 1 KB in (the reserved block): the LUT window is
  // the first 64 KB-aligned address past kPre; the kernel checks the layout
  const size_t pre = lut ? ((1024 + static_cast<size_t>(kPre) + 65535) & ~size_t(65535)) - 1024 + 65536
                         : static_cast<size_t>(kPre) + 1024;
  const size_t smem = pre + static_cast<size_t>(kTS) * NT * kKB * 2 + ring_bytes<WF, NT>() + 1024;
  cudaError_t e = set_smem_limit(tmem_mm_kernel<WF, NT>, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  return launch_pdl(tmem_mm_kernel<WF, NT>, dim3(matmul_ctas()), dim3(kTmThreads), smem, s, map, cmap, smap, P);
}

}  // namespace

bool tmem_mm_supported(const MMArgs& a) {
  if (a.act_fmt != MOE_FMT_BF16 || a.act_row != nullptr || a.E > 1024) return false;
  if (a.out_fmt != MOE_FMT_BF16 && a.out_fmt != MOE_FMT_F32 &&
      !(a.out_fmt == MOE_FMT_MXFP8_BF16 && a.stage == MOE_STAGE_FC1_SWIGLU))
    return false;
  if (a.K % kKB) return false;
  if (a.stage == MOE_STAGE_FC1_SWIGLU ? a.N % 128 : a.N % 256) return false;
  if (a.wkind == kW2) return a.expert_begin == 0 && a.expert_end == a.E && a.K % w2l_sw(a.K) == 0;
  if (a.wkind == kFP8) return a.wslot_of != nullptr;  // the slot map selects (slot < 0: skipped)
  if (a.wkind == kMXFP4) return a.select == 0 || a.select == 2;  // cache slot map (NULL: slot = e)
  return false;
}

cudaError_t launch_tmem_mm(const MMArgs& a, int rows_total, cudaStream_t s) {
  EncodeFn enc = encode_fn();
  if (!enc) return cudaErrorNotSupported;
  TmParams P;
  P.wq = a.wq;
  P.wscale = static_cast<const uint16_t*>(a.wscale);
  P.wslot_of = a.wslot_of;
  P.select_map = a.select_map;
  P.select = a.select;
  P.split = a.split;
  P.offsets = a.offsets;
  P.ebeg = a.expert_begin;
  P.eend = a.expert_end;
  P.E = a.E;
  P.N = a.N;
  P.K = a.K;
  P.fc1 = a.stage == MOE_STAGE_FC1_SWIGLU;
  P.R = P.fc1 ? 2 * a.N : a.N;
  P.out = a.out;
  P.out_fmt = a.out_fmt;
  P.dev_err = a.dev_err;
  P.wait = a.wait;
  // token tile: 128 rows for prefill-sized groups, 32 for decode-sized ones
  // (the decode of each weight block repeats per token tile, so 32-row tiles
  // only pay off when groups are small)
  const int NT = rows_total <= 16 * a.E ? 32 : 128;
  // tokens: [rows_total][K] bf16, box 64 x NT with the 128-byte swizzle
  CUtensorMap map;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(a.K), static_cast<cuuint64_t>(rows_total > 0 ? rows_total : 1)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(a.K) * 2};
  const cuuint32_t box[2] = {kKB, static_cast<cuuint32_t>(NT)};
  const cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(&map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(a.act), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
  CUtensorMap cmap = map, smap = map;  // unused by the formats without TMA-fed codes
  if (a.wkind == kW2) {
    // w2l codes / scales as 2-D byte arrays: one row per (expert, slice, row quad)
    const int SW = w2l_sw(a.K);
    const cuuint64_t qrows = static_cast<cuuint64_t>(a.E) * (a.K / SW) * (P.R / 4);
    const cuuint64_t cd[2] = {static_cast<cuuint64_t>(SW), qrows}, cs[1] = {static_cast<cuuint64_t>(SW)};
    const cuuint64_t sd[2] = {static_cast<cuuint64_t>(SW / 4), qrows}, ss[1] = {static_cast<cuuint64_t>(SW / 4)};
    const cuuint32_t cbox[2] = {64, 32}, sbox[2] = {16, 32};
    if (enc(&cmap, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(a.wq), cd, cs, cbox, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS ||
        enc(&smap, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(a.wscale), sd, ss, sbox, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  if (a.wkind == kMXFP4) {
    // E2M1 nibbles as a 2-D byte array [E slots x R rows][K/2]; box 32 bytes x
    // 128 rows (one weight block), 32-byte swizzle
    const cuuint64_t qd[2] = {static_cast<cuuint64_t>(a.K / 2), static_cast<cuuint64_t>(a.E) * P.R};
    const cuuint64_t qs[1] = {static_cast<cuuint64_t>(a.K / 2)};
    const cuuint32_t qbox[2] = {kKB / 2, 128};
    if (enc(&cmap, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(a.wq), qd, qs, qbox, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_32B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  if (a.wkind == kFP8) {
    // E4M3 workspace as a 2-D byte array [E slots x R rows][K]; box 64 bytes x
    // 128 rows (one weight block), 64-byte swizzle
    const cuuint64_t wd[2] = {static_cast<cuuint64_t>(a.K), static_cast<cuuint64_t>(a.E) * P.R};
    const cuuint64_t ws[1] = {static_cast<cuuint64_t>(a.K)};
    const cuuint32_t wbox[2] = {kKB, 128};
    if (enc(&cmap, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(a.wq), wd, ws, wbox, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  if (a.wkind == kW2)
    return NT == 32 ? launch_tm<kFmtW2, 32>(a, map, cmap, smap, P, s) : launch_tm<kFmtW2, 128>(a, map, cmap, smap, P, s);
  if (a.wkind == kMXFP4)
    return NT == 32 ? launch_tm<kFmtMX4, 32>(a, map, cmap, smap, P, s) : launch_tm<kFmtMX4, 128>(a, map, cmap, smap, P, s);
  return NT == 32 ? launch_tm<kFmtE4M3, 32>(a, map, cmap, smap, P, s)
                  : launch_tm<kFmtE4M3, 128>(a, map, cmap, smap, P, s);
}

}  // namespace moe
