// Grouped expert matmul on the block-scaled FP8 tensor cores
// (tcgen05.mma kind::mxf8f6f4): MXFP8 activation rows (E4M3 codes + one E8M0
// scale per 32 K elements) against
//   * the FP8 workspace ("国产GPU完成MoE大模型Day-0适配" §四): E4M3 weights with
//     the MXFP4 scale folded in, so every weight scale factor is 1.0; or
//   * MXFP4 weights read as they are stored (E2M1 codes + E8M0 scales, the
//     OCP MX block format), with no workspace at all.
// The tensor core multiplies the codes and applies both operands' block
// scales itself; products and sums are those of the definition
// (code_w * 2^Xw * code_x * 2^Xx, fp32 accumulation).
//
// Per tile (expert, pair of 128-row weight blocks, NT tokens) the CTA forms
//     D_b[128 x NT] = W_block_b . X^T          (b = 0, 1)
// (FC1: block 0 = 128 gate rows, block 1 = the matching 128 up rows, so a
// thread of the epilogue holds g and u of one output; FC2: two consecutive
// 128-row blocks), TMEM lane = weight row, column = token.
//
//   warp 0      TMA, one 128-element K stage at a time: the token tile (NT
//               rows x 128 E4M3 bytes) and both weight blocks (128 rows x 128
//               E4M3 bytes, or 128 x 128 E2M1 codes that the copy expands to
//               the MMA's 16-byte form of 16 codes + 8 pad bytes), all with
//               the 128-byte swizzle
//   warps 1, 2  MMA issue, one weight block each: 4 MMAs of K = 32 per stage,
//               the scale byte of k-block ks picked by the instruction
//               descriptor; tcgen05.commit frees the stage
//   warps 4-7   scale factors: per stage, the tokens' E8M0 words (4 k-blocks
//               per 32-bit TMEM cell) written to TMEM with tcgen05.st
//               (token n at lane n mod 32 of every lane quarter, column n/32),
//               and for MXFP4 the weight rows' E8M0 words (row m at lane m,
//               column m/32)
//   warps 8-15  epilogue, two warps per TMEM lane quarter on alternate
//               32-token chunks: tcgen05.ld of D_0 / D_1, SwiGLU for FC1,
//               output rounding (fp32, bf16, or MXFP8: E4M3 codes + E8M0 per
//               32 outputs, the FP8 path's h; block maxima by a butterfly
//               reduce-scatter across the warp), a private shared tile per
//               warp and 16-byte row pieces (no barrier across the warps).  Measured (per-role clock counts): with four
//               epilogue warps and one shuffle reduction per token the
//               epilogue, not the MMAs, set the pace
//   warp 3      allocates and frees TMEM
//
// Tiles are walked round-robin by a persistent grid (one CTA per SM) in the
// order (expert, block pair, token tile): the token tiles of one weight block
// pair are adjacent, so the block is read from HBM once and then from L2.
// Every mbarrier wait is bounded (MOE_DEVERR_TIMEOUT).
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"
#include "internal.cuh"
#include "tc_common.cuh"

namespace moe {

namespace {

constexpr int kMxWarps = 16;
constexpr int kMxThreads = kMxWarps * 32;
constexpr int kKS = 128;        // K elements per stage: 4 MMAs of K = 32, one E8M0 word per row
// pipeline stages: 4 with 128-token tiles; 5 with 32-token tiles, where a
// stage is small (36 KB) and the weight bytes in flight are what bound the
// decode-sized launch (one stage carries 16 KB of packed weights from HBM)
template <int NT>
__host__ __device__ constexpr int mx_stages() { return NT == 32 ? 5 : 4; }
constexpr int kMTab = 12288;    // barriers, flags, tile tables (E <= 1024)
constexpr int kMStg = 16384;    // epilogue staging: 8 warps x [32 tokens][32 outputs] x 2 bytes
constexpr uint32_t kSFCols = 16;  // TMEM scale columns per stage: SFA block 0 (+0), block 1 (+4), SFB (+8)

enum { kAE4M3 = 0, kAE2M1 = 1 };

template <int NT>
__host__ __device__ constexpr int mx_stage_bytes() { return NT * kKS + 2 * 128 * kKS; }
template <int NT>
__host__ __device__ constexpr size_t mx_smem_bytes() {
  return 1024 + kMTab + kMStg + static_cast<size_t>(mx_stages<NT>()) * mx_stage_bytes<NT>();
}
static_assert(mx_smem_bytes<128>() <= 232448 && mx_smem_bytes<32>() <= 232448, "shared memory");

struct MxParams {
  const uint8_t* act_scale;  // E8M0 [rows_total][K/32] of the activation rows
  int rows_total;
  const uint8_t* wscale;     // MXFP4: E8M0 [slots][R][K/32]; FP8 workspace: unused
  const int32_t* wslot_of;   // expert -> weight slot (NULL: slot = e; < 0: skipped)
  const int32_t* offsets;
  int ebeg, eend;
  int E, N, K, R;
  int fc1;
  void* out;
  int out_fmt;               // F32, BF16, or (FC1) MXFP8 with out_scale
  uint8_t* out_scale;
  uint32_t* dev_err;
  long long wait;
};

MOE_D uint32_t ld_u32(const uint8_t* p) { return __ldg(reinterpret_cast<const uint32_t*>(p)); }

MOE_D bool has_ff_byte(uint32_t w) {  // any E8M0 byte 255 (NaN)
  const uint32_t x = ~w;
  return ((x - 0x01010101u) & ~x & 0x80808080u) != 0;
}

template <int AF, int NT, bool kVec>
__global__ void __launch_bounds__(kMxThreads, 1) mx_mm_kernel(const __grid_constant__ CUtensorMap tmap_b,
                                                              const __grid_constant__ CUtensorMap tmap_a,
                                                              const MxParams P) {
  constexpr int kBTile = NT * kKS;        // token bytes per stage
  constexpr int kABlock = 128 * kKS;      // shared bytes of one weight block per stage
  constexpr int kStage = mx_stage_bytes<NT>();
  constexpr int kMS = mx_stages<NT>();
  constexpr uint32_t kATx = AF == kAE2M1 ? 128u * kKS / 2 : 128u * kKS;  // bytes a weight-block copy moves
  constexpr uint32_t kSF0 = 2 * NT;                   // first scale column (after D_0, D_1)
  constexpr uint32_t kSFU = kSF0 + kMS * kSFCols;     // FP8 workspace: the unit weight scales
  constexpr uint32_t kCols = (kSFU + 4 <= 128) ? 128 : ((kSFU + 4 <= 256) ? 256 : 512);
  extern __shared__ __align__(1024) uint8_t smem[];
  const uint32_t base = smem_u32(smem);
  const uint32_t tiles_off = ((base + kMTab + kMStg + 1023u) & ~1023u) - base;
  uint8_t* stages = smem + tiles_off;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem);  // [kMS] stage data landed (TMA)
  uint64_t* empty = full + kMS;                         // [kMS] both blocks' MMAs of the stage done
  uint64_t* sf_full = empty + kMS;                      // [kMS] the stage's scale columns written
  uint64_t* acc_full = sf_full + kMS;
  uint64_t* acc_empty = acc_full + 1;                   // [2] weight block b's accumulator read (8 warps)
  uint32_t* tmem_base_s = reinterpret_cast<uint32_t*>(acc_empty + 2);
  int* flags = reinterpret_cast<int*>(tmem_base_s + 2);
  int* tile_start = flags + 8;          // [E+1]
  int* wslot = tile_start + (P.E + 1);  // [E]
  uint8_t* stg = smem + kMTab;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  {
    uint32_t dyn;
    asm("mov.u32 %0, %%dynamic_smem_size;" : "=r"(dyn));
    if (tiles_off + static_cast<uint32_t>(kMS * kStage) > dyn) {  // launched short: refuse
      if (tid == 0) set_err(P.dev_err, MOE_DEVERR_LAUNCH);
      return;
    }
  }
  const bool fc1 = P.fc1 != 0;
  const int NBLK = fc1 ? P.N / 128 : P.N / 256;
  const int KB = P.K / kKS;
  const int KSB = P.K / 32;  // scale bytes per row

  if (AF == kAE2M1) {
    // the E2M1 copies fill 8 of every 16 bytes; the pad bytes stay zero
    for (int i = tid; i < kMS * 2 * kABlock / 16; i += kMxThreads) {
      const int s = i / (2 * kABlock / 16), r = i - s * (2 * kABlock / 16);
      *reinterpret_cast<uint4*>(stages + s * kStage + kBTile + r * 16) = make_uint4(0, 0, 0, 0);
    }
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  pdl_wait();
  pdl_trigger();
  for (int e = tid; e < P.E; e += kMxThreads) {
    int sl = -1;
    if (e >= P.ebeg && e < P.eend && P.offsets[e + 1] > P.offsets[e]) {
      sl = P.wslot_of ? P.wslot_of[e] : e;
      if (sl >= P.E) {  // beyond the E slots the weight tensor map spans
        set_err(P.dev_err, MOE_DEVERR_BAD_ID);
        sl = -1;
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
    for (int s = 0; s < kMS; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 2);
      mbar_init(&sf_full[s], 4);
    }
    mbar_init(acc_full, 2);
    mbar_init(&acc_empty[0], 8);
    mbar_init(&acc_empty[1], 8);
    flags[0] = 0;
    fence_barrier_init();
  }
  if (warp == 3) {
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
  // first weight row (within the expert) of block b of pair blk
  auto brow = [&](int blk, int b) { return fc1 ? (b ? P.N : 0) + blk * 128 : blk * 256 + b * 128; };
  auto aborted = [&]() { return *reinterpret_cast<volatile int*>(&flags[0]) != 0; };
  auto abort_all = [&]() {
    flags[0] = 1;
    set_err(P.dev_err, MOE_DEVERR_TIMEOUT);
  };

  if (warp == 0) {
    // ================= TMA: token tile + both weight blocks per stage =================
    if (lane == 0) {
      uint32_t L = 0;
      for (int i = blockIdx.x; i < total && !aborted(); i += gridDim.x) {
        int e, blk, mt;
        decode_tile(i, e, blk, mt);
        const int row0 = P.offsets[e] + mt * NT;
        const int r0 = wslot[e] * P.R + brow(blk, 0), r1 = wslot[e] * P.R + brow(blk, 1);
        bool ok = true;
        for (int kb = 0; kb < KB; ++kb, ++L) {
          const int s = L % kMS;
          if (L >= kMS && !mbar_wait(&empty[s], ((L / kMS) - 1) & 1, P.wait)) {
            ok = false;
            break;
          }
          uint8_t* st = stages + s * kStage;
          mbar_arrive_expect_tx(&full[s], kBTile + 2 * kATx);
          tma_load_tile(st, &tmap_b, kb * kKS, row0, &full[s]);
          tma_load_tile(st + kBTile, &tmap_a, kb * kKS, r0, &full[s]);
          tma_load_tile(st + kBTile + kABlock, &tmap_a, kb * kKS, r1, &full[s]);
        }
        if (!ok) {
          abort_all();
          break;
        }
      }
    }
  } else if (warp == 1 || warp == 2) {
    // ================= MMA issue: weight block 0 from warp 1, block 1 from warp 2 =================
    if (lane == 0) {
      const int b = warp - 1;
      uint32_t L = 0;
      int t = 0;
      for (int i = blockIdx.x; i < total && !aborted(); i += gridDim.x, ++t) {
        int e, blk, mt;
        decode_tile(i, e, blk, mt);
        // N of this tile's MMAs: its tokens rounded up to 16
        const int nvalid = min(NT, P.offsets[e + 1] - P.offsets[e] - mt * NT);
        const uint32_t idesc = idesc_mx(AF == kAE2M1 ? 5 : 0, 0, 128, min(NT, (nvalid + 15) & ~15));
        if (t >= 1 && !mbar_wait(&acc_empty[b], (t - 1) & 1, P.wait)) {
          abort_all();
          break;
        }
        tm_fence_after();
        bool ok = true;
        for (int kb = 0; kb < KB; ++kb, ++L) {
          const int s = L % kMS;
          const uint32_t par = (L / kMS) & 1;
          if (!mbar_wait(&full[s], par, P.wait) || !mbar_wait(&sf_full[s], par, P.wait)) {
            ok = false;
            break;
          }
          tm_fence_after();
          const uint32_t sb = smem_u32(stages + s * kStage);
          const uint32_t sa = sb + kBTile + b * kABlock;
          const uint32_t sfa = tmem + (AF == kAE2M1 ? kSF0 + s * kSFCols + 4 * b : kSFU);
          const uint32_t sfb = tmem + kSF0 + s * kSFCols + 8;
#pragma unroll
          for (int ks = 0; ks < kKS / 32; ++ks)
            umma_mx(tmem + static_cast<uint32_t>(b * NT), desc_sw128(sa + ks * 32), desc_sw128(sb + ks * 32),
                    idesc_sf(idesc, ks, ks), sfa, sfb, (kb | ks) != 0);
          umma_commit_to(&empty[s]);
        }
        if (!ok) {
          abort_all();
          break;
        }
        umma_commit_to(acc_full);
      }
    }
  } else if (warp >= 4 && warp < 8) {
    // ================= scale factors into TMEM =================
    // The words of a stage are loaded kPF stages ahead (a register ring), so
    // the round trip of the scale loads (strided rows, from HBM on a weight
    // block's first tile) overlaps the MMAs of the stages in between.
    constexpr int kPF = 8;
    const int q = warp & 3;
    const uint32_t tl = tmem + (static_cast<uint32_t>(32 * q) << 16);
    if (AF == kAE4M3) tm_st1(tl + kSFU + q, 0x7F7F7F7Fu);  // 2^0 for every weight row and k-block
    const int ntile = static_cast<int>(blockIdx.x) < total ? (total - 1 - static_cast<int>(blockIdx.x)) / gridDim.x + 1 : 0;
    const uint32_t Ltot = static_cast<uint32_t>(ntile) * static_cast<uint32_t>(KB);
    // prefetch cursor: tile pi, k-stage pkb
    int pi = blockIdx.x, pkb = 0, p0 = 0;
    const uint8_t* wsa0 = nullptr;
    const uint8_t* wsa1 = nullptr;
    auto rebase = [&]() {
      int e, blk, mt;
      decode_tile(pi, e, blk, mt);
      p0 = P.offsets[e] + mt * NT;
      if (AF == kAE2M1) {
        const size_t r = static_cast<size_t>(wslot[e]) * P.R + 32 * q + lane;
        wsa0 = P.wscale + (r + brow(blk, 0)) * KSB;
        wsa1 = P.wscale + (r + brow(blk, 1)) * KSB;
      }
    };
    if (pi < total) rebase();
    uint32_t w[kPF][4], wa[kPF][2];
    uint32_t nan = 0;
    // one stage's words (4-byte loads; any K)
    auto load = [&](uint32_t (&wd)[4], uint32_t (&wad)[2]) {
      if (pi >= total) return;
      // token n = lane + 32 j of the tile: its 4 E8M0 bytes of this stage
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int p = p0 + lane + 32 * j;
        wd[j] = (j < NT / 32 && p < P.rows_total) ? ld_u32(P.act_scale + static_cast<size_t>(p) * KSB + 4 * pkb)
                                                  : 0x7F7F7F7Fu;
      }
      if (AF == kAE2M1) {
        wad[0] = ld_u32(wsa0 + 4 * pkb);
        wad[1] = ld_u32(wsa1 + 4 * pkb);
      }
      if (++pkb == KB) {
        pkb = 0;
        pi += gridDim.x;
        if (pi < total) rebase();
      }
    };
    // four stages' words of ring entries d0..d0+3 with one 16-byte load per
    // row (K a multiple of 512: a tile has a whole number of 4-stage groups
    // and every row's scale bytes start 16-byte aligned)
    auto load4 = [&](int d0) {
      if (pi >= total) return;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int p = p0 + lane + 32 * j;
        uint4 v = make_uint4(0x7F7F7F7Fu, 0x7F7F7F7Fu, 0x7F7F7F7Fu, 0x7F7F7F7Fu);
        if (j < NT / 32 && p < P.rows_total)
          v = __ldg(reinterpret_cast<const uint4*>(P.act_scale + static_cast<size_t>(p) * KSB + 4 * pkb));
        w[d0][j] = v.x;
        w[d0 + 1][j] = v.y;
        w[d0 + 2][j] = v.z;
        w[d0 + 3][j] = v.w;
      }
      if (AF == kAE2M1) {
        const uint4 a0 = __ldg(reinterpret_cast<const uint4*>(wsa0 + 4 * pkb));
        const uint4 a1 = __ldg(reinterpret_cast<const uint4*>(wsa1 + 4 * pkb));
        wa[d0][0] = a0.x, wa[d0 + 1][0] = a0.y, wa[d0 + 2][0] = a0.z, wa[d0 + 3][0] = a0.w;
        wa[d0][1] = a1.x, wa[d0 + 1][1] = a1.y, wa[d0 + 2][1] = a1.z, wa[d0 + 3][1] = a1.w;
      }
      pkb += 4;
      if (pkb == KB) {
        pkb = 0;
        pi += gridDim.x;
        if (pi < total) rebase();
      }
    };
    if constexpr (kVec) {
      load4(0);
      load4(4);
    } else {
#pragma unroll
      for (int d = 0; d < kPF; ++d) load(w[d], wa[d]);
    }
    bool ok = true;
    for (uint32_t L0 = 0; L0 < Ltot && ok; L0 += kPF) {
      if (__any_sync(0xffffffffu, aborted())) break;  // warp-uniform
#pragma unroll
      for (int d = 0; d < kPF; ++d) {
        const uint32_t L = L0 + d;
        if (L < Ltot && ok) {
          const int s = L % kMS;
          // one decision per warp (the tcgen05.st below are warp-collective)
          ok = __all_sync(0xffffffffu, L < kMS || mbar_wait(&empty[s], ((L / kMS) - 1) & 1, P.wait));
          if (ok) {
            tm_fence_after();  // the MMAs that read these columns are complete
            const uint32_t c0 = tl + kSF0 + s * kSFCols;
            tm_st4(c0 + 8, w[d][0], w[d][1], w[d][2], w[d][3]);
            if (AF == kAE2M1) {
              nan |= (has_ff_byte(wa[d][0]) || has_ff_byte(wa[d][1])) ? 1u : 0u;
              tm_st1(c0 + q, wa[d][0]);
              tm_st1(c0 + 4 + q, wa[d][1]);
            }
            tm_st_wait();
            tm_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&sf_full[s]);
            if constexpr (kVec) {  // a group of four consumed: its entries take the group kPF ahead
              if (d == 3) load4(0);
              if (d == 7) load4(4);
            } else {
              load(w[d], wa[d]);  // the stage kPF ahead
            }
          }
        }
      }
    }
    if (!ok) abort_all();
    if (__any_sync(0xffffffffu, nan != 0) && lane == 0) set_err(P.dev_err, MOE_DEVERR_NAN_SCALE);
  } else if (warp >= 8) {
    // ================= epilogue (8 warps: two per TMEM lane quarter) =================
    // Warps q and q + 4 of the group read lanes 32q..32q+31 (outputs) and
    // take alternate 32-token chunks.  Each warp stages its chunk (32 tokens x
    // its 32 outputs) in a private shared tile and writes it out itself with
    // 16-byte row pieces: no barrier across the epilogue warps.
    const int q = warp & 3;
    const int eh = (warp - 8) >> 2;  // chunk parity
    const uint32_t tlane = static_cast<uint32_t>(32 * q) << 16;
    const bool f32_out = P.out_fmt == MOE_FMT_F32;
    const bool mx_out = P.out_fmt == MOE_FMT_MXFP8;
    const int ob = mx_out ? 1 : 2;         // bytes per output
    uint8_t* wst = stg + (warp - 8) * 2048;  // this warp's tile: [32 tokens][32 outputs]
    int t = 0;
    for (int i = blockIdx.x; i < total; i += gridDim.x, ++t) {
      if (__any_sync(0xffffffffu, aborted())) break;  // warp-uniform
      int e, blk, mt;
      decode_tile(i, e, blk, mt);
      // one decision per warp (the tcgen05.ld below are warp-collective)
      if (!__all_sync(0xffffffffu, mbar_wait(acc_full, t & 1, P.wait))) {
        abort_all();
        break;
      }
      tm_fence_after();
      const int p0 = P.offsets[e] + mt * NT;
      const int nvalid = min(NT, P.offsets[e + 1] - p0);
      // this warp's last chunk: its accumulator reads end there
      const int nch = (nvalid + 31) / 32;
      const int last_c = (nch - 1 - eh) >= 0 ? 32 * (((nch - 1 - eh) & ~1) + eh) : -1;
      auto release = [&](int which) {  // 0 / 1: that block, 2: both
        tm_fence_before();
        __syncwarp();
        if (lane == 0) {
          if (which != 1) mbar_arrive(&acc_empty[0]);
          if (which != 0) mbar_arrive(&acc_empty[1]);
        }
      };
      if (last_c < 0) release(2);  // no chunk for this warp in this tile
      for (int half = 0; half < (fc1 ? 1 : 2); ++half) {
        const int nbase = fc1 ? blk * 128 : blk * 256 + half * 128;
        const int n0 = nbase + 32 * q;  // first output of this warp
        const int n = n0 + lane;        // this lane's output
#pragma unroll 1
        for (int c = 32 * eh; c < nvalid; c += 64) {
          uint32_t r0[32], r1[32];
          if (fc1) {
            tm_ld32(tmem + tlane + static_cast<uint32_t>(c), r0);
            tm_ld32(tmem + tlane + static_cast<uint32_t>(NT + c), r1);
          } else {
            tm_ld32(tmem + tlane + static_cast<uint32_t>(half * NT + c), r0);
          }
          tm_ld_wait();
          if (c == last_c) release(fc1 ? 2 : half);
          float v[32];
#pragma unroll
          for (int j = 0; j < 32; ++j)
            v[j] = fc1 ? silu_fast(__uint_as_float(r0[j])) * __uint_as_float(r1[j]) : __uint_as_float(r0[j]);
          if (f32_out) {
            float* o = static_cast<float*>(P.out);
#pragma unroll
            for (int j = 0; j < 32; ++j)
              if (c + j < nvalid) o[static_cast<size_t>(p0 + c + j) * P.N + n] = v[j];
            continue;
          }
          if (mx_out) {
            // MXFP8: token j's block of 32 outputs is this warp's 32 lanes.
            // Block maxima by a butterfly reduce-scatter: afterwards lane L
            // holds the maximum of token L (31 shuffles for 32 tokens).
            float a[32];
#pragma unroll
            for (int j = 0; j < 32; ++j) a[j] = fabsf(v[j]);
#pragma unroll
            for (int m = 16; m >= 1; m >>= 1) {
              const bool up = (lane & m) != 0;
#pragma unroll
              for (int j = 0; j < m; ++j) {
                const float keep = up ? a[j + m] : a[j];
                const float send = up ? a[j] : a[j + m];
                a[j] = fmaxf(keep, __shfl_xor_sync(0xffffffffu, send, m));
              }
            }
            const int X = mx_scale_exp(a[0]);  // token c + lane
            if (c + lane < nvalid)
              P.out_scale[static_cast<size_t>(p0 + c + lane) * (P.N / 32) + n0 / 32] = static_cast<uint8_t>(X + 127);
            const float inv = exp2i(-X);
#pragma unroll
            for (int j = 0; j < 32; j += 2) {
              const float i0 = __shfl_sync(0xffffffffu, inv, j), i1 = __shfl_sync(0xffffffffu, inv, j + 1);
              const uint16_t two = f32x2_to_e4m3x2(v[j] * i0, v[j + 1] * i1);
              wst[j * 32 + lane] = static_cast<uint8_t>(two & 0xffu);
              wst[(j + 1) * 32 + lane] = static_cast<uint8_t>(two >> 8);
            }
          } else {
            uint16_t* w16 = reinterpret_cast<uint16_t*>(wst);
#pragma unroll
            for (int j = 0; j < 32; j += 2) {
              uint32_t b2;
              asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(b2) : "f"(v[j + 1]), "f"(v[j]));
              w16[j * 32 + lane] = static_cast<uint16_t>(b2 & 0xffffu);
              w16[(j + 1) * 32 + lane] = static_cast<uint16_t>(b2 >> 16);
            }
          }
          __syncwarp();
          // the tile's rows (tokens) as 16-byte pieces: 32 x ob bytes per row
          if (mx_out) {
#pragma unroll 1
            for (int k2 = 0; k2 < 2; ++k2) {
              const int row = (lane >> 1) + 16 * k2, pc = lane & 1;
              if (c + row < nvalid)
                *reinterpret_cast<uint4*>(static_cast<uint8_t*>(P.out) + static_cast<size_t>(p0 + c + row) * P.N +
                                          n0 + pc * 16) = *reinterpret_cast<const uint4*>(wst + row * 32 + pc * 16);
            }
          } else {
#pragma unroll 1
            for (int k2 = 0; k2 < 4; ++k2) {
              const int row = (lane >> 2) + 8 * k2, pc = lane & 3;
              if (c + row < nvalid)
                *reinterpret_cast<uint4*>(static_cast<uint16_t*>(P.out) + static_cast<size_t>(p0 + c + row) * P.N +
                                          n0 + pc * 8) = *reinterpret_cast<const uint4*>(wst + row * 64 + pc * 16);
            }
          }
          __syncwarp();  // the tile is free for the next chunk
        }
      }
    }
  }

  // ---- teardown: every role is done (or gave up); free TMEM
  tm_fence_before();
  __syncthreads();
  if (warp == 3) {
    tm_fence_after();
    tm_dealloc(tmem, kCols);
  }
}

template <int AF, int NT>
cudaError_t launch_mx_t(const CUtensorMap& mb, const CUtensorMap& ma, const MxParams& P, cudaStream_t s) {
  const size_t smem = mx_smem_bytes<NT>();
  if (P.K % 512 == 0 && reinterpret_cast<uintptr_t>(P.act_scale) % 16 == 0) {  // 16-byte scale loads
    cudaError_t e = set_smem_limit(mx_mm_kernel<AF, NT, true>, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    return launch_pdl(mx_mm_kernel<AF, NT, true>, dim3(matmul_ctas()), dim3(kMxThreads), smem, s, mb, ma, P);
  }
  cudaError_t e = set_smem_limit(mx_mm_kernel<AF, NT, false>, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  return launch_pdl(mx_mm_kernel<AF, NT, false>, dim3(matmul_ctas()), dim3(kMxThreads), smem, s, mb, ma, P);
}

}  // namespace

bool mx_mm_supported(const MMArgs& a) {
  if (a.act_fmt != MOE_FMT_MXFP8 || !a.act_scale || a.act_row != nullptr || a.E > 1024) return false;
  if (a.wkind != kFP8 && a.wkind != kMXFP4) return false;
  if (a.wkind == kFP8 && a.wslot_of == nullptr) return false;
  if (a.wkind == kMXFP4 && !(a.select == 0 || a.select == 2)) return false;
  if (a.K % kKS) return false;
  if (a.stage == MOE_STAGE_FC1_SWIGLU ? a.N % 128 : a.N % 256) return false;
  if (a.out_fmt == MOE_FMT_F32 || a.out_fmt == MOE_FMT_BF16) return true;
  return a.out_fmt == MOE_FMT_MXFP8 && a.stage == MOE_STAGE_FC1_SWIGLU && a.out_scale != nullptr;
}

cudaError_t launch_mx_mm(const MMArgs& a, int rows_total, cudaStream_t s) {
  EncodeFn enc = encode_fn();
  if (!enc) return cudaErrorNotSupported;
  MxParams P;
  P.act_scale = a.act_scale;
  P.rows_total = rows_total;
  P.wscale = static_cast<const uint8_t*>(a.wscale);
  P.wslot_of = a.wslot_of;
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
  P.out_scale = a.out_scale;
  P.dev_err = a.dev_err;
  P.wait = a.wait;
  // token tile: 128 rows for prefill-sized groups, 32 for decode-sized ones
  const int NT = rows_total <= 16 * a.E ? 32 : 128;
  const cuuint32_t estr[2] = {1, 1};
  // tokens: E4M3 [rows_total][K], box 128 bytes x NT rows, 128-byte swizzle
  CUtensorMap mb, ma;
  {
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(a.K), static_cast<cuuint64_t>(rows_total > 0 ? rows_total : 1)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(a.K)};
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(kKS), static_cast<cuuint32_t>(NT)};
    if (enc(&mb, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(a.act), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  // weights: [E slots x R rows][K], box 128 K elements x 128 rows, 128-byte
  // swizzle; E2M1 codes (packed two per byte) land as 16 codes + 8 pad bytes
  // per 16 shared bytes, the MMA's form of 4-bit operands
  {
    const bool fp4 = a.wkind == kMXFP4;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(a.K), static_cast<cuuint64_t>(a.E) * P.R};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(fp4 ? a.K / 2 : a.K)};
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(kKS), 128};
    if (enc(&ma, fp4 ? CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B : CU_TENSOR_MAP_DATA_TYPE_UINT8, 2,
            const_cast<uint8_t*>(a.wq), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  if (a.wkind == kMXFP4)
    return NT == 32 ? launch_mx_t<kAE2M1, 32>(mb, ma, P, s) : launch_mx_t<kAE2M1, 128>(mb, ma, P, s);
  return NT == 32 ? launch_mx_t<kAE4M3, 32>(mb, ma, P, s) : launch_mx_t<kAE4M3, 128>(mb, ma, P, s);
}

}  // namespace moe
