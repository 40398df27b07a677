// Decode GEMV for 2-bit codebook experts by shared-memory partial-sum tables.
//
// A code byte holds 4 consecutive weights of a row, each one of the four
// codebook entries {-4,-1,1,4}.  For a fixed token x and a fixed byte
// position p of the row (elements 4p..4p+3), the contribution of that byte to
// a row's dot product is one of 256 values
//     T_p[b] = sum_{i<4} entry(code_i(b)) * x[4p+i],
// the same for every row.  The kernel builds these tables once per (expert,
// token, K slice) and then streams the weight rows, turning every code byte
// into one table lookup: a PRMT forms the shared-memory address straight from
// the byte, an LDS fetches T_p[b], an FADD accumulates.  That is one integer
// op per 4 weights where a register decode needs at least four, which keeps
// the kernel off the integer-pipe ceiling.
//
// Tables: 128 byte positions (a K slice of 512 elements) x 256 entries x fp32
// = 128 KB, lane-interleaved so that the 32 lanes of a warp, each looking up
// its own byte position, hit 32 different banks.  The table sits at a 64 KB
// aligned shared-window address so that byte 1 of every lookup address is
// free for the code byte (one PRMT builds the address).
//
// Work: items (expert e, token t, K slice s, block of RPI weight rows) are
// split into contiguous ranges, one per CTA (all SMs, no clusters).  Per
// item a producer thread streams the rows' slice codes + scales into a ring
// of shared-memory stages (one contiguous bulk copy per 32-row stage in the
// w2l layout); 8 consumer warps look the bytes up, transpose their per-lane
// partials through a small tile and write per-row slice sums to a global
// scratch; an epilogue warp counts the slices of a row block with one atomic
// and, in the CTA that completes it, sums the NSL slices in slice order
// (deterministic), applies SwiGLU for FC1, rounds and stores.  No CTA ever
// waits on another.
//
// Every mbarrier wait is bounded; a timeout sets MOE_DEVERR_TIMEOUT.
#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"
#include "internal.cuh"

namespace moe {

namespace {

constexpr int kLutWarps = 8;                      // consumer warps
constexpr int kLutConsumers = kLutWarps * 32;
constexpr int kLutThreads = kLutConsumers + 64;   // + producer warp + epilogue warp
constexpr int kStageRows = 32;                    // weight rows per ring stage (8 row quads)
constexpr int kMaxStages = 16;
constexpr int kBufs = 8;                          // items the epilogue warp may lag behind
constexpr int kTableBytes = 2 * 256 * 256;        // [j>>1][b][64 slots] fp32
constexpr int kTileBytes = kLutWarps * 32 * 33 * 4;  // per-warp [32 rows][33] transpose tiles
constexpr int kLutSmem = 65536 + kTableBytes + kTileBytes;

struct LutParams {
  const uint16_t* act;
  const int32_t* act_row;
  int act_row_div;
  int act_rows;
  const uint8_t* codes;     // w2l words
  const uint16_t* scales;   // w2l bf16 scales
  const int32_t* select_map;
  int select;
  const int32_t* offsets;
  int E, N, K, R;           // R = weight rows per expert
  int SW, NSL, NLn;         // slice width, slices, active lanes per slice
  int fc1;
  int rpi;                  // weight rows per item (128 or 256)
  int* counters;            // [A][NB] slice arrivals per (row p, block), zero between calls
  float* scratch;           // [A][NB][NSL][RPI] per-slice row sums
  int A;                    // permuted rows the workspace covers
  void* out;
  int out_fmt;
  uint32_t* dev_err;
};

// table address of (byte-in-word j, code byte b, lane l) relative to the table base
MOE_D uint32_t tab_off(int j, uint32_t b, int l) {
  return static_cast<uint32_t>((j >> 1) * 65536 + b * 256 + (j & 1) * 128 + l * 4);
}

// Sum of the four table lookups for one code word (lanebase = table window
// address + 4 * lane, whose byte 1 is zero).
MOE_D float word_sum(uint32_t w, uint32_t lanebase) {
  uint32_t a0, a1, a2, a3;
  asm("prmt.b32 %0, %1, %2, 0x7604;" : "=r"(a0) : "r"(w), "r"(lanebase));
  asm("prmt.b32 %0, %1, %2, 0x7614;" : "=r"(a1) : "r"(w), "r"(lanebase));
  asm("prmt.b32 %0, %1, %2, 0x7624;" : "=r"(a2) : "r"(w), "r"(lanebase));
  asm("prmt.b32 %0, %1, %2, 0x7634;" : "=r"(a3) : "r"(w), "r"(lanebase));
  // plain loads: the tables are fenced by the barrier after they are built
  float t0, t1, t2, t3;
  asm("ld.shared.f32 %0, [%1];" : "=f"(t0) : "r"(a0));
  asm("ld.shared.f32 %0, [%1+128];" : "=f"(t1) : "r"(a1));
  asm("ld.shared.f32 %0, [%1+65536];" : "=f"(t2) : "r"(a2));
  asm("ld.shared.f32 %0, [%1+65664];" : "=f"(t3) : "r"(a3));
  return (t0 + t1) + (t2 + t3);
}

template <int RPI>
__global__ void __launch_bounds__(kLutThreads, 1) w2_lut_kernel(const LutParams P) {
  constexpr int NST = RPI / kStageRows;  // stages per item
  constexpr int V = RPI / 8;             // rows per consumer warp per item (one quad per stage)
  extern __shared__ __align__(1024) uint8_t smem[];
  __shared__ int s_last;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int SW = P.SW, NLn = P.NLn, NSL = P.NSL;
  const int G = SW / 32;                           // scale groups per slice row
  const int codes_stage = kStageRows * SW / 4;     // bytes
  const int scales_stage = kStageRows * G * 2;     // bytes
  const int stage_bytes = codes_stage + scales_stage;

  // ---- shared memory: [barriers][flags][item_start][ring ...][table @ 64K-aligned][tiles]
  const uint32_t base = smem_u32(smem);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem);   // [kMaxStages]
  uint64_t* empty = full + kMaxStages;                   // [kMaxStages]
  uint64_t* pub_bar = empty + kMaxStages;                // [kBufs] 8 consumer warps wrote item it
  uint64_t* free_bar = pub_bar + kBufs;                  // [kBufs] epilogue warp finished item it
  int* flags = reinterpret_cast<int*>(smem + 512);       // [0] abort
  int* item_start = flags + 32;                          // [E+1]
  const uint32_t pre = 512 + 128 + ((4u * (P.E + 1) + 127u) & ~127u);
  const uint32_t table_win = (base + pre + 65535u) & ~65535u;
  int stages = static_cast<int>((table_win - base - pre) / stage_bytes);
  stages = stages > kMaxStages ? kMaxStages : stages;
  uint8_t* ring = smem + pre;
  const uint32_t table_off = table_win - base;

  const bool fc1 = P.fc1 != 0;
  const int outs_item = fc1 ? RPI / 2 : RPI;  // outputs per row block
  const int NB = P.N / outs_item;
  const int per_tok = NSL * NB;               // items per (expert, token)

  if (warp == 0) {  // item_start[e] = items of the selected experts before e
    int run = 0;
    for (int b0 = 0; b0 <= P.E; b0 += 32) {
      const int e = b0 + lane;
      int n = 0;
      if (e < P.E) {
        const int c = P.offsets[e + 1] - P.offsets[e];
        bool sel = c > 0;
        if (sel && P.select == 1) sel = P.select_map[e] < 0;
        if (sel && P.select == 2) sel = P.select_map[e] >= 0;
        if (sel) n = c * per_tok;
      }
      int incl = n;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      if (e <= P.E) item_start[e] = run + incl - n;
      run += __shfl_sync(0xffffffffu, incl, 31);
    }
  }
  if (tid == 0) {
    for (int s = 0; s < kMaxStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kLutWarps);
    }
    for (int b = 0; b < kBufs; ++b) {
      mbar_init(&pub_bar[b], kLutWarps);
      mbar_init(&free_bar[b], 1);
    }
    flags[0] = 0;
    fence_barrier_init();
  }
  __syncthreads();

  // ---- this CTA's contiguous item range; item = (e, t, slice, rb), rb fastest
  const int total = item_start[P.E];
  const int per = (total + gridDim.x - 1) / gridDim.x;
  const int i_beg = min(total, static_cast<int>(blockIdx.x) * per), i_end = min(total, i_beg + per);
  auto decode = [&](int i, int& e, int& t, int& sl, int& rb) {
    int lo = 0, hi = P.E;  // largest e with item_start[e] <= i
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (item_start[mid] <= i) lo = mid; else hi = mid;
    }
    e = lo;
    int loc = i - item_start[e];
    t = loc / per_tok;
    loc -= t * per_tok;
    sl = loc / NB;
    rb = loc - sl * NB;
  };
  auto abort_all = [&]() {
    flags[0] = 1;
    set_err(P.dev_err, MOE_DEVERR_TIMEOUT);
  };
  auto aborted = [&]() { return *reinterpret_cast<volatile int*>(&flags[0]) != 0; };

  // stages are issued in groups of 4, one per producer lane: a multiple of 4 ring slots
  const int S = stages & ~3;

  if (warp == kLutWarps) {
    // ================= producer: lanes 0..3 each issue one 32-row stage of a group of 4 =================
    if (lane < 4 && i_beg < i_end) {
      const int64_t mat_bytes = static_cast<int64_t>(P.R) * (P.K / 4);  // codes bytes per expert
      const int64_t mat_scales = static_cast<int64_t>(P.R) * (P.K / 32);
      const int64_t slice_codes = static_cast<int64_t>(P.R) * SW / 4;
      const int64_t slice_scales = static_cast<int64_t>(P.R) * G;
      const int nstages = (i_end - i_beg) * NST;
      int s0 = 0;
      uint32_t ph = 0;
      bool ok = true;
      int issued = 0;
      for (int L0 = 0; L0 < nstages && ok; L0 += 4) {
        const int L = L0 + lane;
        if (L < nstages) {
          const int i = i_beg + L / NST, st = L % NST;
          int e, t, sl, rb;
          decode(i, e, t, sl, rb);
          int row0;
          if (fc1) row0 = (st < NST / 2) ? rb * (RPI / 2) + st * kStageRows : P.N + rb * (RPI / 2) + (st - NST / 2) * kStageRows;
          else row0 = rb * RPI + st * kStageRows;
          const int slot = s0 + lane;
          if (L >= S && !mbar_wait(&empty[slot], ph ^ 1u)) {
            abort_all();
            ok = false;
          } else if (aborted()) {
            ok = false;
          } else {
            const uint8_t* gc = P.codes + e * mat_bytes + sl * slice_codes + static_cast<int64_t>(row0 / 4) * SW;
            const uint8_t* gs = reinterpret_cast<const uint8_t*>(P.scales + e * mat_scales + sl * slice_scales +
                                                                 static_cast<int64_t>(row0 / 4) * (G * 4));
            uint8_t* d = ring + static_cast<size_t>(slot) * stage_bytes;
            mbar_arrive_expect_tx(&full[slot], stage_bytes);
            bulk_g2s(d, gc, codes_stage, &full[slot]);
            bulk_g2s(d + codes_stage, gs, scales_stage, &full[slot]);
            issued = L + 1;
          }
        }
        ok = __all_sync(0x0000000fu, ok);
        s0 += 4;
        if (s0 == S) {
          s0 = 0;
          ph ^= 1u;
        }
      }
      if (!ok) {  // this lane's copies already issued complete (bounded) before the CTA may leave
        for (int l = lane; l < issued; l += 4)
          if (l + S >= issued) (void)mbar_wait(&full[l % S], (l / S) & 1);
      }
    }
    return;
  }

  if (warp == kLutWarps + 1) {
    // ================= epilogue: slice counting, final sums, SwiGLU =================
    for (int i = i_beg, it = 0; i < i_end; ++i, ++it) {
      int e, t, sl, rb;
      decode(i, e, t, sl, rb);
      const int b = it % kBufs;
      if (!mbar_wait(&pub_bar[b], (it / kBufs) & 1)) {
        abort_all();
        break;
      }
      const int p = P.offsets[e] + t;
      if (p >= P.A) {  // reported by the consumers; nothing was written for it
        __syncwarp();
        if (lane == 0) mbar_arrive(&free_bar[b]);
        continue;
      }
      int* cnt = P.counters + static_cast<size_t>(p) * NB + rb;
      if (lane == 0) {
        // release: this CTA's slice sums (published to this warp through pub_bar)
        // precede the count; acquire: the other slices' sums precede reading them
        int old;
        asm volatile("atom.add.acq_rel.gpu.s32 %0, [%1], 1;" : "=r"(old) : "l"(cnt) : "memory");
        s_last = (old == NSL - 1);
      }
      __syncwarp();
      const bool last = *reinterpret_cast<volatile int*>(&s_last) != 0;
      if (last) {
        const float* sc = P.scratch + (static_cast<size_t>(p) * NB + rb) * NSL * RPI;
        for (int o = lane; o < outs_item; o += 32) {
          float v = 0.f, u = 0.f;
          for (int q = 0; q < NSL; ++q) {
            v += __ldcg(sc + q * RPI + o);
            if (fc1) u += __ldcg(sc + q * RPI + RPI / 2 + o);
          }
          if (fc1) v = silu_f32(v) * u;
          const int n = rb * outs_item + o;
          if (P.out_fmt == MOE_FMT_F32) static_cast<float*>(P.out)[static_cast<size_t>(p) * P.N + n] = v;
          else static_cast<uint16_t*>(P.out)[static_cast<size_t>(p) * P.N + n] = f32_to_bf16_rne(v);
        }
        __syncwarp();
        if (lane == 0) *cnt = 0;  // leave the counters zero for the next call
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&free_bar[b]);
    }
    return;
  }

  // ================= consumers: table lookups over the streamed stages =================
  const uint32_t lanebase = table_win + 4u * static_cast<uint32_t>(lane);
  float* table_f = reinterpret_cast<float*>(smem + table_off);
  float* tile = reinterpret_cast<float*>(smem + table_off + kTableBytes) + warp * (32 * 33);  // [32 rows][33]
  int key_e = -1, key_t = -1, key_s = -1;
  int s = 0;
  uint32_t ph = 0;
  bool failed = false;
  for (int i = i_beg, it = 0; i < i_end; ++i, ++it) {
    int e, t, sl, rb;
    decode(i, e, t, sl, rb);
    int p = P.offsets[e] + t;
    if (p >= P.A) {  // workspace too small for this many rows: report, compute into row 0's slot? no: skip writes
      if (tid == 0) set_err(P.dev_err, MOE_DEVERR_OVERFLOW);
      p = -1;
    }
    if (e != key_e || t != key_t || sl != key_s) {
      // ---- (re)build the partial-sum tables of slice sl for the item's token
      if (named_bar_or(1, kLutConsumers, failed || aborted())) break;  // nobody still reads the old tables
      int row = p < 0 ? 0 : (P.act_row ? P.act_row[p] / P.act_row_div : p);
      if (row < 0 || row >= P.act_rows) {
        if (tid == 0) set_err(P.dev_err, MOE_DEVERR_BAD_ID);
        row = 0;
      }
      const int j = warp & 3, hhalf = warp >> 2;
      if (lane < NLn) {
        const uint2 xv =
            *reinterpret_cast<const uint2*>(P.act + static_cast<size_t>(row) * P.K + sl * SW + 16 * lane + 4 * j);
        const float x0 = __uint_as_float(xv.x << 16), x1 = __uint_as_float(xv.x & 0xffff0000u);
        const float x2 = __uint_as_float(xv.y << 16), x3 = __uint_as_float(xv.y & 0xffff0000u);
        const float cb[4] = {-4.f, -1.f, 1.f, 4.f};
        float plo[16], phi[8];
#pragma unroll
        for (int c1 = 0; c1 < 4; ++c1)
#pragma unroll
          for (int c0 = 0; c0 < 4; ++c0) plo[c0 + 4 * c1] = fmaf(cb[c1], x1, cb[c0] * x0);
#pragma unroll
        for (int h = 0; h < 8; ++h) {  // hi = 8*hhalf + h: code2 = h & 3, code3 = 2*hhalf + (h >> 2)
          const float c3 = hhalf ? cb[2 + (h >> 2)] : cb[h >> 2];
          phi[h] = fmaf(c3, x3, cb[h & 3] * x2);
        }
#pragma unroll
        for (int h = 0; h < 8; ++h) {
          const uint32_t hi = 8 * hhalf + h;
#pragma unroll
          for (int lo = 0; lo < 16; ++lo) table_f[tab_off(j, hi * 16 + lo, lane) / 4] = plo[lo] + phi[h];
        }
      }
      named_bar_sync(1, kLutConsumers);
      key_e = e;
      key_t = t;
      key_s = sl;
    }
    // ---- stream the item's stages: warp w takes row quad w of each stage; a
    // lane's partial of item row (32*st + 4*w + r) goes to tile[4*st + r][lane]
#pragma unroll
    for (int st = 0; st < NST; ++st) {
      if (!failed && !mbar_wait(&full[s], ph)) failed = true;
      const uint8_t* d = ring + static_cast<size_t>(s) * stage_bytes;
      float r4[4] = {0.f, 0.f, 0.f, 0.f};
      if (!failed && lane < NLn) {
        const uint4 w4 = *reinterpret_cast<const uint4*>(d + (warp * NLn + lane) * 16);
        const uint2 s4 = *reinterpret_cast<const uint2*>(d + codes_stage + (warp * G + (lane >> 1)) * 8);
        r4[0] = word_sum(w4.x, lanebase) * __uint_as_float(s4.x << 16);
        r4[1] = word_sum(w4.y, lanebase) * __uint_as_float(s4.x & 0xffff0000u);
        r4[2] = word_sum(w4.z, lanebase) * __uint_as_float(s4.y << 16);
        r4[3] = word_sum(w4.w, lanebase) * __uint_as_float(s4.y & 0xffff0000u);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
#pragma unroll
      for (int r = 0; r < 4; ++r) tile[(st * 4 + r) * 33 + lane] = r4[r];
      if (++s == S) {
        s = 0;
        ph ^= 1u;
      }
    }
    if (failed) {
      abort_all();
      break;
    }
    // ---- row sums: lane v adds up tile row v (its 32 lanes' partials)
    __syncwarp();
    float sum = 0.f;
    if (lane < V) {
      float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
#pragma unroll
      for (int c = 0; c < 32; c += 4) {
        a0 += tile[lane * 33 + c];
        a1 += tile[lane * 33 + c + 1];
        a2 += tile[lane * 33 + c + 2];
        a3 += tile[lane * 33 + c + 3];
      }
      sum = (a0 + a1) + (a2 + a3);
    }
    __syncwarp();
    // ---- slice sums to the scratch; hand the item to the epilogue warp
    const int b = it % kBufs;
    if (it >= kBufs && !mbar_wait(&free_bar[b], ((it / kBufs) - 1) & 1)) {
      abort_all();
      break;
    }
    if (lane < V && p >= 0) {
      const int row = (lane >> 2) * kStageRows + warp * 4 + (lane & 3);
      P.scratch[((static_cast<size_t>(p) * NB + rb) * NSL + sl) * RPI + row] = sum;
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&pub_bar[b]);
  }
}

}  // namespace

// Scratch of the LUT GEMV: slice-arrival counters [rows][NB] (ints, zero
// between calls) then per-slice row sums [rows][NB][NSL][RPI] (fp32).
static void lut_geometry(int stage, int N, int K, int& rpi, int& nb, int& nsl) {
  const bool fc1 = stage == MOE_STAGE_FC1_SWIGLU;
  rpi = (fc1 || N % 256 == 0) ? 256 : 128;
  nb = N / (fc1 ? rpi / 2 : rpi);
  nsl = K / w2l_sw(K);
}

size_t lut_workspace_bytes(int stage, int rows, int N, int K) {
  int rpi, nb, nsl;
  lut_geometry(stage, N, K, rpi, nb, nsl);
  const size_t cnt = (static_cast<size_t>(rows) * nb * sizeof(int) + 255) & ~size_t(255);
  return cnt + static_cast<size_t>(rows) * nb * nsl * rpi * sizeof(float);
}

size_t lut_counter_bytes(int stage, int rows, int N, int K) {
  int rpi, nb, nsl;
  lut_geometry(stage, N, K, rpi, nb, nsl);
  return (static_cast<size_t>(rows) * nb * sizeof(int) + 255) & ~size_t(255);
}

int lut_workspace_rows(int stage, size_t bytes, int N, int K) {
  int rpi, nb, nsl;
  lut_geometry(stage, N, K, rpi, nb, nsl);
  const size_t per = static_cast<size_t>(nb) * sizeof(int) + static_cast<size_t>(nb) * nsl * rpi * sizeof(float);
  int64_t rows = static_cast<int64_t>(bytes / per);
  while (rows > 0 && lut_workspace_bytes(stage, static_cast<int>(rows), N, K) > bytes) --rows;
  return rows > 0x7fffffff ? 0x7fffffff : static_cast<int>(rows);
}

bool lut_supported(const MMArgs& a) {
  if (a.wkind != kW2 || a.act_fmt != MOE_FMT_BF16 || a.out_fmt == MOE_FMT_MXFP8) return false;
  if (a.expert_begin != 0 || a.expert_end != a.E) return false;
  const int SW = w2l_sw(a.K);
  return a.K % SW == 0 && SW % 128 == 0;
}

cudaError_t launch_lut_gemv(const MMArgs& a, void* ws, cudaStream_t s) {
  LutParams P;
  P.act = static_cast<const uint16_t*>(a.act);
  P.act_row = a.act_row;
  P.act_row_div = a.act_row_div;
  P.act_rows = a.act_rows;
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
  P.SW = w2l_sw(a.K);
  P.NSL = a.K / P.SW;
  P.NLn = P.SW / 16;
  int nb, nsl;
  lut_geometry(a.stage, a.N, a.K, P.rpi, nb, nsl);
  P.A = a.ws_rows;
  const size_t cnt = (static_cast<size_t>(a.ws_rows) * nb * sizeof(int) + 255) & ~size_t(255);
  P.counters = static_cast<int*>(ws);
  P.scratch = reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + cnt);
  P.out = a.out;
  P.out_fmt = a.out_fmt;
  P.dev_err = a.dev_err;
  auto kern = P.rpi == 256 ? w2_lut_kernel<256> : w2_lut_kernel<128>;
  static bool attr_done[2] = {false, false};
  if (!attr_done[P.rpi == 256]) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kLutSmem);
    if (e != cudaSuccess) return e;
    attr_done[P.rpi == 256] = true;
  }
  kern<<<device_info().sms, kLutThreads, kLutSmem, s>>>(P);
  return cudaGetLastError();
}

}  // namespace moe
