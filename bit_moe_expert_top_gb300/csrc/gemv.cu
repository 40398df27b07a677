// Grouped expert matmul on CUDA cores: the decode path (few tokens per
// expert, bound by streaming the packed weights from HBM), and the path that
// serves any group size correctly.
//
// Work decomposition: an item is (expert e, block of 32 outputs, range of up
// to kTR permuted rows of the group).  FC1 items read 32 gate + 32 up weight
// rows, FC2 items 32 rows.  A persistent grid walks the item list, which
// every CTA derives from `offsets` on the device (no host sync).
//
// Data movement: one producer thread streams row blocks of the packed weights
// (codes + scales) into a ring of shared-memory stages with 1-D bulk async
// copies completing on mbarriers; 256 consumer threads decode in registers.
// Consumer thread (rho, g) owns the 32-element group g of K for rows rho,
// rho+P, ...; its activations for that group stay in registers for the whole
// stage, so each weight is decoded once and applied to kNT tokens at a time
// with packed fp32x2 FMAs.  Partial dot products of a row are summed across
// the G = K/32 threads through a padded shared-memory tile, in a fixed order.
#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"
#include "internal.cuh"

namespace moe {

namespace {

constexpr int kConsumers = 256;
constexpr int kThreads = kConsumers + 32;
constexpr int kTR = 64;      // permuted rows (tokens) per item
constexpr int kNT = 2;       // tokens per register pass
constexpr int kOutBlk = 32;  // outputs per item

struct GemvParams {
  MMArgs a;
  int rows_total;   // weight rows per expert (2N for FC1, N for FC2)
  int qrow_bytes;   // packed bytes per weight row
  int srow_bytes;   // scale bytes per weight row
  int stages;       // ring depth
  int stage_bytes;  // bytes per ring stage (q + s, 128-aligned parts)
  int sq_bytes;     // q part of a stage
};

template <int WK>
struct WTraits;
template <>
struct WTraits<kW2> {
  static constexpr int kRS = 16;  // weight rows per stage
};
template <>
struct WTraits<kMXFP4> {
  static constexpr int kRS = 16;
};
template <>
struct WTraits<kFP8> {
  static constexpr int kRS = 8;
};

MOE_HD int round_up(int x, int m) { return (x + m - 1) / m * m; }

constexpr int kResPitch = kTR + 1;  // padded: the epilogue reads columns

// Dynamic shared-memory layout, computed identically on host and device.
struct SmemLayout {
  int bars, ring, red, red2, res, items, total;
};
MOE_HD SmemLayout smem_layout(int stages, int stage_bytes, int G, int V, int E) {
  SmemLayout l;
  l.bars = 0;
  l.ring = round_up(2 * stages * 8, 128);
  l.red = l.ring + stages * stage_bytes;
  l.red2 = l.red + round_up(G * (V + 1) * 4, 16);
  l.res = l.red2 + round_up(4 * V * 4, 16);
  l.items = l.res + round_up(2 * kOutBlk * kResPitch * 4, 16);
  l.total = l.items + round_up((E + 1) * 4, 16);
  return l;
}

// Codebook entry of a canonical 2-bit code (ascending {-4,-1,1,4}), built
// from its bits: |entry| = 4 when both bits agree, entry < 0 when bit 1 is 0.
MOE_D float w2_entry(uint32_t c) {
  const uint32_t big = ((c ^ (c >> 1)) & 1u) ^ 1u;
  const uint32_t neg = ((c >> 1) & 1u) ^ 1u;
  return __uint_as_float(0x3F800000u + (big << 24) | (neg << 31));
}

// The two entries of elements 2q, 2q+1 of a canonical code word.
MOE_D float2 w2_pair(uint32_t w, int q) {
  return make_float2(w2_entry(w >> (4 * q)), w2_entry(w >> (4 * q + 2)));
}

// Activations of one 32-element group for one token, as 16 fp32 pairs.
template <int AF>
MOE_D void load_act(const GemvParams& P, int row, int g, float2 (&x)[16]) {
  const int K = P.a.K;
  if (AF == MOE_FMT_BF16) {
    const uint4* src = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(P.a.act) +
                                                      static_cast<size_t>(row) * K + g * 32);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      uint4 v = __ldg(src + i);
      const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) x[i * 4 + j] = make_float2(__uint_as_float(wv[j] << 16), __uint_as_float(wv[j] & 0xffff0000u));
    }
  } else {  // MXFP8
    const uint4* src = reinterpret_cast<const uint4*>(static_cast<const uint8_t*>(P.a.act) +
                                                      static_cast<size_t>(row) * K + g * 32);
    const float sc = exp2i(static_cast<int>(__ldg(P.a.act_scale + static_cast<size_t>(row) * (K / 32) + g)) - 127);
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      uint4 v = __ldg(src + i);
      const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        float2 lo = e4m3x2_to_f32x2(static_cast<uint16_t>(wv[j] & 0xffffu));
        float2 hi = e4m3x2_to_f32x2(static_cast<uint16_t>(wv[j] >> 16));
        x[i * 8 + j * 2] = make_float2(lo.x * sc, lo.y * sc);
        x[i * 8 + j * 2 + 1] = make_float2(hi.x * sc, hi.y * sc);
      }
    }
  }
}

// Dot products of one weight-row group with kNT token groups.  Returns the
// per-token sums including the group scale.
template <int WK>
MOE_D void row_group_dot(const uint8_t* sq, const uint8_t* ss, int rr, int g, int G, const GemvParams& P,
                         const float2 (&x)[kNT][16], float (&part)[kNT], uint32_t& nan_scale) {
  float2 acc[kNT];
#pragma unroll
  for (int t = 0; t < kNT; ++t) acc[t] = make_float2(0.f, 0.f);
  float sc;
  if (WK == kW2) {
    // w2l stage layout: [slice][row quad][lane][4 rows] words, [slice][row quad][group][4 rows] scales
    const int SW = w2l_sw(P.a.K), NLn = SW / 16, Gs = SW / 32, nq = WTraits<kW2>::kRS / 4;
    const int sl = g / Gs, gs = g % Gs, q = rr >> 2, r = rr & 3;
    const uint8_t* wb = sq + ((static_cast<size_t>(sl) * nq + q) * NLn + 2 * gs) * 16 + r * 4;
    const uint2 wv = make_uint2(*reinterpret_cast<const uint32_t*>(wb), *reinterpret_cast<const uint32_t*>(wb + 16));
    sc = bf16_bits_to_f32(
        *reinterpret_cast<const uint16_t*>(ss + ((static_cast<size_t>(sl) * nq + q) * Gs + gs) * 8 + r * 2));
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const uint32_t w = h ? wv.y : wv.x;
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const float2 v = w2_pair(w, q);
#pragma unroll
        for (int t = 0; t < kNT; ++t) acc[t] = ffma2(v, x[t][h * 8 + q], acc[t]);
      }
    }
  } else if (WK == kMXFP4) {
    const uint4 wv = *reinterpret_cast<const uint4*>(sq + static_cast<size_t>(rr) * P.qrow_bytes + g * 16);
    const uint32_t b = ss[static_cast<size_t>(rr) * G + g];
    if (b == 255u) nan_scale = 1u;
    sc = (b == 255u) ? __uint_as_float(0x7fc00000u) : exp2i(static_cast<int>(b) - 127);
    const uint32_t ws[4] = {wv.x, wv.y, wv.z, wv.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float2 v = e2m1x2_to_f32x2((ws[i] >> (8 * j)) & 0xffu);
#pragma unroll
        for (int t = 0; t < kNT; ++t) acc[t] = ffma2(v, x[t][i * 4 + j], acc[t]);
      }
    }
  } else {  // FP8 workspace, scale folded into the bytes
    const uint4* p = reinterpret_cast<const uint4*>(sq + static_cast<size_t>(rr) * P.qrow_bytes + g * 32);
    sc = 1.0f;
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const uint4 wv = p[i];
      const uint32_t ws[4] = {wv.x, wv.y, wv.z, wv.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float2 lo = e4m3x2_to_f32x2(static_cast<uint16_t>(ws[j] & 0xffffu));
        const float2 hi = e4m3x2_to_f32x2(static_cast<uint16_t>(ws[j] >> 16));
#pragma unroll
        for (int t = 0; t < kNT; ++t) {
          acc[t] = ffma2(lo, x[t][i * 8 + j * 2], acc[t]);
          acc[t] = ffma2(hi, x[t][i * 8 + j * 2 + 1], acc[t]);
        }
      }
    }
  }
#pragma unroll
  for (int t = 0; t < kNT; ++t) part[t] = (acc[t].x + acc[t].y) * sc;
}

template <int WK, int AF>
__global__ void __launch_bounds__(kThreads, 1) gemv_kernel(const GemvParams P) {
  constexpr int RS = WTraits<WK>::kRS;
  constexpr int V = RS * kNT;  // partial sums per (stage, chunk)
  const MMArgs& a = P.a;
  const int K = a.K, N = a.N, E = a.E;
  const int G = K / 32;
  const bool fc1 = a.stage == MOE_STAGE_FC1_SWIGLU;
  const int nst = (fc1 ? 2 * kOutBlk : kOutBlk) / RS;  // stages per item
  const int NB = N / kOutBlk;

  extern __shared__ __align__(128) uint8_t smem[];
  const SmemLayout lay = smem_layout(P.stages, P.stage_bytes, G, V, E);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + lay.bars);
  uint64_t* empty = full + P.stages;
  uint8_t* ring = smem + lay.ring;
  float* red = reinterpret_cast<float*>(smem + lay.red);    // [G][V+1]
  float* red2 = reinterpret_cast<float*>(smem + lay.red2);  // [4][V]
  float* res = reinterpret_cast<float*>(smem + lay.res);    // [2*kOutBlk][kResPitch]
  int* item_start = reinterpret_cast<int*>(smem + lay.items);  // [E+1]
  __shared__ int s_abort;

  const int tid = threadIdx.x;
  // ---- item list (every thread of the CTA derives the same one)
  if (tid < 32) {
    int run = 0;
    for (int base = 0; base <= E; base += 32) {
      const int e = base + tid;
      int n = 0;
      if (e < E && e >= a.expert_begin && e < a.expert_end) {
        const int c = a.offsets[e + 1] - a.offsets[e];
        bool sel = c > 0;
        if (sel && a.select == 1) sel = a.select_map[e] < 0;
        if (sel && a.select == 2) sel = a.select_map[e] >= 0;
        if (sel) n = ((c + kTR - 1) / kTR) * NB;
      }
      int incl = n;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        int t = __shfl_up_sync(0xffffffffu, incl, o);
        if (tid >= o) incl += t;
      }
      if (e <= E) item_start[e] = run + incl - n;
      run += __shfl_sync(0xffffffffu, incl, 31);
    }
  }
  if (tid == 0) {
    s_abort = 0;
    for (int s = 0; s < P.stages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kConsumers / 32);
    }
    fence_barrier_init();
  }
  __syncthreads();
  const int total = item_start[E];

  auto decode_item = [&](int i, int& e, int& nb, int& r) {
    int lo = 0, hi = E;  // largest e with item_start[e] <= i
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (item_start[mid] <= i) lo = mid; else hi = mid;
    }
    e = lo;
    const int local = i - item_start[e];
    const int c = a.offsets[e + 1] - a.offsets[e];
    const int nr = (c + kTR - 1) / kTR;
    nb = local / nr;
    r = local - nb * nr;
  };

  if (tid >= kConsumers) {
    // ================= producer =================
    if (tid != kConsumers) return;
    uint32_t L = 0;
    for (int i = blockIdx.x; i < total; i += gridDim.x) {
      int e, nb, r;
      decode_item(i, e, nb, r);
      const int slot = a.wslot_of ? a.wslot_of[e] : e;
      for (int st = 0; st < nst; ++st, ++L) {
        int row0;
        if (fc1) row0 = (st < nst / 2) ? nb * kOutBlk + st * RS : N + nb * kOutBlk + (st - nst / 2) * RS;
        else row0 = nb * kOutBlk + st * RS;
        const int s = L % P.stages;
        if (L >= static_cast<uint32_t>(P.stages)) {
          if (!mbar_wait(&empty[s], ((L / P.stages) - 1) & 1, a.wait)) {
            set_err(a.dev_err, MOE_DEVERR_TIMEOUT);
            return;
          }
        }
        if (*reinterpret_cast<volatile int*>(&s_abort)) return;
        const size_t grow = static_cast<size_t>(slot) * P.rows_total + row0;
        uint8_t* dq = ring + static_cast<size_t>(s) * P.stage_bytes;
        const uint32_t qb = RS * P.qrow_bytes, sb = RS * P.srow_bytes;
        mbar_arrive_expect_tx(&full[s], qb + sb);
        if (WK == kW2) {
          // one copy per K slice: RS rows of a slice are contiguous in the w2l layout
          const int SW = w2l_sw(K), nsl = K / SW;
          const uint32_t qs = RS * SW / 4, ssz = RS * (SW / 32) * 2;
          const uint8_t* wq_e = a.wq + static_cast<size_t>(slot) * P.rows_total * P.qrow_bytes;
          const uint8_t* ws_e = static_cast<const uint8_t*>(a.wscale) + static_cast<size_t>(slot) * P.rows_total * P.srow_bytes;
          for (int sl = 0; sl < nsl; ++sl) {
            bulk_g2s(dq + sl * qs, wq_e + (static_cast<size_t>(sl) * P.rows_total + row0) * (SW / 4), qs, &full[s]);
            bulk_g2s(dq + P.sq_bytes + sl * ssz,
                     ws_e + (static_cast<size_t>(sl) * P.rows_total + row0) * (SW / 32) * 2, ssz, &full[s]);
          }
        } else {
          bulk_g2s(dq, a.wq + grow * P.qrow_bytes, qb, &full[s]);
          if (sb) bulk_g2s(dq + P.sq_bytes, static_cast<const uint8_t*>(a.wscale) + grow * P.srow_bytes, sb, &full[s]);
        }
      }
    }
    return;
  }

  // ================= consumers =================
  const int warp = tid >> 5, lane = tid & 31;
  const int Prow = kConsumers / G >= 1 ? kConsumers / G : 1;  // rows in parallel
  const bool active = tid < Prow * G;
  const int g = tid % G, rho = tid / G;
  uint32_t nan_scale = 0;
  uint32_t L = 0;
  for (int i = blockIdx.x; i < total; i += gridDim.x) {
    int e, nb, r;
    decode_item(i, e, nb, r);
    const int p0 = a.offsets[e] + r * kTR;
    const int ntok = min(kTR, a.offsets[e + 1] - p0);
    for (int st = 0; st < nst; ++st, ++L) {
      const int s = L % P.stages;
      const bool ok = mbar_wait(&full[s], (L / P.stages) & 1, a.wait);
      const uint8_t* sq = ring + static_cast<size_t>(s) * P.stage_bytes;
      const uint8_t* ss = sq + P.sq_bytes;
      bool abort_now = !ok;
      for (int c0 = 0; c0 < ntok; c0 += kNT) {
        float2 x[kNT][16];
        if (active && !abort_now) {
#pragma unroll
          for (int t = 0; t < kNT; ++t) {
            if (c0 + t < ntok) {
              const int p = p0 + c0 + t;
              const int row = a.act_row ? a.act_row[p] / a.act_row_div : p;
              load_act<AF>(P, row, g, x[t]);
            } else {
#pragma unroll
              for (int j = 0; j < 16; ++j) x[t][j] = make_float2(0.f, 0.f);
            }
          }
          for (int rr = rho; rr < RS; rr += Prow) {
            float part[kNT];
            row_group_dot<WK>(sq, ss, rr, g, G, P, x, part, nan_scale);
#pragma unroll
            for (int t = 0; t < kNT; ++t) red[g * (V + 1) + rr * kNT + t] = part[t];
          }
        }
        // all consumers agree on abort (a timed-out wait anywhere aborts all)
        abort_now = named_bar_or(1, kConsumers, abort_now);
        if (abort_now) break;
        // sum the G partials of each (row, token): 4 parts of G/4 each, then combine
        {
          const int idx = tid % V, part_id = tid / V;
          const int nparts = kConsumers / V;  // V <= 64 -> >= 4 parts
          if (part_id < 4) {
            const int per = (G + 3) / 4;
            const int g0 = part_id * per, g1 = min(G, g0 + per);
            float s0 = 0.f, s1 = 0.f;
            int gg = g0;
            for (; gg + 1 < g1; gg += 2) {
              s0 += red[gg * (V + 1) + idx];
              s1 += red[(gg + 1) * (V + 1) + idx];
            }
            if (gg < g1) s0 += red[gg * (V + 1) + idx];
            red2[part_id * V + idx] = s0 + s1;
          }
          (void)nparts;
        }
        named_bar_sync(1, kConsumers);
        if (tid < V) {
          const int rr = tid / kNT, t = tid % kNT;
          float v = (red2[tid] + red2[V + tid]) + (red2[2 * V + tid] + red2[3 * V + tid]);
          const int orow = st * RS + rr;  // row within the item's 2*kOutBlk (FC1) or kOutBlk
          if (c0 + t < ntok) res[orow * kResPitch + c0 + t] = v;
        }
        named_bar_sync(1, kConsumers);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
      if (abort_now) {
        if (tid == 0) {
          s_abort = 1;
          set_err(a.dev_err, MOE_DEVERR_TIMEOUT);
        }
        return;
      }
    }
    // ---- epilogue: one warp per token, lane = output column
    for (int t = warp; t < ntok; t += kConsumers / 32) {
      const int p = p0 + t;
      const int n = nb * kOutBlk + lane;
      float v;
      if (fc1) {
        const float gv = res[lane * kResPitch + t], uv = res[(kOutBlk + lane) * kResPitch + t];
        v = silu_f32(gv) * uv;
      } else {
        v = res[lane * kResPitch + t];
      }
      if (a.out_fmt == MOE_FMT_F32) {
        static_cast<float*>(a.out)[static_cast<size_t>(p) * N + n] = v;
      } else if (a.out_fmt == MOE_FMT_BF16) {
        static_cast<uint16_t*>(a.out)[static_cast<size_t>(p) * N + n] = f32_to_bf16_rne(v);
      } else {  // MXFP8 along N, one block of 32 per item
        float amax = fabsf(v);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
        const int X = mx_scale_exp(amax);
        const float sv = v * exp2i(-X);
        const float nbv = __shfl_down_sync(0xffffffffu, sv, 1);
        const uint16_t two = f32x2_to_e4m3x2(sv, nbv);
        if ((lane & 1) == 0)
          *reinterpret_cast<uint16_t*>(static_cast<uint8_t*>(a.out) + static_cast<size_t>(p) * N + n) = two;
        if (lane == 0) a.out_scale[static_cast<size_t>(p) * (N / 32) + nb] = static_cast<uint8_t>(X + 127);
      }
    }
    named_bar_sync(1, kConsumers);  // res is reused by the next item
  }
  if (nan_scale) set_err(a.dev_err, MOE_DEVERR_NAN_SCALE);
}

template <int WK, int AF>
cudaError_t launch_t(const GemvParams& P0, cudaStream_t s) {
  GemvParams P = P0;
  constexpr int RS = WTraits<WK>::kRS;
  constexpr int V = RS * kNT;
  const int G = P.a.K / 32;
  const DeviceInfo& di = device_info();
  const int budget = static_cast<int>(di.smem_optin) - 1024;
  const SmemLayout fixed = smem_layout(0, P.stage_bytes, G, V, P.a.E);
  int stages = (budget - fixed.total - 256) / P.stage_bytes;
  stages = stages > 8 ? 8 : stages;
  if (stages < 2) return cudaErrorInvalidConfiguration;
  P.stages = stages;
  const SmemLayout lay = smem_layout(stages, P.stage_bytes, G, V, P.a.E);
  cudaError_t e = set_smem_limit(gemv_kernel<WK, AF>, lay.total);
  if (e != cudaSuccess) return e;
  gemv_kernel<WK, AF><<<di.sms, kThreads, lay.total, s>>>(P);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_gemv(const MMArgs& a, cudaStream_t s) {
  if (a.mode == MOE_MODE_SPLIT) {
    // groups of one row on the table GEMV, larger ones on the tensor core;
    // the two launches cover disjoint experts (so disjoint output rows)
    MMArgs v = a, g = a;
    v.mode = MOE_MODE_GEMV;
    v.split = 1;
    g.mode = MOE_MODE_GEMM;
    g.split = 2;
    if (a.wkind == kW2 && a.ws && a.ws_rows > 0 && lut_supported(v) && tmem_mm_supported(g)) {
      const cudaError_t e = launch_tmem_mm(g, a.act_rows, s);
      return e != cudaSuccess ? e : launch_lut_gemv(v, a.ws, s);
    }
    MMArgs all = a;  // a shape either side does not take: every group on the GEMV
    all.mode = MOE_MODE_GEMV;
    return launch_gemv(all, s);
  }
  // AUTO: the tensor-core GEMM for prefill-sized calls over permuted rows; the
  // GEMV for decode-sized ones (one 128-row tile per expert would be mostly idle)
  const bool want_gemm =
      a.mode == MOE_MODE_GEMM || (a.mode == MOE_MODE_AUTO && a.act_row == nullptr && a.act_rows >= 2048);
  if (want_gemm && mx_mm_supported(a)) return launch_mx_mm(a, a.act_rows, s);
  if (want_gemm && tmem_mm_supported(a)) return launch_tmem_mm(a, a.act_rows, s);
  if (a.out_fmt == MOE_FMT_MXFP8_BF16) return cudaErrorNotSupported;  // tensor-core path only
  if (want_gemm && gemm_supported(a)) return launch_gemm_tc(a, a.act_rows, s);
  if (a.ws && a.ws_rows > 0 && lut_supported(a)) return launch_lut_gemv(a, a.ws, s);
  return launch_gemv_generic(a, s);
}

cudaError_t launch_gemv_generic(const MMArgs& a, cudaStream_t s) {
  GemvParams P;
  P.a = a;
  const bool fc1 = a.stage == MOE_STAGE_FC1_SWIGLU;
  P.rows_total = fc1 ? 2 * a.N : a.N;
  int rs;
  switch (a.wkind) {
    case kW2:
      P.qrow_bytes = a.K / 4;
      P.srow_bytes = (a.K / 32) * 2;
      rs = WTraits<kW2>::kRS;
      break;
    case kMXFP4:
      P.qrow_bytes = a.K / 2;
      P.srow_bytes = a.K / 32;
      rs = WTraits<kMXFP4>::kRS;
      break;
    default:
      P.qrow_bytes = a.K;
      P.srow_bytes = 0;
      rs = WTraits<kFP8>::kRS;
      break;
  }
  P.sq_bytes = round_up(rs * P.qrow_bytes, 128);
  P.stage_bytes = P.sq_bytes + round_up(rs * P.srow_bytes, 128);
  P.stages = 0;
  const bool mx = a.act_fmt == MOE_FMT_MXFP8;
  switch (a.wkind) {
    case kW2: return mx ? launch_t<kW2, MOE_FMT_MXFP8>(P, s) : launch_t<kW2, MOE_FMT_BF16>(P, s);
    case kMXFP4: return mx ? launch_t<kMXFP4, MOE_FMT_MXFP8>(P, s) : launch_t<kMXFP4, MOE_FMT_BF16>(P, s);
    default: return mx ? launch_t<kFP8, MOE_FMT_MXFP8>(P, s) : launch_t<kFP8, MOE_FMT_BF16>(P, s);
  }
}

}  // namespace moe
