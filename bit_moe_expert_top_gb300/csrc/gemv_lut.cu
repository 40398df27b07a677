// Decode GEMV for 2-bit codebook experts by shared-memory partial-sum tables.
//
// A code byte holds 4 consecutive weights of a row, each one of the four
// codebook entries {-4,-1,1,4}.  For a fixed token x and a fixed byte
// position p of the row (elements 4p..4p+3), the contribution of that byte to
// a row's dot product is one of 256 values
//     T_p[b] = sum_{i<4} entry(code_i(b)) * x[4p+i],
// the same for every row.  The kernel builds these tables once per (token,
// K slice) and then streams the weight rows, turning every code byte into one
// table lookup: a PRMT forms the shared-memory address straight from the
// byte, an LDS fetches T_p[b], an FADD accumulates.  That is one integer op
// per 4 weights where a register decode needs at least four.
//
// Tables: one K slice of 512 elements = 128 byte positions x 256 entries x
// fp32 = 128 KB.  The slice is 32 code words per row; lane l of a warp always
// handles word l, and the table of word l's four byte positions sits in bank
// l, so a warp's 32 lookups never conflict.  The table starts at a 64 KB
// aligned shared-window address so that byte 1 of every lookup address is
// free for the code byte (one PRMT builds the address).
//
// Work: units (permuted row p, K slice s, batch of 16 weight rows) in
// (p, s, batch) order, split into one contiguous range per CTA (one CTA per
// SM).  A CTA walks its range segment by segment (one segment = one (p, s)
// table) with 16 warps; a warp takes every 16th batch of the segment.  Per
// batch a lane loads its word of 4 row quads straight from global memory
// (one 16-byte load per quad: the w2l layout puts word l of a quad's 4 rows
// side by side) plus the 4 matching bf16 scales, and issues the loads of its
// next batch while it consumes the current one.  (Bulk copies of a few KB
// into a shared ring stream far slower on this part, and would also spend
// shared-memory bandwidth twice.)  A shuffle reduce-scatter turns the 32
// lanes x 16 rows of partials into one slice sum per row (held by two
// lanes), which the warp stores to a global scratch with plain stores: no
// atomics and no fences, so nothing ever waits for the loads in flight.  A second, small kernel (launched as a programmatic dependent of
// the first) sums each row's slices in slice order (deterministic), applies
// SwiGLU for FC1, rounds and stores.  Neither kernel waits on another CTA.
#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"
#include "internal.cuh"
#include "layer_args.cuh"
#include "route_common.cuh"

namespace moe {

namespace {

constexpr int kLutWarps = 16;                // (20 or 24 warps with fewer registers each measured slower)
constexpr int kLutThreads = kLutWarps * 32;
constexpr int kBuildWarps = 16;               // warps that build a segment's tables
constexpr int kBR = 16;                       // weight rows per batch (4 row quads; 32-row batches measured slower)
constexpr int kSW = 512;                      // K elements per slice
constexpr int kPrologue = 26896;              // shared bytes below the table window
constexpr int kTableBytes = 2 * 65536;        // [j>>1][b][j&1][32 lanes] fp32
constexpr int kLutSmem = kPrologue + 65536 + kTableBytes;
constexpr int kMaxE = 1024;
// prologue layout: pref [E+1] ints, then the CTA's segment table and the
// double-buffered activation slice of the table builds
constexpr int kXBufOff = 4352;                // bf16 [2][kSW]
static_assert(4 * (kMaxE + 1) <= kXBufOff, "prologue overflow");
constexpr int kSlotTabOff = 8192;             // int [E]: weight slot of each expert
constexpr int kOffTabOff = 12288;             // int [E+1]: offsets[e], the first permuted row of expert e
static_assert(kXBufOff + 2 * kSW * 2 <= kSlotTabOff && kSlotTabOff + 4 * kMaxE <= kOffTabOff, "prologue overflow");
constexpr int kSegTabOff = 16640;             // int4 [kSegCap]: (permuted row, token row or -1, weight slot, slice)
constexpr int kSegCap = 128;
static_assert(kOffTabOff + 4 * (kMaxE + 1) <= kSegTabOff, "prologue overflow");
// the single-launch decode layer's routing and grouping (A = T*k <= kLayerA)
constexpr int kLayerA = 256;
constexpr int kLayerIds = 18688;              // int [kLayerA]: ids
constexpr int kLayerW = kLayerIds + 4 * kLayerA;      // float [kLayerA]: w
constexpr int kLayerPerm = kLayerW + 4 * kLayerA;     // int [kLayerA]: perm
constexpr int kLayerInv = kLayerPerm + 4 * kLayerA;   // int [kLayerA]: inv
constexpr int kLayerOffs = kLayerInv + 4 * kLayerA;   // int [kMaxE + 1]: offsets
static_assert(kSegTabOff + 16 * kSegCap <= kLayerIds && kLayerOffs + 4 * (kMaxE + 1) <= kPrologue, "prologue overflow");

struct LutParams {
  const uint16_t* act;
  const int32_t* act_row;
  int act_row_div;
  int act_rows;
  const uint8_t* codes;     // w2l words
  const uint16_t* scales;   // w2l bf16 scales
  const int32_t* select_map;
  int select;
  const int32_t* wslot;     // expert -> slot of the weight arrays (NULL: slot = expert)
  int slot_lo, slot_hi;     // with wslot: only experts whose slot lies in [slot_lo, slot_hi)
  int split;                // 1: only groups of fewer than kSplitRows rows
  int layer;                // single-launch layer: bit 0 offsets, bit 1 act_row from its shared-memory arrays
  const int32_t* offsets;
  int E, N, K, R;           // R = weight rows per expert
  int NSL;                  // K slices
  int NB;                   // row batches per permuted row (FC1: N/8, FC2: N/16)
  int fc1;
  int* rows_hdr;            // [0]: selected rows; then prow[A]: permuted row of selected row i, or -1
  float* scratch;           // [A][NB][NSL][kBR] per-slice row sums
  int A;                    // permuted rows the scratch covers
  void* out;
  int out_fmt;
  uint32_t* dev_err;
};

MOE_D float2 fadd2(float2 a, float2 b) {
  unsigned long long ra = *reinterpret_cast<unsigned long long*>(&a);
  unsigned long long rb = *reinterpret_cast<unsigned long long*>(&b);
  unsigned long long rd;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(rd) : "l"(ra), "l"(rb));
  return *reinterpret_cast<float2*>(&rd);
}

MOE_D float2 fmul2(float2 a, float2 b) {
  unsigned long long ra = *reinterpret_cast<unsigned long long*>(&a);
  unsigned long long rb = *reinterpret_cast<unsigned long long*>(&b);
  unsigned long long rd;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(rd) : "l"(ra), "l"(rb));
  return *reinterpret_cast<float2*>(&rd);
}

// The four table entries of one code word (lanebase = table window address +
// 4 * lane, whose byte 1 is zero): byte k of the word indexes the table of
// byte position 4*lane + k.
MOE_D float4 word_lookup(uint32_t w, uint32_t lanebase) {
  uint32_t a0, a1, a2, a3;
  asm("prmt.b32 %0, %1, %2, 0x7604;" : "=r"(a0) : "r"(w), "r"(lanebase));
  asm("prmt.b32 %0, %1, %2, 0x7614;" : "=r"(a1) : "r"(w), "r"(lanebase));
  asm("prmt.b32 %0, %1, %2, 0x7624;" : "=r"(a2) : "r"(w), "r"(lanebase));
  asm("prmt.b32 %0, %1, %2, 0x7634;" : "=r"(a3) : "r"(w), "r"(lanebase));
  float4 t;
  asm volatile("ld.shared.f32 %0, [%1];" : "=f"(t.x) : "r"(a0));
  asm volatile("ld.shared.f32 %0, [%1+128];" : "=f"(t.y) : "r"(a1));
  asm volatile("ld.shared.f32 %0, [%1+65536];" : "=f"(t.z) : "r"(a2));
  asm volatile("ld.shared.f32 %0, [%1+65664];" : "=f"(t.w) : "r"(a3));
  return t;
}

// Scaled word sums of two rows (words wa, wb; bf16 scales packed in sc as
// lo = row a, hi = row b), with packed fp32x2 adds.
MOE_D float2 word_pair(uint32_t wa, uint32_t wb, uint32_t sc, uint32_t lanebase) {
  const float4 ta = word_lookup(wa, lanebase);
  const float4 tb = word_lookup(wb, lanebase);
  const float2 s01 = fadd2(make_float2(ta.x, tb.x), make_float2(ta.y, tb.y));
  const float2 s23 = fadd2(make_float2(ta.z, tb.z), make_float2(ta.w, tb.w));
  return fmul2(fadd2(s01, s23), make_float2(__uint_as_float(sc << 16), __uint_as_float(sc & 0xffff0000u)));
}

// 8-byte asynchronous global -> shared copy (completion by cp.async groups).
MOE_D void cp_async8(uint32_t dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(dst), "l"(src) : "memory");
}
MOE_D void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
MOE_D void cp_async_wait1() { asm volatile("cp.async.wait_group 1;" ::: "memory"); }

MOE_D uint4 ldg_stream(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

MOE_D uint2 ldg_stream2(const void* p) {
  uint2 v;
  asm volatile("ld.global.nc.L1::no_allocate.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "l"(p));
  return v;
}

// One reduce-scatter level over the row pairs v[0..2H) (pair i = rows 2i,
// 2i+1): lanes with bit m set keep the upper half and add the partner's upper
// half; the others keep the lower half.
template <int H>
MOE_D void rs_level2(float2* v, int lane, int m) {
  const bool up = (lane & m) != 0;
#pragma unroll
  for (int i = 0; i < H; ++i) {
    const float2 keep = up ? v[i + H] : v[i];
    const float2 send = up ? v[i] : v[i + H];
    float2 got;
    got.x = __shfl_xor_sync(0xffffffffu, send.x, m);
    got.y = __shfl_xor_sync(0xffffffffu, send.y, m);
    v[i] = fadd2(keep, got);
  }
}

// Shared-memory prologue of one call (FC1 or FC2) by one CTA: the selected
// rows before each expert (pref), each expert's weight slot and first
// permuted row.  Reads only the grouping (offsets) and the expert maps.
MOE_D void lut_prologue(const LutParams& P, uint8_t* smem) {
  int* pref = reinterpret_cast<int*>(smem);  // [E+1] selected permuted rows before expert e
  int* slot_tab = reinterpret_cast<int*>(smem + kSlotTabOff);  // [E] weight slot of expert e
  int* off_s = reinterpret_cast<int*>(smem + kOffTabOff);      // [E+1] offsets
  const int32_t* offsets = (P.layer & 1) ? reinterpret_cast<const int32_t*>(smem + kLayerOffs) : P.offsets;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  // ---- selected rows per expert, exclusive prefix: every thread loads the
  // counts of experts 2t and 2t+1 at once (one round trip), then a block scan
  {
    __shared__ int warp_tot[kLutWarps];
    int n[2] = {0, 0};
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int e = 2 * tid + h;
      if (e < P.E) {
        const int lo = offsets[e], hi = offsets[e + 1];
        const int c = hi - lo;
        const int sm = P.select ? P.select_map[e] : 0;
        const int ws = P.wslot ? P.wslot[e] : e;
        bool sel = c > 0;
        if (sel && P.select == 1) sel = sm < 0;
        if (sel && P.select == 2) sel = sm >= 0;
        if (sel && P.split == 1) sel = c < kSplitRows;
        if (P.wslot) sel = sel && ws >= P.slot_lo && ws < P.slot_hi;
        slot_tab[e] = ws;
        off_s[e] = lo;
        if (e == P.E - 1) off_s[P.E] = hi;
        if (sel) n[h] = c;
      }
    }
    const int local = n[0] + n[1];
    int incl = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    if (lane == 31) warp_tot[warp] = incl;
    __syncthreads();
    int before = 0;
    for (int w2 = 0; w2 < warp; ++w2) before += warp_tot[w2];
    const int excl = before + incl - local;
    if (2 * tid <= P.E) pref[2 * tid] = excl;
    if (2 * tid + 1 <= P.E) pref[2 * tid + 1] = excl + n[0];
    if (tid == kLutThreads - 1) pref[P.E] = excl + local;  // the total (also for E = 1024)
  }
  __syncthreads();
}

// The permuted row of every selected row, for the summing step (-1 where
// the row is skipped: beyond the scratch, or a bad token index); global.
MOE_D void lut_rows(const LutParams& P, const uint8_t* smem) {
  const int* pref = reinterpret_cast<const int*>(smem);
  const int* off_s = reinterpret_cast<const int*>(smem + kOffTabOff);
  const int32_t* act_row = (P.layer & 2) ? reinterpret_cast<const int32_t*>(smem + kLayerPerm) : P.act_row;
  const int tid = threadIdx.x;
  {
    const int nsel = pref[P.E];
    if (blockIdx.x == 0 && tid == 0) P.rows_hdr[0] = nsel;
    const int lim = min(nsel, P.A);
    for (int i = blockIdx.x * kLutThreads + tid; i < lim; i += gridDim.x * kLutThreads) {
      int lo = 0, hi = P.E;
      while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (pref[mid] <= i) lo = mid; else hi = mid;
      }
      const int p = off_s[lo] + (i - pref[lo]);
      bool ok = p < P.A;
      if (ok) {
        const int row = act_row ? act_row[p] / P.act_row_div : p;
        ok = row >= 0 && row < P.act_rows;
      }
      P.rows_hdr[1 + i] = ok ? p : -1;
    }
  }
}

// The table GEMV of one call (FC1 or FC2) by one CTA of the persistent grid,
// after lut_prologue.
MOE_D void lut_main(const LutParams& P, uint8_t* smem) {
  int* pref = reinterpret_cast<int*>(smem);
  int* slot_tab = reinterpret_cast<int*>(smem + kSlotTabOff);
  const int* off_s = reinterpret_cast<const int*>(smem + kOffTabOff);
  const int32_t* act_row = (P.layer & 2) ? reinterpret_cast<const int32_t*>(smem + kLayerPerm) : P.act_row;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t base = smem_u32(smem);
  const uint32_t table_win = (base + kPrologue + 65535u) & ~65535u;
  float* table_f = reinterpret_cast<float*>(smem + (table_win - base));
  const uint32_t lanebase = table_win + 4u * static_cast<uint32_t>(lane);
  const int NSL = P.NSL, NB = P.NB;
  const bool fc1 = P.fc1 != 0;

  // ---- this CTA's unit range; unit = (selected row, slice, batch), batch fastest
  const int64_t per_row = static_cast<int64_t>(NSL) * NB;
  const int64_t total = static_cast<int64_t>(pref[P.E]) * per_row;
  const int64_t u_beg = total * blockIdx.x / gridDim.x;
  const int64_t u_end = total * (blockIdx.x + 1) / gridDim.x;
  if (u_beg >= u_end) return;

  const int64_t mat_codes = static_cast<int64_t>(P.R) * (P.K / 4);    // bytes per expert
  const int64_t mat_scales = static_cast<int64_t>(P.R) * (P.K / 32);  // bf16 per expert
  const int64_t slice_codes = static_cast<int64_t>(P.R) * (kSW / 4);
  const int64_t slice_scales = static_cast<int64_t>(P.R) * (kSW / 32);
  // byte offsets of a batch's four row quads from its first: FC1 batches are
  // quads 2rb, 2rb+1 (gate rows) and N/4 + 2rb, N/4 + 2rb + 1 (up rows); FC2
  // batches quads 4rb .. 4rb+3.  A quad is 512 code bytes and 128 scale bytes.
  const uint32_t cstep = fc1 ? 1024u : 2048u, sstep = fc1 ? 256u : 512u;
  const uint32_t chi = fc1 ? static_cast<uint32_t>(P.N) * 128u : 1024u;
  const uint32_t shi = fc1 ? static_cast<uint32_t>(P.N) * 32u : 256u;
  const uint32_t sum_step = static_cast<uint32_t>(NSL) * kBR;           // scratch floats per batch

  uint4 v[4];
  uint2 sc[4];
  float2 acc[8];  // row pairs (2i, 2i+1) of the batch

  auto expert_of = [&](int psel) {  // largest e with pref[e] <= psel
    int lo = 0, hi = P.E;
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (pref[mid] <= psel) lo = mid; else hi = mid;
    }
    return lo;
  };
  auto issue = [&](const uint8_t* gc, const uint8_t* gs, int rb) {
    const uint8_t* c0 = gc + static_cast<uint32_t>(rb) * cstep;
    const uint8_t* c2 = c0 + chi;
    const uint8_t* s0 = gs + static_cast<uint32_t>(rb) * sstep;
    const uint8_t* s2 = s0 + shi;
    v[0] = ldg_stream(c0);
    v[1] = ldg_stream(c0 + 512);
    v[2] = ldg_stream(c2);
    v[3] = ldg_stream(c2 + 512);
    sc[0] = ldg_stream2(s0);
    sc[1] = ldg_stream2(s0 + 128);
    sc[2] = ldg_stream2(s2);
    sc[3] = ldg_stream2(s2 + 128);
  };

  // ---- the CTA's segments (one per (selected row, slice) table): their
  // permuted row and token row, looked up once for all of them in parallel
  // (a lookup per segment would stall every warp at each table build), and
  // each segment's 512 activations brought into shared memory by cp.async
  // one segment ahead
  const int64_t seg_first = u_beg / NB;
  const int64_t seg_last = (u_end - 1) / NB;
  const int64_t nseg = seg_last - seg_first + 1;
  int4* seg_tab = reinterpret_cast<int4*>(smem + kSegTabOff);
  const uint16_t* xbuf = reinterpret_cast<const uint16_t*>(smem + kXBufOff);
  // (p, row, weight slot, slice; row = -1 if the segment is skipped)
  auto seg_lookup = [&](int64_t sg) -> int4 {
    const int ps = static_cast<int>(sg / NSL);
    const int sl = static_cast<int>(sg - static_cast<int64_t>(ps) * NSL);
    const int ee = expert_of(ps);
    const int pp = off_s[ee] + (ps - pref[ee]);
    if (pp >= P.A) {  // the scratch does not cover this row: report and skip
      set_err(P.dev_err, MOE_DEVERR_OVERFLOW);
      return make_int4(pp, -1, slot_tab[ee], sl);
    }
    const int rr = act_row ? act_row[pp] / P.act_row_div : pp;
    if (rr < 0 || rr >= P.act_rows) {
      set_err(P.dev_err, MOE_DEVERR_BAD_ID);
      return make_int4(pp, -1, slot_tab[ee], sl);
    }
    return make_int4(pp, rr, slot_tab[ee], sl);
  };
  for (int i = tid; i < nseg && i < kSegCap; i += kLutThreads) seg_tab[i] = seg_lookup(seg_first + i);
  __syncthreads();
  auto seg_info = [&](int64_t sg) -> int4 {
    const int64_t i = sg - seg_first;
    return i < kSegCap ? seg_tab[i] : seg_lookup(sg);
  };
  // activations of segment sg into buffer sg & 1: 128 threads x 8 bytes; one
  // cp.async group per call on every thread (empty where nothing is copied)
  auto prefetch_x = [&](int64_t sg) {
    if (sg <= seg_last && tid < kSW / 4) {
      const int4 si = seg_info(sg);
      if (si.y >= 0) {
        const int sl = si.w;
        cp_async8(smem_u32(xbuf) + static_cast<uint32_t>(((sg - seg_first) & 1) * kSW * 2 + 8 * tid),
                  P.act + static_cast<size_t>(si.y) * P.K + sl * kSW + 4 * tid);
      }
    }
    cp_async_commit();
  };
  // segment sg: its weight pointers and the end of the CTA's batches in it
  // (batch indices inside a segment are 32-bit: NB <= K/8)
  auto seg_ptrs = [&](int64_t sg, const uint8_t*& gc, const uint8_t*& gs) {
    const int4 si = seg_info(sg);
    gc = P.codes + si.z * mat_codes + si.w * slice_codes + lane * 16;
    gs = reinterpret_cast<const uint8_t*>(P.scales + si.z * mat_scales + si.w * slice_scales) + (lane >> 1) * 8;
  };
  auto seg_hi = [&](int64_t sg) { return sg == seg_last ? static_cast<int>(u_end - sg * NB) : NB; };
  prefetch_x(seg_first);
  prefetch_x(seg_first + 1);
  // A warp's units: the CTA's units u_beg, u_beg + 1, ... go round-robin to
  // the 16 warps (unit u to warp (u - u_beg) mod 16), so that every warp
  // gets the same number of batches within one; in a segment (one (row,
  // slice) table) a warp takes every 16th batch.  The loads of a warp's next
  // unit go out while the current one is consumed, also across a segment
  // boundary; the row checks (which need global loads) only gate the table
  // build and the stores, never the weight loads.
  int64_t seg = seg_first;
  const uint8_t* gcodes;
  const uint8_t* gscales;
  seg_ptrs(seg, gcodes, gscales);
  int rb_hi = seg_hi(seg);
  int rb = static_cast<int>(u_beg - seg * NB) + warp;
  bool pending = false;
  if (rb < rb_hi) {
    issue(gcodes, gscales, rb);
    pending = true;
  }
  while (true) {
    const bool has_next = seg < seg_last;
    const uint8_t* ncodes = gcodes;
    const uint8_t* nscales = gscales;
    int nrb_hi = 0;
    // this warp's first batch of the next segment
    const int nrb_first = (warp - static_cast<int>(((seg + 1) * NB - u_beg) & 15)) & 15;
    if (has_next) {
      seg_ptrs(seg + 1, ncodes, nscales);
      nrb_hi = seg_hi(seg + 1);
    }
    const int4 si = seg_info(seg);
    const bool valid = si.y >= 0;
    const int s = si.w;
    float* const sbase = P.scratch + (static_cast<size_t>(si.x) * NB * NSL + s) * kBR + (lane >> 1);
    if (!pending && rb < rb_hi) {
      issue(gcodes, gscales, rb);
      pending = true;
    }

    // ---- (re)build the tables for (row, s): warp w writes byte-in-word j = w & 3
    // and code bytes b in [64*(w>>2), +64); lane l is byte position 4l + j
    cp_async_wait1();  // this segment's activations have landed (the next one's may be in flight)
    __syncthreads();  // nobody still reads the previous segment's tables
    if (valid && warp < kBuildWarps) {
      const int j = warp & 3, bq = warp >> 2;
      const uint2 xv = *reinterpret_cast<const uint2*>(xbuf + ((seg - seg_first) & 1) * kSW + 16 * lane + 4 * j);
      const float x0 = __uint_as_float(xv.x << 16), x1 = __uint_as_float(xv.x & 0xffff0000u);
      const float x2 = __uint_as_float(xv.y << 16), x3 = __uint_as_float(xv.y & 0xffff0000u);
      const float cb[4] = {-4.f, -1.f, 1.f, 4.f};
      const float c3 = bq == 0 ? -4.f : bq == 1 ? -1.f : bq == 2 ? 1.f : 4.f;  // code 3 of b = b >> 6 = bq
      float plo[16];
#pragma unroll
      for (int c1 = 0; c1 < 4; ++c1)
#pragma unroll
        for (int c0 = 0; c0 < 4; ++c0) plo[c0 + 4 * c1] = fmaf(cb[c1], x1, cb[c0] * x0);
      float* tw = table_f + (j >> 1) * 16384 + (j & 1) * 32 + lane;
#pragma unroll
      for (int c2 = 0; c2 < 4; ++c2) {
        const float ph = fmaf(c3, x3, cb[c2] * x2);
        const int b0 = bq * 64 + c2 * 16;
#pragma unroll
        for (int l4 = 0; l4 < 16; ++l4) tw[(b0 + l4) * 64] = plo[l4] + ph;
      }
    }
    __syncthreads();
    prefetch_x(seg + 2);  // into the buffer this build has finished reading

    bool more = false;
    if (rb < rb_hi) {
      while (true) {
        // the warp's next unit: the same segment, or its first batch of the next
        const int rb_same = rb + kLutWarps;
        const bool same = rb_same < rb_hi;
        int rbn = rb_same;
        const uint8_t* nc = gcodes;
        const uint8_t* ns = gscales;
        more = same;
        if (!same) {
          rbn = nrb_first;
          more = has_next && nrb_first < nrb_hi;
          nc = ncodes;
          ns = nscales;
        }
        if (valid) {
          const uint8_t* c0 = nc + static_cast<uint32_t>(rbn) * cstep;
          const uint8_t* s0 = ns + static_cast<uint32_t>(rbn) * sstep;
          const uint8_t* const cq[4] = {c0, c0 + 512, c0 + chi, c0 + chi + 512};
          const uint8_t* const sq[4] = {s0, s0 + 128, s0 + shi, s0 + shi + 128};
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const uint4 w4 = v[q];
            const uint2 s4 = sc[q];
            acc[2 * q] = word_pair(w4.x, w4.y, s4.x, lanebase);
            acc[2 * q + 1] = word_pair(w4.z, w4.w, s4.y, lanebase);
            if (more) {  // the next unit's loads go out while this one is consumed
              v[q] = ldg_stream(cq[q]);
              sc[q] = ldg_stream2(sq[q]);
            }
          }
          // ---- reduce-scatter: afterwards lanes 2r and 2r + 1 hold the slice
          // sum of batch row r
          rs_level2<4>(acc, lane, 16);
          rs_level2<2>(acc, lane, 8);
          rs_level2<1>(acc, lane, 4);
          const bool hi = (lane & 2) != 0;
          const float keep = hi ? acc[0].y : acc[0].x;
          const float send = hi ? acc[0].x : acc[0].y;
          float sum = keep + __shfl_xor_sync(0xffffffffu, send, 2);
          sum += __shfl_xor_sync(0xffffffffu, sum, 1);
          if ((lane & 1) == 0) __stcg(sbase + static_cast<uint32_t>(rb) * sum_step, sum);
        } else if (more) {
          issue(nc, ns, rbn);
        }
        if (!same) break;
        rb = rb_same;
      }
    }
    pending = more;
    if (!has_next) break;
    // ---- advance to the next segment
    ++seg;
    gcodes = ncodes;
    gscales = nscales;
    rb_hi = nrb_hi;
    rb = nrb_first;
  }
}

MOE_D void lut_run(const LutParams& P, uint8_t* smem) {
  lut_prologue(P, smem);
  lut_rows(P, smem);
  lut_main(P, smem);
}

__global__ void __launch_bounds__(kLutThreads, 1) w2_lut_kernel(const LutParams P) {
  extern __shared__ __align__(1024) uint8_t smem[];
  pdl_wait();  // offsets, activations and the scratch belong to earlier kernels
  pdl_trigger();
  lut_run(P, smem);
}

// The NSL (<= kMaxSlices) slice sums at sp (stride kBR) added in slice
// order; every load is issued before the first add.
constexpr int kMaxSlices = 16;  // K <= 8192
MOE_D float slice_total(const float* sp, int NSL) {
  float v[kMaxSlices];
#pragma unroll
  for (int q = 0; q < kMaxSlices; ++q) v[q] = q < NSL ? __ldcg(sp + q * kBR) : 0.f;
  float t = 0.f;
#pragma unroll
  for (int q = 0; q < kMaxSlices; ++q)
    if (q < NSL) t += v[q];
  return t;
}

// One output of the finishing step: the NSL slice sums of selected row i,
// output n, added in slice order, SwiGLU for FC1, in t; returns the output's
// element index, or -1 where the row is skipped.
MOE_D int64_t finish_value(const LutParams& P, int i, int n, float& t) {
  const int NSL = P.NSL, NB = P.NB;
  const int p = __ldcg(P.rows_hdr + 1 + i);
  if (p < 0) return -1;
  if (P.fc1) {  // batch n/8: rows 0..7 gate rows, 8..15 the matching up rows
    const float* sp = P.scratch + (static_cast<size_t>(p) * NB + (n >> 3)) * NSL * kBR + (n & 7);
    const float g = slice_total(sp, NSL);
    const float u = slice_total(sp + 8, NSL);
    t = silu_f32(g) * u;
  } else {
    const float* sp = P.scratch + (static_cast<size_t>(p) * NB + (n >> 4)) * NSL * kBR + (n & 15);
    t = slice_total(sp, NSL);
  }
  return static_cast<int64_t>(p) * P.N + n;
}

MOE_D void finish_store(const LutParams& P, int64_t o, float t) {
  if (P.out_fmt == MOE_FMT_F32) static_cast<float*>(P.out)[o] = t;
  else static_cast<uint16_t*>(P.out)[o] = f32_to_bf16_rne(t);
}

MOE_D void finish_one(const LutParams& P, int i, int n) {
  float t;
  const int64_t o = finish_value(P, i, n, t);
  if (o >= 0) finish_store(P, o, t);
}

// Sums the NSL slice sums of every output in slice order, applies SwiGLU for
// FC1, rounds and stores.  Block (i, j) takes selected rows i, i + gridDim.x,
// ... and outputs [256 j, 256 j + 256); one thread per output.
__global__ void __launch_bounds__(256) w2_lut_finish_kernel(const LutParams P) {
  // everything read here is written by the preceding (primary) grid
  pdl_wait();
  pdl_trigger();
  const int n = blockIdx.y * 256 + threadIdx.x;
  if (n >= P.N) return;
  const int lim = min(__ldcg(P.rows_hdr), P.A);
  for (int i = blockIdx.x; i < lim; i += gridDim.x) finish_one(P, i, n);
}

// ------------------------------------------------------------------ one launch for FC1 and FC2
// All CTAs of a cooperative launch (every CTA resident: one per SM) meet
// here.  The counter is zero when the launch starts; barrier k completes when
// it reaches k * gridDim.x.  The wait is bounded: past the limit the CTA
// records MOE_DEVERR_TIMEOUT and the kernel returns (the others then time out
// too).
// The barrier in two halves, so that a CTA can do work of its own between
// its arrival and its wait.
MOE_D void grid_arrive(unsigned int* cnt) {
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();  // this CTA's results before its arrival
    atomicAdd(cnt, 1u);
  }
}

MOE_D bool grid_wait(unsigned int* cnt, unsigned int target, long long limit, uint32_t* dev_err) {
  __shared__ int s_ok;
  if (threadIdx.x == 0) {
    const long long t0 = clock64();
    int ok = 1;
    while (true) {
      unsigned int v;
      asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(cnt) : "memory");
      if (v >= target) break;
      if (clock64() - t0 > limit) {
        ok = 0;
        set_err(dev_err, MOE_DEVERR_TIMEOUT);
        break;
      }
      __nanosleep(64);
    }
    s_ok = ok;
  }
  __syncthreads();
  asm volatile("fence.acq_rel.gpu;" ::: "memory");  // the other CTAs' results are visible to every thread
  return s_ok != 0;
}

MOE_D bool grid_barrier(unsigned int* cnt, unsigned int target, long long limit, uint32_t* dev_err) {
  grid_arrive(cnt);
  return grid_wait(cnt, target, limit, dev_err);
}

// The finishing step over the whole grid, two outputs per thread and round
// (both outputs' loads go out before either is added up).
MOE_D void finish_grid(const LutParams& P) {
  const int lim = min(__ldcg(P.rows_hdr), P.A);
  const int64_t total = static_cast<int64_t>(lim) * P.N;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; idx < total; idx += 2 * stride) {
    const int64_t idx2 = idx + stride;
    float t1 = 0.f, t2 = 0.f;
    const int64_t o1 = finish_value(P, static_cast<int>(idx / P.N), static_cast<int>(idx % P.N), t1);
    const int64_t o2 = idx2 < total ? finish_value(P, static_cast<int>(idx2 / P.N), static_cast<int>(idx2 % P.N), t2) : -1;
    if (o1 >= 0) finish_store(P, o1, t1);
    if (o2 >= 0) finish_store(P, o2, t2);
  }
}

// FC1 + SwiGLU and FC2 of the 2-bit decode layer in one persistent launch:
// FC1 tables, barrier, FC1 slice sums -> h, barrier, FC2 tables (on h),
// barrier, FC2 slice sums -> y.  Same arithmetic and order as the two calls.
__global__ void __launch_bounds__(kLutThreads, 1) w2_decode_fused_kernel(const LutParams P1, const LutParams P2,
                                                                        unsigned int* bar, long long wait) {
  extern __shared__ __align__(1024) uint8_t smem[];
  pdl_wait();
  pdl_trigger();
  lut_run(P1, smem);
  grid_arrive(bar);
  // FC2's shared-memory prologue needs only the grouping: it runs while the
  // other CTAs finish FC1 (FC1 no longer reads this CTA's shared memory)
  lut_prologue(P2, smem);
  if (!grid_wait(bar, gridDim.x, wait, P1.dev_err)) return;
  finish_grid(P1);
  if (!grid_barrier(bar, 2 * gridDim.x, wait, P1.dev_err)) return;
  lut_rows(P2, smem);  // after every CTA's FC1 sums have read the row list
  lut_main(P2, smem);
  if (!grid_barrier(bar, 3 * gridDim.x, wait, P1.dev_err)) return;
  finish_grid(P2);
  // leave the counter at zero for the next launch: the last CTA to arrive
  // here (every other CTA is past its last barrier wait) resets it
  if (threadIdx.x == 0 && atomicAdd(bar, 1u) == 4 * gridDim.x - 1) atomicExch(bar, 0u);
}

// ------------------------------------------------------------------ one launch for the decode layer
constexpr int kLayerK = 16;  // experts per token at most

struct LayerParams {
  const float* logits;  // [T][E]
  int T, E, k;
  int32_t* ids;         // [T][k] out
  float* w;             // [T][k] out
  int32_t* offsets;     // [E+1] out
  int32_t* perm;        // [A] out
  int32_t* inv;         // [A] out
  uint16_t* y;          // bf16 [A][H] out
  void* out;            // [T][H] out, out_fmt
  int out_fmt;
  uint32_t* dev_err;
};

// Routing and grouping of the whole step by one CTA into its shared memory
// (every CTA computes the same; CTA 0 also writes them out): route_token per
// token (the routing kernel's arithmetic), then moe_permute's stable
// counting sort (rows of one expert in increasing assignment order).
template <int NPL>
MOE_D void layer_route(const LayerParams& L, uint8_t* smem) {
  int* ids_s = reinterpret_cast<int*>(smem + kLayerIds);
  float* w_s = reinterpret_cast<float*>(smem + kLayerW);
  int* perm_s = reinterpret_cast<int*>(smem + kLayerPerm);
  int* inv_s = reinterpret_cast<int*>(smem + kLayerInv);
  int* offs_s = reinterpret_cast<int*>(smem + kLayerOffs);
  const uint32_t base = smem_u32(smem);
  int* cnt = reinterpret_cast<int*>(smem + (((base + kPrologue + 65535u) & ~65535u) - base));  // the table window, free here
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int A = L.T * L.k, E = L.E;
  bool nan = false;
  for (int t = warp; t < L.T; t += kLutWarps) {
    int id;
    float wt;
    nan |= route_token<NPL>(L.logits + static_cast<size_t>(t) * E, E, L.k, lane, id, wt);
    if (lane < L.k) {
      ids_s[t * L.k + lane] = id;
      w_s[t * L.k + lane] = wt;
    }
  }
  if (nan && lane == 0 && blockIdx.x == 0) set_err(L.dev_err, MOE_DEVERR_NAN_LOGIT);
  for (int e = tid; e < E; e += kLutThreads) cnt[e] = 0;
  __syncthreads();
  for (int a = tid; a < A; a += kLutThreads) atomicAdd(&cnt[ids_s[a]], 1);
  __syncthreads();
  {  // offsets: exclusive scan of the counts, experts 2t and 2t+1 per thread
    __shared__ int lay_wsum[kLutWarps];
    const int n0 = 2 * tid < E ? cnt[2 * tid] : 0;
    const int n1 = 2 * tid + 1 < E ? cnt[2 * tid + 1] : 0;
    int incl = n0 + n1;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    if (lane == 31) lay_wsum[warp] = incl;
    __syncthreads();
    int before = 0;
    for (int w2 = 0; w2 < warp; ++w2) before += lay_wsum[w2];
    const int excl = before + incl - n0 - n1;
    if (2 * tid <= E) offs_s[2 * tid] = excl;
    if (2 * tid + 1 <= E) offs_s[2 * tid + 1] = excl + n0;
    if (tid == kLutThreads - 1) offs_s[E] = excl + n0 + n1;  // the total (also for E = 1024)
  }
  __syncthreads();
  for (int a = tid; a < A; a += kLutThreads) {  // stable: rank among the expert's earlier assignments
    const int e = ids_s[a];
    int r = 0;
    for (int b2 = 0; b2 < a; ++b2) r += ids_s[b2] == e;
    const int pos = offs_s[e] + r;
    perm_s[pos] = a;
    inv_s[a] = pos;
  }
  __syncthreads();
  if (blockIdx.x == 0) {
    for (int a = tid; a < A; a += kLutThreads) {
      L.ids[a] = ids_s[a];
      L.w[a] = w_s[a];
      L.perm[a] = perm_s[a];
      L.inv[a] = inv_s[a];
    }
    for (int e = tid; e <= E; e += kLutThreads) L.offsets[e] = offs_s[e];
  }
}

// FC2's summing step and the weighted combine in one pass: output n of token
// t sums the slices of its k rows (y, rounded to bf16 and stored) and adds
// them up in slot order as moe_combine does (out = sum_j w_j * y_j, fmaf from
// zero).  Every row is one token's slot, so each y element is written once.
MOE_D void layer_finish(const LutParams& P, const LayerParams& L, const uint8_t* smem) {
  const float* w_s = reinterpret_cast<const float*>(smem + kLayerW);
  const int* inv_s = reinterpret_cast<const int*>(smem + kLayerInv);
  const int H = P.N, NSL = P.NSL, NB = P.NB, k = L.k;
  const int64_t total = static_cast<int64_t>(L.T) * H;
  for (int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; idx < total;
       idx += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int t = static_cast<int>(idx / H), n = static_cast<int>(idx % H);
    float v[kLayerK];
#pragma unroll
    for (int j = 0; j < kLayerK; ++j) {  // every slot's loads before the first store
      v[j] = 0.f;
      if (j < k) {
        const int p = inv_s[t * k + j];
        v[j] = slice_total(P.scratch + (static_cast<size_t>(p) * NB + (n >> 4)) * NSL * kBR + (n & 15), NSL);
      }
    }
    float acc = 0.f;
#pragma unroll
    for (int j = 0; j < kLayerK; ++j) {
      if (j < k) {
        const int p = inv_s[t * k + j];
        const uint16_t yb = f32_to_bf16_rne(v[j]);
        L.y[static_cast<size_t>(p) * H + n] = yb;
        acc = fmaf(w_s[t * k + j], __uint_as_float(static_cast<uint32_t>(yb) << 16), acc);
      }
    }
    if (L.out_fmt == MOE_FMT_F32) static_cast<float*>(L.out)[static_cast<size_t>(t) * H + n] = acc;
    else static_cast<uint16_t*>(L.out)[static_cast<size_t>(t) * H + n] = f32_to_bf16_rne(acc);
  }
}

// FC1's summing step of the single-launch layer over the whole grid: every
// row is valid and selected row i is permuted row i (all experts, all
// rows), so no row list is read; two outputs per thread and round.
MOE_D void finish_grid_all(const LutParams& P, int A) {
  const int64_t total = static_cast<int64_t>(A) * P.N;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; idx < total; idx += 2 * stride) {
    const int64_t idx2 = idx + stride;
    const int p1 = static_cast<int>(idx / P.N), n1 = static_cast<int>(idx % P.N);
    const float* s1 = P.scratch + (static_cast<size_t>(p1) * P.NB + (n1 >> 3)) * P.NSL * kBR + (n1 & 7);
    const float g1 = slice_total(s1, P.NSL), u1 = slice_total(s1 + 8, P.NSL);
    float g2 = 0.f, u2 = 0.f;
    int p2 = 0, n2 = 0;
    if (idx2 < total) {
      p2 = static_cast<int>(idx2 / P.N);
      n2 = static_cast<int>(idx2 % P.N);
      const float* s2 = P.scratch + (static_cast<size_t>(p2) * P.NB + (n2 >> 3)) * P.NSL * kBR + (n2 & 7);
      g2 = slice_total(s2, P.NSL);
      u2 = slice_total(s2 + 8, P.NSL);
    }
    finish_store(P, static_cast<int64_t>(p1) * P.N + n1, silu_f32(g1) * u1);
    if (idx2 < total) finish_store(P, static_cast<int64_t>(p2) * P.N + n2, silu_f32(g2) * u2);
  }
}

// The whole 2-bit decode layer in one persistent launch: routing and
// grouping (every CTA, shared memory), FC1 tables, barrier, FC1 sums -> h,
// barrier, FC2 tables, barrier, FC2 sums -> y with the combine -> out.  Same
// arithmetic and order as moe_route, moe_permute, moe_w2_decode_fused and
// moe_combine.
template <int NPL>
__global__ void __launch_bounds__(kLutThreads, 1) w2_decode_layer_kernel(const LayerParams L, const LutParams P1,
                                                                        const LutParams P2, unsigned int* bar,
                                                                        long long wait) {
  extern __shared__ __align__(1024) uint8_t smem[];
  pdl_wait();
  pdl_trigger();
  layer_route<NPL>(L, smem);
  lut_prologue(P1, smem);  // (no row list: the summing steps below index rows directly)
  lut_main(P1, smem);
  grid_arrive(bar);
  lut_prologue(P2, smem);
  if (!grid_wait(bar, gridDim.x, wait, P1.dev_err)) return;
  finish_grid_all(P1, L.T * L.k);
  if (!grid_barrier(bar, 2 * gridDim.x, wait, P1.dev_err)) return;
  lut_main(P2, smem);
  if (!grid_barrier(bar, 3 * gridDim.x, wait, P1.dev_err)) return;
  layer_finish(P2, L, smem);
  if (threadIdx.x == 0 && atomicAdd(bar, 1u) == 4 * gridDim.x - 1) atomicExch(bar, 0u);
}

}  // namespace

// Scratch of the table GEMV: a row header (the selected-row count, then the
// permuted row of each selected row; 256-byte padded) and the per-slice row
// sums [rows][NB][NSL][kBR] (fp32).  Everything is written before it is read;
// no initial contents needed.  NB = N/8 batches for FC1 (8 gate + 8 up rows
// each), N/16 for FC2.
// nsl = 0 (no table GEMV, no workspace) unless K is a multiple of the slice.
static void lut_geometry(int stage, int N, int K, int& nb, int& nsl) {
  nb = stage == MOE_STAGE_FC1_SWIGLU ? N / 8 : N / 16;
  nsl = K % kSW == 0 ? K / kSW : 0;
}

static size_t lut_header_bytes(int rows) { return (static_cast<size_t>(rows + 1) * sizeof(int) + 255) & ~size_t(255); }

size_t lut_workspace_bytes(int stage, int rows, int N, int K) {
  int nb, nsl;
  lut_geometry(stage, N, K, nb, nsl);
  if (nsl == 0 || rows <= 0) return 0;
  return lut_header_bytes(rows) + static_cast<size_t>(rows) * nb * nsl * kBR * sizeof(float);
}

int lut_workspace_rows(int stage, size_t bytes, int N, int K) {
  int nb, nsl;
  lut_geometry(stage, N, K, nb, nsl);
  if (nsl == 0) return 0;
  const size_t per = static_cast<size_t>(nb) * nsl * kBR * sizeof(float) + sizeof(int);
  int64_t rows = static_cast<int64_t>(bytes / per);
  if (rows > 0x7ffffffe) rows = 0x7ffffffe;
  while (rows > 0 && lut_workspace_bytes(stage, static_cast<int>(rows), N, K) > bytes) --rows;
  return static_cast<int>(rows);
}

bool lut_supported(const MMArgs& a) {
  if (a.wkind != kW2 || a.act_fmt != MOE_FMT_BF16) return false;
  if (a.out_fmt != MOE_FMT_BF16 && a.out_fmt != MOE_FMT_F32) return false;
  if (a.expert_begin != 0 || a.expert_end != a.E || a.E > kMaxE) return false;
  return a.K % kSW == 0 && a.N % 32 == 0;
}

static LutParams lut_params(const MMArgs& a, void* ws) {
  LutParams P;
  P.act = static_cast<const uint16_t*>(a.act);
  P.act_row = a.act_row;
  P.act_row_div = a.act_row_div;
  P.act_rows = a.act_rows;
  P.codes = a.wq;
  P.scales = static_cast<const uint16_t*>(a.wscale);
  P.select_map = a.select_map;
  P.select = a.select;
  P.wslot = a.wslot_of;
  P.slot_lo = a.slot_lo;
  P.slot_hi = a.slot_hi;
  P.split = a.split;
  P.layer = 0;
  P.offsets = a.offsets;
  P.E = a.E;
  P.N = a.N;
  P.K = a.K;
  P.fc1 = a.stage == MOE_STAGE_FC1_SWIGLU;
  P.R = P.fc1 ? 2 * a.N : a.N;
  lut_geometry(a.stage, a.N, a.K, P.NB, P.NSL);
  P.A = a.ws_rows;
  P.rows_hdr = static_cast<int*>(ws);
  P.scratch = reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + lut_header_bytes(a.ws_rows));
  P.out = a.out;
  P.out_fmt = a.out_fmt;
  P.dev_err = a.dev_err;
  return P;
}

cudaError_t launch_lut_gemv(const MMArgs& a, void* ws, cudaStream_t s) {
  const LutParams P = lut_params(a, ws);
  cudaError_t e = set_smem_limit(w2_lut_kernel, kLutSmem);
  if (e != cudaSuccess) return e;
  e = launch_pdl(w2_lut_kernel, dim3(matmul_ctas()), dim3(kLutThreads), kLutSmem, s, P);
  if (e != cudaSuccess) return e;
  // the finishing kernel as a programmatic dependent: its launch overlaps the
  // main kernel's tail; its pdl_wait orders the scratch reads
  const dim3 fgrid(static_cast<unsigned>(a.ws_rows < 4096 ? a.ws_rows : 4096), static_cast<unsigned>((a.N + 255) / 256));
  return launch_pdl(w2_lut_finish_kernel, fgrid, dim3(256), 0, s, P);
}

cudaError_t launch_w2_decode_fused(const MMArgs& fc1, const MMArgs& fc2, void* ws, cudaStream_t s) {
  unsigned int* bar = static_cast<unsigned int*>(ws);
  void* lws = static_cast<uint8_t*>(ws) + 256;
  const LutParams P1 = lut_params(fc1, lws), P2 = lut_params(fc2, lws);
  cudaError_t e = set_smem_limit(w2_decode_fused_kernel, kLutSmem);
  if (e != cudaSuccess) return e;
  // cooperative: every CTA is resident at once (one per SM), which the
  // grid-wide barriers need; programmatic: the launch overlaps the
  // predecessor's tail (the kernel's griddepcontrol.wait orders its reads)
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(device_info().sms);
  cfg.blockDim = dim3(kLutThreads);
  cfg.dynamicSmemBytes = kLutSmem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, w2_decode_fused_kernel, P1, P2, bar, fc1.wait);
}

bool layer_supported(int T, int E, int k) { return T * k <= kLayerA && k <= kLayerK && k <= 32 && E <= kMaxE; }

cudaError_t launch_w2_decode_layer(const LayerArgs& la, const MMArgs& fc1, const MMArgs& fc2, void* ws,
                                   cudaStream_t s) {
  unsigned int* bar = static_cast<unsigned int*>(ws);
  void* lws = static_cast<uint8_t*>(ws) + 256;
  LutParams P1 = lut_params(fc1, lws), P2 = lut_params(fc2, lws);
  P1.layer = 3;  // FC1 reads token rows through the grouping's perm
  P2.layer = 1;
  LayerParams L;
  L.logits = la.logits;
  L.T = la.T;
  L.E = la.E;
  L.k = la.k;
  L.ids = la.ids;
  L.w = la.w;
  L.offsets = la.offsets;
  L.perm = la.perm;
  L.inv = la.inv;
  L.y = static_cast<uint16_t*>(la.y);
  L.out = la.out;
  L.out_fmt = la.out_fmt;
  L.dev_err = fc1.dev_err;
  auto kern = la.E <= 128 ? w2_decode_layer_kernel<4>
              : la.E <= 256 ? w2_decode_layer_kernel<8>
              : la.E <= 512 ? w2_decode_layer_kernel<16>
                            : w2_decode_layer_kernel<32>;
  cudaError_t e = set_smem_limit(kern, kLutSmem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(device_info().sms);
  cfg.blockDim = dim3(kLutThreads);
  cfg.dynamicSmemBytes = kLutSmem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, kern, L, P1, P2, bar, fc1.wait);
}

}  // namespace moe
