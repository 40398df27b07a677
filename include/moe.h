/*
 * libmoe — low-bit routed-expert FFN for one GB300 (sm_103a).
 *
 * The layer (vLLM-Moet README, release v2026.11.03-r23 notes: "FC1 + SwiGLU +
 * MXFP8 quant, FC2"; blog "这个项目我们能学到什么?": 2-bit codebook {-4,-1,1,4}
 * experts and an FP4 delta cache of hot experts; "国产GPU完成MoE大模型Day-0适配"
 * §四: MXFP4 weights converted online into a reused FP8 workspace):
 *
 *   moe_route      top-k softmax routing of router logits
 *   moe_permute    stable grouping of the T*k assignments by expert (+ optional
 *                  gather of activation rows, bf16 or MXFP8-quantised)
 *   moe_w2_mm      expert FC1+SwiGLU or FC2 on 2-bit codebook weights
 *   moe_mxfp4_mm   expert FC1+SwiGLU or FC2 on MXFP4 weights (delta cache) or
 *                  on the FP8 workspace
 *   mxfp4_to_fp8_ws  MXFP4 -> E4M3 conversion into the caller's workspace
 *   moe_combine    out[t] = sum_j w[t,j] * y[inv[t*k+j]]
 *
 * Conventions shared by every call
 * --------------------------------
 *  - Notation: T tokens, E experts, H hidden, I expert intermediate, k experts
 *    per token, A = T*k assignments, a = t*k + j (j = slot in the top-k).
 *  - Every pointer argument is a DEVICE pointer owned by the caller, unless the
 *    comment says "host".  The library never allocates or frees device memory;
 *    the one device memory it keeps is the fixed scratch array of
 *    moe_w2_mm_noalloc, part of its module image.  Buffers must not alias unless a comment allows it.
 *  - Every call is asynchronous on `stream` (a cudaStream_t passed as void*;
 *    NULL = the legacy default stream) and never synchronises the host, except
 *    moe_get_error.
 *  - Every call returns MOE_OK or a status below.  On MOE_ERR_CUDA the CUDA
 *    error text is available from moe_last_error_string() (per thread).
 *  - Data errors found on the device never trap: kernels OR MOE_DEVERR_* bits
 *    into the caller's `dev_err` word (a uint32 in device memory, which the
 *    caller zeroes; may be NULL to ignore) and carry on.  Read with
 *    moe_get_error.
 *  - Thread-safe: the only host-side global state is a per-device property
 *    cache, a per-device record of the kernels whose shared-memory limit was
 *    raised, the bounded-wait limit (moe_set_wait_limit), the side-SM
 *    reservation (moe_set_side_sms) and the per-device
 *    address of moe_w2_mm_noalloc's scratch.
 *  - Every on-chip wait of a pipeline (mbarrier phases) is bounded: a wait
 *    that runs past the limit makes its kernel stop, set MOE_DEVERR_TIMEOUT and
 *    return, so a fault in the pipeline never hangs the GPU.
 *
 * Canonical weight layout (what callers store; parity is stated against it)
 * ---------------------------------------------------------------------------
 *  - W1 of expert e: [2I][H] row-major, K = H contiguous; rows 0..I-1 are the
 *    gate projection, rows I..2I-1 the up projection.
 *  - W2 of expert e: [H][I] row-major, K = I contiguous.
 *  - Experts are stacked on a leading dimension: W1 [E][2I][H], W2 [E][H][I].
 *  - 2-bit codebook: code c in 0..3 is the c-th entry of {-4,-1,1,4}; 4 codes
 *    per byte, element i of a row at bits 2*(i%4) of byte i/4; one fp16 scale
 *    per 32 consecutive K elements, [rows][K/32].  The dequantised weight is
 *    entry * RNE_bf16(scale) (exact in bf16).
 *  - MXFP4 (OCP MX v1.0): E2M1 nibbles, element 2i in the LOW nibble of byte
 *    i; one E8M0 byte per 32 consecutive K elements, [rows][K/32]; value =
 *    E2M1 * 2^(E8M0-127); E8M0 = 255 is NaN.
 *  - moe_w2_mm reads the 2-bit weights in the "w2l" kernel layout written once
 *    by moe_w2_repack (same byte sizes; see there).
 *
 * Shape limits: 1 <= k <= E <= 1024, k <= 32; H and I multiples of 128;
 * T*k < 2^31.
 */
#ifndef BIT_MOE_EXPERT_TOP_MOE_H
#define BIT_MOE_EXPERT_TOP_MOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MOE_ABI_VERSION 1

#if defined(__GNUC__)
#define MOE_API __attribute__((visibility("default")))
#else
#define MOE_API
#endif

/* status codes */
#define MOE_OK 0
#define MOE_ERR_ARG 1          /* NULL / misaligned pointer, bad shape or enum     */
#define MOE_ERR_WS_SMALL 2     /* workspace smaller than the *_workspace_size query */
#define MOE_ERR_UNSUPPORTED 3  /* device is not sm_103 / sm_100 family, or format combination not built */
#define MOE_ERR_CUDA 4         /* a CUDA call failed; see moe_last_error_string()   */

/* bits a kernel ORs into *dev_err */
#define MOE_DEVERR_BAD_ID 0x1u       /* expert id outside [0, E)                        */
#define MOE_DEVERR_NAN_LOGIT 0x2u    /* NaN router logit (ranked below every number)    */
#define MOE_DEVERR_NAN_SCALE 0x4u    /* E8M0 scale byte 255 (NaN) in MXFP4 weights      */
#define MOE_DEVERR_TIMEOUT 0x8u      /* a bounded on-chip wait gave up; outputs invalid */
#define MOE_DEVERR_OVERFLOW 0x10u    /* an expert group exceeded a kernel's row limit   */
#define MOE_DEVERR_LAUNCH 0x20u      /* a kernel found its launch short of what its layout
                                        needs (dynamic shared memory) and did nothing   */

/* activation / output formats */
#define MOE_FMT_NONE 0
#define MOE_FMT_BF16 1   /* uint16 bf16 bit patterns, [rows][cols]                       */
#define MOE_FMT_F32 2    /* float, [rows][cols]                                          */
#define MOE_FMT_MXFP8 3  /* E4M3 bytes [rows][cols] + E8M0 bytes [rows][cols/32] (OCP MX)  */
#define MOE_FMT_MXFP8_BF16 4  /* MXFP8-quantised values (OCP MX rounding, as MOE_FMT_MXFP8)
                                 stored as bf16 [rows][cols]: each element is q * 2^X exactly
                                 (for |values| >= 2^-133).  The tensor-core path's form of
                                 MXFP8 activations: its matmul reads bf16. */

/* expert matmul stage */
#define MOE_STAGE_FC1_SWIGLU 1  /* h[p][n] = silu(g)*u, g/u = gate/up rows of W1, n < I */
#define MOE_STAGE_FC2 2         /* y[p][n] = W2 row n . h[p],               n < H       */

/* expert matmul mode */
#define MOE_MODE_AUTO 0  /* GEMV for small groups, tensor-core GEMM for large ones */
#define MOE_MODE_GEMV 1  /* CUDA-core grouped GEMV (any group size)               */
#define MOE_MODE_GEMM 2  /* tcgen05 tensor-core grouped GEMM                      */
#define MOE_MODE_SPLIT 3 /* moe_w2_mm only: per group, GEMV for one row, GEMM for more */

/* Library version (MOE_ABI_VERSION). */
MOE_API int moe_version(void);

/* Text of the last MOE_ERR_* raised on the calling host thread ("" if none).
 * The pointer stays valid until the next library call on this thread. */
MOE_API const char* moe_last_error_string(void);

/* Synchronises `stream`, then copies the device word *dev_err to the host
 * word *bits (host pointer).  The device word is left unchanged. */
MOE_API int moe_get_error(const uint32_t* dev_err, void* stream, uint32_t* bits);

/* Sets the bounded-wait limit, in SM clock cycles, that expert-matmul
 * launches made after this call pass to their kernels (cycles <= 0 restores
 * the default, 3e9 cycles, about 1.5 s at 2 GHz).  Returns the previous
 * limit.  Process-wide; host only. */
MOE_API long long moe_set_wait_limit(long long cycles);

/* Reserves n SMs of the device for the copy kernels that run on a side
 * stream beside the expert matmuls: the MXFP4 -> FP8 workspace conversion of
 * the next expert batch ("国产GPU完成MoE大模型Day-0适配" §四: conversion
 * overlapped with the current batch's matmuls on another stream) and the copy
 * of routed host-resident experts into device slots (moe_cache_fill; the blog
 * "这个项目我们能学到什么?", "GPU作为专家缓存").  With 0 < n < the SM count,
 * the persistent matmul kernels launched after this call (moe_w2_mm /
 * moe_w2_mm_slots on the table GEMV, moe_w2_mm / moe_mxfp4_mm in GEMM mode)
 * take one CTA per remaining SM, and mxfp4_to_fp8_ws / moe_cache_fill launch
 * n CTAs that hold one SM each, so the two share the GPU whatever order they
 * start in; results are unchanged (every tile, row and block is computed the
 * same way).  0 (the default) gives every launch the whole GPU.  Returns the
 * previous value, or -1 (setting unchanged) for n < 0 or n > 1024.
 * Process-wide; host only. */
MOE_API int moe_set_side_sms(int n);

/* Self-test of the bounded wait (no counterpart in the pages): launches one
 * warp that waits, with limit `cycles` (1 .. 3e9), on a shared-memory
 * mbarrier that nothing ever arrives on, using the pipelines' wait.  When the
 * limit runs out the kernel ORs MOE_DEVERR_TIMEOUT into *dev_err and returns;
 * the context stays usable.  No copy or MMA is in flight in that kernel. */
MOE_API int moe_check_bounded_wait(long long cycles, uint32_t* dev_err, void* stream);

/* ------------------------------------------------------------------ routing
 * Top-k softmax routing (vLLM-Moet README line table: 384 routed experts per
 * layer; "top-8 softmax routing").
 *   logits  float [T][E]
 *   ids     int32 [T][k]  out: experts ordered by (logit desc, id asc); NaN
 *                         logits rank below every number (sets NAN_LOGIT)
 *   w       float [T][k]  out: w_j = exp(l_j - l_0) / sum_j' exp(l_j' - l_0)
 *                         (softmax renormalised over the k selected; sums to 1)
 * T = 0 is a no-op. */
MOE_API int moe_route(const float* logits, int T, int E, int k, int32_t* ids, float* w,
              uint32_t* dev_err, void* stream);

/* ------------------------------------------------------------------ grouping
 * Stable counting sort of the A = T*k assignments by expert id: the
 * per-expert token groups the expert matmuls run on (vLLM-Moet README,
 * release v2026.11.03-r23 notes: the prefill MoE step; the MXFP8 gather
 * is its "MXFP8 quant" of the activations).
 *   ids      int32 [T][k]   expert of each assignment (ids outside [0,E) set
 *                           BAD_ID; such an assignment gets inv = -1 and no row)
 *   offsets  int32 [E+1]    out: group e occupies permuted rows
 *                           offsets[e] .. offsets[e+1]-1; offsets[0] = 0
 *   perm     int32 [A]      out: perm[p] = assignment a of permuted row p, rows of
 *                           one group in increasing a
 *   inv      int32 [A]      out: inv[perm[p]] = p
 *   x        bf16 [T][H]    optional activations (NULL when act_fmt = NONE)
 *   act_fmt  MOE_FMT_NONE: no gather; MOE_FMT_BF16: x_perm[p] = x[perm[p]/k]
 *            (MOE_FMT_MXFP8_BF16: the same rows MXFP8-rounded, stored as bf16);
 *            (bf16 [A][H]); MOE_FMT_MXFP8: x_perm[p] = MXFP8(x[perm[p]/k]),
 *            E4M3 [A][H] + E8M0 x_perm_scale [A][H/32] (OCP MX: per block of 32,
 *            scale 2^(floor(log2 amax) - 8), elements RNE + saturate).
 *   ws       unused (pass NULL, 0); kept so the signature stays stable.
 * Deterministic and atomics-free in its outputs. */
MOE_API size_t moe_permute_workspace_size(int T, int k, int E);
MOE_API int moe_permute(const int32_t* ids, int T, int k, int E,
                int32_t* offsets, int32_t* perm, int32_t* inv,
                const uint16_t* x, int H, int act_fmt, void* x_perm, uint8_t* x_perm_scale,
                void* ws, size_t ws_bytes, uint32_t* dev_err, void* stream);

/* rows[a] = rows_perm[inv[a]] for a < A (the inverse of the gather; no page
 * has it: the identity unpermute(permute(x)) = x is a test of the grouping).  fmt is
 * MOE_FMT_BF16 or MOE_FMT_F32; cols elements per row.  A test helper. */
MOE_API int moe_unpermute(const void* rows_perm, int fmt, const int32_t* inv, int A, int cols,
                  void* rows, void* stream);

/* ------------------------------------------------------------------ weights
 * Rewrite canonical 2-bit weights (blog "这个项目我们能学到什么?": codebook
 * {-4,-1,1,4}, one fp16 scale per 32) into the w2l kernel layout (run once,
 * at load).
 *   codes   uint8 [mats][R][K/4] canonical;   scales fp16 [mats][R][K/32]
 *   codes_k uint8 [mats][R][K/4] out;         scales_k bf16 [mats][R][K/32] out
 * w2l keeps the canonical code bytes but moves whole 32-bit words (16
 * elements): K is cut into slices of SW elements (SW = K if K <= 512, else the
 * largest of 512/256/128 dividing K); word (row, slice s, lane l) — elements
 * s*SW + 16l .. +15 of the row — is stored at word index
 *   s*(R*SW/16) + (row/4)*(4*SW/16) + 4l + row%4
 * of its matrix, and scale (row, slice s, group g of the slice) at
 *   s*(R*SW/32) + (row/4)*(4*SW/32) + 4g + row%4,
 * converted to RNE_bf16(fp16 scale) (the scale the dequantised weights use).
 * Any block of 4n rows of one slice is then contiguous.  `mats` counts the
 * stacked matrices (E), R the rows of one (2I for W1, H for W2); R % 4 == 0. */
MOE_API int moe_w2_repack(const uint8_t* codes, const uint16_t* scales, int64_t mats, int R, int K,
                  uint8_t* codes_k, uint16_t* scales_k, void* stream);

/* Exact dequantised values (bf16 bit patterns [mats][R][K]) of w2l weights
 * (the same blog's 2-bit codebook experts):
 * entry * RNE_bf16(scale), the values the expert matmuls compute with. */
MOE_API int moe_dequant_w2(const uint8_t* codes_k, const uint16_t* scales_k, int64_t mats, int R, int K,
                   uint16_t* out_bf16, void* stream);

/* Exact dequantised MXFP4 values (OCP MX v1.0 E2M1 x E8M0; the vLLM-Moet
 * README's MXFP4 experts) as float [rows][K] (NaN where the scale is 255). */
MOE_API int moe_dequant_mxfp4(const uint8_t* e2m1, const uint8_t* e8m0, int64_t rows, int K,
                      float* out_f32, void* stream);

/* MXFP4 -> FP8 workspace ("国产GPU完成MoE大模型Day-0适配" §四: weights stay MXFP4,
 * the needed expert blocks are converted online into a preallocated FP8
 * workspace that is reused).
 *   e2m1, e8m0  MXFP4 matrices stacked [n_src][rows][K/2], [n_src][rows][K/32]
 *   experts     int32 [n_experts] (device): source matrix index of each converted expert
 *   ws_slots    int32 [n_experts] (device): destination slot of each
 *   ws          uint8 workspace; slot s is the E4M3 matrix at ws + s*rows*K
 *               (scale folded in: byte = E4M3_RNE_satfinite(E2M1 * 2^(E8M0-127)),
 *               0x7F where the scale is NaN, which also sets NAN_SCALE)
 *   ws_bytes    capacity; every slot must fit (checked on the device: a slot
 *               that does not fit sets OVERFLOW and is skipped)
 * Exact for every code when E8M0-127 lies in [-8, 6]. */
MOE_API int mxfp4_to_fp8_ws(const uint8_t* e2m1, const uint8_t* e8m0, const int32_t* experts, int n_experts,
                    int rows, int K, uint8_t* ws, size_t ws_bytes, const int32_t* ws_slots,
                    uint32_t* dev_err, void* stream);

/* ------------------------------------------------------------------ expert matmuls
 * The expert FFN (vLLM-Moet README, release v2026.11.03-r23 notes: "FC1 +
 * SwiGLU + MXFP8 quant, FC2"; line table: 2-bit codebook experts, 384 per
 * layer) on low-bit weights dequantised inside the matmul.
 * For every expert e whose group is non-empty and selected (see below), for
 * every permuted row p of the group (offsets[e] <= p < offsets[e+1]):
 *   activation row a_p = act row (act_row ? act_row[p] / act_row_div : p), K elements;
 *   act holds act_rows rows (T for token rows read through act_row, A for
 *   permuted rows); a row index outside [0, act_rows) sets BAD_ID
 *   FC1_SWIGLU: g_n = W1_e[n] . a_p, u_n = W1_e[N+n] . a_p (fp32);
 *               out[p][n] = silu(g_n) * u_n, n < N (N = I); weights have 2N rows
 *   FC2:        out[p][n] = W2_e[n] . a_p, n < N (N = H); weights have N rows
 * Formats: act_fmt BF16 or MXFP8 (act_scale = E8M0 [rows][K/32]); out_fmt BF16
 * or F32, and MXFP8 for FC1 (out_scale receives E8M0 [rows][N/32]); FC1 on the
 * tensor-core path (GEMM) also takes out_fmt MXFP8_BF16 (h MXFP8-rounded, as
 * bf16), the form its FC2 reads.  Rounding:
 * out = RNE of the fp32 result into out_fmt.  Rows of unselected experts are
 * left untouched.  A call whose activation has no rows (act_rows == 0, e.g.
 * an empty token batch) checks its scalar arguments and otherwise does
 * nothing: its buffers may be empty and their pointers NULL.  This holds for
 * every expert-matmul entry point (moe_w2_mm, moe_w2_mm_noalloc,
 * moe_w2_decode_fused, moe_mxfp4_mm, moe_w2_mm_slots).
 * Modes: GEMV = CUDA-core kernels (2-bit with a workspace and K a multiple
 * of 512: shared-memory partial-sum tables with K split in 512-element
 * slices over CTAs; otherwise, and for MXFP4 / FP8: register decode); GEMM =
 * tcgen05 tensor-core kernel with the dequantised weights in tensor memory,
 * for 2-bit, MXFP4 and FP8-workspace weights, on bf16 activations already
 * permuted (act_row must be NULL), K a multiple of 64, N a multiple of 128
 * (FC1) or 256 (FC2); 2-bit FC2 with N a multiple of 128 only goes to an
 * older tcgen05 kernel with the weights in shared memory; a call that fits
 * neither runs as GEMV (MXFP8_BF16 output excepted: MOE_ERR_UNSUPPORTED).
 * AUTO = GEMM when act_row is NULL, act_rows >= 2048 and the shape is
 * supported, else GEMV.
 * SPLIT (moe_w2_mm only; act_row must be NULL): groups of one row go to the
 * table GEMV (which streams an expert's weights once per row) and groups of
 * two rows or more to the tensor-core GEMM (once per expert for all its rows
 * in a 32- or 128-row token tile), as two launches over disjoint experts;
 * needs a workspace and a shape both take, else every group runs as GEMV.
 * Each row's result is that of the path its group took.
 *   ws, ws_bytes (moe_w2_mm): scratch of the 2-bit GEMV, at least
 *        moe_w2_mm_workspace_size(stage, A, N, K) bytes for A permuted rows,
 *        256-byte aligned.  Its contents on entry do not matter (every value
 *        is written before it is read), so FC1 and FC2 may share one.  The
 *        size query returns 0 for shapes the table GEMV does not take (K not
 *        a multiple of 512): a workspace passed with those is ignored.
 *        With ws == NULL the 2-bit GEMV uses the slower register-decode kernel.
 *        A row beyond the workspace's capacity sets OVERFLOW and is skipped.
 *        Calls that share one workspace must not overlap on the GPU.
 *   ws (moe_mxfp4_mm): unused (NULL, 0).
 */
MOE_API size_t moe_w2_mm_workspace_size(int stage, int rows, int N, int K);

MOE_API int moe_w2_mm(int stage, int mode,
              const void* act, int act_fmt, const uint8_t* act_scale, int act_rows,
              const int32_t* act_row, int act_row_div,
              const uint8_t* codes_k, const uint16_t* scales_k,  /* w2l [E][rows][K/4], [E][rows][K/32] */
              const int32_t* offsets, const int32_t* expert_slot, /* nullable: skip e with expert_slot[e] >= 0 */
              int E, int N, int K,
              void* out, int out_fmt, uint8_t* out_scale,
              void* ws, size_t ws_bytes, uint32_t* dev_err, void* stream);

/* moe_w2_mm_noalloc: the 2-bit table GEMV of moe_w2_mm (decode), run on a
 * scratch array that the library holds itself.  None of the pages has a
 * counterpart: it exists for callers that cannot pass a workspace, e.g. C host
 * code with no device allocator of its own, or a serving engine that has given
 * all spare device memory to its KV cache and may not allocate while decoding.
 * The call allocates and frees nothing.
 *
 * Computes exactly what moe_w2_mm computes with mode GEMV and a workspace
 * (same kernel, same summation order: the outputs are bit-identical), with
 *   act     bf16 [act_rows][K] (act_fmt is BF16; act_row / act_row_div as in
 *           moe_w2_mm); out_fmt BF16 or F32 (no MXFP8 output)
 *   rows    the number of permuted rows the call covers (offsets[E], e.g. T*k);
 *           a row p >= rows sets OVERFLOW and is skipped
 * Limit: moe_w2_mm_workspace_size(stage, rows, N, K) must not exceed
 * MOE_W2_NOALLOC_SCRATCH_BYTES (16 MiB: 127 rows of FC1 at H=4096, I=2048, or
 * 255 rows of FC2), else MOE_ERR_WS_SMALL.  Shapes the table GEMV does not
 * take (K not a multiple of its slice width) give MOE_ERR_UNSUPPORTED.
 * Set-up: the first call on a device, with that device current, looks up the
 * scratch's device address (cudaGetSymbolAddress, which may load the module);
 * make that first call before any stream capture.  The address is cached per
 * device until the process exits: after cudaDeviceReset on a device the
 * cached address is stale, so do not call this entry point there again.  Nothing in the scratch
 * needs to start at zero, so a call issues no copy or memset.
 * One scratch per device: calls that overlap on the GPU (other streams or
 * threads) race on it and give wrong results; serialise them. */
#define MOE_W2_NOALLOC_SCRATCH_BYTES (16u << 20)

MOE_API int moe_w2_mm_noalloc(int stage,
                      const void* act, int act_rows, const int32_t* act_row, int act_row_div,
                      const uint8_t* codes_k, const uint16_t* scales_k,
                      const int32_t* offsets, const int32_t* expert_slot,
                      int E, int N, int K, int rows,
                      void* out, int out_fmt, uint32_t* dev_err, void* stream);

/* FC1 + SwiGLU and FC2 of a 2-bit decode step in ONE kernel launch (vLLM-Moet
 * README, "MoET hybrid": the decode MoE runs inside a captured CUDA graph;
 * here the two expert matmuls and their summing steps are one persistent
 * cooperative kernel, every CTA resident, with grid-wide barriers between
 * FC1's tables, FC1's sums, FC2's tables and FC2's sums).  Computes exactly
 * moe_w2_mm(FC1, GEMV, x via act_row -> h bf16) then moe_w2_mm(FC2, GEMV,
 * h -> y): same kernels' arithmetic and summation order, bit-identical h and y.
 *   x         bf16 [act_rows][H] token rows, read through act_row / act_row_div
 *             (as moe_w2_mm); h bf16 [rows][I] out; y [rows][H] out in y_fmt
 *             (BF16 or F32); rows = offsets[E]
 *   codes1/scales1, codes2/scales2  w2l weights of W1 [E][2I][H/4] and W2
 *   expert_slot  nullable: experts with expert_slot[e] >= 0 are skipped
 *   ws        >= moe_w2_decode_fused_workspace_size(rows, H, I) bytes,
 *             256-byte aligned; its first 4 bytes are the barrier counter,
 *             which must be zero before the first call (e.g. a zero-filled
 *             workspace) and which every call leaves at zero; the rest is the
 *             table GEMV's scratch shared by both stages.  Calls that share
 *             one workspace must not overlap on the GPU
 * H and I multiples of 512, else MOE_ERR_UNSUPPORTED.  Every grid barrier is a
 * bounded wait (MOE_DEVERR_TIMEOUT, then the kernel returns); after a timeout
 * the counter is left non-zero and must be zeroed again before the next call. */
MOE_API size_t moe_w2_decode_fused_workspace_size(int rows, int H, int I);
MOE_API int moe_w2_decode_fused(const void* x, int act_rows, const int32_t* act_row, int act_row_div,
                        const uint8_t* codes1, const uint16_t* scales1, const uint8_t* codes2,
                        const uint16_t* scales2, const int32_t* offsets, const int32_t* expert_slot,
                        int E, int H, int I, void* h, void* y, int y_fmt, void* ws, size_t ws_bytes,
                        uint32_t* dev_err, void* stream);

/* One whole 2-bit decode layer step in ONE kernel launch (vLLM-Moet README,
 * "MoET hybrid": the decode MoE inside a captured CUDA graph; here routing,
 * grouping, both expert matmuls and the combine are one persistent
 * cooperative kernel).  Computes exactly
 *   moe_route(logits -> ids, w), moe_permute(ids -> offsets, perm, inv; no
 *   gather), moe_w2_decode_fused(x via perm / k -> h, y bf16),
 *   moe_combine(y, w, inv -> out)
 * with the same arithmetic and order: every output is bit-identical to
 * those four calls.  Every CTA routes and groups the whole step in its own
 * shared memory; the combine runs inside FC2's summing step.
 *   logits   float [T][E]; x bf16 [T][H]
 *   codes1/scales1, codes2/scales2  w2l weights of W1 [E][2I][H/4] and W2
 *   ids int32 [T][k], w float [T][k], offsets int32 [E+1], perm / inv int32
 *            [T*k], h bf16 [T*k][I], y bf16 [T*k][H]: out, as the four calls
 *            write them; out [T][H] in out_fmt (BF16 or F32)
 *   ws       >= moe_w2_decode_layer_workspace_size(T, k, H, I) bytes, the
 *            workspace of moe_w2_decode_fused for T*k rows (same barrier
 *            counter rule: zero before the first call, left at zero)
 * Limits: T*k <= 256, k <= 16, E <= 1024, H and I multiples of 512, else
 * MOE_ERR_UNSUPPORTED (T*k, k) or MOE_ERR_ARG (E, k > E).  T = 0 zeroes
 * offsets and launches nothing.  A NaN logit sets NAN_LOGIT, as moe_route
 * does.  Grid barriers are bounded waits (MOE_DEVERR_TIMEOUT). */
MOE_API size_t moe_w2_decode_layer_workspace_size(int T, int k, int H, int I);
MOE_API int moe_w2_decode_layer(const float* logits, const void* x, int T, int E, int k,
                        const uint8_t* codes1, const uint16_t* scales1, const uint8_t* codes2,
                        const uint16_t* scales2, int H, int I, int32_t* ids, float* w, int32_t* offsets,
                        int32_t* perm, int32_t* inv, void* h, void* y, void* out, int out_fmt, void* ws,
                        size_t ws_bytes, uint32_t* dev_err, void* stream);

/* As moe_w2_mm for MXFP4 weights (blog "这个项目我们能学到什么?": the FP4
 * delta cache of hot experts; OCP MX E2M1 + E8M0), or for FP8 workspace
 * weights ("国产GPU完成MoE大模型Day-0适配" §四: the matmul reads the reused FP8
 * workspace).  With MXFP8 activations on the tensor-core path (mode GEMM or
 * AUTO at prefill sizes, act_row NULL, K a multiple of 128) both weight forms
 * run on the block-scaled FP8 tensor core (tcgen05 kind::mxf8f6f4: E4M3 or
 * E2M1 codes with their E8M0 block scales, MXFP8 tokens), and FC1 may write h
 * as MXFP8 (out_scale E8M0 [rows][N/32]).
 * Weight source, exactly one of:
 *   e2m1/e8m0 non-NULL: MXFP4 slots [S][rows][K/2], [S][rows][K/32]; expert e
 *       uses slot expert_slot[e] (experts with expert_slot[e] < 0 are skipped;
 *       expert_slot NULL means slot = e).  Slots are below E; on the
 *       tensor-core path a slot >= E sets MOE_DEVERR_BAD_ID and its expert is
 *       skipped.
 *   fp8_ws non-NULL: E4M3 workspace, expert e uses slot ws_slot_of_expert[e]
 *       (rows*K bytes per slot, as written by mxfp4_to_fp8_ws); experts with a
 *       negative slot are skipped.  Slots are below E (a workspace holds at
 *       most one slot per expert); on the tensor-core path (MOE_MODE_GEMM) a
 *       slot >= E sets MOE_DEVERR_BAD_ID and its expert is skipped.
 * Only experts e in [expert_begin, expert_end) are processed. */
MOE_API int moe_mxfp4_mm(int stage, int mode,
                 const void* act, int act_fmt, const uint8_t* act_scale, int act_rows,
                 const int32_t* act_row, int act_row_div,
                 const uint8_t* e2m1, const uint8_t* e8m0,
                 const uint8_t* fp8_ws, const int32_t* ws_slot_of_expert,
                 const int32_t* offsets, const int32_t* expert_slot,
                 int expert_begin, int expert_end,
                 int E, int N, int K,
                 void* out, int out_fmt, uint8_t* out_scale,
                 void* ws, size_t ws_bytes, uint32_t* dev_err, void* stream);

/* ------------------------------------------------------------------ FP4 delta cache
 * Which experts hold an MXFP4 slot of the delta cache, kept on the device and
 * updated between steps from the routing, with no host sync (blog
 * "这个项目我们能学到什么?" on vLLM-Moet: the hottest experts are kept at FP4
 * precision over the 2-bit base; "GPU作为专家缓存": the GPU holds the hot
 * experts).  The policy is this library's reading (the pages fix it nowhere):
 *   counts   uint32 [E] (in/out): per-expert hotness, an integer moving
 *            average of routed assignments: c <- c - (c >> decay_shift) + n_e,
 *            n_e = offsets[e+1] - offsets[e] of this step; decay_shift >= 31
 *            keeps the cumulative count; saturates at 2^32 - 1.  Zero them
 *            once before the first call.
 *   the cached set is the S experts of largest count, ties to the lowest id;
 *   slot_expert int32 [S] (in/out): expert held by slot s, -1 = empty; a
 *            cached expert that stays in the set keeps its slot, experts that
 *            leave free theirs, experts that enter take the free slots in
 *            ascending order, hottest first.  (Entries >= E set BAD_ID and are
 *            treated as empty.)
 *   expert_slot int32 [E] (out): the inverse map, -1 = not cached: the map
 *            moe_w2_mm / moe_mxfp4_mm take as expert_slot.
 *   promoted int32 [S] (out): the expert that entered slot s in this call, -1
 *            where the slot kept its expert or stays empty; moe_cache_fill
 *            copies exactly these.
 * 1 <= S <= E <= 1024.  One small kernel; stream-ordered with the steps. */
MOE_API int moe_cache_select(const int32_t* offsets, int E, uint32_t* counts, int decay_shift, int S,
                     int32_t* expert_slot, int32_t* slot_expert, int32_t* promoted,
                     uint32_t* dev_err, void* stream);

/* ------------------------------------------------------------------ host-resident experts
 * Experts kept in host memory, staged into device memory per step (blog
 * "这个项目我们能学到什么?" on vLLM-Moet: the GPU as a cache of hot experts,
 * the rest fetched as needed; vLLM-Moet README, "MoET hybrid"): a pool of
 * R + S weight slots in device memory, slots [0, R) hold resident experts,
 * slots [R, R + S) are staging slots refilled every step.
 *   res_slot    int32 [E]: resident slot of each expert, -1 = host-resident
 *               (an entry >= R sets BAD_ID and counts as host-resident)
 *   weight_slot int32 [E] (out): the slot each routed expert is read from
 *               this step: its resident slot, or R + j for the j-th routed
 *               host-resident expert (ascending expert id); -1 when more than
 *               S host-resident experts are routed (OVERFLOW; skipped)
 *   staged      int32 [S] (out): the expert to copy into staging slot R + j,
 *               -1 = unused; pass it to moe_cache_fill with the store's
 *               arrays as src and the pool's slot-R addresses as dst
 * 1 <= E <= 1024, 1 <= S <= 1024.  One small kernel. */
MOE_API int moe_stage_select(const int32_t* offsets, int E, const int32_t* res_slot, int R, int S,
                     int32_t* weight_slot, int32_t* staged, uint32_t* dev_err, void* stream);

/* The 2-bit table GEMV of moe_w2_mm (stage FC1 or FC2, bf16 activations,
 * BF16 or F32 output) with the weights addressed through a slot map: expert
 * e is read from slot weight_slot[e] of the w2l arrays codes_k / scales_k
 * (slot-major, the per-expert sizes of moe_w2_repack), and only experts whose
 * slot lies in [slot_lo, slot_hi) are computed (rows of the others are left
 * untouched), so the resident and the staged experts of a step can run as two
 * calls around the staging copy.  Outputs are bit-identical to moe_w2_mm's
 * for the same rows.  Needs the table GEMV's shapes (K a multiple of 512,
 * else MOE_ERR_UNSUPPORTED) and its workspace (ws, ws_bytes as moe_w2_mm). */
MOE_API int moe_w2_mm_slots(int stage, const void* act, int act_rows, const int32_t* act_row, int act_row_div,
                    const uint8_t* codes_k, const uint16_t* scales_k, const int32_t* offsets,
                    const int32_t* weight_slot, int slot_lo, int slot_hi, int E, int N, int K,
                    void* out, int out_fmt, void* ws, size_t ws_bytes, uint32_t* dev_err, void* stream);

/* Copies the stored weights of each promoted expert into its slot: for every
 * slot s with promoted[s] = e >= 0 and every array a < n_arrays (at most 4,
 * e.g. W1 nibbles, W1 scales, W2 nibbles, W2 scales):
 *   dst[a] + s * bytes[a]  <-  src[a] + e * bytes[a]        (bytes[a] bytes)
 * src, dst and bytes are HOST arrays of n_arrays entries; src[a] and dst[a]
 * point to device-accessible memory: device memory, or pinned host memory
 * mapped into the device's address space (the expert store may stay in host
 * memory and be read over the CPU-GPU link).  Pointers 16-byte aligned,
 * bytes[a] a multiple of 16.  Slots that were not promoted are not touched,
 * so steps that use other slots may follow on the same stream. */
MOE_API int moe_cache_fill(const int32_t* promoted, int S, int n_arrays, const void* const* src, void* const* dst,
                   const size_t* bytes, void* stream);

/* ------------------------------------------------------------------ combine
 * The weighted combine of the routed experts' outputs (the top-k softmax
 * weights of moe_route; vLLM-Moet README line table, top-k routing):
 * out[t][n] = sum_{j=0..k-1} w[t][j] * y[inv[t*k+j]][n], accumulated in fp32 in
 * ascending j, then rounded to out_fmt (BF16 or F32).  One owner per output
 * row: deterministic, no atomics.  Assignments with inv < 0 contribute nothing.
 *   y    [A][H] in y_fmt (BF16 or F32), permuted row order */
MOE_API int moe_combine(const void* y, int y_fmt, const float* w, const int32_t* inv,
                int T, int k, int H, void* out, int out_fmt, void* stream);

#ifdef __cplusplus
}
#endif
#endif
