// Internal launch interface between the C-ABI layer (abi.cu) and the kernel
// translation units.  Plain types only.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"

namespace moe {

// Launch `kernel` as a programmatic dependent of the preceding work in `s`:
// its launch and any prologue before pdl_wait() overlap the predecessor's
// tail (captured into CUDA graphs as programmatic edges).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                       Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

struct DeviceInfo {
  int device = -1;
  int sms = 0;
  int major = 0, minor = 0;
  size_t smem_optin = 0;
};
// Cached properties of the current device.
const DeviceInfo& device_info();

// Raises `kernel`'s dynamic shared-memory limit to `bytes` on the current
// device, once per (device, kernel, size); thread-safe.
cudaError_t set_smem_limit(const void* kernel, int bytes);
template <typename K>
cudaError_t set_smem_limit(K* kernel, int bytes) {
  return set_smem_limit(reinterpret_cast<const void*>(kernel), bytes);
}

// The bounded-wait limit (SM clock cycles) that launches pass to their
// kernels (moe_set_wait_limit).
long long wait_limit();

// SMs reserved on this device for the side-stream copy kernels (workspace
// conversion, expert cache fill; moe_set_side_sms; 0: none), and the CTAs of
// a persistent matmul (one per SM that is not reserved).
int side_sms();
int matmul_ctas();

// ---- route / permute / combine (route_permute.cu)
cudaError_t launch_route(const float* logits, int T, int E, int k, int32_t* ids, float* w, uint32_t* dev_err,
                         cudaStream_t s);
cudaError_t launch_permute(const int32_t* ids, int T, int k, int E, int32_t* offsets, int32_t* perm, int32_t* inv,
                           void* ws, size_t ws_bytes, uint32_t* dev_err, cudaStream_t s);
// workspace of the multi-CTA grouping (0: the single-CTA kernel does it)
size_t permute_workspace_bytes(int A, int E);
cudaError_t launch_gather(const uint16_t* x, const int32_t* inv, int T, int k, int H, int act_fmt, void* x_perm,
                          uint8_t* x_perm_scale, cudaStream_t s);
cudaError_t launch_unpermute(const void* rows_perm, int fmt, const int32_t* inv, int A, int cols, void* rows,
                             cudaStream_t s);
cudaError_t launch_combine(const void* y, int y_fmt, const float* w, const int32_t* inv, int T, int k, int H,
                           void* out, int out_fmt, cudaStream_t s);

// ---- weight formats (convert.cu)
cudaError_t launch_w2_repack(const uint8_t* codes, const uint16_t* scales, int64_t mats, int64_t R, int K,
                             uint8_t* codes_k, uint16_t* scales_k, cudaStream_t s);
cudaError_t launch_dequant_w2(const uint8_t* codes_k, const uint16_t* scales_k, int64_t mats, int64_t R, int K,
                              uint16_t* out, cudaStream_t s);
cudaError_t launch_dequant_mxfp4(const uint8_t* e2m1, const uint8_t* e8m0, int64_t rows, int K, float* out,
                                 cudaStream_t s);
cudaError_t launch_mxfp4_to_fp8(const uint8_t* e2m1, const uint8_t* e8m0, const int32_t* experts, int n_experts,
                                int rows, int K, uint8_t* ws, size_t ws_bytes, const int32_t* ws_slots,
                                uint32_t* dev_err, cudaStream_t s);

// ---- expert matmuls on CUDA cores (gemv.cu)
enum WeightKind { kW2 = 0, kMXFP4 = 1, kFP8 = 2 };

// MOE_MODE_SPLIT: groups of this many rows or more go to the tensor-core
// kernel (one pass over the expert's weights for all its rows), smaller ones
// to the table GEMV (one pass per row).
constexpr int kSplitRows = 2;

struct MMArgs {
  int stage;  // MOE_STAGE_*
  const void* act;
  int act_fmt;
  const uint8_t* act_scale;
  int act_rows;               // rows of act (bounds of the gathered row index)
  void* ws;                   // caller workspace (LUT GEMV scratch), may be NULL
  size_t ws_bytes;
  int ws_rows;                // permuted rows the workspace covers
  int mode;                   // MOE_MODE_*
  const int32_t* act_row;
  int act_row_div;
  int wkind;                  // WeightKind
  const uint8_t* wq;          // codes / nibbles / e4m3 bytes, [slots][rows][K*bits/8]
  const void* wscale;         // bf16 (w2k) or E8M0 [slots][rows][K/32]; NULL for FP8
  const int32_t* wslot_of;    // expert -> weight slot (nullable: slot = e)
  int slot_lo, slot_hi;       // 2-bit table GEMV with wslot_of: experts whose slot is in [slot_lo, slot_hi)
  const int32_t* select_map;  // per-expert map read by `select`
  int select;                 // 0: all experts; 1: experts with select_map[e] < 0 (the
                              // 2-bit pass skips delta-cached experts); 2: select_map[e] >= 0
  int split;                  // 0: every group; 1: groups of fewer than kSplitRows rows;
                              // 2: groups of kSplitRows rows or more (MOE_MODE_SPLIT halves)
  const int32_t* offsets;
  int expert_begin, expert_end;
  int E, N, K;
  void* out;
  int out_fmt;
  uint8_t* out_scale;
  uint32_t* dev_err;
  long long wait;             // bounded-wait limit in SM clock cycles
};
// Dispatch: the shared-memory LUT GEMV for 2-bit weights when the shape allows,
// else the generic CUDA-core kernel.
cudaError_t launch_gemv(const MMArgs& a, cudaStream_t s);
cudaError_t launch_gemv_generic(const MMArgs& a, cudaStream_t s);
bool lut_supported(const MMArgs& a);
size_t lut_workspace_bytes(int stage, int rows, int N, int K);
int lut_workspace_rows(int stage, size_t bytes, int N, int K);
cudaError_t launch_lut_gemv(const MMArgs& a, void* ws, cudaStream_t s);
// FC1 and FC2 of the table GEMV in one cooperative launch; ws = 256 bytes of
// barrier counter, then the table GEMV's workspace (shared by both stages)
cudaError_t launch_w2_decode_fused(const MMArgs& fc1, const MMArgs& fc2, void* ws, cudaStream_t s);
bool gemm_supported(const MMArgs& a);
cudaError_t launch_gemm_tc(const MMArgs& a, int rows_total, cudaStream_t s);
// tensor-core grouped matmul with the dequantised weights in TMEM (gemm_tmem.cu)
bool tmem_mm_supported(const MMArgs& a);
// block-scaled FP8 tensor-core matmul on MXFP8 activations (gemm_mx.cu)
bool mx_mm_supported(const MMArgs& a);
cudaError_t launch_mx_mm(const MMArgs& a, int rows_total, cudaStream_t s);
cudaError_t launch_tmem_mm(const MMArgs& a, int rows_total, cudaStream_t s);

// ---- FP4 delta-cache management (cache.cu)
cudaError_t launch_cache_select(const int32_t* offsets, int E, uint32_t* counts, int decay_shift, int S,
                                int32_t* expert_slot, int32_t* slot_expert, int32_t* promoted, uint32_t* dev_err,
                                cudaStream_t s);
cudaError_t launch_stage_select(const int32_t* offsets, int E, const int32_t* res_slot, int R, int S,
                                int32_t* weight_slot, int32_t* staged, uint32_t* dev_err, cudaStream_t s);
cudaError_t launch_cache_fill(const int32_t* promoted, int S, int n, const void* const* src, void* const* dst,
                              const size_t* bytes, cudaStream_t s);

// ---- diagnostics (diag.cu)
// One warp waits with the pipelines' bounded wait, limit `cycles`, on a
// shared-memory mbarrier nobody arrives on; sets MOE_DEVERR_TIMEOUT.
cudaError_t launch_bounded_wait_check(long long cycles, uint32_t* dev_err, cudaStream_t s);

// ---- the table GEMV on the library's own fixed scratch (noalloc.cu)
// Device address of the scratch array on the current device (looked up on the
// first call per device).
cudaError_t noalloc_scratch(void** ptr);
// Runs launch_lut_gemv on that scratch for `rows` permuted rows; the caller
// has checked that the rows fit.
cudaError_t launch_lut_gemv_noalloc(MMArgs a, int rows, cudaStream_t s);

}  // namespace moe
