// C ABI of libmoe: argument validation, dispatch, error reporting.
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <vector>

#include "../../include/moe.h"
#include "internal.cuh"
#include "layer_args.cuh"

namespace moe {

namespace {
thread_local char g_err[512] = {0};

int fail(int code, const char* fmt, const char* detail = nullptr) {
  if (detail) std::snprintf(g_err, sizeof(g_err), fmt, detail);
  else std::snprintf(g_err, sizeof(g_err), "%s", fmt);
  return code;
}

int cuda_status(cudaError_t e, const char* where) {
  if (e == cudaSuccess) {
    g_err[0] = 0;
    return MOE_OK;
  }
  std::snprintf(g_err, sizeof(g_err), "%s: %s", where, cudaGetErrorString(e));
  // the dispatchers answer cudaErrorNotSupported for a combination no kernel
  // takes (e.g. MXFP8_BF16 output off the tensor-core path)
  return e == cudaErrorNotSupported ? MOE_ERR_UNSUPPORTED : MOE_ERR_CUDA;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

std::mutex g_dev_mu;
DeviceInfo g_dev[64];
}  // namespace

const DeviceInfo& device_info() {
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) dev = 0;
  std::lock_guard<std::mutex> lk(g_dev_mu);
  DeviceInfo& d = g_dev[dev];
  if (d.device != dev) {
    cudaDeviceProp p;
    if (cudaGetDeviceProperties(&p, dev) == cudaSuccess) {
      d.sms = p.multiProcessorCount;
      d.major = p.major;
      d.minor = p.minor;
      d.smem_optin = p.sharedMemPerBlockOptin;
      d.device = dev;
    }
  }
  return d;
}

namespace {
struct SmemLimit {
  int device;
  const void* kernel;
  int bytes;
};
std::mutex g_smem_mu;
std::vector<SmemLimit> g_smem;
std::atomic<long long> g_wait{kWaitCycles};
std::atomic<int> g_side_sms{0};
}  // namespace

cudaError_t set_smem_limit(const void* kernel, int bytes) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lk(g_smem_mu);
  for (const SmemLimit& l : g_smem)
    if (l.device == dev && l.kernel == kernel && l.bytes >= bytes) return cudaSuccess;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e != cudaSuccess) return e;
  g_smem.push_back({dev, kernel, bytes});
  return cudaSuccess;
}

long long wait_limit() { return g_wait.load(std::memory_order_relaxed); }

int side_sms() {
  const int n = g_side_sms.load(std::memory_order_relaxed);
  const int sms = device_info().sms;
  return n > 0 && n < sms ? n : 0;
}

int matmul_ctas() { return device_info().sms - side_sms(); }

static int check_device() {
  const DeviceInfo& d = device_info();
  if (d.device < 0) return fail(MOE_ERR_CUDA, "no CUDA device");
  if (d.major != 10) return fail(MOE_ERR_UNSUPPORTED, "libmoe is built for sm_103a (Blackwell datacenter) only");
  return MOE_OK;
}

}  // namespace moe

using namespace moe;

extern "C" {

int moe_version(void) { return MOE_ABI_VERSION; }

const char* moe_last_error_string(void) { return g_err; }

int moe_get_error(const uint32_t* dev_err, void* stream, uint32_t* bits) {
  if (!dev_err || !bits) return fail(MOE_ERR_ARG, "moe_get_error: NULL pointer");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_status(e, "moe_get_error(sync)");
  e = cudaMemcpy(bits, dev_err, sizeof(uint32_t), cudaMemcpyDeviceToHost);
  return cuda_status(e, "moe_get_error(copy)");
}

long long moe_set_wait_limit(long long cycles) {
  if (cycles <= 0) cycles = kWaitCycles;
  return g_wait.exchange(cycles);
}

int moe_set_side_sms(int n) {
  if (n < 0 || n > 1024) return -1;
  return g_side_sms.exchange(n);
}

int moe_check_bounded_wait(long long cycles, uint32_t* dev_err, void* stream) {
  if (cycles < 1 || cycles > kWaitCycles || !dev_err) return fail(MOE_ERR_ARG, "moe_check_bounded_wait: bad args");
  if (int r = check_device()) return r;
  return cuda_status(launch_bounded_wait_check(cycles, dev_err, static_cast<cudaStream_t>(stream)),
                     "moe_check_bounded_wait");
}

int moe_route(const float* logits, int T, int E, int k, int32_t* ids, float* w, uint32_t* dev_err, void* stream) {
  if (T < 0 || E < 1 || E > 1024 || k < 1 || k > 32 || k > E) return fail(MOE_ERR_ARG, "moe_route: bad shape");
  if (T == 0) return MOE_OK;
  if (!logits || !ids || !w) return fail(MOE_ERR_ARG, "moe_route: NULL pointer");
  if (int r = check_device()) return r;
  return cuda_status(launch_route(logits, T, E, k, ids, w, dev_err, static_cast<cudaStream_t>(stream)), "moe_route");
}

size_t moe_permute_workspace_size(int T, int k, int E) {
  if (T <= 0 || k < 1 || E < 1 || E > 1024 || static_cast<int64_t>(T) * k >= (1LL << 31)) return 0;
  return permute_workspace_bytes(T * k, E);
}

int moe_permute(const int32_t* ids, int T, int k, int E, int32_t* offsets, int32_t* perm, int32_t* inv,
                const uint16_t* x, int H, int act_fmt, void* x_perm, uint8_t* x_perm_scale, void* ws,
                size_t ws_bytes, uint32_t* dev_err, void* stream) {
  if (T < 0 || E < 1 || E > 1024 || k < 1 || k > 32 || k > E || static_cast<int64_t>(T) * k >= (1LL << 31))
    return fail(MOE_ERR_ARG, "moe_permute: bad shape");
  if (!offsets || (T > 0 && (!ids || !perm || !inv))) return fail(MOE_ERR_ARG, "moe_permute: NULL pointer");
  if (act_fmt != MOE_FMT_NONE) {
    if (act_fmt != MOE_FMT_BF16 && act_fmt != MOE_FMT_MXFP8 && act_fmt != MOE_FMT_MXFP8_BF16)
      return fail(MOE_ERR_ARG, "moe_permute: act_fmt");
    if (H <= 0 || H % 128) return fail(MOE_ERR_ARG, "moe_permute: H must be a positive multiple of 128");
    if (T > 0 && (!x || !x_perm || !aligned(x, 16) || !aligned(x_perm, 16)))
      return fail(MOE_ERR_ARG, "moe_permute: x / x_perm NULL or not 16-byte aligned");
    if (act_fmt == MOE_FMT_MXFP8 && T > 0 && !x_perm_scale) return fail(MOE_ERR_ARG, "moe_permute: x_perm_scale");
  }
  if (int r = check_device()) return r;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (ws && !aligned(ws, 16)) return fail(MOE_ERR_ARG, "moe_permute: ws not 16-byte aligned");
  cudaError_t e = launch_permute(ids, T, k, E, offsets, perm, inv, ws, ws_bytes, dev_err, s);
  if (e == cudaSuccess && act_fmt != MOE_FMT_NONE) e = launch_gather(x, inv, T, k, H, act_fmt, x_perm, x_perm_scale, s);
  return cuda_status(e, "moe_permute");
}

int moe_unpermute(const void* rows_perm, int fmt, const int32_t* inv, int A, int cols, void* rows, void* stream) {
  if (A < 0 || cols <= 0 || (fmt != MOE_FMT_BF16 && fmt != MOE_FMT_F32)) return fail(MOE_ERR_ARG, "moe_unpermute: bad args");
  if ((cols * (fmt == MOE_FMT_F32 ? 4 : 2)) % 16) return fail(MOE_ERR_ARG, "moe_unpermute: row bytes must be a multiple of 16");
  if (A == 0) return MOE_OK;
  if (!rows_perm || !inv || !rows || !aligned(rows_perm, 16) || !aligned(rows, 16))
    return fail(MOE_ERR_ARG, "moe_unpermute: NULL or misaligned pointer");
  if (int r = check_device()) return r;
  return cuda_status(launch_unpermute(rows_perm, fmt, inv, A, cols, rows, static_cast<cudaStream_t>(stream)),
                     "moe_unpermute");
}

int moe_w2_repack(const uint8_t* codes, const uint16_t* scales, int64_t mats, int R, int K, uint8_t* codes_k,
                  uint16_t* scales_k, void* stream) {
  if (mats < 0 || R < 0 || R % 4 || K <= 0 || K % 128) return fail(MOE_ERR_ARG, "moe_w2_repack: bad shape");
  if (mats == 0 || R == 0) return MOE_OK;
  if (!codes || !scales || !codes_k || !scales_k || !aligned(codes, 4) || !aligned(codes_k, 4) ||
      !aligned(scales, 2) || !aligned(scales_k, 2))
    return fail(MOE_ERR_ARG, "moe_w2_repack: NULL or misaligned pointer");
  if (int r = check_device()) return r;
  return cuda_status(launch_w2_repack(codes, scales, mats, R, K, codes_k, scales_k, static_cast<cudaStream_t>(stream)),
                     "moe_w2_repack");
}

int moe_dequant_w2(const uint8_t* codes_k, const uint16_t* scales_k, int64_t mats, int R, int K, uint16_t* out_bf16,
                   void* stream) {
  if (mats < 0 || R < 0 || R % 4 || K <= 0 || K % 128) return fail(MOE_ERR_ARG, "moe_dequant_w2: bad shape");
  if (mats == 0 || R == 0) return MOE_OK;
  if (!codes_k || !scales_k || !out_bf16 || !aligned(codes_k, 4)) return fail(MOE_ERR_ARG, "moe_dequant_w2: pointer");
  if (int r = check_device()) return r;
  return cuda_status(launch_dequant_w2(codes_k, scales_k, mats, R, K, out_bf16, static_cast<cudaStream_t>(stream)),
                     "moe_dequant_w2");
}

int moe_dequant_mxfp4(const uint8_t* e2m1, const uint8_t* e8m0, int64_t rows, int K, float* out_f32, void* stream) {
  if (rows < 0 || K <= 0 || K % 32) return fail(MOE_ERR_ARG, "moe_dequant_mxfp4: bad shape");
  if (rows == 0) return MOE_OK;
  if (!e2m1 || !e8m0 || !out_f32 || !aligned(e2m1, 16)) return fail(MOE_ERR_ARG, "moe_dequant_mxfp4: pointer");
  if (int r = check_device()) return r;
  return cuda_status(launch_dequant_mxfp4(e2m1, e8m0, rows, K, out_f32, static_cast<cudaStream_t>(stream)),
                     "moe_dequant_mxfp4");
}

int mxfp4_to_fp8_ws(const uint8_t* e2m1, const uint8_t* e8m0, const int32_t* experts, int n_experts, int rows, int K,
                    uint8_t* ws, size_t ws_bytes, const int32_t* ws_slots, uint32_t* dev_err, void* stream) {
  if (n_experts < 0 || rows < 0 || K <= 0 || K % 32) return fail(MOE_ERR_ARG, "mxfp4_to_fp8_ws: bad shape");
  if (n_experts == 0 || rows == 0) return MOE_OK;
  if (!e2m1 || !e8m0 || !experts || !ws || !ws_slots || !aligned(e2m1, 16) || !aligned(ws, 16))
    return fail(MOE_ERR_ARG, "mxfp4_to_fp8_ws: NULL or misaligned pointer");
  if (ws_bytes < static_cast<size_t>(rows) * K) return fail(MOE_ERR_WS_SMALL, "mxfp4_to_fp8_ws: workspace below one slot");
  if (int r = check_device()) return r;
  return cuda_status(launch_mxfp4_to_fp8(e2m1, e8m0, experts, n_experts, rows, K, ws, ws_bytes, ws_slots, dev_err,
                                         static_cast<cudaStream_t>(stream)),
                     "mxfp4_to_fp8_ws");
}

// Argument checks shared by the expert-matmul calls.  Returns MOE_OK, a
// status, or kNoRows when the activation has no rows: the call then does
// nothing (its buffers may be empty, their pointers NULL).
constexpr int kNoRows = -1;

static int check_mm(const char* who, int stage, int mode, const void* act, int act_fmt, const uint8_t* act_scale,
                    int act_rows, const int32_t* offsets, int E, int N, int K, const void* out, int out_fmt,
                    const uint8_t* out_scale) {
  if (stage != MOE_STAGE_FC1_SWIGLU && stage != MOE_STAGE_FC2) return fail(MOE_ERR_ARG, "%s: bad stage", who);
  if (mode < MOE_MODE_AUTO || mode > MOE_MODE_SPLIT) return fail(MOE_ERR_ARG, "%s: bad mode", who);
  if (E < 1 || E > 1024 || N <= 0 || K <= 0 || N % 128 || K % 128 || K > 8192)
    return fail(MOE_ERR_ARG, "%s: bad shape (N, K multiples of 128, K <= 8192, 1 <= E <= 1024)", who);
  if (act_fmt != MOE_FMT_BF16 && act_fmt != MOE_FMT_MXFP8) return fail(MOE_ERR_ARG, "%s: act_fmt", who);
  if (out_fmt != MOE_FMT_BF16 && out_fmt != MOE_FMT_F32 && out_fmt != MOE_FMT_MXFP8 && out_fmt != MOE_FMT_MXFP8_BF16)
    return fail(MOE_ERR_ARG, "%s: out_fmt", who);
  if (out_fmt == MOE_FMT_MXFP8_BF16 && stage != MOE_STAGE_FC1_SWIGLU)
    return fail(MOE_ERR_ARG, "%s: MXFP8_BF16 output is for FC1", who);
  if (out_fmt == MOE_FMT_MXFP8 && stage != MOE_STAGE_FC1_SWIGLU)
    return fail(MOE_ERR_ARG, "%s: MXFP8 output is for FC1", who);
  if (act_rows < 0) return fail(MOE_ERR_ARG, "%s: act_rows < 0", who);
  if (act_rows == 0) return kNoRows;
  if (act_fmt == MOE_FMT_MXFP8 && (!act_scale || !aligned(act_scale, 4)))
    return fail(MOE_ERR_ARG, "%s: act_scale NULL or not 4-byte aligned", who);
  if (!act || !offsets || !out || !aligned(act, 16)) return fail(MOE_ERR_ARG, "%s: NULL or misaligned pointer", who);
  if (out_fmt == MOE_FMT_MXFP8 && !out_scale) return fail(MOE_ERR_ARG, "%s: MXFP8 output needs out_scale", who);
  return check_device();
}

size_t moe_w2_mm_workspace_size(int stage, int rows, int N, int K) {
  if ((stage != MOE_STAGE_FC1_SWIGLU && stage != MOE_STAGE_FC2) || rows < 0 || N <= 0 || K <= 0 || N % 128 ||
      K % 128)
    return 0;
  return lut_workspace_bytes(stage, rows, N, K);
}

int moe_w2_mm(int stage, int mode, const void* act, int act_fmt, const uint8_t* act_scale, int act_rows,
              const int32_t* act_row, int act_row_div, const uint8_t* codes_k, const uint16_t* scales_k, const int32_t* offsets,
              const int32_t* expert_slot, int E, int N, int K, void* out, int out_fmt, uint8_t* out_scale, void* ws,
              size_t ws_bytes, uint32_t* dev_err, void* stream) {
  if (int r = check_mm("moe_w2_mm", stage, mode, act, act_fmt, act_scale, act_rows, offsets, E, N, K, out, out_fmt, out_scale))
    return r == kNoRows ? MOE_OK : r;
  if (!codes_k || !scales_k || !aligned(codes_k, 16) || !aligned(scales_k, 16))
    return fail(MOE_ERR_ARG, "moe_w2_mm: weights NULL or not 16-byte aligned");
  if (act_rows < 0) return fail(MOE_ERR_ARG, "moe_w2_mm: act_rows < 0");
  if (act_row && act_row_div < 1) return fail(MOE_ERR_ARG, "moe_w2_mm: act_row_div < 1");
  if (mode == MOE_MODE_SPLIT && act_row) return fail(MOE_ERR_ARG, "moe_w2_mm: MOE_MODE_SPLIT reads permuted rows (act_row NULL)");
  MMArgs a{};
  a.stage = stage;
  a.act = act;
  a.act_fmt = act_fmt;
  a.act_scale = act_scale;
  a.act_rows = act_rows;
  a.mode = mode;
  a.act_row = act_row;
  a.act_row_div = act_row ? act_row_div : 1;
  a.wkind = kW2;
  a.wq = codes_k;
  a.wscale = scales_k;
  // the workspace only serves the table GEMV; shapes it does not take need none
  const bool table_shape = lut_workspace_bytes(stage, 1, N, K) > 0;  // K a multiple of 512
  a.ws = (ws && ws_bytes && table_shape) ? ws : nullptr;
  a.ws_bytes = a.ws ? ws_bytes : 0;
  a.ws_rows = a.ws ? lut_workspace_rows(stage, ws_bytes, N, K) : 0;
  if (a.ws && !aligned(ws, 256)) return fail(MOE_ERR_ARG, "moe_w2_mm: ws must be 256-byte aligned");
  if (a.ws && a.ws_rows < 1) return fail(MOE_ERR_WS_SMALL, "moe_w2_mm: workspace below one row");
  a.wslot_of = nullptr;  // 2-bit weights are indexed by expert
  a.select_map = expert_slot;
  a.select = expert_slot ? 1 : 0;
  a.offsets = offsets;
  a.expert_begin = 0;
  a.expert_end = E;
  a.E = E;
  a.N = N;
  a.K = K;
  a.out = out;
  a.out_fmt = out_fmt;
  a.out_scale = out_scale;
  a.dev_err = dev_err;
  a.wait = wait_limit();
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  return cuda_status(launch_gemv(a, s), "moe_w2_mm");
}

int moe_w2_mm_noalloc(int stage, const void* act, int act_rows, const int32_t* act_row, int act_row_div,
                      const uint8_t* codes_k, const uint16_t* scales_k, const int32_t* offsets,
                      const int32_t* expert_slot, int E, int N, int K, int rows, void* out, int out_fmt,
                      uint32_t* dev_err, void* stream) {
  if (int r = check_mm("moe_w2_mm_noalloc", stage, MOE_MODE_GEMV, act, MOE_FMT_BF16, nullptr, act_rows, offsets, E, N, K, out,
                       out_fmt, nullptr))
    return r == kNoRows ? MOE_OK : r;
  if (out_fmt == MOE_FMT_MXFP8) return fail(MOE_ERR_ARG, "moe_w2_mm_noalloc: out_fmt must be BF16 or F32");
  if (!codes_k || !scales_k || !aligned(codes_k, 16) || !aligned(scales_k, 16))
    return fail(MOE_ERR_ARG, "moe_w2_mm_noalloc: weights NULL or not 16-byte aligned");
  if (act_rows < 0 || rows < 0) return fail(MOE_ERR_ARG, "moe_w2_mm_noalloc: act_rows or rows < 0");
  if (act_row && act_row_div < 1) return fail(MOE_ERR_ARG, "moe_w2_mm_noalloc: act_row_div < 1");
  if (rows == 0) return MOE_OK;
  MMArgs a{};
  a.stage = stage;
  a.act = act;
  a.act_fmt = MOE_FMT_BF16;
  a.act_rows = act_rows;
  a.mode = MOE_MODE_GEMV;
  a.act_row = act_row;
  a.act_row_div = act_row ? act_row_div : 1;
  a.wkind = kW2;
  a.wq = codes_k;
  a.wscale = scales_k;
  a.select_map = expert_slot;
  a.select = expert_slot ? 1 : 0;
  a.offsets = offsets;
  a.expert_begin = 0;
  a.expert_end = E;
  a.E = E;
  a.N = N;
  a.K = K;
  a.out = out;
  a.out_fmt = out_fmt;
  a.dev_err = dev_err;
  a.wait = wait_limit();
  // the shape first: a shape the table GEMV does not take is unsupported
  // whatever its size
  if (!lut_supported(a))
    return fail(MOE_ERR_UNSUPPORTED, "moe_w2_mm_noalloc: K is not a multiple of the table GEMV's slice width");
  const size_t need = lut_workspace_bytes(stage, rows, N, K);
  if (need > MOE_W2_NOALLOC_SCRATCH_BYTES) {
    std::snprintf(g_err, sizeof(g_err),
                  "moe_w2_mm_noalloc: %d rows need %zu bytes of scratch, above the fixed %u bytes; use moe_w2_mm "
                  "with a workspace",
                  rows, need, MOE_W2_NOALLOC_SCRATCH_BYTES);
    return MOE_ERR_WS_SMALL;
  }
  return cuda_status(launch_lut_gemv_noalloc(a, rows, static_cast<cudaStream_t>(stream)), "moe_w2_mm_noalloc");
}

size_t moe_w2_decode_fused_workspace_size(int rows, int H, int I) {
  if (rows <= 0 || H <= 0 || I <= 0 || H % 128 || I % 128) return 0;
  const size_t a = lut_workspace_bytes(MOE_STAGE_FC1_SWIGLU, rows, I, H);
  const size_t b = lut_workspace_bytes(MOE_STAGE_FC2, rows, H, I);
  if (a == 0 || b == 0) return 0;
  return 256 + (a > b ? a : b);
}

int moe_w2_decode_fused(const void* x, int act_rows, const int32_t* act_row, int act_row_div, const uint8_t* codes1,
                        const uint16_t* scales1, const uint8_t* codes2, const uint16_t* scales2,
                        const int32_t* offsets, const int32_t* expert_slot, int E, int H, int I, void* h, void* y,
                        int y_fmt, void* ws, size_t ws_bytes, uint32_t* dev_err, void* stream) {
  if (int r = check_mm("moe_w2_decode_fused", MOE_STAGE_FC1_SWIGLU, MOE_MODE_GEMV, x, MOE_FMT_BF16, nullptr, act_rows, offsets,
                       E, I, H, h, MOE_FMT_BF16, nullptr))
    return r == kNoRows ? MOE_OK : r;
  if (!y || !aligned(h, 16) || (y_fmt != MOE_FMT_BF16 && y_fmt != MOE_FMT_F32))
    return fail(MOE_ERR_ARG, "moe_w2_decode_fused: h / y / y_fmt");
  if (!codes1 || !scales1 || !codes2 || !scales2 || !aligned(codes1, 16) || !aligned(scales1, 16) ||
      !aligned(codes2, 16) || !aligned(scales2, 16))
    return fail(MOE_ERR_ARG, "moe_w2_decode_fused: weights NULL or not 16-byte aligned");
  if (act_rows < 0 || (act_row && act_row_div < 1)) return fail(MOE_ERR_ARG, "moe_w2_decode_fused: act rows");
  if (!ws || !aligned(ws, 256) || ws_bytes <= 256) return fail(MOE_ERR_ARG, "moe_w2_decode_fused: workspace");
  MMArgs a1{}, a2{};
  for (MMArgs* a : {&a1, &a2}) {
    a->act_fmt = MOE_FMT_BF16;
    a->mode = MOE_MODE_GEMV;
    a->wkind = kW2;
    a->select_map = expert_slot;
    a->select = expert_slot ? 1 : 0;
    a->offsets = offsets;
    a->expert_begin = 0;
    a->expert_end = E;
    a->E = E;
    a->dev_err = dev_err;
    a->wait = wait_limit();
  }
  a1.stage = MOE_STAGE_FC1_SWIGLU;
  a1.act = x;
  a1.act_rows = act_rows;
  a1.act_row = act_row;
  a1.act_row_div = act_row ? act_row_div : 1;
  a1.wq = codes1;
  a1.wscale = scales1;
  a1.N = I;
  a1.K = H;
  a1.out = h;
  a1.out_fmt = MOE_FMT_BF16;
  a2.stage = MOE_STAGE_FC2;
  a2.act = h;
  a2.act_rows = 0x7fffffff;  // h rows are the permuted rows themselves
  a2.act_row = nullptr;
  a2.act_row_div = 1;
  a2.wq = codes2;
  a2.wscale = scales2;
  a2.N = H;
  a2.K = I;
  a2.out = y;
  a2.out_fmt = y_fmt;
  if (!lut_supported(a1) || !lut_supported(a2))
    return fail(MOE_ERR_UNSUPPORTED, "moe_w2_decode_fused: H and I must be multiples of 512");
  const size_t lws = ws_bytes - 256;
  for (MMArgs* a : {&a1, &a2}) {
    a->ws = static_cast<uint8_t*>(ws) + 256;
    a->ws_bytes = lws;
    a->ws_rows = lut_workspace_rows(a->stage, lws, a->N, a->K);
    if (a->ws_rows < 1) return fail(MOE_ERR_WS_SMALL, "moe_w2_decode_fused: workspace below one row");
  }
  return cuda_status(launch_w2_decode_fused(a1, a2, ws, static_cast<cudaStream_t>(stream)), "moe_w2_decode_fused");
}

size_t moe_w2_decode_layer_workspace_size(int T, int k, int H, int I) {
  if (T <= 0 || k <= 0 || static_cast<int64_t>(T) * k > 0x7fffffff) return 0;
  return moe_w2_decode_fused_workspace_size(T * k, H, I);
}

int moe_w2_decode_layer(const float* logits, const void* x, int T, int E, int k, const uint8_t* codes1,
                        const uint16_t* scales1, const uint8_t* codes2, const uint16_t* scales2, int H, int I,
                        int32_t* ids, float* w, int32_t* offsets, int32_t* perm, int32_t* inv, void* h, void* y,
                        void* out, int out_fmt, void* ws, size_t ws_bytes, uint32_t* dev_err, void* stream) {
  if (T < 0 || E < 1 || E > 1024 || k < 1 || k > E) return fail(MOE_ERR_ARG, "moe_w2_decode_layer: bad shape");
  if (!offsets) return fail(MOE_ERR_ARG, "moe_w2_decode_layer: offsets NULL");
  if (out_fmt != MOE_FMT_BF16 && out_fmt != MOE_FMT_F32) return fail(MOE_ERR_ARG, "moe_w2_decode_layer: out_fmt");
  if (H <= 0 || I <= 0) return fail(MOE_ERR_ARG, "moe_w2_decode_layer: H / I");
  if (int r = check_device()) return r;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (T == 0)  // no assignments: every group empty, nothing else to write
    return cuda_status(cudaMemsetAsync(offsets, 0, sizeof(int32_t) * (E + 1), s), "moe_w2_decode_layer");
  if (!logits || !x || !ids || !w || !perm || !inv || !h || !y || !out || !aligned(x, 16) || !aligned(h, 16))
    return fail(MOE_ERR_ARG, "moe_w2_decode_layer: NULL pointer, or x / h not 16-byte aligned");
  if (!codes1 || !scales1 || !codes2 || !scales2 || !aligned(codes1, 16) || !aligned(scales1, 16) ||
      !aligned(codes2, 16) || !aligned(scales2, 16))
    return fail(MOE_ERR_ARG, "moe_w2_decode_layer: weights NULL or not 16-byte aligned");
  if (!ws || !aligned(ws, 256) || ws_bytes <= 256) return fail(MOE_ERR_ARG, "moe_w2_decode_layer: workspace");
  if (!layer_supported(T, E, k))
    return fail(MOE_ERR_UNSUPPORTED, "moe_w2_decode_layer: T*k above 256 or k above 16");
  const int A = T * k;
  MMArgs a1{}, a2{};
  for (MMArgs* a : {&a1, &a2}) {
    a->act_fmt = MOE_FMT_BF16;
    a->mode = MOE_MODE_GEMV;
    a->wkind = kW2;
    a->offsets = nullptr;  // the grouping's, in the kernel's shared memory
    a->expert_begin = 0;
    a->expert_end = E;
    a->E = E;
    a->dev_err = dev_err;
    a->wait = wait_limit();
  }
  a1.stage = MOE_STAGE_FC1_SWIGLU;
  a1.act = x;
  a1.act_rows = T;
  a1.act_row = nullptr;  // the grouping's perm, in shared memory
  a1.act_row_div = k;
  a1.wq = codes1;
  a1.wscale = scales1;
  a1.N = I;
  a1.K = H;
  a1.out = h;
  a1.out_fmt = MOE_FMT_BF16;
  a2.stage = MOE_STAGE_FC2;
  a2.act = h;
  a2.act_rows = 0x7fffffff;  // h rows are the permuted rows themselves
  a2.act_row = nullptr;
  a2.act_row_div = 1;
  a2.wq = codes2;
  a2.wscale = scales2;
  a2.N = H;
  a2.K = I;
  a2.out = y;
  a2.out_fmt = MOE_FMT_BF16;
  if (!lut_supported(a1) || !lut_supported(a2))
    return fail(MOE_ERR_UNSUPPORTED, "moe_w2_decode_layer: H and I must be multiples of 512");
  const size_t lws = ws_bytes - 256;
  for (MMArgs* a : {&a1, &a2}) {
    a->ws = static_cast<uint8_t*>(ws) + 256;
    a->ws_bytes = lws;
    a->ws_rows = lut_workspace_rows(a->stage, lws, a->N, a->K);
    if (a->ws_rows < A) return fail(MOE_ERR_WS_SMALL, "moe_w2_decode_layer: workspace below T*k rows");
  }
  LayerArgs la;
  la.logits = logits;
  la.T = T;
  la.E = E;
  la.k = k;
  la.ids = ids;
  la.w = w;
  la.offsets = offsets;
  la.perm = perm;
  la.inv = inv;
  la.y = y;
  la.out = out;
  la.out_fmt = out_fmt;
  return cuda_status(launch_w2_decode_layer(la, a1, a2, ws, s), "moe_w2_decode_layer");
}

int moe_mxfp4_mm(int stage, int mode, const void* act, int act_fmt, const uint8_t* act_scale, int act_rows,
                 const int32_t* act_row, int act_row_div, const uint8_t* e2m1, const uint8_t* e8m0, const uint8_t* fp8_ws,
                 const int32_t* ws_slot_of_expert, const int32_t* offsets, const int32_t* expert_slot,
                 int expert_begin, int expert_end, int E, int N, int K, void* out, int out_fmt, uint8_t* out_scale,
                 void* ws, size_t ws_bytes, uint32_t* dev_err, void* stream) {
  (void)ws;
  (void)ws_bytes;
  if (mode == MOE_MODE_SPLIT) return fail(MOE_ERR_ARG, "moe_mxfp4_mm: MOE_MODE_SPLIT is for 2-bit weights");
  if (int r = check_mm("moe_mxfp4_mm", stage, mode, act, act_fmt, act_scale, act_rows, offsets, E, N, K, out, out_fmt, out_scale))
    return r == kNoRows ? MOE_OK : r;
  if (act_row && act_row_div < 1) return fail(MOE_ERR_ARG, "moe_mxfp4_mm: act_row_div < 1");
  if (act_rows < 0) return fail(MOE_ERR_ARG, "moe_mxfp4_mm: act_rows < 0");
  if (expert_begin < 0 || expert_end > E || expert_begin > expert_end)
    return fail(MOE_ERR_ARG, "moe_mxfp4_mm: bad expert range");
  const bool use_fp8 = fp8_ws != nullptr;
  if (use_fp8 == (e2m1 != nullptr)) return fail(MOE_ERR_ARG, "moe_mxfp4_mm: give exactly one of e2m1 / fp8_ws");
  MMArgs a{};
  a.stage = stage;
  a.act = act;
  a.act_fmt = act_fmt;
  a.act_scale = act_scale;
  a.act_rows = act_rows;
  a.mode = mode;
  a.act_row = act_row;
  a.act_row_div = act_row ? act_row_div : 1;
  if (use_fp8) {
    if (!ws_slot_of_expert || !aligned(fp8_ws, 16)) return fail(MOE_ERR_ARG, "moe_mxfp4_mm: FP8 workspace args");
    a.wkind = kFP8;
    a.wq = fp8_ws;
    a.wscale = nullptr;
    a.wslot_of = ws_slot_of_expert;
    a.select_map = ws_slot_of_expert;
    a.select = 2;
  } else {
    if (!e8m0 || !aligned(e2m1, 16) || !aligned(e8m0, 16)) return fail(MOE_ERR_ARG, "moe_mxfp4_mm: MXFP4 weights");
    a.wkind = kMXFP4;
    a.wq = e2m1;
    a.wscale = e8m0;
    a.wslot_of = expert_slot;
    a.select_map = expert_slot;
    a.select = expert_slot ? 2 : 0;
  }
  a.offsets = offsets;
  a.expert_begin = expert_begin;
  a.expert_end = expert_end;
  a.E = E;
  a.N = N;
  a.K = K;
  a.out = out;
  a.out_fmt = out_fmt;
  a.out_scale = out_scale;
  a.dev_err = dev_err;
  a.wait = wait_limit();
  return cuda_status(launch_gemv(a, static_cast<cudaStream_t>(stream)), "moe_mxfp4_mm");
}

int moe_cache_select(const int32_t* offsets, int E, uint32_t* counts, int decay_shift, int S, int32_t* expert_slot,
                     int32_t* slot_expert, int32_t* promoted, uint32_t* dev_err, void* stream) {
  if (E < 1 || E > 1024 || S < 1 || S > E || decay_shift < 0) return fail(MOE_ERR_ARG, "moe_cache_select: bad shape");
  if (!offsets || !counts || !expert_slot || !slot_expert || !promoted)
    return fail(MOE_ERR_ARG, "moe_cache_select: NULL pointer");
  if (int r = check_device()) return r;
  return cuda_status(launch_cache_select(offsets, E, counts, decay_shift, S, expert_slot, slot_expert, promoted,
                                         dev_err, static_cast<cudaStream_t>(stream)),
                     "moe_cache_select");
}

int moe_stage_select(const int32_t* offsets, int E, const int32_t* res_slot, int R, int S, int32_t* weight_slot,
                     int32_t* staged, uint32_t* dev_err, void* stream) {
  if (E < 1 || E > 1024 || R < 0 || S < 1 || S > 1024) return fail(MOE_ERR_ARG, "moe_stage_select: bad shape");
  if (!offsets || !res_slot || !weight_slot || !staged) return fail(MOE_ERR_ARG, "moe_stage_select: NULL pointer");
  if (int r = check_device()) return r;
  return cuda_status(launch_stage_select(offsets, E, res_slot, R, S, weight_slot, staged, dev_err,
                                         static_cast<cudaStream_t>(stream)),
                     "moe_stage_select");
}

int moe_w2_mm_slots(int stage, const void* act, int act_rows, const int32_t* act_row, int act_row_div,
                    const uint8_t* codes_k, const uint16_t* scales_k, const int32_t* offsets,
                    const int32_t* weight_slot, int slot_lo, int slot_hi, int E, int N, int K, void* out, int out_fmt,
                    void* ws, size_t ws_bytes, uint32_t* dev_err, void* stream) {
  if (int r = check_mm("moe_w2_mm_slots", stage, MOE_MODE_GEMV, act, MOE_FMT_BF16, nullptr, act_rows, offsets, E, N, K, out,
                       out_fmt, nullptr))
    return r == kNoRows ? MOE_OK : r;
  if (out_fmt != MOE_FMT_BF16 && out_fmt != MOE_FMT_F32) return fail(MOE_ERR_ARG, "moe_w2_mm_slots: out_fmt");
  if (!codes_k || !scales_k || !weight_slot || !aligned(codes_k, 16) || !aligned(scales_k, 16))
    return fail(MOE_ERR_ARG, "moe_w2_mm_slots: weights / slot map NULL or misaligned");
  if (act_rows < 0 || slot_lo < 0 || slot_hi < slot_lo) return fail(MOE_ERR_ARG, "moe_w2_mm_slots: bad rows / slots");
  if (act_row && act_row_div < 1) return fail(MOE_ERR_ARG, "moe_w2_mm_slots: act_row_div < 1");
  if (!ws || !aligned(ws, 256)) return fail(MOE_ERR_ARG, "moe_w2_mm_slots: needs a 256-byte aligned workspace");
  MMArgs a{};
  a.stage = stage;
  a.act = act;
  a.act_fmt = MOE_FMT_BF16;
  a.act_rows = act_rows;
  a.mode = MOE_MODE_GEMV;
  a.act_row = act_row;
  a.act_row_div = act_row ? act_row_div : 1;
  a.wkind = kW2;
  a.wq = codes_k;
  a.wscale = scales_k;
  a.wslot_of = weight_slot;
  a.slot_lo = slot_lo;
  a.slot_hi = slot_hi;
  a.offsets = offsets;
  a.expert_begin = 0;
  a.expert_end = E;
  a.E = E;
  a.N = N;
  a.K = K;
  a.out = out;
  a.out_fmt = out_fmt;
  a.dev_err = dev_err;
  a.wait = wait_limit();
  if (!lut_supported(a))
    return fail(MOE_ERR_UNSUPPORTED, "moe_w2_mm_slots: K is not a multiple of the table GEMV's slice width");
  a.ws = ws;
  a.ws_bytes = ws_bytes;
  a.ws_rows = lut_workspace_rows(stage, ws_bytes, N, K);
  if (a.ws_rows < 1) return fail(MOE_ERR_WS_SMALL, "moe_w2_mm_slots: workspace below one row");
  return cuda_status(launch_lut_gemv(a, ws, static_cast<cudaStream_t>(stream)), "moe_w2_mm_slots");
}

int moe_cache_fill(const int32_t* promoted, int S, int n_arrays, const void* const* src, void* const* dst,
                   const size_t* bytes, void* stream) {
  if (S < 1 || n_arrays < 1 || n_arrays > 4 || !promoted || !src || !dst || !bytes)
    return fail(MOE_ERR_ARG, "moe_cache_fill: bad arguments");
  for (int a = 0; a < n_arrays; ++a) {
    if (!src[a] || !dst[a] || !aligned(src[a], 16) || !aligned(dst[a], 16) || bytes[a] == 0 || bytes[a] % 16)
      return fail(MOE_ERR_ARG, "moe_cache_fill: array pointers must be 16-byte aligned, sizes multiples of 16");
  }
  if (int r = check_device()) return r;
  return cuda_status(launch_cache_fill(promoted, S, n_arrays, src, dst, bytes, static_cast<cudaStream_t>(stream)),
                     "moe_cache_fill");
}

int moe_combine(const void* y, int y_fmt, const float* w, const int32_t* inv, int T, int k, int H, void* out,
                int out_fmt, void* stream) {
  if (T < 0 || k < 1 || k > 32 || H <= 0 || H % 128) return fail(MOE_ERR_ARG, "moe_combine: bad shape");
  if ((y_fmt != MOE_FMT_BF16 && y_fmt != MOE_FMT_F32) || (out_fmt != MOE_FMT_BF16 && out_fmt != MOE_FMT_F32))
    return fail(MOE_ERR_ARG, "moe_combine: format");
  if (T == 0) return MOE_OK;
  if (!y || !w || !inv || !out || !aligned(y, 16) || !aligned(out, 16))
    return fail(MOE_ERR_ARG, "moe_combine: NULL or misaligned pointer");
  if (int r = check_device()) return r;
  return cuda_status(launch_combine(y, y_fmt, w, inv, T, k, H, out, out_fmt, static_cast<cudaStream_t>(stream)),
                     "moe_combine");
}

}  // extern "C"
