"""ctypes binding of libmoe.so (argument marshalling only).

Each function has the name of the C entry point it calls and takes torch
tensors (device memory) plus plain ints; every computation happens in the
library's CUDA kernels.  The library must have been built in-tree
(``python -m bit_moe_expert_top_gb300.build``); there is no fallback: loading
fails loudly when it is missing.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmoe.so")

MOE_OK, MOE_ERR_ARG, MOE_ERR_WS_SMALL, MOE_ERR_UNSUPPORTED, MOE_ERR_CUDA = 0, 1, 2, 3, 4
DEVERR_BAD_ID, DEVERR_NAN_LOGIT, DEVERR_NAN_SCALE, DEVERR_TIMEOUT, DEVERR_OVERFLOW, DEVERR_LAUNCH = 1, 2, 4, 8, 16, 32
FMT_NONE, FMT_BF16, FMT_F32, FMT_MXFP8, FMT_MXFP8_BF16 = 0, 1, 2, 3, 4
STAGE_FC1_SWIGLU, STAGE_FC2 = 1, 2
MODE_AUTO, MODE_GEMV, MODE_GEMM, MODE_SPLIT = 0, 1, 2, 3

# every entry point declared in include/moe.h
EXPORTS = ["moe_version", "moe_last_error_string", "moe_get_error", "moe_set_wait_limit", "moe_set_side_sms",
           "moe_check_bounded_wait", "moe_route", "moe_permute_workspace_size",
           "moe_permute", "moe_unpermute", "moe_w2_repack", "moe_dequant_w2", "moe_dequant_mxfp4",
           "mxfp4_to_fp8_ws", "moe_w2_mm_workspace_size", "moe_w2_mm", "moe_w2_mm_noalloc", "moe_mxfp4_mm",
           "moe_combine", "moe_cache_select", "moe_cache_fill", "moe_stage_select", "moe_w2_mm_slots",
           "moe_w2_decode_fused_workspace_size", "moe_w2_decode_fused", "moe_w2_decode_layer_workspace_size",
           "moe_w2_decode_layer"]
W2_NOALLOC_SCRATCH_BYTES = 16 << 20


class MoEError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"libmoe status {code}: {msg}")
        self.code = code


_P, _I, _L, _S = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t
_SIGS = {
    "moe_version": (_I, []),
    "moe_last_error_string": (ctypes.c_char_p, []),
    "moe_get_error": (_I, [_P, _P, _P]),
    "moe_set_wait_limit": (_L, [_L]),
    "moe_set_side_sms": (_I, [_I]),
    "moe_check_bounded_wait": (_I, [_L, _P, _P]),
    "moe_route": (_I, [_P, _I, _I, _I, _P, _P, _P, _P]),
    "moe_permute_workspace_size": (_S, [_I, _I, _I]),
    "moe_permute": (_I, [_P, _I, _I, _I, _P, _P, _P, _P, _I, _I, _P, _P, _P, _S, _P, _P]),
    "moe_unpermute": (_I, [_P, _I, _P, _I, _I, _P, _P]),
    "moe_w2_repack": (_I, [_P, _P, _L, _I, _I, _P, _P, _P]),
    "moe_dequant_w2": (_I, [_P, _P, _L, _I, _I, _P, _P]),
    "moe_dequant_mxfp4": (_I, [_P, _P, _L, _I, _P, _P]),
    "mxfp4_to_fp8_ws": (_I, [_P, _P, _P, _I, _I, _I, _P, _S, _P, _P, _P]),
    "moe_w2_mm_workspace_size": (_S, [_I, _I, _I, _I]),
    "moe_w2_mm": (_I, [_I, _I, _P, _I, _P, _I, _P, _I, _P, _P, _P, _P, _I, _I, _I, _P, _I, _P, _P, _S, _P, _P]),
    "moe_w2_mm_noalloc": (_I, [_I, _P, _I, _P, _I, _P, _P, _P, _P, _I, _I, _I, _I, _P, _I, _P, _P]),
    "moe_mxfp4_mm": (_I, [_I, _I, _P, _I, _P, _I, _P, _I, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _P, _I,
                          _P, _P, _S, _P, _P]),
    "moe_combine": (_I, [_P, _I, _P, _P, _I, _I, _I, _P, _I, _P]),
    "moe_cache_select": (_I, [_P, _I, _P, _I, _I, _P, _P, _P, _P, _P]),
    "moe_cache_fill": (_I, [_P, _I, _I, _P, _P, _P, _P]),
    "moe_stage_select": (_I, [_P, _I, _P, _I, _I, _P, _P, _P, _P]),
    "moe_w2_decode_fused_workspace_size": (_S, [_I, _I, _I]),
    "moe_w2_decode_fused": (_I, [_P, _I, _P, _I, _P, _P, _P, _P, _P, _P, _I, _I, _I, _P, _P, _I, _P, _S, _P, _P]),
    "moe_w2_decode_layer_workspace_size": (_S, [_I, _I, _I, _I]),
    "moe_w2_decode_layer": (_I, [_P, _P, _I, _I, _I, _P, _P, _P, _P, _I, _I, _P, _P, _P, _P, _P, _P, _P, _P, _I,
                                 _P, _S, _P, _P]),
    "moe_w2_mm_slots": (_I, [_I, _P, _I, _P, _I, _P, _P, _P, _P, _I, _I, _I, _I, _I, _P, _I, _P, _S, _P, _P]),
}

_lib: Optional[ctypes.CDLL] = None


def lib() -> ctypes.CDLL:
    """Load libmoe.so (once).  Raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"libmoe.so not built at {LIB_PATH}; run python -m bit_moe_expert_top_gb300.build")
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGS.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _lib = L
    return _lib


def _ptr(t) -> Optional[int]:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(rc: int):
    if rc != MOE_OK:
        raise MoEError(rc, lib().moe_last_error_string().decode(errors="replace"))


# ---------------------------------------------------------------- entry points

def moe_version() -> int:
    return lib().moe_version()


def moe_get_error(dev_err: torch.Tensor, stream=None) -> int:
    bits = ctypes.c_uint32(0)
    _check(lib().moe_get_error(_ptr(dev_err), _stream(stream), ctypes.addressof(bits)))
    return int(bits.value)


def moe_set_wait_limit(cycles: int) -> int:
    return int(lib().moe_set_wait_limit(cycles))


def moe_set_side_sms(n: int) -> int:
    return int(lib().moe_set_side_sms(n))


def moe_check_bounded_wait(cycles, dev_err, stream=None):
    _check(lib().moe_check_bounded_wait(cycles, _ptr(dev_err), _stream(stream)))


def moe_route(logits, k, ids, w, dev_err=None, stream=None):
    T, E = logits.shape
    _check(lib().moe_route(_ptr(logits), T, E, k, _ptr(ids), _ptr(w), _ptr(dev_err), _stream(stream)))


def moe_permute_workspace_size(T, k, E) -> int:
    return int(lib().moe_permute_workspace_size(T, k, E))


def moe_permute(ids, E, offsets, perm, inv, x=None, act_fmt=FMT_NONE, x_perm=None, x_perm_scale=None,
                ws=None, ws_bytes=0, dev_err=None, stream=None):
    T, k = ids.shape
    H = x.shape[1] if x is not None else 0
    _check(lib().moe_permute(_ptr(ids), T, k, E, _ptr(offsets), _ptr(perm), _ptr(inv), _ptr(x), H, act_fmt,
                             _ptr(x_perm), _ptr(x_perm_scale), _ptr(ws), ws_bytes, _ptr(dev_err), _stream(stream)))


def moe_unpermute(rows_perm, fmt, inv, rows, stream=None):
    A, cols = rows_perm.shape
    _check(lib().moe_unpermute(_ptr(rows_perm), fmt, _ptr(inv), A, cols, _ptr(rows), _stream(stream)))


def moe_w2_repack(codes, scales, mats, R, K, codes_k, scales_k, stream=None):
    _check(lib().moe_w2_repack(_ptr(codes), _ptr(scales), mats, R, K, _ptr(codes_k), _ptr(scales_k),
                               _stream(stream)))


def moe_dequant_w2(codes_k, scales_k, mats, R, K, out_bf16, stream=None):
    _check(lib().moe_dequant_w2(_ptr(codes_k), _ptr(scales_k), mats, R, K, _ptr(out_bf16), _stream(stream)))


def moe_dequant_mxfp4(e2m1, e8m0, rows, K, out_f32, stream=None):
    _check(lib().moe_dequant_mxfp4(_ptr(e2m1), _ptr(e8m0), rows, K, _ptr(out_f32), _stream(stream)))


def mxfp4_to_fp8_ws(e2m1, e8m0, experts, rows, K, ws, ws_slots, dev_err=None, stream=None, ws_bytes=None):
    n = experts.numel()
    nbytes = ws.numel() * ws.element_size() if ws_bytes is None else ws_bytes
    _check(lib().mxfp4_to_fp8_ws(_ptr(e2m1), _ptr(e8m0), _ptr(experts), n, rows, K, _ptr(ws), nbytes,
                                 _ptr(ws_slots), _ptr(dev_err), _stream(stream)))


def moe_w2_mm_workspace_size(stage, rows, N, K) -> int:
    return int(lib().moe_w2_mm_workspace_size(stage, rows, N, K))


def moe_w2_mm(stage, act, act_fmt, codes_k, scales_k, offsets, E, N, K, out, out_fmt, act_scale=None,
              act_row=None, act_row_div=1, expert_slot=None, out_scale=None, mode=MODE_AUTO, ws=None,
              dev_err=None, stream=None):
    nbytes = 0 if ws is None else ws.numel() * ws.element_size()
    _check(lib().moe_w2_mm(stage, mode, _ptr(act), act_fmt, _ptr(act_scale), act.shape[0], _ptr(act_row),
                           act_row_div,
                           _ptr(codes_k), _ptr(scales_k), _ptr(offsets), _ptr(expert_slot), E, N, K, _ptr(out),
                           out_fmt, _ptr(out_scale), _ptr(ws), nbytes, _ptr(dev_err), _stream(stream)))


def moe_w2_mm_noalloc(stage, act, codes_k, scales_k, offsets, E, N, K, rows, out, out_fmt, act_row=None,
                      act_row_div=1, expert_slot=None, dev_err=None, stream=None):
    """moe_w2_mm's table GEMV on the library's own fixed scratch (bf16 act)."""
    _check(lib().moe_w2_mm_noalloc(stage, _ptr(act), act.shape[0], _ptr(act_row), act_row_div, _ptr(codes_k),
                                   _ptr(scales_k), _ptr(offsets), _ptr(expert_slot), E, N, K, rows, _ptr(out),
                                   out_fmt, _ptr(dev_err), _stream(stream)))


def moe_mxfp4_mm(stage, act, act_fmt, offsets, E, N, K, out, out_fmt, e2m1=None, e8m0=None, fp8_ws=None,
                 ws_slot_of_expert=None, act_scale=None, act_row=None, act_row_div=1, expert_slot=None,
                 expert_begin=0, expert_end=None, out_scale=None, mode=MODE_AUTO, dev_err=None, stream=None):
    expert_end = E if expert_end is None else expert_end
    _check(lib().moe_mxfp4_mm(stage, mode, _ptr(act), act_fmt, _ptr(act_scale), act.shape[0], _ptr(act_row),
                              act_row_div,
                              _ptr(e2m1), _ptr(e8m0), _ptr(fp8_ws), _ptr(ws_slot_of_expert), _ptr(offsets),
                              _ptr(expert_slot), expert_begin, expert_end, E, N, K, _ptr(out), out_fmt,
                              _ptr(out_scale), None, 0, _ptr(dev_err), _stream(stream)))


def moe_combine(y, y_fmt, w, inv, T, k, H, out, out_fmt, stream=None):
    _check(lib().moe_combine(_ptr(y), y_fmt, _ptr(w), _ptr(inv), T, k, H, _ptr(out), out_fmt, _stream(stream)))


def moe_cache_select(offsets, counts, decay_shift, expert_slot, slot_expert, promoted, dev_err=None, stream=None):
    E = counts.numel()
    S = slot_expert.numel()
    _check(lib().moe_cache_select(_ptr(offsets), E, _ptr(counts), decay_shift, S, _ptr(expert_slot),
                                  _ptr(slot_expert), _ptr(promoted), _ptr(dev_err), _stream(stream)))


def moe_cache_fill(promoted, srcs, dsts, nbytes, stream=None):
    """srcs / dsts: device-accessible base addresses (tensors or ints); nbytes:
    bytes per expert / slot of each array."""
    n = len(srcs)
    S = promoted.numel()
    src_arr = (ctypes.c_void_p * n)(*[_ptr(t) for t in srcs])
    dst_arr = (ctypes.c_void_p * n)(*[_ptr(t) for t in dsts])
    by_arr = (ctypes.c_size_t * n)(*[int(b) for b in nbytes])
    _check(lib().moe_cache_fill(_ptr(promoted), S, n, src_arr, dst_arr, by_arr, _stream(stream)))


def moe_stage_select(offsets, res_slot, R, weight_slot, staged, dev_err=None, stream=None):
    E = res_slot.numel()
    _check(lib().moe_stage_select(_ptr(offsets), E, _ptr(res_slot), R, staged.numel(), _ptr(weight_slot),
                                  _ptr(staged), _ptr(dev_err), _stream(stream)))


def moe_w2_mm_slots(stage, act, codes_k, scales_k, offsets, weight_slot, slot_lo, slot_hi, E, N, K, out, out_fmt,
                    ws, act_row=None, act_row_div=1, dev_err=None, stream=None):
    nbytes = ws.numel() * ws.element_size()
    _check(lib().moe_w2_mm_slots(stage, _ptr(act), act.shape[0], _ptr(act_row), act_row_div, _ptr(codes_k),
                                 _ptr(scales_k), _ptr(offsets), _ptr(weight_slot), slot_lo, slot_hi, E, N, K,
                                 _ptr(out), out_fmt, _ptr(ws), nbytes, _ptr(dev_err), _stream(stream)))


def moe_w2_decode_fused_workspace_size(rows, H, I) -> int:
    return int(lib().moe_w2_decode_fused_workspace_size(rows, H, I))


def moe_w2_decode_fused(x, codes1, scales1, codes2, scales2, offsets, E, H, I, h, y, y_fmt, ws, act_row=None,
                        act_row_div=1, expert_slot=None, dev_err=None, stream=None):
    nbytes = ws.numel() * ws.element_size()
    _check(lib().moe_w2_decode_fused(_ptr(x), x.shape[0], _ptr(act_row), act_row_div, _ptr(codes1), _ptr(scales1),
                                     _ptr(codes2), _ptr(scales2), _ptr(offsets), _ptr(expert_slot), E, H, I,
                                     _ptr(h), _ptr(y), y_fmt, _ptr(ws), nbytes, _ptr(dev_err), _stream(stream)))


def moe_w2_decode_layer_workspace_size(T, k, H, I) -> int:
    return int(lib().moe_w2_decode_layer_workspace_size(T, k, H, I))


def moe_w2_decode_layer(logits, x, k, codes1, scales1, codes2, scales2, H, I, ids, w, offsets, perm, inv, h, y, out,
                        out_fmt, ws, dev_err=None, stream=None):
    T, E = logits.shape
    nbytes = 0 if ws is None else ws.numel() * ws.element_size()
    _check(lib().moe_w2_decode_layer(_ptr(logits), _ptr(x), T, E, k, _ptr(codes1), _ptr(scales1), _ptr(codes2),
                                     _ptr(scales2), H, I, _ptr(ids), _ptr(w), _ptr(offsets), _ptr(perm), _ptr(inv),
                                     _ptr(h), _ptr(y), _ptr(out), out_fmt, _ptr(ws), nbytes, _ptr(dev_err),
                                     _stream(stream)))
