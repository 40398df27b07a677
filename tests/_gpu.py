"""Helpers shared by the GPU parity tests: device upload and the oracle runs
on the same seeded inputs."""
import numpy as np
import torch

from bit_moe_expert_top_gb300 import _lib as L
from bit_moe_expert_top_gb300 import synth
from bit_moe_expert_top_gb300.layer import MoELayer
from oracle import codecs as C
from oracle import moe as M

DEV = "cuda"

# Output tolerances of the layer (max |err| / RMS(out)): bf16 profile and the
# FP8 workspace profile.
TOL_BF16 = 2e-2
TOL_FP8 = 6e-2
# Routing weights: fp32 expf (<= 2 ulp) + sum + divide against the fp64
# softmax rounded once: a few ulp of 1.0.
TOL_W = 1e-6


def dev(a, dtype=None):
    t = torch.from_numpy(np.ascontiguousarray(a))
    if dtype is not None:
        t = t.view(dtype)
    return t.to(DEV)


def host(t):
    return t.cpu().numpy()


def bf16_to_f64(t):
    return C.bf16_bits_to_f64(host(t).view(np.uint16))


def make_layer(w, seed=0, out_fmt=L.FMT_F32, mode=L.MODE_GEMV, layer=0, direct=False):
    """(MoELayer, oracle expert accessor, profile).  direct: MXFP4 experts
    multiplied as stored (no FP8 workspace)."""
    if w.weights == "w2":
        raw = synth.make_w2_layer(w, seed, layer)
        ml = MoELayer("w2", w.E, w.H, w.I, w.k, w2=raw, out_fmt=out_fmt, mode=mode)
        return ml, M.w2_expert_weights(*raw), "bf16"
    if w.weights == "mixed":
        raw = synth.make_w2_layer(w, seed, layer)
        mx = synth.make_mxfp4_layer(w, n=w.n_hot, seed=seed, layer=layer)
        slot = synth.hot_experts(w, seed)
        ml = MoELayer("mixed", w.E, w.H, w.I, w.k, w2=raw, mx=mx, expert_slot=slot, out_fmt=out_fmt, mode=mode)
        acc = M.mixed_expert_weights(M.w2_expert_weights(*raw), M.mxfp4_expert_weights(*mx), slot)
        return ml, acc, "bf16"
    mx = synth.make_mxfp4_layer(w, seed=seed, layer=layer)
    if direct:
        ml = MoELayer("mxfp4", w.E, w.H, w.I, w.k, mx=mx, out_fmt=out_fmt, mode=mode)
        return ml, M.mxfp4_expert_weights(*mx), "fp8"
    ml = MoELayer("fp8", w.E, w.H, w.I, w.k, mx=mx, out_fmt=out_fmt, mode=mode,
                  fp8_batch=max(1, min(16, w.E // 4)))
    return ml, M.fp8_expert_weights(*mx), "fp8"


def run_layer(ml, x_bits, logits):
    x = dev(x_bits.view(np.int16))
    lg = dev(logits)
    b = ml.buffers(x.shape[0])
    out = ml.step(x, lg, b)
    torch.cuda.synchronize()
    return out, b


def rel_err(got, want):
    want = np.asarray(want, dtype=np.float64)
    rms = float(np.sqrt(np.mean(want ** 2)))
    return float(np.max(np.abs(np.asarray(got, dtype=np.float64) - want))) / rms, rms
