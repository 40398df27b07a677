"""The mixed decode layer with its delta-cache (MXFP4) experts on the
block-scaled FP8 tensor core (cache_fp8: MXFP8 token rows and an MXFP8 h for
those experts; the 2-bit experts unchanged, in bf16), through the C ABI
(GPU), against the oracle's per-expert profile (fp8 for the cache experts,
bf16 for the others): routing bit-exact, the layer output at the FP8 gate,
and the 2-bit experts' y rows bit-identical to the all-bf16 mixed layer's."""
import numpy as np
import pytest
import torch

from bit_moe_expert_top_gb300 import _lib as L
from bit_moe_expert_top_gb300 import synth
from bit_moe_expert_top_gb300.layer import MoELayer
from oracle import moe as M

from tests._gpu import TOL_FP8, dev, host, rel_err

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("case", ["small", "full size, sampled tokens"])
def test_cache_fp8_mixed_layer(case):
    w = synth.get_workload("mixed_decode")
    tok = [3, 60]
    if case == "small":
        w = w.replace(E=24, H=512, I=256, k=4, T=48, n_hot=6)
        tok = list(range(w.T))
    raw = synth.make_w2_layer(w)
    mx = synth.make_mxfp4_layer(w, n=w.n_hot)
    slot = synth.hot_experts(w)
    bf = MoELayer("mixed", w.E, w.H, w.I, w.k, w2=raw, mx=mx, expert_slot=slot, out_fmt=L.FMT_F32)
    f8 = MoELayer("mixed", w.E, w.H, w.I, w.k, w2=raw, mx=mx, expert_slot=slot, out_fmt=L.FMT_F32,
                  cache_fp8=True)
    x = synth.make_x(w)
    lg = synth.make_logits(w, x_bits=x)
    xd, ld = dev(x.view(np.int16)), dev(lg)
    bb, b8 = bf.buffers(w.T), f8.buffers(w.T)
    bf.step(xd, ld, bb)
    out = f8.step(xd, ld, b8)
    torch.cuda.synchronize()
    assert L.moe_get_error(b8.dev_err) == 0
    off = host(b8.offsets)
    cached_rows = np.zeros(w.T * w.k, bool)
    for e in np.nonzero(slot >= 0)[0]:
        cached_rows[off[e]:off[e + 1]] = True
    assert cached_rows.any() and (~cached_rows).any()
    keep = torch.from_numpy(~cached_rows).cuda()
    assert torch.equal(b8.y[keep], bb.y[keep])  # the 2-bit experts' rows: the same table GEMV
    acc = M.mixed_expert_weights(M.w2_expert_weights(*raw), M.mxfp4_expert_weights(*mx), slot)
    ref = M.layer(x, lg, w.k, acc, tokens=tok, expert_profile=lambda e: "fp8" if slot[e] >= 0 else "bf16")
    assert np.array_equal(host(b8.ids), ref["ids"])
    err, rms = rel_err(host(out)[tok], ref["out"])
    assert rms > 0 and err <= TOL_FP8, err
