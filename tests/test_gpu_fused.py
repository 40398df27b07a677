"""FC1 + SwiGLU and FC2 of the 2-bit decode step in one cooperative launch
(moe_w2_decode_fused), through the C ABI (GPU): bit-identical h, y and layer
output to the two table-GEMV calls, and the oracle's gate."""
import numpy as np
import pytest
import torch

from bit_moe_expert_top_gb300 import _lib as L
from bit_moe_expert_top_gb300 import synth
from bit_moe_expert_top_gb300.layer import MoELayer
from oracle import moe as M

from tests._gpu import TOL_BF16, dev, host, rel_err

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("name", ["small", "decode", "mixed_decode_sized"])
def test_fused_decode_bit_identical_to_two_calls(name):
    if name == "small":
        w = synth.get_workload("tiny").replace(E=24, H=1024, I=512, k=4, T=13, logits="uniform")
    elif name == "decode":
        w = synth.get_workload("decode")
    else:  # 64 tokens, Zipf routing: several rows per expert
        w = synth.get_workload("prefill_bf16").replace(T=64)
    raw = synth.make_w2_layer(w)
    two = MoELayer("w2", w.E, w.H, w.I, w.k, w2=raw, out_fmt=L.FMT_F32, mode=L.MODE_GEMV, fused=False)
    one = MoELayer("w2", w.E, w.H, w.I, w.k, w2=raw, out_fmt=L.FMT_F32, mode=L.MODE_GEMV, fused=True,
                   single_launch=False)
    for bi in range(2):
        x = synth.make_x(w, 0, tid_offset=bi)
        lg = synth.make_logits(w, 0, x_bits=x, tid_offset=bi)
        xd, ld = dev(x.view(np.int16)), dev(lg)
        b2, b1 = two.buffers(w.T), one.buffers(w.T)
        assert b1.fws is not None and b2.fws is None
        o2 = two.step(xd, ld, b2)
        o1 = one.step(xd, ld, b1)
        torch.cuda.synchronize()
        assert L.moe_get_error(b1.dev_err) == 0
        assert torch.equal(b1.h, b2.h) and torch.equal(b1.y, b2.y) and torch.equal(o1, o2)
        tok = [0, w.T - 1]
        ref = M.layer(x, lg, w.k, M.w2_expert_weights(*raw), profile="bf16", tokens=tok)
        err, _ = rel_err(host(o1)[tok], ref["out"])
        assert err <= TOL_BF16


def test_fused_decode_repeats_and_captures():
    """Repeated launches (the barrier counter is zeroed by each call) and a
    captured graph give the same bits."""
    w = synth.get_workload("decode")
    ml = MoELayer("w2", w.E, w.H, w.I, w.k, w2=synth.make_w2_layer(w), out_fmt=L.FMT_BF16, mode=L.MODE_GEMV,
                  fused=True, single_launch=False)
    x = dev(synth.make_x(w).view(np.int16))
    lg = dev(synth.make_logits(w))
    b = ml.buffers(w.T)
    first = ml.step(x, lg, b).clone()
    for _ in range(3):
        assert torch.equal(ml.step(x, lg, b), first)
    g = ml.capture(w.T)
    assert torch.equal(g.run(x, lg), first)
    assert L.moe_get_error(b.dev_err) == 0


def test_mxfp4_decode_on_the_block_scaled_tensor_core():
    """The decode shapes with MXFP4 experts multiplied as stored (MXFP8 tokens,
    32-token tiles, one tile per expert): sampled tokens at the FP8 gate."""
    from tests._gpu import TOL_FP8, make_layer, run_layer
    w = synth.get_workload("decode").replace(weights="mxfp4")
    ml, acc, prof = make_layer(w, direct=True)
    x = synth.make_x(w)
    lg = synth.make_logits(w, x_bits=x)
    out, b = run_layer(ml, x, lg)
    assert L.moe_get_error(b.dev_err) == 0
    tok = [0, 3, 7]
    ref = M.layer(x, lg, w.k, acc, profile=prof, tokens=tok)
    err, _ = rel_err(host(out)[tok], ref["out"])
    assert err <= TOL_FP8
