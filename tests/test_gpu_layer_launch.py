"""The whole 2-bit decode step in one launch (moe_w2_decode_layer), through
the C ABI (GPU): every output (ids, w, offsets, perm, inv, h, y, out)
bit-identical to the four calls it replaces (moe_route, moe_permute,
moe_w2_decode_fused, moe_combine) at the decode workload and at edge shapes
(k not a power of two, one token, the largest T*k, E = 1024, tied and NaN
logits, T = 0), repeats and a captured graph, and the oracle's gate."""
import numpy as np
import pytest
import torch

from bit_moe_expert_top_gb300 import _lib as L
from bit_moe_expert_top_gb300 import synth
from bit_moe_expert_top_gb300.layer import MoELayer
from oracle import moe as M

from tests._gpu import TOL_BF16, dev, host, rel_err

pytestmark = pytest.mark.gpu

CASES = {
    "decode": dict(),
    "odd k": dict(E=24, H=1024, I=512, k=3, T=13),
    "one token": dict(E=8, H=512, I=512, k=2, T=1),
    "largest": dict(E=1024, H=512, I=512, k=16, T=16),
    "E 129..256": dict(E=200, H=512, I=1024, k=6, T=10),
    "E 257..512": dict(E=257, H=512, I=512, k=5, T=7),
}


def _pair(w, raw, out_fmt):
    four = MoELayer("w2", w.E, w.H, w.I, w.k, w2=raw, out_fmt=out_fmt, mode=L.MODE_GEMV, fused=True,
                    single_launch=False)
    one = MoELayer("w2", w.E, w.H, w.I, w.k, w2=raw, out_fmt=out_fmt, mode=L.MODE_GEMV, fused=True,
                   single_launch=True)
    return four, one


def _same(b1, b4):
    for f in ("ids", "w", "offsets", "perm", "inv", "h", "y", "out"):
        assert torch.equal(getattr(b1, f), getattr(b4, f)), f
    assert L.moe_get_error(b1.dev_err) == L.moe_get_error(b4.dev_err)


@pytest.mark.parametrize("out_fmt", [L.FMT_BF16, L.FMT_F32], ids=["bf16 out", "f32 out"])
@pytest.mark.parametrize("case", list(CASES))
def test_single_launch_bit_identical_to_four_calls(case, out_fmt):
    w = synth.get_workload("decode").replace(**CASES[case])
    if case != "decode":
        w = w.replace(logits="uniform")
    raw = synth.make_w2_layer(w)
    four, one = _pair(w, raw, out_fmt)
    for bi in range(2):
        x = synth.make_x(w, 0, tid_offset=bi)
        lg = synth.make_logits(w, 0, x_bits=x, tid_offset=bi)
        xd, ld = dev(x.view(np.int16)), dev(lg)
        b4, b1 = four.buffers(w.T), one.buffers(w.T)
        o4 = four.step(xd, ld, b4)
        o1 = one.step(xd, ld, b1)
        torch.cuda.synchronize()
        assert L.moe_get_error(b1.dev_err) == 0
        _same(b1, b4)
        if bi == 0:
            tok = [0, w.T - 1]
            ref = M.layer(x, lg, w.k, M.w2_expert_weights(*raw), profile="bf16", tokens=tok)
            assert np.array_equal(host(b1.ids), ref["ids"])
            err, _ = rel_err(host(o1).astype(np.float64)[tok] if out_fmt == L.FMT_F32 else
                             _bf16_host(o1)[tok], ref["out"])
            assert err <= TOL_BF16


def _bf16_host(t):
    from oracle import codecs as C
    return C.bf16_bits_to_f64(host(t).view(np.uint16))


def test_single_launch_ties_and_nan_logits():
    """Logits on a coarse grid (many ties: the lower expert id wins) and a
    NaN in one token's row (ranked below every number, NAN_LOGIT set)."""
    w = synth.get_workload("decode").replace(E=64, H=512, I=512, k=4, T=8, logits="uniform")
    raw = synth.make_w2_layer(w)
    four, one = _pair(w, raw, L.FMT_F32)
    x = synth.make_x(w)
    lg = np.round(synth.make_logits(w, x_bits=x) * 4) / 4
    lg[3, 5] = np.nan
    xd, ld = dev(x.view(np.int16)), dev(lg.astype(np.float32))
    b4, b1 = four.buffers(w.T), one.buffers(w.T)
    four.step(xd, ld, b4)
    one.step(xd, ld, b1)
    torch.cuda.synchronize()
    assert L.moe_get_error(b1.dev_err) == L.DEVERR_NAN_LOGIT
    _same(b1, b4)
    ids, _, _ = M.route(lg.astype(np.float32), w.k)
    assert np.array_equal(host(b1.ids), ids)


def test_single_launch_repeats_capture_and_empty_step():
    w = synth.get_workload("decode")
    raw = synth.make_w2_layer(w)
    _, one = _pair(w, raw, L.FMT_BF16)
    x = dev(synth.make_x(w).view(np.int16))
    lg = dev(synth.make_logits(w))
    b = one.buffers(w.T)
    first = one.step(x, lg, b).clone()
    for _ in range(3):  # the barrier counter is left at zero by every launch
        assert torch.equal(one.step(x, lg, b), first)
    g = one.capture(w.T)
    assert torch.equal(g.run(x, lg), first)
    assert L.moe_get_error(b.dev_err) == 0
    # T = 0: offsets zeroed, nothing launched
    b0 = one.buffers(0)
    b0.offsets.fill_(7)
    out = one.step(torch.empty((0, w.H), dtype=torch.int16, device="cuda"),
                   torch.empty((0, w.E), dtype=torch.float32, device="cuda"), b0)
    torch.cuda.synchronize()
    assert out.shape[0] == 0 and int(b0.offsets.abs().sum()) == 0


def test_single_launch_limits():
    """Shapes beyond the one-launch limits are refused with UNSUPPORTED (the
    layer then takes the four calls)."""
    w = synth.get_workload("decode").replace(E=64, H=512, I=512, k=4, T=65)  # T*k = 260 > 256
    raw = synth.make_w2_layer(w)
    four, one = _pair(w, raw, L.FMT_F32)
    b = one.buffers(w.T)
    n = L.moe_w2_decode_layer_workspace_size(w.T, w.k, w.H, w.I)
    ws = torch.zeros((n + 3) // 4, dtype=torch.int32, device="cuda")
    lg = dev(synth.make_logits(w))
    x = dev(synth.make_x(w).view(np.int16))
    with pytest.raises(L.MoEError) as ei:
        L.moe_w2_decode_layer(lg, x, w.k, one.c1k, one.s1k, one.c2k, one.s2k, w.H, w.I, b.ids, b.w, b.offsets,
                              b.perm, b.inv, b.h, b.y, b.out, L.FMT_F32, ws, dev_err=b.dev_err)
    assert ei.value.code == L.MOE_ERR_UNSUPPORTED
    b4 = four.buffers(w.T)
    o4 = four.step(x, lg, b4)
    o1 = one.step(x, lg, b)  # falls back to the four calls
    torch.cuda.synchronize()
    assert torch.equal(o1, o4)
