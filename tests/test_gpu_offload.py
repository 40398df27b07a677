"""Host-resident 2-bit experts staged per step into a device pool
(moe_stage_select + moe_cache_fill from pinned host memory +
moe_w2_mm_slots), through the C ABI (GPU).

The staging choice is checked against its definition written out here; the
layer with most experts in host memory must give the same bits as the layer
with every expert in device memory (same kernel, same summation order per
row), and match the oracle."""
import numpy as np
import pytest
import torch

from bit_moe_expert_top_gb300 import _lib as L
from bit_moe_expert_top_gb300 import synth
from bit_moe_expert_top_gb300.layer import MoELayer
from oracle import moe as M

from tests._gpu import DEV, TOL_BF16, dev, host, rel_err

pytestmark = pytest.mark.gpu


def _staging_by_definition(off, res, R, S):
    """Routed experts without a resident slot, in ascending id, take staging
    slots R, R+1, ...; beyond S of them they are skipped (-1)."""
    cnt = np.diff(off)
    ws = np.array(res, dtype=np.int64)
    staged = np.full(S, -1, np.int64)
    j = 0
    for e in range(cnt.size):
        if cnt[e] > 0 and res[e] < 0:
            if j < S:
                ws[e] = R + j
                staged[j] = e
            else:
                ws[e] = -1
            j += 1
    return ws, staged, j > S


@pytest.mark.parametrize("E,R,S", [(48, 20, 64), (384, 192, 64), (40, 10, 3), (8, 0, 8)])
def test_stage_select_matches_its_definition(E, R, S):
    g = np.random.default_rng(E + R)
    res = np.full(E, -1, np.int32)
    res[g.permutation(E)[:R]] = np.arange(R, dtype=np.int32)
    d_res = dev(res)
    ws = torch.empty(E, dtype=torch.int32, device=DEV)
    st = torch.empty(S, dtype=torch.int32, device=DEV)
    for _ in range(5):
        sizes = g.poisson(0.4, size=E)
        off = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32)
        err = torch.zeros(1, dtype=torch.int32, device=DEV)
        L.moe_stage_select(dev(off), d_res, R, ws, st, dev_err=err)
        want_ws, want_st, over = _staging_by_definition(off, res, R, S)
        routed = np.diff(off) > 0
        assert np.array_equal(host(ws)[routed], want_ws[routed])
        assert np.array_equal(host(st), want_st)
        assert bool(L.moe_get_error(err) & L.DEVERR_OVERFLOW) == over


def _pair(w, resident, S=64, side_sms=0):
    raw = synth.make_w2_layer(w)
    full = MoELayer("w2", w.E, w.H, w.I, w.k, w2=raw, out_fmt=L.FMT_F32, mode=L.MODE_GEMV)
    off = MoELayer("w2host", w.E, w.H, w.I, w.k, w2=raw, out_fmt=L.FMT_F32, mode=L.MODE_GEMV,
                   resident=resident, stage_slots=S, side_sms=side_sms)
    return raw, full, off


@pytest.mark.parametrize("name,frac,side", [("small", 0.4, 0), ("decode", 0.5, 0), ("small", 0.4, 12),
                                            ("decode", 0.5, 16)])
def test_host_resident_layer_bit_identical_to_device_layer(name, frac, side):
    """side: SMs reserved for the staging copy, the resident experts' FC1 and
    FC2 running beside it on the others (moe_set_side_sms)."""
    w = (synth.get_workload("tiny").replace(E=48, H=1024, I=512, k=4, T=16, logits="uniform") if name == "small"
         else synth.get_workload("decode"))
    resident = list(range(0, w.E, int(round(1 / frac))))        # every other / every 2.5th expert on the device
    raw, full, offl = _pair(w, resident, side_sms=side)
    assert offl.R == len(resident) and offl.store[0].is_pinned()
    for bi in range(2):
        x = synth.make_x(w, 0, tid_offset=bi)
        lg = synth.make_logits(w, 0, x_bits=x, tid_offset=bi)
        xd, ld = dev(x.view(np.int16)), dev(lg)
        bf, bo = full.buffers(w.T), offl.buffers(w.T)
        out_f = full.step(xd, ld, bf)
        out_o = offl.step(xd, ld, bo)
        torch.cuda.synchronize()
        assert L.moe_get_error(bo.dev_err) == 0
        off = host(bo.offsets)
        cold = int(np.sum((np.diff(off) > 0) & (host(offl.res_slot) < 0)))
        assert cold > 0                                          # some routed experts came over the link
        assert torch.equal(out_o, out_f)
        assert torch.equal(bo.y, bf.y)
        assert L.moe_set_side_sms(0) == 0                        # the layer restored the setting
        tok = [0, w.T - 1]
        ref = M.layer(x, lg, w.k, M.w2_expert_weights(*raw), profile="bf16", tokens=tok)
        err, _ = rel_err(host(out_o)[tok], ref["out"])
        assert err <= TOL_BF16


def test_host_resident_layer_overflow_is_flagged():
    """More routed host-resident experts than staging slots: OVERFLOW, and the
    skipped experts' rows are left alone (no wrong weights are read)."""
    w = synth.get_workload("tiny").replace(E=32, H=512, I=512, k=4, T=16, logits="uniform")
    raw, full, offl = _pair(w, resident=[0, 1], S=2)
    x = dev(synth.make_x(w).view(np.int16))
    lg = dev(synth.make_logits(w))
    b = offl.buffers(w.T)
    offl.step(x, lg, b)
    torch.cuda.synchronize()
    assert L.moe_get_error(b.dev_err) & L.DEVERR_OVERFLOW
