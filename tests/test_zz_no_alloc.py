"""moe_w2_mm_noalloc (the table GEMV on the library's own fixed scratch)
against moe_w2_mm with a caller workspace, through the C ABI.

The file sorts last so that it also runs after every other GPU test in one
process; it passes alone as well.  Two calls in a row on each shape: the
second finds the scratch as the first left it."""
import numpy as np
import pytest
import torch

from bit_moe_expert_top_gb300 import _lib as L
from bit_moe_expert_top_gb300 import synth
from tests._gpu import TOL_BF16, dev, make_layer

pytestmark = pytest.mark.gpu


def _check_close(got, want):
    """max |got - want| <= TOL_BF16 * RMS(want) (the layer's bf16 bar); the two
    entry points run the same kernel in the same order, so the values are also
    expected to be identical."""
    g = got.view(torch.bfloat16).double().cpu().numpy()
    w = want.view(torch.bfloat16).double().cpu().numpy()
    rms = float(np.sqrt(np.mean(w ** 2)))
    assert rms > 0
    assert float(np.max(np.abs(g - w))) <= TOL_BF16 * rms
    assert torch.equal(got, want)


SMALL = dict(E=6, H=1024, I=512, k=3, T=21, logits="uniform")   # several slices and batches, ragged


def _routed(name, seed):
    w = synth.get_workload("tiny").replace(**SMALL) if name == "small" else synth.get_workload(name)
    ml, _, _ = make_layer(w, seed=seed, out_fmt=L.FMT_BF16, mode=L.MODE_GEMV)
    x = dev(synth.make_x(w, seed).view(np.int16))
    lg = dev(synth.make_logits(w, seed))
    b = ml.buffers(w.T)
    L.moe_route(lg, w.k, b.ids, b.w, b.dev_err)
    L.moe_permute(b.ids, w.E, b.offsets, b.perm, b.inv, dev_err=b.dev_err)
    torch.cuda.synchronize()
    return w, ml, x, b


@pytest.mark.parametrize("name", ["small", "decode"])
def test_noalloc_matches_workspace_entry(name):
    w, ml, x, b = _routed(name, seed=5)
    E, H, I, k, A = w.E, w.H, w.I, w.k, w.T * w.k
    assert b.ws is not None
    # the existing entry point, with the caller's workspace
    h_ref = torch.empty_like(b.h)
    y_ref = torch.empty_like(b.y)
    L.moe_w2_mm(L.STAGE_FC1_SWIGLU, x, L.FMT_BF16, ml.c1k, ml.s1k, b.offsets, E, I, H, h_ref, L.FMT_BF16,
                act_row=b.perm, act_row_div=k, mode=L.MODE_GEMV, ws=b.ws, dev_err=b.dev_err)
    L.moe_w2_mm(L.STAGE_FC2, h_ref, L.FMT_BF16, ml.c2k, ml.s2k, b.offsets, E, H, I, y_ref, L.FMT_BF16,
                mode=L.MODE_GEMV, ws=b.ws, dev_err=b.dev_err)
    torch.cuda.synchronize()
    free_before = None
    for call in range(2):
        h = torch.full_like(b.h, 0x7FC0)       # bf16 NaN: every row must be rewritten
        y = torch.full_like(b.y, 0x7FC0)
        torch.cuda.synchronize()
        if call == 1:
            free_before = torch.cuda.mem_get_info()[0]
        L.moe_w2_mm_noalloc(L.STAGE_FC1_SWIGLU, x, ml.c1k, ml.s1k, b.offsets, E, I, H, A, h, L.FMT_BF16,
                            act_row=b.perm, act_row_div=k, dev_err=b.dev_err)
        L.moe_w2_mm_noalloc(L.STAGE_FC2, h, ml.c2k, ml.s2k, b.offsets, E, H, I, A, y, L.FMT_BF16,
                            dev_err=b.dev_err)
        torch.cuda.synchronize()
        if call == 1:
            # once the module is loaded, a call takes no device memory
            assert torch.cuda.mem_get_info()[0] == free_before
        _check_close(h, h_ref)
        _check_close(y, y_ref)
    assert L.moe_get_error(b.dev_err) == 0


def test_noalloc_rejects_rows_beyond_the_fixed_scratch():
    w, ml, x, b = _routed("decode", seed=6)
    E, H, I = w.E, w.H, w.I
    rows = 1
    while L.moe_w2_mm_workspace_size(L.STAGE_FC1_SWIGLU, rows + 1, I, H) <= L.W2_NOALLOC_SCRATCH_BYTES:
        rows += 1
    big = torch.empty((rows + 1, I), dtype=torch.int16, device="cuda")
    with pytest.raises(L.MoEError) as ei:
        L.moe_w2_mm_noalloc(L.STAGE_FC1_SWIGLU, x, ml.c1k, ml.s1k, b.offsets, E, I, H, rows + 1, big, L.FMT_BF16,
                            act_row=b.perm, act_row_div=w.k, dev_err=b.dev_err)
    assert ei.value.code == L.MOE_ERR_WS_SMALL
    assert "scratch" in str(ei.value)


def test_k_not_a_multiple_of_the_slice_width():
    """K = 640 (a multiple of 128, not of the table GEMV's 512-element slice):
    the workspace query answers 0, moe_w2_mm runs the register-decode GEMV
    (a workspace passed anyway is ignored) and matches the oracle's exact
    sums, and moe_w2_mm_noalloc refuses the shape as unsupported (not as a
    small scratch), whatever the row count."""
    from oracle import codecs as C
    from oracle import moe as M
    w = synth.get_workload("tiny").replace(E=4, H=640, I=256, k=2, T=9, logits="uniform")
    assert L.moe_w2_mm_workspace_size(L.STAGE_FC1_SWIGLU, 64, w.I, w.H) == 0
    assert L.moe_w2_mm_workspace_size(L.STAGE_FC2, 64, w.H, 640) == 0
    ml, acc, _ = make_layer(w, seed=1, out_fmt=L.FMT_F32, mode=L.MODE_GEMV)
    x = synth.make_x(w, 1)
    lg = synth.make_logits(w, 1)
    ids, _, _ = M.route(lg, w.k)
    off, perm, _ = M.permute(ids, w.E)
    A = w.T * w.k
    h = torch.empty((A, w.I), dtype=torch.float32, device="cuda")
    junk_ws = torch.empty(1 << 20, dtype=torch.uint8, device="cuda")
    L.moe_w2_mm(L.STAGE_FC1_SWIGLU, dev(x.view(np.int16)), L.FMT_BF16, ml.c1k, ml.s1k, dev(off), w.E, w.I, w.H, h,
                L.FMT_F32, act_row=dev(perm), act_row_div=w.k, mode=L.MODE_GEMV, ws=junk_ws)
    torch.cuda.synchronize()
    xp = C.bf16_bits_to_f64(x)[perm // w.k]
    want = np.zeros((A, w.I))
    for e in range(w.E):
        r = slice(off[e], off[e + 1])
        if off[e] != off[e + 1]:
            W1 = acc(e)[0]
            want[r] = M.silu(C.to_f32(xp[r] @ W1[:w.I].T)) * C.to_f32(xp[r] @ W1[w.I:].T)
    rms = np.sqrt(np.mean(want ** 2))
    assert np.max(np.abs(h.double().cpu().numpy() - want)) <= 1e-4 * rms
    out = torch.empty((100000, w.I), dtype=torch.int16, device="cuda")
    for rows in (A, 100000):
        with pytest.raises(L.MoEError) as ei:
            L.moe_w2_mm_noalloc(L.STAGE_FC1_SWIGLU, dev(x.view(np.int16)), ml.c1k, ml.s1k, dev(off), w.E, w.I, w.H,
                                rows, out, L.FMT_BF16, act_row=dev(perm), act_row_div=w.k)
        assert ei.value.code == L.MOE_ERR_UNSUPPORTED
