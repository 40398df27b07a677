"""The 2-bit table GEMV (MODE_GEMV with a workspace) stage by stage, through
the C ABI (GPU).

FC1 and FC2 with fp32 outputs are compared element by element with the exact
(fp64) sums of the same bf16 operands, at 1e-4 * RMS: that checks the table
arithmetic, the K-slice split and the slice-ordered final sums free of bf16
rounding flips.  Shapes span several K slices, several row batches per CTA
and CTA ranges that cut segments anywhere.  Also: the workspace is left zero,
a workspace that covers fewer rows flags OVERFLOW and leaves the uncovered
rows alone, and the register-decode kernel (no workspace) agrees."""
import numpy as np
import pytest
import torch

from bit_moe_expert_top_gb300 import _lib as L
from bit_moe_expert_top_gb300 import synth
from oracle import codecs as C
from oracle import moe as M

from tests._gpu import DEV, dev, host, make_layer

pytestmark = pytest.mark.gpu

SHAPES = [(6, 1024, 512, 3, 37), (4, 512, 512, 2, 90), (9, 1536, 1024, 4, 21), (40, 512, 1024, 8, 3)]


def _setup(E, H, I, k, T, seed=0):
    w = synth.get_workload("tiny").replace(E=E, H=H, I=I, k=k, T=T, logits="uniform")
    ml, acc, _ = make_layer(w, seed, mode=L.MODE_GEMV)
    x = synth.make_x(w, seed)
    logits = synth.make_logits(w, seed, x_bits=x)
    ids, _, _ = M.route(logits, k)
    off, perm, inv = M.permute(ids, E)
    return w, ml, acc, x, off, perm


def _want(acc, x, off, perm, k, E, H, I):
    """fp32 h = silu(g)*u from exact sums, and exact y on the bf16-rounded h."""
    A = perm.size
    xp = C.bf16_bits_to_f64(x)[perm // k]
    want_h = np.zeros((A, I))
    for e in range(E):
        rows = slice(off[e], off[e + 1])
        if off[e] == off[e + 1]:
            continue
        W1, _ = acc(e)
        g = C.to_f32(xp[rows] @ W1[:I].T)
        u = C.to_f32(xp[rows] @ W1[I:].T)
        want_h[rows] = M.silu(g) * u
    h_bits = C.f32_to_bf16_bits(want_h.astype(np.float32))
    hval = C.bf16_bits_to_f64(h_bits)
    want_y = np.zeros((A, H))
    for e in range(E):
        rows = slice(off[e], off[e + 1])
        if off[e] != off[e + 1]:
            want_y[rows] = hval[rows] @ acc(e)[1].T
    return want_h, h_bits, want_y


def _ws(rows, N_fc1, K_fc1, N_fc2, K_fc2):
    """A workspace full of garbage (NaN patterns): its contents must not matter."""
    n = max(L.moe_w2_mm_workspace_size(L.STAGE_FC1_SWIGLU, rows, N_fc1, K_fc1),
            L.moe_w2_mm_workspace_size(L.STAGE_FC2, rows, N_fc2, K_fc2))
    return torch.full(((n + 3) // 4,), 0x7FC01234, dtype=torch.int32, device=DEV)


@pytest.mark.parametrize("E,H,I,k,T", SHAPES)
def test_lut_stages_exact_sums(E, H, I, k, T):
    w, ml, acc, x, off, perm = _setup(E, H, I, k, T)
    A = T * k
    want_h, h_bits, want_y = _want(acc, x, off, perm, k, E, H, I)
    d_off, d_perm, d_x = dev(off), dev(perm), dev(x.view(np.int16))
    ws = _ws(A, I, H, H, I)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    for use_ws in (ws, None):       # table GEMV, then the register-decode kernel
        h32 = torch.empty((A, I), dtype=torch.float32, device=DEV)
        L.moe_w2_mm(L.STAGE_FC1_SWIGLU, d_x, L.FMT_BF16, ml.c1k, ml.s1k, d_off, E, I, H, h32, L.FMT_F32,
                    act_row=d_perm, act_row_div=k, mode=L.MODE_GEMV, ws=use_ws, dev_err=err)
        y32 = torch.empty((A, H), dtype=torch.float32, device=DEV)
        L.moe_w2_mm(L.STAGE_FC2, dev(h_bits.view(np.int16)), L.FMT_BF16, ml.c2k, ml.s2k, d_off, E, H, I, y32,
                    L.FMT_F32, mode=L.MODE_GEMV, ws=use_ws, dev_err=err)
        torch.cuda.synchronize()
        rms_h = np.sqrt(np.mean(want_h ** 2))
        assert np.max(np.abs(host(h32).astype(np.float64) - want_h)) <= 1e-4 * rms_h
        rms_y = np.sqrt(np.mean(want_y ** 2))
        assert np.max(np.abs(host(y32).astype(np.float64) - want_y)) <= 1e-4 * rms_y
    assert L.moe_get_error(err) == 0


def test_lut_small_workspace_flags_overflow():
    E, H, I, k, T = 6, 1024, 512, 3, 37
    w, ml, acc, x, off, perm = _setup(E, H, I, k, T, seed=3)
    A = T * k
    cap = A - 17
    d_off, d_perm, d_x = dev(off), dev(perm), dev(x.view(np.int16))
    full = _ws(A, I, H, H, I)
    ref = torch.empty((A, I), dtype=torch.int16, device=DEV)
    L.moe_w2_mm(L.STAGE_FC1_SWIGLU, d_x, L.FMT_BF16, ml.c1k, ml.s1k, d_off, E, I, H, ref, L.FMT_BF16,
                act_row=d_perm, act_row_div=k, mode=L.MODE_GEMV, ws=full)
    n = L.moe_w2_mm_workspace_size(L.STAGE_FC1_SWIGLU, cap, I, H)
    small = torch.full(((n + 3) // 4,), -1, dtype=torch.int32, device=DEV)
    got = torch.full((A, I), 0x7FC0, dtype=torch.int16, device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    L.moe_w2_mm(L.STAGE_FC1_SWIGLU, d_x, L.FMT_BF16, ml.c1k, ml.s1k, d_off, E, I, H, got, L.FMT_BF16,
                act_row=d_perm, act_row_div=k, mode=L.MODE_GEMV, ws=small, dev_err=err)
    assert L.moe_get_error(err) & L.DEVERR_OVERFLOW
    assert torch.equal(got[:cap], ref[:cap])
    assert bool((got[cap:] == 0x7FC0).all())


def test_lut_skips_delta_cached_experts():
    """expert_slot[e] >= 0: the 2-bit pass leaves those experts' rows alone."""
    E, H, I, k, T = 8, 512, 512, 2, 40
    w, ml, acc, x, off, perm = _setup(E, H, I, k, T, seed=4)
    A = T * k
    slot = np.full(E, -1, dtype=np.int32)
    slot[[1, 5]] = [0, 1]
    want_h, _, _ = _want(acc, x, off, perm, k, E, H, I)
    got = torch.full((A, I), float("nan"), dtype=torch.float32, device=DEV)
    L.moe_w2_mm(L.STAGE_FC1_SWIGLU, dev(x.view(np.int16)), L.FMT_BF16, ml.c1k, ml.s1k, dev(off), E, I, H, got,
                L.FMT_F32, act_row=dev(perm), act_row_div=k, expert_slot=dev(slot), mode=L.MODE_GEMV,
                ws=_ws(A, I, H, H, I))
    g = host(got).astype(np.float64)
    rms = np.sqrt(np.mean(want_h ** 2))
    for e in range(E):
        rows = slice(off[e], off[e + 1])
        if slot[e] >= 0:
            assert np.isnan(g[rows]).all()
        else:
            assert np.max(np.abs(g[rows] - want_h[rows]), initial=0.0) <= 1e-4 * rms
