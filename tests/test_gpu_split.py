"""moe_w2_mm with MOE_MODE_SPLIT, through the C ABI (GPU): groups of one row on
the table GEMV, groups of two rows or more on the tensor-core kernel, in one
call over disjoint experts.

Checks, on group sizes chosen to cover 0, 1, 2, a few and more than one
32-row token tile, with some experts delta-cached (skipped):
  * FC1 and FC2 with fp32 outputs against the exact (fp64) sums of the same
    bf16 operands, element by element;
  * every row equal, bit for bit, to the path its group was sent to (the
    whole call in GEMV mode for one-row groups, in GEMM mode for the rest);
  * rows of skipped experts untouched.
"""
import numpy as np
import pytest
import torch

from bit_moe_expert_top_gb300 import _lib as L
from bit_moe_expert_top_gb300 import synth
from oracle import codecs as C
from oracle import moe as M

from tests._gpu import DEV, dev, host, make_layer

pytestmark = pytest.mark.gpu

# fp32 accumulation over K products against the exact sum: a few ulp per
# sqrt(K) terms, far inside this bound at K <= 2048
STAGE_TOL = 1e-4

SIZES = [0, 1, 2, 1, 5, 0, 33, 1, 3, 70, 1, 2, 0, 1, 9, 1]   # 16 experts, 130 rows
CACHED = [3, 6, 14]                                          # delta-cache slots: skipped by the 2-bit pass


def _case(H, I, sizes, cached=CACHED):
    E = len(sizes)
    w = synth.get_workload("tiny").replace(E=E, H=H, I=I, k=1, T=int(sum(sizes)), logits="uniform")
    ml, acc, _ = make_layer(w, mode=L.MODE_GEMV)
    off = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32)
    slot = np.full(E, -1, np.int32)
    slot[cached] = np.arange(len(cached), dtype=np.int32)
    return w, ml, acc, off, slot


def _run(ml, stage, act_bits, off, slot, N, K, mode, fill):
    E = len(off) - 1
    A = int(off[-1])
    out = torch.full((A, N), fill, dtype=torch.float32, device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    codes, scales = (ml.c1k, ml.s1k) if stage == L.STAGE_FC1_SWIGLU else (ml.c2k, ml.s2k)
    ws = torch.empty(L.moe_w2_mm_workspace_size(stage, A, N, K), dtype=torch.uint8, device=DEV)
    L.moe_w2_mm(stage, dev(act_bits.view(np.int16)), L.FMT_BF16, codes, scales, dev(off), E, N, K, out, L.FMT_F32,
                expert_slot=dev(slot), mode=mode, ws=ws, dev_err=err)
    torch.cuda.synchronize()
    assert L.moe_get_error(err) == 0
    return host(out)


@pytest.mark.parametrize("H,I", [(1024, 512), (512, 2048)])
def test_split_mode_matches_exact_sums_and_its_paths(H, I):
    w, ml, acc, off, slot = _case(H, I, SIZES)
    E, A = len(SIZES), int(off[-1])
    x_bits = synth.make_x(w)                                  # A permuted rows (k = 1)
    xp = C.bf16_bits_to_f64(x_bits)
    sizes = np.diff(off)
    row_group = np.repeat(np.arange(E), sizes)
    skipped = np.isin(row_group, CACHED)
    single = (sizes[row_group] == 1) & ~skipped
    multi = (sizes[row_group] >= 2) & ~skipped
    assert single.any() and multi.any() and skipped.any()

    # FC1 (SwiGLU, fp32 out) against the exact sums
    h = _run(ml, L.STAGE_FC1_SWIGLU, x_bits, off, slot, I, H, L.MODE_SPLIT, np.nan)
    want_h = np.zeros((A, I))
    for e in range(E):
        rows = slice(off[e], off[e + 1])
        if e in CACHED or sizes[e] == 0:
            continue
        W1, _ = acc(e)
        want_h[rows] = M.silu(C.to_f32(xp[rows] @ W1[:I].T)) * C.to_f32(xp[rows] @ W1[I:].T)
    rms = np.sqrt(np.mean(want_h[~skipped] ** 2))
    assert np.max(np.abs(h[~skipped].astype(np.float64) - want_h[~skipped])) <= STAGE_TOL * rms
    assert np.all(np.isnan(h[skipped]))                       # cached experts' rows untouched

    # each row is the result of the path its group took, bit for bit
    h_gemv = _run(ml, L.STAGE_FC1_SWIGLU, x_bits, off, slot, I, H, L.MODE_GEMV, np.nan)
    h_gemm = _run(ml, L.STAGE_FC1_SWIGLU, x_bits, off, slot, I, H, L.MODE_GEMM, np.nan)
    assert np.array_equal(h[single].view(np.uint32), h_gemv[single].view(np.uint32))
    assert np.array_equal(h[multi].view(np.uint32), h_gemm[multi].view(np.uint32))

    # FC2 on the oracle's bf16 h
    h_bits = C.f32_to_bf16_bits(want_h.astype(np.float32))
    hv = C.bf16_bits_to_f64(h_bits)
    y = _run(ml, L.STAGE_FC2, h_bits, off, slot, H, I, L.MODE_SPLIT, np.nan)
    want_y = np.zeros((A, H))
    for e in range(E):
        if e in CACHED or sizes[e] == 0:
            continue
        rows = slice(off[e], off[e + 1])
        want_y[rows] = hv[rows] @ acc(e)[1].T
    rms = np.sqrt(np.mean(want_y[~skipped] ** 2))
    assert np.max(np.abs(y[~skipped].astype(np.float64) - want_y[~skipped])) <= STAGE_TOL * rms
    assert np.all(np.isnan(y[skipped]))
    y_gemv = _run(ml, L.STAGE_FC2, h_bits, off, slot, H, I, L.MODE_GEMV, np.nan)
    y_gemm = _run(ml, L.STAGE_FC2, h_bits, off, slot, H, I, L.MODE_GEMM, np.nan)
    assert np.array_equal(y[single].view(np.uint32), y_gemv[single].view(np.uint32))
    assert np.array_equal(y[multi].view(np.uint32), y_gemm[multi].view(np.uint32))


def test_split_mode_all_single_and_all_multi():
    """Only one-row groups (the tensor-core launch has no tile) and only larger
    groups (the table GEMV has no row): both halves cope with an empty share."""
    for sizes in ([1, 1, 0, 1, 1, 1, 1, 0], [2, 4, 0, 3, 40, 2, 2, 7]):
        w, ml, acc, off, _ = _case(512, 512, sizes, cached=[])
        slot = np.full(len(sizes), -1, np.int32)
        x_bits = synth.make_x(w)
        got = _run(ml, L.STAGE_FC1_SWIGLU, x_bits, off, slot, 512, 512, L.MODE_SPLIT, np.nan)
        ref = _run(ml, L.STAGE_FC1_SWIGLU, x_bits, off, slot, 512, 512,
                   L.MODE_GEMV if max(sizes) == 1 else L.MODE_GEMM, np.nan)
        assert np.array_equal(got.view(np.uint32), ref.view(np.uint32))


def test_split_mode_rejects_gathered_rows_and_mxfp4():
    w, ml, _, off, slot = _case(512, 512, [1, 2], cached=[])
    A = int(off[-1])
    x = dev(synth.make_x(w).view(np.int16))
    out = torch.empty((A, 512), dtype=torch.float32, device=DEV)
    perm = dev(np.arange(A, dtype=np.int32))
    with pytest.raises(RuntimeError):
        L.moe_w2_mm(L.STAGE_FC1_SWIGLU, x, L.FMT_BF16, ml.c1k, ml.s1k, dev(off), 2, 512, 512, out, L.FMT_F32,
                    act_row=perm, mode=L.MODE_SPLIT)
    q = torch.zeros((2, 1024, 256), dtype=torch.uint8, device=DEV)
    s = torch.full((2, 1024, 16), 127, dtype=torch.uint8, device=DEV)
    with pytest.raises(RuntimeError):
        L.moe_mxfp4_mm(L.STAGE_FC1_SWIGLU, x, L.FMT_BF16, dev(off), 2, 512, 512, out, L.FMT_F32, e2m1=q, e8m0=s,
                       mode=L.MODE_SPLIT)


def test_mixed_layer_with_split_matches_oracle():
    """The mixed layer (cache experts on the tensor core) with its 2-bit calls
    in SPLIT mode: layer output against the oracle at the bf16 gate."""
    from bit_moe_expert_top_gb300.layer import MoELayer
    from tests._gpu import TOL_BF16, rel_err, run_layer

    w = synth.get_workload("mixed_decode").replace(E=128, H=512, I=512, k=4, T=32, n_hot=16)
    raw = synth.make_w2_layer(w, 0, 0)
    mx = synth.make_mxfp4_layer(w, n=w.n_hot, seed=0, layer=0)
    slot = synth.hot_experts(w, 0)
    ml = MoELayer("mixed", w.E, w.H, w.I, w.k, w2=raw, mx=mx, expert_slot=slot, out_fmt=L.FMT_F32,
                  mode=L.MODE_AUTO, split=True)
    assert ml.mx_tensor_path() and ml.split
    x = synth.make_x(w)
    lg = synth.make_logits(w, x_bits=x)
    out, b = run_layer(ml, x, lg)
    assert L.moe_get_error(b.dev_err) == 0
    cnt = np.diff(host(b.offsets))
    assert np.any((cnt == 1) & (slot < 0)) and np.any((cnt >= 2) & (slot < 0))  # both halves of the split ran
    acc = M.mixed_expert_weights(M.w2_expert_weights(*raw), M.mxfp4_expert_weights(*mx), slot)
    ref = M.layer(x, lg, w.k, acc, profile="bf16")
    err, _ = rel_err(host(out), ref["out"])
    assert err <= TOL_BF16
