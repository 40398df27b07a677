"""Parity of the tcgen05 tensor-core expert matmuls (MODE_GEMM) against the
oracle, through the C ABI (GPU).

Two kinds of checks:
  * the whole layer at the problem's output gate (max|err| <= 2e-2 * RMS) on
    shapes with several 128-row tiles per group, partial tiles, BN = 128 and
    256 output blocks and K slices of 128 / 384 / 512;
  * FC1 and FC2 alone with fp32 outputs against the exact (fp64) sums of the
    same bf16 operands, element by element at 1e-4 * RMS: this checks the
    tensor-core arithmetic itself, free of the bf16 rounding flips that an
    accumulation-order difference can cause in h and y.
"""
import numpy as np
import pytest
import torch

from bit_moe_expert_top_gb300 import _lib as L
from bit_moe_expert_top_gb300 import synth
from oracle import codecs as C
from oracle import moe as M

from tests._gpu import DEV, dev, host, make_layer
from tests.test_gpu_layer import _check_full, _check_sampled

pytestmark = pytest.mark.gpu


def test_gemm_tiny_full_parity():
    # stricter than the method's bf16 gate: holds while no bf16 rounding of h
    # differs from the oracle's (the epilogue's SiLU refines its reciprocal)
    err = _check_full(synth.get_workload("tiny"), mode=L.MODE_GEMM)
    assert err < 1e-3


@pytest.mark.parametrize("E,H,I,k,T", [(16, 1024, 512, 4, 100), (4, 512, 256, 4, 301), (8, 256, 128, 8, 1),
                                       (3, 384, 640, 3, 77), (4, 512, 384, 4, 250)])
def test_gemm_tiles_and_ragged_tail(E, H, I, k, T):
    w = synth.get_workload("tiny").replace(E=E, H=H, I=I, k=k, T=T, logits="uniform")
    _check_full(w, mode=L.MODE_GEMM)


@pytest.mark.parametrize("E,H,I,k,T", [(4, 512, 384, 2, 400), (8, 1024, 512, 4, 260), (3, 384, 640, 3, 77)])
def test_gemm_stages_exact_sums(E, H, I, k, T):
    w = synth.get_workload("tiny").replace(E=E, H=H, I=I, k=k, T=T, logits="uniform")
    ml, acc, _ = make_layer(w, mode=L.MODE_GEMM)
    x = synth.make_x(w)
    logits = synth.make_logits(w, x_bits=x)
    ids, _, _ = M.route(logits, k)
    off, perm, inv = M.permute(ids, E)
    A = T * k
    xp = C.bf16_bits_to_f64(x)[perm // k]                       # permuted activation rows
    xp_bits = C.f32_to_bf16_bits(xp.astype(np.float32))
    d_off = dev(off)
    # FC1 with fp32 output: h_f32 = silu(g) * u, g/u exact sums rounded once to fp32
    h32 = torch.empty((A, I), dtype=torch.float32, device=DEV)
    L.moe_w2_mm(L.STAGE_FC1_SWIGLU, dev(xp_bits.view(np.int16)), L.FMT_BF16, ml.c1k, ml.s1k, d_off, E, I, H, h32,
                L.FMT_F32, mode=L.MODE_GEMM)
    want_h = np.zeros((A, I))
    for e in range(E):
        rows = slice(off[e], off[e + 1])
        W1, W2 = acc(e)
        g = C.to_f32(xp[rows] @ W1[:I].T)
        u = C.to_f32(xp[rows] @ W1[I:].T)
        want_h[rows] = M.silu(g) * u
    got_h = host(h32).astype(np.float64)
    rms_h = np.sqrt(np.mean(want_h ** 2))
    assert np.max(np.abs(got_h - want_h)) <= 1e-4 * rms_h
    # FC2 with fp32 output on bf16 h (the oracle's h)
    h_bits = C.f32_to_bf16_bits(want_h.astype(np.float32))
    hval = C.bf16_bits_to_f64(h_bits)
    y32 = torch.empty((A, H), dtype=torch.float32, device=DEV)
    L.moe_w2_mm(L.STAGE_FC2, dev(h_bits.view(np.int16)), L.FMT_BF16, ml.c2k, ml.s2k, d_off, E, H, I, y32,
                L.FMT_F32, mode=L.MODE_GEMM)
    want_y = np.zeros((A, H))
    for e in range(E):
        rows = slice(off[e], off[e + 1])
        want_y[rows] = hval[rows] @ acc(e)[1].T
    rms_y = np.sqrt(np.mean(want_y ** 2))
    assert np.max(np.abs(host(y32).astype(np.float64) - want_y)) <= 1e-4 * rms_y


@pytest.mark.parametrize("E,H,I,k,T", [(4, 512, 384, 2, 400), (8, 1024, 512, 4, 260)])
def test_gemm_fc1_bf16_h_rounding(E, H, I, k, T):
    """FC1 with bf16 output against h = silu(g) * u rounded once to bf16 from
    the exact (fp64) sums g, u (each rounded to fp32): every element equal, or
    one bf16 step away where the epilogue's fp32 SiLU (hardware exponential,
    refined reciprocal; a few ulp) lands on the other side of a rounding
    midpoint, plus the fp32 accumulation's absolute error (~1e-7 RMS, which is
    many bf16 steps of an h whose u nearly cancels); differences are rare."""
    w = synth.get_workload("tiny").replace(E=E, H=H, I=I, k=k, T=T, logits="uniform")
    ml, acc, _ = make_layer(w, mode=L.MODE_GEMM)
    x = synth.make_x(w)
    ids, _, _ = M.route(synth.make_logits(w, x_bits=x), k)
    off, perm, _ = M.permute(ids, E)
    A = T * k
    xp = C.bf16_bits_to_f64(x)[perm // k]
    xp_bits = C.f32_to_bf16_bits(xp.astype(np.float32))
    h = torch.empty((A, I), dtype=torch.int16, device=DEV)
    L.moe_w2_mm(L.STAGE_FC1_SWIGLU, dev(xp_bits.view(np.int16)), L.FMT_BF16, ml.c1k, ml.s1k, dev(off), E, I, H, h,
                L.FMT_BF16, mode=L.MODE_GEMM)
    want = np.zeros((A, I))
    for e in range(E):
        rows = slice(off[e], off[e + 1])
        W1, _ = acc(e)
        want[rows] = M.silu(C.to_f32(xp[rows] @ W1[:I].T)) * C.to_f32(xp[rows] @ W1[I:].T)
    want_bits = C.f32_to_bf16_bits(want.astype(np.float32))
    got_bits = host(h).view(np.uint16)
    wv, gv = C.bf16_bits_to_f64(want_bits), C.bf16_bits_to_f64(got_bits)
    rms_h = np.sqrt(np.mean(want ** 2))
    ulp = 2.0 ** (np.floor(np.log2(np.maximum(np.abs(wv), 1e-30))) - 7)   # bf16: 8 significant bits
    assert np.all(np.abs(gv - wv) <= ulp + 1e-5 * rms_h)
    assert np.mean(got_bits != want_bits) < 2e-3


def test_gemm_prefill_bf16_full_size_sampled():
    _check_sampled("prefill_bf16", [0, 4099, 8191], mode=L.MODE_GEMM)


@pytest.mark.parametrize("E,H,I,k,T", [(12, 512, 256, 4, 90), (8, 1024, 512, 8, 300), (5, 768, 384, 2, 77),
                                       (16, 512, 256, 2, 20)])  # the last: decode-sized groups, 32-token tiles
def test_fp8_workspace_gemm_full_parity(E, H, I, k, T):
    """FP8-workspace experts on the tensor-core path: MXFP8-rounded bf16
    activation rows, E4M3 weights decoded into TMEM, FC1 writes h
    MXFP8-rounded (the oracle's fp8 profile)."""
    w = synth.get_workload("prefill_fp8").replace(E=E, H=H, I=I, k=k, T=T)
    _check_full(w, mode=L.MODE_GEMM)


@pytest.mark.parametrize("E,H,I,k,T,n_hot", [(24, 512, 256, 4, 48, 6), (40, 1024, 512, 8, 200, 12)])
def test_mixed_delta_cache_tensor_path_full_parity(E, H, I, k, T, n_hot):
    """Mixed layer with the MXFP4 cache experts on the tensor-core path
    (E2M1 LUT decode into TMEM, 32-token tiles) and the 2-bit experts on
    the table GEMV."""
    w = synth.get_workload("mixed_decode").replace(E=E, H=H, I=I, k=k, T=T, n_hot=n_hot)
    _check_full(w, mode=L.MODE_AUTO)


def test_gemm_decode_sized_groups_full_parity():
    """Few tokens per expert: 32-token tiles, most of each tile past the group end."""
    w = synth.get_workload("tiny").replace(E=64, H=512, I=256, k=2, T=40, logits="uniform")
    _check_full(w, mode=L.MODE_GEMM)


def test_mxfp8_bf16_output_off_the_tensor_path_is_unsupported():
    """FC1's MXFP8_BF16 output exists only on the tensor-core path: asked of
    the GEMV it is refused as unsupported, not run and not a CUDA error."""
    w = synth.get_workload("tiny")
    ml, _, _ = make_layer(w, mode=L.MODE_GEMV)
    b = ml.buffers(w.T)
    x = dev(synth.make_x(w).view(np.int16))
    L.moe_route(dev(synth.make_logits(w)), w.k, b.ids, b.w, b.dev_err)
    L.moe_permute(b.ids, w.E, b.offsets, b.perm, b.inv, dev_err=b.dev_err)
    h = torch.empty((w.T * w.k, w.I), dtype=torch.int16, device=DEV)
    with pytest.raises(L.MoEError) as ei:
        L.moe_w2_mm(L.STAGE_FC1_SWIGLU, x, L.FMT_BF16, ml.c1k, ml.s1k, b.offsets, w.E, w.I, w.H, h,
                    L.FMT_MXFP8_BF16, act_row=b.perm, act_row_div=w.k, mode=L.MODE_GEMV, ws=b.ws,
                    dev_err=b.dev_err)
    assert ei.value.code == L.MOE_ERR_UNSUPPORTED
