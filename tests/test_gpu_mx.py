"""The block-scaled FP8 tensor-core expert matmul (kind::mxf8f6f4) against the
oracle, through the C ABI (GPU).

MXFP8 activation rows (E4M3 codes + one E8M0 per 32) times either the FP8
workspace (E4M3 weights, scale folded in) or MXFP4 weights read directly
(E2M1 codes + E8M0 scales).  Stage checks compare every output element with
exact sums of the same operands (fp32 outputs) on launches where every CTA
takes several tiles (128- and 32-token tiles); FC1's MXFP8 output is
compared with the OCP MX rounding of h from exact sums; whole layers are
held to the FP8 profile's gate, at small sizes on every element and at the
full prefill_fp8 size on sampled tokens and on every row of the three
largest expert groups."""
import numpy as np
import pytest
import torch

from bit_moe_expert_top_gb300 import _lib as L
from bit_moe_expert_top_gb300 import synth
from oracle import codecs as C
from oracle import moe as M

from tests._gpu import DEV, dev, host, make_layer, run_layer
from tests.test_gpu_layer import _check_full, _check_sampled
from tests.test_gpu_multitile import MULTI, _compare, _exact_fc1, _nt, _sms, _tiles, _weights

pytestmark = pytest.mark.gpu


def _mxfp8_rows(w, A, K, seed, tid):
    """Seeded MXFP8 activation rows [A, K]: E4M3 codes uniform over the finite
    codes, E8M0 scales uniform in [120, 130] (an input recipe)."""
    g = synth.rng_for(seed, w.wid, 9000 + tid)
    q = g.integers(0, 256, size=(A, K), dtype=np.uint8)
    q[(q & 0x7F) == 0x7F] = 0x38          # no NaN code
    s = g.integers(120, 131, size=(A, K // 32), dtype=np.uint8)
    return q, s


def _mx_values(q, s):
    return C.e4m3_value(q) * np.repeat(C.e8m0_value(s), 32, axis=1)


def _mm(fmt, d, stage, act, act_scale, off, E, N, K, out, out_fmt=L.FMT_F32, out_scale=None, ebeg=0, eend=None):
    i = "1" if stage == L.STAGE_FC1_SWIGLU else "2"
    if fmt == "mx4":
        L.moe_mxfp4_mm(stage, act, L.FMT_MXFP8, off, E, N, K, out, out_fmt, e2m1=d["q" + i], e8m0=d["e" + i],
                       act_scale=act_scale, out_scale=out_scale, mode=L.MODE_GEMM)
    else:
        L.moe_mxfp4_mm(stage, act, L.FMT_MXFP8, off, E, N, K, out, out_fmt, fp8_ws=d["ws" + i],
                       ws_slot_of_expert=d["slot"], act_scale=act_scale, out_scale=out_scale,
                       expert_begin=ebeg, expert_end=E if eend is None else eend, mode=L.MODE_GEMM)


@pytest.mark.parametrize("fmt", ["fp8", "mx4"])
@pytest.mark.parametrize("shape", ["t128", "t32"])
def test_mx_stages_every_element(fmt, shape):
    w = synth.get_workload("prefill_fp8").replace(logits="uniform", **MULTI[shape])
    E, H, I, k = w.E, w.H, w.I, w.k
    A = w.T * k
    x = synth.make_x(w)
    ids, _, _ = M.route(synth.make_logits(w, x_bits=x), k)
    off, _, _ = M.permute(ids, E)
    nt = _nt(A, E)
    assert _tiles(off, nt, I // 128) >= 3 * _sms()      # every CTA takes several FC1 tiles
    d, acc = _weights(fmt, w)
    xq, xs = _mxfp8_rows(w, A, H, 0, 1)
    hq, hs = _mxfp8_rows(w, A, I, 0, 2)
    d_off = dev(off)
    h32 = torch.full((A, I), float("nan"), dtype=torch.float32, device=DEV)
    _mm(fmt, d, L.STAGE_FC1_SWIGLU, dev(xq), dev(xs), d_off, E, I, H, h32)
    y32 = torch.full((A, H), float("nan"), dtype=torch.float32, device=DEV)
    _mm(fmt, d, L.STAGE_FC2, dev(hq), dev(hs), d_off, E, H, I, y32)
    torch.cuda.synchronize()
    xv, hv = _mx_values(xq, xs), _mx_values(hq, hs)
    want_h = np.zeros((A, I))
    want_y = np.zeros((A, H))
    for e in range(E):
        rows = slice(off[e], off[e + 1])
        if off[e] == off[e + 1]:
            continue
        W1, W2 = acc(e)
        want_h[rows] = _exact_fc1(xv[rows], W1, I)
        want_y[rows] = hv[rows] @ W2.T
    _compare(host(h32), want_h, H)
    _compare(host(y32), want_y, I)


@pytest.mark.parametrize("fmt", ["fp8", "mx4"])
def test_mx_fc1_mxfp8_output(fmt):
    """FC1 with MXFP8 output (the FP8 path's h): per token and block of 32
    outputs, the E8M0 scale and the E4M3 codes of the OCP MX rounding of
    h = silu(g) * u (exact sums).  Identical but where the kernel's fp32 h
    (another summation order, hardware exponential) sits on the other side of
    a rounding point: then the decoded value is one E4M3 step away (or the
    block scale one binade away); such cases are rare."""
    w = synth.get_workload("prefill_fp8").replace(logits="uniform", **MULTI["t128"])
    E, H, I, k = w.E, w.H, w.I, w.k
    A = w.T * k
    x = synth.make_x(w)
    ids, _, _ = M.route(synth.make_logits(w, x_bits=x), k)
    off, _, _ = M.permute(ids, E)
    d, acc = _weights(fmt, w)
    xq, xs = _mxfp8_rows(w, A, H, 0, 3)
    hq = torch.empty((A, I), dtype=torch.uint8, device=DEV)
    hs = torch.empty((A, I // 32), dtype=torch.uint8, device=DEV)
    _mm(fmt, d, L.STAGE_FC1_SWIGLU, dev(xq), dev(xs), dev(off), E, I, H, hq, L.FMT_MXFP8, out_scale=hs)
    torch.cuda.synchronize()
    xv = _mx_values(xq, xs)
    want = np.zeros((A, I))
    for e in range(E):
        rows = slice(off[e], off[e + 1])
        if off[e] != off[e + 1]:
            want[rows] = _exact_fc1(xv[rows], acc(e)[0], I)
    wq, ws = C.mxfp8_quantize(C.to_f32(want))
    gq, gs = host(hq), host(hs)
    assert np.mean(gs != ws) < 1e-3
    assert np.mean(gq != wq) < 5e-3
    got_v = C.mxfp8_dequantize(gq, gs)
    want_v = C.mxfp8_dequantize(wq, ws)
    blk_amax = np.repeat(np.abs(want).reshape(A, I // 32, 32).max(axis=2), 32, axis=1)
    # one E4M3 step (3 mantissa bits) of the block's largest value, at most
    assert np.all(np.abs(got_v - want_v) <= 2.0 ** -3 * blk_amax + 1e-30)


@pytest.mark.parametrize("E,H,I,k,T", [(12, 512, 256, 4, 90), (8, 1024, 512, 8, 300), (16, 512, 256, 2, 20)])
@pytest.mark.parametrize("direct", [False, True])
def test_fp8_layers_on_the_block_scaled_tensor_core(E, H, I, k, T, direct):
    """Whole FP8-profile layers (MXFP8 gather, FC1 with MXFP8 h, FC2, combine)
    on the block-scaled tensor core: the FP8 workspace path and the direct
    MXFP4 path, every output element at the FP8 gate."""
    w = synth.get_workload("prefill_fp8").replace(E=E, H=H, I=I, k=k, T=T)
    _check_full(w, mode=L.MODE_GEMM, direct=direct)


def test_direct_mxfp4_layer_nan_scale_flagged():
    w = synth.get_workload("prefill_fp8").replace(E=4, H=256, I=128, k=2, T=8, e8m0_lo=255, e8m0_hi=255)
    from tests._gpu import make_layer, run_layer
    ml, _, _ = make_layer(w, direct=True)
    x = synth.make_x(w)
    _, b = run_layer(ml, x, synth.make_logits(w, x_bits=x))
    assert L.moe_get_error(b.dev_err) & L.DEVERR_NAN_SCALE


@pytest.mark.parametrize("direct", [False, True])
def test_prefill_fp8_full_size_sampled_tensor_core(direct):
    _check_sampled("prefill_fp8", [7, 9000, 16383], mode=L.MODE_GEMM, direct=direct)


@pytest.mark.parametrize("fmt", ["fp8", "mx4"])
def test_prefill_fp8_full_size_largest_groups_every_row(fmt):
    """prefill_fp8's full size in the layer's launch configuration (FP8
    workspace: expert batches of 16; direct: one launch over all experts):
    FC1 and FC2 (fp32 outputs) on every row of the three largest groups
    against exact sums, on seeded MXFP8 rows."""
    w = synth.get_workload("prefill_fp8")
    E, H, I, k = w.E, w.H, w.I, w.k
    A = w.T * k
    x = synth.make_x(w)
    ids, _, _ = M.route(synth.make_logits(w, x_bits=x), k)
    off, _, _ = M.permute(ids, E)
    cnt = np.diff(off)
    big = [int(e) for e in np.argsort(-cnt, kind="stable")[:3]]
    d, acc = _weights(fmt, w)
    xq, xs = _mxfp8_rows(w, A, H, 0, 4)
    hq, hs = _mxfp8_rows(w, A, I, 0, 5)
    d_off = dev(off)
    h32 = torch.empty((A, I), dtype=torch.float32, device=DEV)
    y32 = torch.empty((A, H), dtype=torch.float32, device=DEV)
    dxq, dxs, dhq, dhs = dev(xq), dev(xs), dev(hq), dev(hs)
    ranges = [(b0, min(E, b0 + 16)) for b0 in range(0, E, 16)] if fmt == "fp8" else [(0, E)]
    for b0, b1 in ranges:
        _mm(fmt, d, L.STAGE_FC1_SWIGLU, dxq, dxs, d_off, E, I, H, h32, ebeg=b0, eend=b1)
        _mm(fmt, d, L.STAGE_FC2, dhq, dhs, d_off, E, H, I, y32, ebeg=b0, eend=b1)
    torch.cuda.synchronize()
    got_h, got_y = host(h32), host(y32)
    for e in big:
        rows = np.arange(off[e], off[e + 1])
        assert rows.size > 300
        W1, W2 = acc(e)
        _compare(got_h[rows], _exact_fc1(_mx_values(xq[rows], xs[rows]), W1, I), H)
        _compare(got_y[rows], _mx_values(hq[rows], hs[rows]) @ W2.T, I)


def test_conversion_on_reserved_sms_is_bit_identical():
    """mxfp4_to_fp8_ws with SMs reserved (moe_set_side_sms): the same
    bytes as the whole-GPU conversion, flags included; the setting is
    restored afterwards."""
    g = np.random.default_rng(5)
    n_exp, rows, K = 6, 256, 512
    q = g.integers(0, 256, size=(n_exp, rows, K // 2), dtype=np.uint8)
    s = g.integers(110, 135, size=(n_exp, rows, K // 32), dtype=np.uint8)
    s[3, 7, 2] = 255                                              # one NaN scale
    experts = np.array([5, 0, 3, 2], dtype=np.int32)
    slots = np.array([1, 3, 0, 2], dtype=np.int32)
    outs = []
    for n in (0, 7):
        prev = L.moe_set_side_sms(n)
        try:
            ws = torch.full((4, rows, K), 0xAB, dtype=torch.uint8, device=DEV)
            err = torch.zeros(1, dtype=torch.int32, device=DEV)
            L.mxfp4_to_fp8_ws(dev(q), dev(s), dev(experts), rows, K, ws, dev(slots), dev_err=err)
            outs.append((host(ws), L.moe_get_error(err)))
        finally:
            L.moe_set_side_sms(prev)
    assert np.array_equal(outs[0][0], outs[1][0])
    assert outs[0][1] == outs[1][1] and outs[0][1] & L.DEVERR_NAN_SCALE
    assert L.moe_set_side_sms(0) == 0


def test_fp8_layer_with_reserved_conversion_sms_is_bit_identical():
    """The FP8-workspace layer with SMs reserved for the side-stream
    conversion (smaller matmul grid, conversion beside it): output, h and y
    bit-identical to the layer without the reservation."""
    w = synth.get_workload("prefill_fp8").replace(E=48, H=1024, I=512, T=700, k=4)
    ml, _, _ = make_layer(w, out_fmt=L.FMT_BF16, mode=L.MODE_GEMM)
    x = synth.make_x(w)
    lg = synth.make_logits(w, x_bits=x)
    outs = []
    for conv in (0, 20):
        ml.side_sms = conv
        out, b = run_layer(ml, x, lg)
        assert L.moe_get_error(b.dev_err) == 0
        outs.append((out.clone(), b.h.clone(), b.y.clone()))
    for a, c in zip(outs[0], outs[1]):
        assert torch.equal(a, c)
    assert L.moe_set_side_sms(0) == 0                     # the layer restored the setting
