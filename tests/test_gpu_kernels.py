"""Per-kernel parity against the oracle through the C ABI (GPU).

Bit-exact: routing ids, grouping (offsets/perm/inv), dequantised weights, the
FP8 workspace bytes and the MXFP8 activation codes.  Tolerances: routing
weights (TOL_W) and the combine (fp32 sums in the same order)."""
import numpy as np
import pytest
import torch

from bit_moe_expert_top_gb300 import _lib as L
from bit_moe_expert_top_gb300 import synth
from oracle import codecs as C
from oracle import moe as M

from tests._gpu import DEV, TOL_W, dev, host

pytestmark = pytest.mark.gpu


def test_library_version():
    assert L.moe_version() == 1


# ----------------------------------------------------------------- weights

def test_w2_repack_dequant_exhaustive():
    """Every byte value in every position, with normal, subnormal and rounding-tie scales."""
    rows, K = 64, 2048
    g = np.random.default_rng(5)
    codes = np.tile(np.arange(256, dtype=np.uint8), rows * K // 4 // 256).reshape(rows, K // 4)
    codes = np.roll(codes, 3, axis=1) ^ g.integers(0, 256, codes.shape, dtype=np.uint8)
    codes[:32] = np.tile(np.arange(256, dtype=np.uint8), 32 * K // 4 // 256).reshape(32, K // 4)
    scales = np.abs(g.standard_normal((rows, K // 32)).astype(np.float32) * 0.02).astype(np.float16)
    scales[0, :8] = np.array([6e-8, 1e-5, 1.0 + 2 ** -8, 0.0, 65504, 1e-7, 3.0, 1.0 + 3 * 2 ** -9], np.float16)
    ck = torch.empty((rows, K // 4), dtype=torch.uint8, device=DEV)
    sk = torch.empty((rows, K // 32), dtype=torch.int16, device=DEV)
    L.moe_w2_repack(dev(codes), dev(scales.view(np.int16)), 1, rows, K, ck, sk)
    out = torch.empty((rows, K), dtype=torch.int16, device=DEV)
    L.moe_dequant_w2(ck, sk, 1, rows, K, out)
    got = C.bf16_bits_to_f64(host(out).view(np.uint16))
    want = C.decode_w2(codes, scales)
    assert np.array_equal(got, want)


def test_mxfp4_dequant_exhaustive():
    rows, K = 32, 256
    nib = np.arange(256, dtype=np.uint8)
    q = np.tile(nib, rows * K // 2 // 256).reshape(rows, K // 2)
    s = (np.arange(rows * K // 32) % 256).astype(np.uint8).reshape(rows, K // 32)
    out = torch.empty((rows, K), dtype=torch.float32, device=DEV)
    L.moe_dequant_mxfp4(dev(q), dev(s), rows, K, out)
    got = host(out)
    want = C.decode_mxfp4(q, s).astype(np.float32)     # exact, or +-inf beyond fp32's range
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], want[~nan])
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(want[~nan]))


def test_mxfp4_to_fp8_ws_exhaustive_and_slots():
    """All 16 codes x all 256 scale bytes, converted into non-identity slots."""
    rows, K = 256, 128                      # 256 rows: scale byte = row
    nib = np.arange(16, dtype=np.uint8)
    row = np.tile(nib[0::2] | (nib[1::2] << 4), K // 16)      # 64 bytes
    q = np.stack([np.tile(row, (rows, 1)), np.tile(row[::-1], (rows, 1))])  # 2 source matrices
    s = np.stack([np.repeat(np.arange(256, dtype=np.uint8)[:, None], K // 32, 1)] * 2)
    ws = torch.full((4, rows, K), 0xAA, dtype=torch.uint8, device=DEV)
    experts = dev(np.array([1, 0], np.int32))
    slots = dev(np.array([3, 1], np.int32))
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    L.mxfp4_to_fp8_ws(dev(q), dev(s), experts, rows, K, ws, slots, dev_err=err)
    got = host(ws)
    assert np.array_equal(got[3], C.mxfp4_to_e4m3(q[1], s[1]))
    assert np.array_equal(got[1], C.mxfp4_to_e4m3(q[0], s[0]))
    assert (got[0] == 0xAA).all() and (got[2] == 0xAA).all()
    assert L.moe_get_error(err) & L.DEVERR_NAN_SCALE          # row 255 has the NaN scale


def test_fp8_ws_overflow_is_reported_not_written():
    rows, K = 32, 128
    q = np.zeros((1, rows, K // 2), np.uint8)
    s = np.full((1, rows, K // 32), 127, np.uint8)
    ws = torch.zeros((1, rows, K), dtype=torch.uint8, device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    L.mxfp4_to_fp8_ws(dev(q), dev(s), dev(np.array([0], np.int32)), rows, K, ws, dev(np.array([1], np.int32)),
                      dev_err=err)
    assert L.moe_get_error(err) & L.DEVERR_OVERFLOW


# ----------------------------------------------------------------- routing

@pytest.mark.parametrize("name", ["tiny", "decode", "mixed_decode", "prefill_fp8"])
def test_route_matches_oracle(name):
    w = synth.get_workload(name)
    T = min(w.T, 2048)
    logits = synth.make_logits(w, T=T)
    ids, wt, _ = M.route(logits, w.k)
    gi = torch.empty((T, w.k), dtype=torch.int32, device=DEV)
    gw = torch.empty((T, w.k), dtype=torch.float32, device=DEV)
    L.moe_route(dev(logits), w.k, gi, gw)
    assert np.array_equal(host(gi), ids)
    assert np.max(np.abs(host(gw) - wt)) <= TOL_W
    assert np.max(np.abs(host(gw).astype(np.float64).sum(1) - 1)) <= 1e-6


def test_route_ties_nan_and_k_equals_e():
    g = np.random.default_rng(2)
    T, E = 300, 24
    logits = (g.integers(0, 3, (T, E)) * 0.5).astype(np.float32)
    logits[7, :] = 0.0
    logits[9, 4] = np.nan
    logits[11, :] = np.nan
    for k in (1, 5, E):
        ids, wt, _ = M.route(logits, k)
        gi = torch.empty((T, k), dtype=torch.int32, device=DEV)
        gw = torch.empty((T, k), dtype=torch.float32, device=DEV)
        err = torch.zeros(1, dtype=torch.int32, device=DEV)
        L.moe_route(dev(logits), k, gi, gw, dev_err=err)
        assert np.array_equal(host(gi), ids)
        fin = np.isfinite(wt).all(1)
        assert np.max(np.abs(host(gw)[fin] - wt[fin])) <= TOL_W
        assert L.moe_get_error(err) & L.DEVERR_NAN_LOGIT


def test_route_zero_tokens_and_bad_args():
    gi = torch.empty((1, 2), dtype=torch.int32, device=DEV)
    gw = torch.empty((1, 2), dtype=torch.float32, device=DEV)
    L.moe_route(torch.empty((0, 8), dtype=torch.float32, device=DEV), 2, gi, gw)   # no-op
    with pytest.raises(L.MoEError) as ei:
        L.moe_route(torch.zeros((4, 8), dtype=torch.float32, device=DEV), 9, gi, gw)
    assert ei.value.code == L.MOE_ERR_ARG


# ----------------------------------------------------------------- grouping

@pytest.mark.parametrize("E,T,k", [(8, 16, 2), (384, 8, 8), (384, 64, 8), (384, 8192, 8), (256, 16384, 8),
                                   (5, 1, 5), (1024, 3, 32), (7, 1000, 1), (1024, 9000, 4), (3, 4099, 2)])
def test_permute_matches_oracle(E, T, k):
    g = np.random.default_rng(E * 7 + T)
    logits = g.random((T, E)).astype(np.float32)
    logits[:, 1] += 2.0                               # one hot expert, many empty ones
    ids, _, _ = M.route(logits, k)
    off, perm, inv = M.permute(ids, E)
    A = T * k
    nws = L.moe_permute_workspace_size(T, k, E)
    assert (nws > 0) == (A >= 8192)                   # large groupings run on many CTAs
    for use_ws in ([False, True] if nws else [False]):
        go = torch.full((E + 1,), -7, dtype=torch.int32, device=DEV)
        gp = torch.full((A,), -7, dtype=torch.int32, device=DEV)
        gv = torch.full((A,), -7, dtype=torch.int32, device=DEV)
        ws = torch.full(((nws + 3) // 4,), -7, dtype=torch.int32, device=DEV) if use_ws else None
        L.moe_permute(dev(ids), E, go, gp, gv, ws=ws, ws_bytes=nws if use_ws else 0)
        assert np.array_equal(host(go), off)
        assert np.array_equal(host(gp), perm)
        assert np.array_equal(host(gv), inv)


def test_permute_bad_ids_flagged():
    ids = np.array([[0, 1], [2, 9], [-1, 3]], np.int32)
    go = torch.empty(5, dtype=torch.int32, device=DEV)
    gp = torch.full((6,), -7, dtype=torch.int32, device=DEV)
    gv = torch.empty(6, dtype=torch.int32, device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    L.moe_permute(dev(ids), 4, go, gp, gv, dev_err=err)
    assert L.moe_get_error(err) & L.DEVERR_BAD_ID
    o = host(go)
    assert o[-1] == 4 and list(np.diff(o)) == [1, 1, 1, 1]
    v = host(gv)
    assert v[3] == -1 and v[4] == -1
    assert sorted(host(gp)[:4].tolist()) == [0, 1, 2, 5]


def test_permute_gather_bf16_and_unpermute_identity():
    w = synth.get_workload("tiny").replace(T=37, E=6, k=3, H=384)
    x = synth.make_x(w)
    ids, _, _ = M.route(synth.make_logits(w.replace(logits="uniform")), w.k)
    A = w.A
    go = torch.empty(w.E + 1, dtype=torch.int32, device=DEV)
    gp = torch.empty(A, dtype=torch.int32, device=DEV)
    gv = torch.empty(A, dtype=torch.int32, device=DEV)
    xp = torch.empty((A, w.H), dtype=torch.int16, device=DEV)
    L.moe_permute(dev(ids), w.E, go, gp, gv, x=dev(x.view(np.int16)), act_fmt=L.FMT_BF16, x_perm=xp)
    _, perm, _ = M.permute(ids, w.E)
    assert np.array_equal(host(xp).view(np.uint16), M.gather_rows(x, perm, w.k))
    back = torch.empty((A, w.H), dtype=torch.int16, device=DEV)
    L.moe_unpermute(xp, L.FMT_BF16, gv, back)
    assert np.array_equal(host(back).view(np.uint16), np.repeat(x, w.k, axis=0))


def test_permute_gather_mxfp8_matches_oracle():
    w = synth.get_workload("prefill_fp8").replace(T=40, E=16)
    x = synth.make_x(w)
    x[3, :64] = 0                                   # an all-zero block
    x[5, 32:64] = 0x0001                            # subnormal bf16 block
    x[6, 5] = 0x7F00                                # huge value in a block
    ids, _, _ = M.route(synth.make_logits(w), w.k)
    A = w.A
    go = torch.empty(w.E + 1, dtype=torch.int32, device=DEV)
    gp = torch.empty(A, dtype=torch.int32, device=DEV)
    gv = torch.empty(A, dtype=torch.int32, device=DEV)
    q = torch.empty((A, w.H), dtype=torch.uint8, device=DEV)
    sc = torch.empty((A, w.H // 32), dtype=torch.uint8, device=DEV)
    L.moe_permute(dev(ids), w.E, go, gp, gv, x=dev(x.view(np.int16)), act_fmt=L.FMT_MXFP8, x_perm=q,
                  x_perm_scale=sc)
    _, perm, _ = M.permute(ids, w.E)
    xq, xs = C.mxfp8_quantize(C.bf16_bits_to_f64(x))
    assert np.array_equal(host(q), xq[perm // w.k])
    assert np.array_equal(host(sc), xs[perm // w.k])


# ----------------------------------------------------------------- combine

@pytest.mark.parametrize("yfmt", [L.FMT_BF16, L.FMT_F32])
def test_combine_matches_oracle(yfmt):
    g = np.random.default_rng(9)
    T, k, H, E = 50, 4, 512, 12
    ids, wt, _ = M.route(g.random((T, E)).astype(np.float32), k)
    off, perm, inv = M.permute(ids, E)
    yv = g.standard_normal((T * k, H)).astype(np.float32)
    if yfmt == L.FMT_BF16:
        ybits = C.f32_to_bf16_bits(yv)
        yd = dev(ybits.view(np.int16))
        yval = C.bf16_bits_to_f64(ybits)
    else:
        yd = dev(yv)
        yval = yv.astype(np.float64)
    out = torch.empty((T, H), dtype=torch.float32, device=DEV)
    L.moe_combine(yd, yfmt, dev(wt), dev(inv), T, k, H, out, L.FMT_F32)
    want = M.combine(M.unpermute(yval, inv).reshape(T, k, H), wt)
    rms = np.sqrt(np.mean(want ** 2))
    assert np.max(np.abs(host(out) - want)) <= 1e-6 * rms
    outb = torch.empty((T, H), dtype=torch.int16, device=DEV)
    L.moe_combine(yd, yfmt, dev(wt), dev(inv), T, k, H, outb, L.FMT_BF16)
    ob = C.bf16_bits_to_f64(host(outb).view(np.uint16))
    assert np.max(np.abs(ob - C.rne_bf16(want))) <= 2 ** -7 * np.max(np.abs(want))


# ----------------------------------------------------------------- error paths

def test_bounded_wait_expires_and_reports_timeout():
    """A wait that nothing ends gives up after its limit, reports
    MOE_DEVERR_TIMEOUT and returns; the context stays usable (a routing call
    afterwards is still exact)."""
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    L.moe_check_bounded_wait(2_000_000, err)          # ~1 ms of SM clocks
    assert L.moe_get_error(err) == L.DEVERR_TIMEOUT
    w = synth.get_workload("tiny")
    lg = synth.make_logits(w)
    ids = torch.empty((w.T, w.k), dtype=torch.int32, device=DEV)
    wt = torch.empty((w.T, w.k), dtype=torch.float32, device=DEV)
    err2 = torch.zeros(1, dtype=torch.int32, device=DEV)
    L.moe_route(dev(lg), w.k, ids, wt, err2)
    assert L.moe_get_error(err2) == 0
    assert np.array_equal(host(ids), M.route(lg, w.k)[0])


def test_wait_limit_setting_round_trips():
    """moe_set_wait_limit returns the previous limit; <= 0 restores the default."""
    prev = L.moe_set_wait_limit(12345)
    try:
        assert L.moe_set_wait_limit(0) == 12345
        assert L.moe_set_wait_limit(0) == 3_000_000_000
    finally:
        L.moe_set_wait_limit(prev)


def test_bounded_wait_check_rejects_bad_limits():
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    for cyc in (0, -5, 3_000_000_001):
        with pytest.raises(L.MoEError) as ei:
            L.moe_check_bounded_wait(cyc, err)
        assert ei.value.code == L.MOE_ERR_ARG
