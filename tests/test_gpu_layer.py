"""Whole-layer parity against the oracle through the C ABI (GPU).

Small shapes are compared on every output element (and on the per-assignment
FC2 rows); the full-size workloads on sampled tokens that the oracle computes
one by one, plus properties that hold at any size."""
import numpy as np
import pytest
import torch

from bit_moe_expert_top_gb300 import _lib as L
from bit_moe_expert_top_gb300 import synth
from oracle import codecs as C
from oracle import moe as M

from tests._gpu import TOL_BF16, TOL_FP8, bf16_to_f64, dev, host, make_layer, rel_err, run_layer

pytestmark = pytest.mark.gpu


def _check_full(w, seed=0, mode=L.MODE_GEMV, direct=False):
    ml, acc, prof = make_layer(w, seed, mode=mode, direct=direct)
    x = synth.make_x(w, seed)
    logits = synth.make_logits(w, seed, x_bits=x)
    out, b = run_layer(ml, x, logits)
    ref = M.layer(x, logits, w.k, acc, profile=prof)
    assert np.array_equal(host(b.ids), ref["ids"])
    err, rms = rel_err(host(out), ref["out"])
    assert rms > 0
    assert err <= (TOL_FP8 if prof == "fp8" else TOL_BF16), err
    # per-assignment FC2 rows (bf16): identical but where an fp32 accumulation-
    # order difference flips a bf16 rounding of h or y (rare; each flip moves y
    # by about one bf16 ulp of h times a W2 row)
    y = bf16_to_f64(b.y)[host(b.inv)].reshape(w.T, w.k, w.H)
    diff = np.abs(y - ref["y"])
    # tensor-core accumulation rounds differently from an fp32 FMA chain: more flips
    tensor = mode == L.MODE_GEMM or (w.weights == "mixed" and mode == L.MODE_AUTO)
    assert np.mean(diff > 0) < (0.05 if prof == "fp8" else (3e-2 if tensor else 2e-3))
    rms_y = np.sqrt(np.mean(ref["y"] ** 2))
    if prof == "fp8":
        assert np.max(diff) <= TOL_FP8 * rms_y
    else:   # one bf16 ulp of the element itself, plus a flipped h's share
        assert np.all(diff <= 2.0 ** -7 * np.abs(ref["y"]) + 1e-2 * rms_y)
    return err


def test_tiny_layer_full_parity():
    err = _check_full(synth.get_workload("tiny"))
    assert err < 1e-4


@pytest.mark.parametrize("E,H,I,k,T", [(16, 1024, 512, 4, 100), (4, 512, 256, 2, 301), (8, 256, 128, 8, 1),
                                       (3, 384, 640, 3, 77)])
def test_w2_layer_tiles_and_ragged_tail(E, H, I, k, T):
    w = synth.get_workload("tiny").replace(E=E, H=H, I=I, k=k, T=T, logits="uniform")
    _check_full(w)


def test_mixed_layer_small_full_parity():
    w = synth.get_workload("mixed_decode").replace(E=24, H=512, I=256, k=4, T=48, n_hot=6)
    _check_full(w)


def test_fp8_layer_small_full_parity():
    w = synth.get_workload("prefill_fp8").replace(E=12, H=512, I=256, k=4, T=90)
    _check_full(w)


def test_fp8_layer_nan_scale_flagged():
    w = synth.get_workload("prefill_fp8").replace(E=4, H=256, I=128, k=2, T=8, e8m0_lo=255, e8m0_hi=255)
    ml, acc, prof = make_layer(w)
    x = synth.make_x(w)
    out, b = run_layer(ml, x, synth.make_logits(w, x_bits=x))
    assert L.moe_get_error(b.dev_err) & L.DEVERR_NAN_SCALE


def _check_sampled(name, tokens, seed=0, mode=L.MODE_GEMV, direct=False):
    w = synth.get_workload(name)
    ml, acc, prof = make_layer(w, seed, mode=mode, direct=direct)
    x = synth.make_x(w, seed)
    logits = synth.make_logits(w, seed, x_bits=x)
    out, b = run_layer(ml, x, logits)
    o = host(out)
    assert np.isfinite(o).all()
    assert L.moe_get_error(b.dev_err) == 0
    ids, wt, _ = M.route(logits, w.k)
    assert np.array_equal(host(b.ids), ids)
    off, perm, inv = M.permute(ids, w.E)
    assert np.array_equal(host(b.offsets), off) and np.array_equal(host(b.perm), perm)
    ref = M.layer(x, logits, w.k, acc, profile=prof, tokens=tokens)
    err, rms = rel_err(o[ref["tokens"]], ref["out"])
    assert err <= (TOL_FP8 if prof == "fp8" else TOL_BF16), err
    # deterministic: a second run gives identical bits
    out2, _ = run_layer(ml, x, logits)
    assert torch.equal(out, out2)
    return err


def test_decode_full_size_sampled():
    _check_sampled("decode", [0, 3, 7])


def test_mixed_decode_full_size_sampled():
    _check_sampled("mixed_decode", [0, 41])


def test_mixed_decode_full_size_sampled_tensor_path():
    """The default (AUTO) mixed layer: cache experts on the tensor cores."""
    _check_sampled("mixed_decode", [3, 60], mode=L.MODE_AUTO)


@pytest.mark.parametrize("name,mode", [("mixed_decode", L.MODE_AUTO), ("prefill_fp8", L.MODE_GEMM),
                                       ("decode", L.MODE_GEMV)])
def test_layer_repeat_bit_identical(name, mode):
    """Several steps on the same inputs give the same bits (the table GEMV
    adds its slice sums in slice order; the tensor-core matmul's TMA weight
    rings (MXFP4 nibbles, E4M3 bytes, 2-bit codes) hand a slot back to the
    producer only after its words are consumed).  Releasing it right after the
    shared-memory reads were issued let the next TMA overwrite the slot first
    on some steps (seen as 3-10 differing rows of h on the mixed layer)."""
    w = synth.get_workload(name)
    if name == "prefill_fp8":  # two expert batches through the E4M3 workspace ring, 128-token tiles
        w = w.replace(E=32, H=1024, I=512, T=512)
    ml, _, _ = make_layer(w, 0, mode=mode)
    x = dev(synth.make_x(w, 0).view(np.int16))
    lg = dev(synth.make_logits(w, 0))
    b = ml.buffers(w.T)
    first = ml.step(x, lg, b).clone()
    for _ in range(5):
        assert torch.equal(ml.step(x, lg, b), first)
    assert L.moe_get_error(b.dev_err) == 0


def test_prefill_bf16_full_size_sampled():
    _check_sampled("prefill_bf16", [0, 4099, 8191])


def test_prefill_fp8_full_size_sampled():
    _check_sampled("prefill_fp8", [5, 16383])


@pytest.mark.parametrize("name,mode", [("decode", L.MODE_GEMV), ("tiny", L.MODE_GEMM)])
def test_captured_layer_graph_matches_the_eager_step(name, mode):
    """MoELayer.capture: the whole step replayed from one CUDA graph gives the
    eager step's bits, for a second batch copied into the graph's inputs
    too, and matches the oracle."""
    w = synth.get_workload(name)
    ml, acc, prof = make_layer(w, 0, mode=mode)
    g = ml.capture(w.T)
    for bi in range(2):
        x = synth.make_x(w, 0, tid_offset=bi)
        lg = synth.make_logits(w, 0, x_bits=x, tid_offset=bi)
        xd, ld = dev(x.view(np.int16)), dev(lg)
        out_g = g.run(xd, ld).clone()
        b = ml.buffers(w.T)
        out_e = ml.step(xd, ld, b)
        torch.cuda.synchronize()
        assert torch.equal(out_g, out_e)
        tok = [0, w.T - 1]
        ref = M.layer(x, lg, w.k, acc, profile=prof, tokens=tok)
        err, _ = rel_err(host(out_g)[tok], ref["out"])
        assert err <= TOL_BF16
