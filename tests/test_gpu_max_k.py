"""The expert matmuls at the largest K the C ABI accepts (8192), through the
C ABI (GPU): FC1 with H = 8192 and FC2 with I = 8192, every output element
against the exact sums of the same operands (fp32 outputs), for the
tensor-core kernel in its three weight formats and for the 2-bit table GEMV
(16 K slices per row); and whole layers on the block-scaled FP8 paths at
H = 8192 against the oracle's FP8 profile.
"""
import numpy as np
import pytest
import torch

from bit_moe_expert_top_gb300 import _lib as L
from bit_moe_expert_top_gb300 import synth
from oracle import codecs as C

from tests._gpu import DEV, dev, host
from tests.test_gpu_layer import _check_full
from tests.test_gpu_multitile import _compare, _exact_fc1, _h_input, _mm, _routing, _weights

pytestmark = pytest.mark.gpu

KMAX = 8192


def _shape(fmt, which):
    base = "tiny" if fmt == "w2" else "prefill_fp8"
    dims = dict(H=KMAX, I=256) if which == "fc1" else dict(H=256, I=KMAX)
    return synth.get_workload(base).replace(E=4, k=2, T=64, logits="uniform", **dims)


def _stage(w, acc, which, call):
    """Run one stage through `call(stage, act, off, N, K, out)` and compare
    every element with the exact sums."""
    x, off, perm = _routing(w)
    E, H, I, A = w.E, w.H, w.I, w.T * w.k
    if which == "fc1":
        xp = C.bf16_bits_to_f64(x)[perm // w.k]
        xp_bits = C.f32_to_bf16_bits(xp.astype(np.float32))
        out = torch.empty((A, I), dtype=torch.float32, device=DEV)
        call(L.STAGE_FC1_SWIGLU, dev(xp_bits.view(np.int16)), dev(off), I, H, out)
        want = np.zeros((A, I))
        for e in range(E):
            rows = slice(off[e], off[e + 1])
            want[rows] = _exact_fc1(xp[rows], acc(e)[0], I)
        _compare(host(out), want, H)
    else:
        hin = _h_input(w, A)
        hv = C.bf16_bits_to_f64(hin)
        out = torch.empty((A, H), dtype=torch.float32, device=DEV)
        call(L.STAGE_FC2, dev(hin.view(np.int16)), dev(off), H, I, out)
        want = np.zeros((A, H))
        for e in range(E):
            rows = slice(off[e], off[e + 1])
            want[rows] = hv[rows] @ acc(e)[1].T
        _compare(host(out), want, I)


@pytest.mark.parametrize("which", ["fc1", "fc2"])
@pytest.mark.parametrize("fmt", ["w2", "fp8", "mx4"])
def test_max_k_tensor_core_stages(fmt, which):
    w = _shape(fmt, which)
    d, acc = _weights(fmt, w)
    _stage(w, acc, which, lambda st, act, off, N, K, out: _mm(fmt, d, st, act, off, w.E, N, K, out))


@pytest.mark.parametrize("which", ["fc1", "fc2"])
def test_max_k_table_gemv_stages(which):
    w = _shape("w2", which)
    d, acc = _weights("w2", w)
    ml = d["ml"]
    A = w.T * w.k

    def call(stage, act, off, N, K, out):
        codes, scales = (ml.c1k, ml.s1k) if stage == L.STAGE_FC1_SWIGLU else (ml.c2k, ml.s2k)
        ws = torch.empty(L.moe_w2_mm_workspace_size(stage, A, N, K), dtype=torch.uint8, device=DEV)
        assert ws.numel() > 0                                  # the table GEMV takes this shape
        err = torch.zeros(1, dtype=torch.int32, device=DEV)
        L.moe_w2_mm(stage, act, L.FMT_BF16, codes, scales, off, w.E, N, K, out, L.FMT_F32, mode=L.MODE_GEMV,
                    ws=ws, dev_err=err)
        assert L.moe_get_error(err) == 0
    _stage(w, acc, which, call)


@pytest.mark.parametrize("direct", [True, False], ids=["MXFP4 direct", "FP8 workspace"])
def test_max_k_block_scaled_layers(direct):
    w = synth.get_workload("prefill_fp8").replace(E=4, H=KMAX, I=256, k=2, T=160, logits="uniform")
    _check_full(w, mode=L.MODE_GEMM, direct=direct)
