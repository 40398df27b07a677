"""Degenerate shapes of the whole layer on every weight path, through the C
ABI (GPU), against the oracle at the problem's output gates:

  * one expert (E = 1, k = 1): every token in one group, the layer reduces
    to a dense SwiGLU MLP;
  * every expert routed by every token (k = E): E groups of T rows, the
    combine sums k outputs per token;
  * an empty batch (T = 0): the step runs, flags nothing, returns no rows.
"""
import numpy as np
import pytest
import torch

from bit_moe_expert_top_gb300 import _lib as L
from bit_moe_expert_top_gb300 import synth
from oracle import moe as M

from tests._gpu import TOL_BF16, TOL_FP8, host, make_layer, rel_err, run_layer

pytestmark = pytest.mark.gpu

# (label, workload, make_layer mode, direct MXFP4)
PATHS = [
    ("w2 table GEMV (fused decode)", "tiny", L.MODE_GEMV, False),
    ("w2 tensor core", "tiny", L.MODE_GEMM, False),
    ("mixed, cache on the tensor core", "mixed_decode", L.MODE_AUTO, False),
    ("MXFP4 block-scaled", "prefill_fp8", L.MODE_GEMM, True),
    ("FP8 workspace", "prefill_fp8", L.MODE_GEMM, False),
]


def _workload(base, E, k, T):
    w = synth.get_workload(base).replace(E=E, H=512, I=512, k=k, T=T, logits="uniform")
    if w.weights == "mixed":
        w = w.replace(n_hot=max(1, E // 2))
    return w


def _run_against_oracle(w, mode, direct):
    ml, acc, prof = make_layer(w, mode=mode, direct=direct)
    x = synth.make_x(w)
    lg = synth.make_logits(w, x_bits=x)
    out, b = run_layer(ml, x, lg)
    assert L.moe_get_error(b.dev_err) == 0
    ref = M.layer(x, lg, w.k, acc, profile=prof)
    assert np.array_equal(host(b.ids), ref["ids"])
    err, rms = rel_err(host(out).astype(np.float64), ref["out"])
    assert rms > 0
    assert err <= (TOL_FP8 if prof == "fp8" else TOL_BF16), err


@pytest.mark.parametrize("label,base,mode,direct", PATHS, ids=[p[0] for p in PATHS])
def test_single_expert_layer(label, base, mode, direct):
    _run_against_oracle(_workload(base, E=1, k=1, T=40), mode, direct)


@pytest.mark.parametrize("label,base,mode,direct", PATHS, ids=[p[0] for p in PATHS])
def test_every_expert_routed(label, base, mode, direct):
    w = _workload(base, E=4, k=4, T=24)
    ids, _, _ = M.route(synth.make_logits(w, x_bits=synth.make_x(w)), w.k)
    assert np.array_equal(np.bincount(ids.ravel(), minlength=w.E), np.full(w.E, w.T))
    _run_against_oracle(w, mode, direct)


@pytest.mark.parametrize("label,base,mode,direct", PATHS, ids=[p[0] for p in PATHS])
def test_empty_batch(label, base, mode, direct):
    w = _workload(base, E=8, k=2, T=0)
    ml, _, _ = make_layer(w, mode=mode, direct=direct)
    x = torch.empty((0, w.H), dtype=torch.int16, device="cuda")
    lg = torch.empty((0, w.E), dtype=torch.float32, device="cuda")
    b = ml.buffers(0)
    out = ml.step(x, lg, b)
    torch.cuda.synchronize()
    assert out.shape[0] == 0
    assert L.moe_get_error(b.dev_err) == 0
