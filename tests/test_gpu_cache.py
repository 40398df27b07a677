"""FP4 delta-cache management on the device (moe_cache_select /
moe_cache_fill) against the oracle's policy, through the C ABI (GPU).

A sequence of mixed layer steps with Zipf-skewed routing: after every step
the counts, the slot maps and the promotion list must equal the oracle's
bit for bit; every filled slot must hold exactly the stored MXFP4 bytes of
its expert (from device memory, and from pinned host memory read over the
CPU-GPU link); and the next step, run with the updated map, must match the
oracle's layer under the same map at the method's bf16 gate."""
import numpy as np
import pytest
import torch

from bit_moe_expert_top_gb300 import _lib as L
from bit_moe_expert_top_gb300 import synth
from bit_moe_expert_top_gb300.layer import MoELayer
from oracle import cache as K
from oracle import moe as M

from tests._gpu import DEV, TOL_BF16, dev, host, rel_err

pytestmark = pytest.mark.gpu


def _cache_state(E, S):
    return (torch.zeros(E, dtype=torch.int32, device=DEV), torch.full((E,), -1, dtype=torch.int32, device=DEV),
            torch.full((S,), -1, dtype=torch.int32, device=DEV), torch.empty(S, dtype=torch.int32, device=DEV))


def test_cache_select_matches_the_policy_on_random_counts():
    """The selection kernel alone, many random steps (ties, decay, E = 1024)."""
    g = np.random.default_rng(11)
    for E, S, d in [(40, 8, 31), (384, 64, 2), (1024, 100, 1), (7, 7, 31), (64, 1, 0)]:
        counts, es, se, pr = _cache_state(E, S)
        c_o = np.zeros(E, np.uint32)
        es_o = np.full(E, -1, np.int32)
        se_o = np.full(S, -1, np.int32)
        err = torch.zeros(1, dtype=torch.int32, device=DEV)
        for _ in range(12):
            sizes = g.poisson(g.uniform(0, 3, size=E)).astype(np.int64)
            off = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32)
            L.moe_cache_select(dev(off), counts, d, es, se, pr, dev_err=err)
            c_o, es_o, se_o, pr_o = K.step(c_o, es_o, se_o, off, d)
            assert np.array_equal(host(counts).view(np.uint32), c_o)
            assert np.array_equal(host(es), es_o)
            assert np.array_equal(host(se), se_o)
            assert np.array_equal(host(pr), pr_o)
        assert L.moe_get_error(err) == 0


@pytest.mark.parametrize("host_store", [False, True])
def test_cache_promotion_through_layer_steps(host_store):
    w = synth.get_workload("mixed_decode").replace(E=48, H=512, I=512, k=4, T=24, n_hot=8)
    E, S, k = w.E, w.n_hot, w.k
    raw = synth.make_w2_layer(w)
    mx_all = synth.make_mxfp4_layer(w, n=E)            # the MXFP4 store: every expert
    # the layer starts with an empty cache: slot arrays zero, no expert mapped
    cache0 = tuple(np.zeros((S,) + a.shape[1:], a.dtype) for a in mx_all)
    ml = MoELayer("mixed", E, w.H, w.I, k, w2=raw, mx=cache0, expert_slot=np.full(E, -1, np.int32),
                  out_fmt=L.FMT_F32, mode=L.MODE_AUTO)
    if host_store:
        store = [torch.from_numpy(a).pin_memory() for a in mx_all]
    else:
        store = [dev(a) for a in mx_all]
    ml.attach_store(store, decay_shift=31)
    dsts = [ml.q1, ml.e1, ml.q2, ml.e2]
    es, se, pr = ml.expert_slot, ml.slot_expert, ml.promoted
    c_o = np.zeros(E, np.uint32)
    es_o = np.full(E, -1, np.int32)
    se_o = np.full(S, -1, np.int32)
    w2_acc = M.w2_expert_weights(*raw)
    mx_acc = M.mxfp4_expert_weights(*mx_all)
    promoted_total = 0
    for step in range(6):
        wz = w.replace(zipf_beta=0.5, zipf_s=1.1)
        x = synth.make_x(wz, 0, tid_offset=step)
        logits = synth.make_logits(wz, step, x_bits=x, tid_offset=step)
        b = ml.buffers(w.T)
        out = ml.step(dev(x.view(np.int16)), dev(logits), b)
        torch.cuda.synchronize()
        # the step used the map of the previous update
        acc = (lambda es_now: (lambda e: mx_acc(e) if es_now[e] >= 0 else w2_acc(e)))(es_o.copy())
        ref = M.layer(x, logits, k, acc, profile="bf16")
        err, _ = rel_err(host(out), ref["out"])
        assert err <= TOL_BF16, (step, err)
        assert L.moe_get_error(b.dev_err) == 0
        # update the cache from this step's grouping, then fill the new slots
        ml.update_cache(b)
        torch.cuda.synchronize()
        c_o, es_o, se_o, pr_o = K.step(c_o, es_o, se_o, host(b.offsets), 31)
        assert np.array_equal(host(es), es_o) and np.array_equal(host(se), se_o)
        assert np.array_equal(host(pr), pr_o)
        promoted_total += int((pr_o >= 0).sum())
        for s in range(S):                               # slot contents = the expert's stored bytes
            e = int(se_o[s])
            if e >= 0:
                for a, dst in zip(mx_all, dsts):
                    assert np.array_equal(host(dst[s]), a[e]), (step, s, e)
    assert promoted_total > S                            # the hot set moved during the sequence
