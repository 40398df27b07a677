"""Pins for the oracle's routing, grouping and layer (no GPU).

The layer is checked against formulations written separately here:
  * routing by brute force (Python sort with the tie rule, math.exp softmax);
  * grouping by counting loops and invariants (permutation, stability,
    unpermute(gather(x)) == x);
  * a dense formulation out_t = sum_e G[t,e] FFN_e(x_t) over ALL experts with
    a dense gate matrix, in torch float64 with torch's own bf16 / e4m3 casts;
  * the E=1, k=1 reduction to a dense SwiGLU MLP;
  * a closed form (all codes +1, one scale) and an invariant (identical
    experts => output equals that expert's output).
"""
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

from bit_moe_expert_top_gb300 import synth
from oracle import codecs as C
from oracle import moe as M


# --------------------------------------------------------------------------- routing

def _route_bruteforce(logits, k):
    T, E = logits.shape
    ids = np.zeros((T, k), np.int64)
    w = np.zeros((T, k))
    for t in range(T):
        row = [float(v) for v in logits[t]]
        key = lambda e: (1 if math.isnan(row[e]) else 0, -row[e] if not math.isnan(row[e]) else 0.0, e)
        order = sorted(range(E), key=key)[:k]
        ids[t] = order
        sel = [row[e] if not math.isnan(row[e]) else -math.inf for e in order]
        z = [math.exp(v - sel[0]) for v in sel]
        s = sum(z)
        w[t] = [v / s for v in z]
    return ids, w


@pytest.mark.parametrize("seed", range(6))
def test_route_bruteforce_with_ties(seed):
    g = np.random.default_rng(seed)
    T, E = 40, 9
    logits = g.integers(0, 4, (T, E)).astype(np.float32) * np.float32(0.25)   # many ties
    logits[3, 2] = np.nan
    for k in (1, 2, 3, E):
        ids, w, anynan = M.route(logits, k)
        bi, bw = _route_bruteforce(logits, k)
        assert np.array_equal(ids, bi)
        assert np.allclose(w, bw, rtol=0, atol=2e-7)
        assert anynan
        assert np.all(np.abs(w.astype(np.float64).sum(1) - 1) <= 1e-6)


def test_route_special_cases():
    E, k = 16, 8
    ids, w, _ = M.route(np.zeros((3, E), np.float32), k)
    assert (ids == np.arange(k)).all() and np.all(w == np.float32(1.0 / k))
    L = np.zeros((1, E), np.float32)
    L[0, 11] = 100.0
    ids, w, _ = M.route(L, k)
    assert ids[0, 0] == 11 and w[0, 0] == np.float32(1.0) and list(ids[0, 1:]) == list(range(7))
    ids, w, _ = M.route(np.random.default_rng(0).random((5, E)).astype(np.float32), E)
    assert all(sorted(r) == list(range(E)) for r in ids)


# --------------------------------------------------------------------------- grouping

def test_permute_invariants_and_bruteforce():
    g = np.random.default_rng(1)
    for E, T, k in [(8, 16, 2), (384, 64, 8), (5, 1, 5), (7, 0, 2)]:
        ids = np.array([g.choice(E, k, replace=False) for _ in range(T)]).reshape(T, k).astype(np.int32)
        off, perm, inv = M.permute(ids, E)
        A = T * k
        counts = [0] * E
        for a in range(A):
            counts[ids.reshape(-1)[a]] += 1
        assert list(np.diff(off)) == counts and off[0] == 0 and off[-1] == A
        assert sorted(perm.tolist()) == list(range(A))
        want = [a for e in range(E) for a in range(A) if ids.reshape(-1)[a] == e]
        assert perm.tolist() == want
        assert all(inv[perm[p]] == p for p in range(A))
        x = g.standard_normal((T, 4))
        xp = M.gather_rows(x, perm, k)
        back = M.unpermute(xp, inv)
        assert np.array_equal(back, np.repeat(x, k, axis=0))


# --------------------------------------------------------------------------- layer

def _bf16(t):
    return t.to(torch.float32).to(torch.bfloat16).to(torch.float64)


def _f32(t):
    return t.to(torch.float32).to(torch.float64)


def _dense_layer(x_bits, logits, k, W1s, W2s):
    """out_t = sum_e G[t,e] FFN_e(x_t): every expert evaluated on every token."""
    x = torch.from_numpy((x_bits.astype(np.uint32) << 16).view(np.float32)).to(torch.float64)
    T, E = logits.shape
    bi, bw = _route_bruteforce(logits, k)
    G = torch.zeros(T, E, dtype=torch.float64)
    for t in range(T):
        for j in range(k):
            G[t, bi[t, j]] = float(np.float32(bw[t, j]))
    out = torch.zeros(T, x.shape[1], dtype=torch.float64)
    I = W2s[0].shape[1]
    for e in range(E):
        W1 = torch.from_numpy(W1s[e])
        W2 = torch.from_numpy(W2s[e])
        gt = _f32(x @ W1[:I].T)
        up = _f32(x @ W1[I:].T)
        h = _bf16(gt * torch.sigmoid(gt) * up)
        y = _bf16(h @ W2.T)
        out += G[:, e:e + 1] * y
    return out.to(torch.float32).numpy()


def _tiny_weights(w, seed=0):
    c1, s1, c2, s2 = synth.make_w2_layer(w, seed)
    W1s = [C.decode_w2(c1[e], s1[e]) for e in range(w.E)]
    W2s = [C.decode_w2(c2[e], s2[e]) for e in range(w.E)]
    return (c1, s1, c2, s2), W1s, W2s


def test_layer_matches_dense_formulation_tiny():
    w = synth.get_workload("tiny")
    x = synth.make_x(w)
    logits = synth.make_logits(w, x_bits=x)
    raw, W1s, W2s = _tiny_weights(w)
    res = M.layer(x, logits, w.k, M.w2_expert_weights(*raw))
    dense = _dense_layer(x, logits, w.k, W1s, W2s)
    rms = float(np.sqrt(np.mean(dense.astype(np.float64) ** 2)))
    assert rms > 0
    assert np.max(np.abs(res["out"] - dense)) <= 1e-6 * rms


def test_layer_token_subset_matches_full():
    w = synth.get_workload("tiny")
    x = synth.make_x(w)
    logits = synth.make_logits(w, x_bits=x)
    raw, _, _ = _tiny_weights(w)
    full = M.layer(x, logits, w.k, M.w2_expert_weights(*raw))
    sub = M.layer(x, logits, w.k, M.w2_expert_weights(*raw), tokens=[3, 0, 15])
    assert np.array_equal(sub["out"], full["out"][[3, 0, 15]])


def test_single_expert_reduces_to_dense_swiglu():
    w = synth.get_workload("tiny").replace(E=1, k=1, T=5)
    x = synth.make_x(w)
    logits = np.zeros((w.T, 1), np.float32)
    raw, W1s, W2s = _tiny_weights(w)
    res = M.layer(x, logits, 1, M.w2_expert_weights(*raw))
    xt = torch.from_numpy((x.astype(np.uint32) << 16).view(np.float32)).double()
    W1 = torch.from_numpy(W1s[0])
    W2 = torch.from_numpy(W2s[0])
    gate, up = torch.nn.functional.linear(xt, W1).to(torch.float32).double().chunk(2, dim=-1)
    h = (F.silu(gate) * up).float().bfloat16().double()
    y = torch.nn.functional.linear(h, W2).float().bfloat16().float().numpy()
    assert np.array_equal(res["out"], y)


def test_closed_form_all_plus_one():
    """codes all +1 (code 2 = 0b10 -> byte 0xAA) and one scale s:
    g = u = b*sum(x) with b = bf16(s); h = bf16(silu(g)*g); y_n = bf16(b*sum_i h_i)."""
    w = synth.get_workload("tiny").replace(E=1, k=1, T=3)
    H, I = w.H, w.I
    s = np.float16(0.0123)
    c1 = np.full((1, 2 * I, H // 4), 0xAA, np.uint8)
    c2 = np.full((1, H, I // 4), 0xAA, np.uint8)
    s1 = np.full((1, 2 * I, H // 32), s, np.float16)
    s2 = np.full((1, H, I // 32), s, np.float16)
    x = synth.make_x(w)
    res = M.layer(x, np.zeros((w.T, 1), np.float32), 1, M.w2_expert_weights(c1, s1, c2, s2))
    b = float(torch.tensor(float(s)).bfloat16().float())
    for t in range(w.T):
        xv = (x[t].astype(np.uint32) << 16).view(np.float32).astype(np.float64)
        gsum = float(np.float32(b * math.fsum(xv)))
        hval = float(torch.tensor(gsum / (1 + math.exp(-gsum)) * gsum, dtype=torch.float32).bfloat16().float())
        yval = float(torch.tensor(b * hval * I, dtype=torch.float32).bfloat16().float())
        assert np.all(res["out"][t] == np.float32(yval))


def test_identical_experts_invariant():
    w = synth.get_workload("tiny").replace(E=6, k=3)
    x = synth.make_x(w)
    logits = synth.make_logits(w, x_bits=x)
    c1, s1, c2, s2 = synth.make_w2_layer(w)
    for e in range(1, w.E):
        c1[e], s1[e], c2[e], s2[e] = c1[0], s1[0], c2[0], s2[0]
    res = M.layer(x, logits, w.k, M.w2_expert_weights(c1, s1, c2, s2))
    one = M.layer(x, np.zeros((w.T, 1), np.float32), 1, M.w2_expert_weights(c1, s1, c2, s2))
    rms = np.sqrt(np.mean(one["out"].astype(np.float64) ** 2))
    assert np.max(np.abs(res["out"] - one["out"])) <= 1e-6 * rms


def _mxfp8_torch(a):
    """Independent MXFP8 conversion along the last axis (torch e4m3 cast after
    clamping; scale exponent by search)."""
    a = np.asarray(a, dtype=np.float64)
    out = np.zeros_like(a)
    for idx in np.ndindex(a.shape[:-1]):
        row = a[idx]
        for b0 in range(0, row.size, 32):
            blk = row[b0:b0 + 32]
            amax = float(np.max(np.abs(blk)))
            if amax == 0:
                X = -127
            else:
                X = math.frexp(amax)[1] - 1 - 8
            sc = np.clip(blk * 2.0 ** -X, -448, 448)
            q = torch.from_numpy(sc.astype(np.float32)).to(torch.float8_e4m3fn).to(torch.float64).numpy()
            out[idx + (slice(b0, b0 + 32),)] = q * 2.0 ** X
    return out


def test_fp8_profile_single_expert_against_torch():
    w = synth.get_workload("tiny").replace(E=1, k=1, T=4, weights="mxfp4")
    q1, s1, q2, s2 = synth.make_mxfp4_layer(w)
    x = synth.make_x(w)
    res = M.layer(x, np.zeros((w.T, 1), np.float32), 1, M.fp8_expert_weights(q1, s1, q2, s2), profile="fp8")
    W1 = torch.from_numpy(C.decode_mxfp4(q1[0], s1[0])).float().to(torch.float8_e4m3fn).double()
    W2 = torch.from_numpy(C.decode_mxfp4(q2[0], s2[0])).float().to(torch.float8_e4m3fn).double()
    xt = torch.from_numpy(_mxfp8_torch((x.astype(np.uint32) << 16).view(np.float32)))
    gate, up = (xt @ W1.T).float().double().chunk(2, dim=-1)
    h = (F.silu(gate) * up).float().double()
    hq = torch.from_numpy(_mxfp8_torch(h.numpy()))
    y = (hq @ W2.T).float().bfloat16().float().numpy()
    assert np.array_equal(res["out"], y)


def test_mixed_accessor_routes_hot_experts_to_mxfp4():
    w = synth.get_workload("tiny").replace(E=6, k=2, n_hot=2, weights="mixed", logits="zipf")
    slot = synth.hot_experts(w)
    assert (slot >= 0).sum() == 2
    raw = synth.make_w2_layer(w)
    mx = synth.make_mxfp4_layer(w, n=2)
    get = M.mixed_expert_weights(M.w2_expert_weights(*raw), M.mxfp4_expert_weights(*mx), slot)
    for e in range(w.E):
        W1, _ = get(e)
        if slot[e] >= 0:
            assert np.array_equal(W1, C.decode_mxfp4(mx[0][slot[e]], mx[1][slot[e]]))
        else:
            assert np.array_equal(W1, C.decode_w2(raw[0][e], raw[1][e]))


def test_per_expert_profile_selects_each_experts_rows():
    """expert_profile: every assignment's y is the one its expert's profile
    gives (fp8 for the delta-cache experts, bf16 for the 2-bit ones), taken
    from full runs in each single profile, and the output is their combine."""
    w = synth.get_workload("tiny").replace(E=6, k=3, T=10, n_hot=2, weights="mixed", logits="zipf")
    slot = synth.hot_experts(w)
    raw = synth.make_w2_layer(w)
    mx = synth.make_mxfp4_layer(w, n=2)
    get = M.mixed_expert_weights(M.w2_expert_weights(*raw), M.mxfp4_expert_weights(*mx), slot)
    x = synth.make_x(w)
    lg = synth.make_logits(w, x_bits=x)
    mixed = M.layer(x, lg, w.k, get, expert_profile=lambda e: "fp8" if slot[e] >= 0 else "bf16")
    bf = M.layer(x, lg, w.k, get, profile="bf16")
    fp = M.layer(x, lg, w.k, get, profile="fp8")
    cached = slot[mixed["ids"]] >= 0
    assert cached.any() and (~cached).any()
    want_y = np.where(cached[:, :, None], fp["y"], bf["y"])
    assert np.array_equal(mixed["y"], want_y)
    assert not np.array_equal(fp["y"][cached], bf["y"][cached])   # the profiles really differ there
    out = np.zeros((w.T, w.H))
    for t in range(w.T):
        for j in range(w.k):
            out[t] += float(mixed["w"][t, j]) * want_y[t, j]
    assert np.allclose(mixed["out"], out, rtol=1e-6, atol=0)  # fp32 of the fp64 sum (summation order aside)
