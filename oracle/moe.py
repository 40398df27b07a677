"""The routed-expert FFN written out from its definition.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

Notation: T tokens, E experts, H hidden, I expert intermediate, k experts per
token, A = T*k assignments a = t*k + j (j = slot in the token's top-k).

The layer (vLLM-Moet README, release v2026.11.03-r23 notes: the prefill MoE is
"FC1 + SwiGLU + MXFP8 quant, FC2"; the routed experts are 384 per layer in the
README's line table):

    ids, w   = top-k softmax routing of the router logits
    for every assignment (t, j):  e = ids[t, j]
        g = W1_e[gate] x_t ,  u = W1_e[up] x_t          (FC1, gate/up)
        h = silu(g) * u                                  (SwiGLU)
        y = W2_e h                                       (FC2)
    out_t = sum_j w[t, j] * y(t, j)                      (weighted combine)

Precision profiles (where the definition rounds):

  * "bf16" (2-bit and MXFP4 experts): weights are the exact dequantised
    values (bf16-representable), x is bf16; g, u are fp32; h = RNE_bf16(silu(g)*u);
    y = RNE_bf16(W2 h); out = fp32(sum_j w_j y_j).
  * "fp8" (MXFP4 converted to an FP8 workspace, "国产GPU完成MoE大模型Day-0适配"
    §四): weights are the E4M3 workspace values; x is MXFP8-quantised per
    token in blocks of 32 along H; g, u fp32; h = fp32(silu(g)*u) is
    MXFP8-quantised along I; y = RNE_bf16(W2 h_q); out as above.
  * per expert (``expert_profile``): each expert's rows follow the profile
    named for that expert, e.g. the delta cache's MXFP4 experts in "fp8"
    (FP8 as the compute precision of MXFP4 experts, §四) and the 2-bit
    experts in "bf16"; the combine is unchanged.

Each dot product is accumulated in fp64 and rounded once to fp32.
"""
from __future__ import annotations

from typing import Callable, Dict, Iterable, Optional, Tuple

import numpy as np

from . import codecs as C

# ---------------------------------------------------------------------------
# routing
# ---------------------------------------------------------------------------


def route(logits: np.ndarray, k: int) -> Tuple[np.ndarray, np.ndarray, bool]:
    """Top-k softmax routing (384 routed experts per layer, top-k per token:
    vLLM-Moet README line table; "top-8 softmax routing" of the problem).

    Experts are ordered by (logit descending, expert id ascending): equal
    logits go to the lowest id.  NaN ranks below every number and raises the
    error flag.  The slot-j weight is the softmax over the k selected logits,
        w_j = exp(l_j - l_0) / sum_j' exp(l_j' - l_0),
    i.e. the full softmax renormalised over the top-k; the weights of a token
    sum to 1.  Returns (ids int32 [T,k], w fp32 [T,k], any_nan)."""
    L = np.asarray(logits, dtype=np.float32)
    T, E = L.shape
    assert 1 <= k <= E
    lf = L.astype(np.float64)
    nan = np.isnan(lf)
    key_val = np.where(nan, np.inf, -lf)          # ascending sort of -logit; NaN last
    eid = np.broadcast_to(np.arange(E), (T, E))
    order = np.lexsort((eid, key_val, nan), axis=-1)
    ids = order[:, :k].astype(np.int32)
    sel = np.take_along_axis(lf, ids.astype(np.int64), axis=1)
    sel = np.where(np.isnan(sel), -np.inf, sel)
    z = np.exp(sel - sel[:, :1])
    w = (z / z.sum(axis=1, keepdims=True)).astype(np.float32)
    return ids, w, bool(nan.any())


# ---------------------------------------------------------------------------
# grouping of assignments by expert
# ---------------------------------------------------------------------------


def permute(ids: np.ndarray, E: int):
    """Stable grouping of the A assignments by expert.

    perm lists the assignments a = t*k + j sorted by (expert, a); offsets[e] is
    the first position of expert e's group (exclusive prefix sum of the group
    sizes, offsets[E] = A); inv[perm[p]] = p.  Returns (offsets int32 [E+1],
    perm int32 [A], inv int32 [A])."""
    flat = np.asarray(ids, dtype=np.int64).reshape(-1)
    A = flat.size
    assert flat.size == 0 or (flat.min() >= 0 and flat.max() < E)
    counts = np.bincount(flat, minlength=E)
    offsets = np.zeros(E + 1, dtype=np.int64)
    offsets[1:] = np.cumsum(counts)
    perm = np.argsort(flat, kind="stable")
    inv = np.empty(A, dtype=np.int64)
    inv[perm] = np.arange(A)
    return offsets.astype(np.int32), perm.astype(np.int32), inv.astype(np.int32)


def gather_rows(x: np.ndarray, perm: np.ndarray, k: int) -> np.ndarray:
    """x_perm[p] = x[perm[p] // k]: each permuted row is its token's activation."""
    return np.asarray(x)[np.asarray(perm, dtype=np.int64) // k]


def unpermute(rows_perm: np.ndarray, inv: np.ndarray) -> np.ndarray:
    """rows[a] = rows_perm[inv[a]] (assignment order)."""
    return np.asarray(rows_perm)[np.asarray(inv, dtype=np.int64)]


# ---------------------------------------------------------------------------
# expert FFN
# ---------------------------------------------------------------------------


def silu(g: np.ndarray) -> np.ndarray:
    """silu(g) = g / (1 + exp(-g)) = g * sigmoid(g)."""
    g = np.asarray(g, dtype=np.float64)
    with np.errstate(over="ignore"):
        return g / (1.0 + np.exp(-g))


def expert_ffn_bf16(x: np.ndarray, W1: np.ndarray, W2: np.ndarray) -> np.ndarray:
    """Profile "bf16": x float64 [n,H] (bf16 values), W1 float64 [2I,H] (gate
    rows first, then up), W2 float64 [H,I].  Returns y float64 [n,H] holding
    bf16 values."""
    I = W2.shape[1]
    g = C.to_f32(x @ W1[:I].T)
    u = C.to_f32(x @ W1[I:].T)
    h = C.rne_bf16(silu(g) * u)
    return C.rne_bf16(h @ W2.T)


def expert_ffn_fp8(x: np.ndarray, W1: np.ndarray, W2: np.ndarray) -> np.ndarray:
    """Profile "fp8": W1 / W2 are the E4M3 workspace values (float64); x float64
    [n,H] bf16 values is MXFP8-quantised along H; h (fp32) is MXFP8-quantised
    along I before FC2 ("FC1 + SwiGLU + MXFP8 quant, FC2")."""
    I = W2.shape[1]
    xq, xs = C.mxfp8_quantize(x)
    xd = C.mxfp8_dequantize(xq, xs)
    g = C.to_f32(xd @ W1[:I].T)
    u = C.to_f32(xd @ W1[I:].T)
    h = C.to_f32(silu(g) * u)
    hq, hs = C.mxfp8_quantize(h)
    hd = C.mxfp8_dequantize(hq, hs)
    return C.rne_bf16(hd @ W2.T)


# ---------------------------------------------------------------------------
# combine and the whole layer
# ---------------------------------------------------------------------------


def combine(y: np.ndarray, w: np.ndarray) -> np.ndarray:
    """out[t] = sum_j w[t,j] * y[t,j], fp32 result.  y float64 [T,k,H] in
    assignment order, w [T,k]."""
    return C.to_f32(np.einsum("tj,tjh->th", np.asarray(w, dtype=np.float64), y))


ExpertWeights = Callable[[int], Tuple[np.ndarray, np.ndarray]]


def layer(x_bits: np.ndarray, logits: np.ndarray, k: int, expert_weights: ExpertWeights,
          profile: str = "bf16", tokens: Optional[Iterable[int]] = None,
          expert_profile: Optional[Callable[[int], str]] = None) -> Dict[str, np.ndarray]:
    """The routed-expert FFN for the tokens ``tokens`` (default all).

    ``expert_weights(e)`` returns the dequantised (W1 [2I,H], W2 [H,I]) float64
    values of expert e in the profile's weight format.  Routing runs over all
    tokens; the FFN and combine only over the requested ones.  Each expert's
    weights are fetched once.  ``expert_profile(e)``, if given, names the
    profile of expert e (overriding ``profile``).  Returns dict(ids, w,
    y [n,k,H], out fp32 [n,H], tokens)."""
    ids, w, _ = route(logits, k)
    T = ids.shape[0]
    tok = np.arange(T) if tokens is None else np.asarray(list(tokens), dtype=np.int64)
    x = C.bf16_bits_to_f64(np.asarray(x_bits)[tok])
    sub_ids = ids[tok]
    H = x.shape[1]
    y = np.zeros((tok.size, k, H))
    ffns = {"bf16": expert_ffn_bf16, "fp8": expert_ffn_fp8}
    for e in np.unique(sub_ids):
        rows, slots = np.nonzero(sub_ids == e)
        W1, W2 = expert_weights(int(e))
        ffn = ffns[expert_profile(int(e)) if expert_profile else profile]
        y[rows, slots] = ffn(x[rows], W1, W2)
    out = combine(y, w[tok])
    return dict(ids=ids, w=w, y=y, out=out, tokens=tok)


# ---------------------------------------------------------------------------
# weight accessors for the canonical storage formats
# ---------------------------------------------------------------------------


def w2_expert_weights(codes1, scales1, codes2, scales2) -> ExpertWeights:
    """Accessor over stacked 2-bit experts (see include/moe.h for the layout)."""
    def get(e):
        return C.decode_w2(codes1[e], scales1[e]), C.decode_w2(codes2[e], scales2[e])
    return get


def mxfp4_expert_weights(q1, s1, q2, s2) -> ExpertWeights:
    def get(e):
        return C.decode_mxfp4(q1[e], s1[e]), C.decode_mxfp4(q2[e], s2[e])
    return get


def fp8_expert_weights(q1, s1, q2, s2) -> ExpertWeights:
    """Experts stored as MXFP4 and used through the FP8 workspace: the weight
    values are those of the converted E4M3 bytes."""
    def get(e):
        return (C.e4m3_value(C.mxfp4_to_e4m3(q1[e], s1[e])),
                C.e4m3_value(C.mxfp4_to_e4m3(q2[e], s2[e])))
    return get


def mixed_expert_weights(w2: ExpertWeights, mx: ExpertWeights, slot: np.ndarray) -> ExpertWeights:
    """FP4 delta cache: an expert with slot[e] >= 0 is served by the MXFP4
    entry in that slot, every other expert by its 2-bit weights (the hot
    experts "kept at FP4 precision" over the 2-bit base: blog
    "这个项目我们能学到什么?" on vLLM-Moet)."""
    def get(e):
        s = int(slot[e])
        return mx(s) if s >= 0 else w2(e)
    return get
