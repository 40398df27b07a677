"""Seeded synthetic inputs for the low-bit routed-expert FFN.

This module is shared by the CUDA path's tests/bench and by the CPU oracle's
tests.  It holds only input recipes (shapes, value distributions, seeds) and
none of the layer's arithmetic: no decoding, routing, rounding or matmul of
the method happens here.  Every array is produced on the host with NumPy's
PCG64 generator seeded by ``SeedSequence([seed, workload_id, tensor_id])`` so
both sides receive byte-identical inputs.

Workloads follow the problem statement of the vLLM-Moet pages (2-bit codebook
experts with an FP4 delta cache; MXFP4 experts converted online into an FP8
workspace as in "Day-0 adaptation ... §四"):

===============  ===  ====  ====  =  =====  ======================================
name             E    H     I     k  T      weights / routing
===============  ===  ====  ====  =  =====  ======================================
tiny             8    256   128   2  16     2-bit; logits = x . Wr^T, Wr N(0,1)*0.1
decode           384  4096  2048  8  8      2-bit; logits U(0,1)
mixed_decode     384  4096  2048  8  64     2-bit base + 64 hottest as MXFP4; Zipf(1.1)
prefill_bf16     384  4096  2048  8  8192   2-bit; Zipf(1.1) logits
prefill_fp8      256  7168  2048  8  16384  MXFP4 (E8M0 in [-8,-4]); logits U(0,1)
===============  ===  ====  ====  =  =====  ======================================

Canonical weight layout (the library's ABI layout, see include/moe.h):
  * W1 of an expert is [2I][H] row-major: rows 0..I-1 gate, rows I..2I-1 up.
  * W2 of an expert is [H][I] row-major.
  * 2-bit codes: 4 per byte, element i of a row at bits 2*(i%4) of byte i//4.
    fp16 scales [rows][K/32].
  * MXFP4: 2 E2M1 nibbles per byte, element 2i in the low nibble; E8M0 bytes
    [rows][K/32].
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import numpy as np

__all__ = ["Workload", "WORKLOADS", "get_workload", "rng_for", "make_x", "make_logits",
           "make_w2_expert", "make_w2_layer", "make_mxfp4_expert", "make_mxfp4_layer",
           "zipf_ranks", "hot_experts"]


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    wid: int          # id folded into every seed
    E: int
    H: int
    I: int
    k: int
    T: int
    weights: str      # "w2" | "mixed" | "mxfp4"
    logits: str       # "router" | "uniform" | "zipf"
    n_hot: int = 0    # experts held as MXFP4 delta-cache entries ("mixed")
    zipf_s: float = 1.1
    zipf_beta: float = 0.03
    e8m0_lo: int = 119  # E8M0 bytes drawn uniformly in [lo, hi]  (2^-8 .. 2^-4)
    e8m0_hi: int = 123
    scale_sigma: float = 0.02

    @property
    def A(self) -> int:
        return self.T * self.k

    def replace(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


WORKLOADS = {
    w.name: w for w in [
        Workload("tiny", 1, 8, 256, 128, 2, 16, "w2", "router"),
        Workload("decode", 2, 384, 4096, 2048, 8, 8, "w2", "uniform"),
        Workload("mixed_decode", 3, 384, 4096, 2048, 8, 64, "mixed", "zipf", n_hot=64),
        Workload("prefill_bf16", 4, 384, 4096, 2048, 8, 8192, "w2", "zipf"),
        Workload("prefill_fp8", 5, 256, 7168, 2048, 8, 16384, "mxfp4", "uniform"),
    ]
}

# tensor ids inside one workload's seed space
_TID_X, _TID_LOGITS, _TID_ROUTER, _TID_RANK = 1, 2, 3, 4
_TID_W2_BASE, _TID_MX_BASE = 1000, 500000


def get_workload(name: str, **overrides) -> Workload:
    w = WORKLOADS[name]
    return w.replace(**overrides) if overrides else w


def rng_for(seed: int, wid: int, tid: int) -> np.random.Generator:
    return np.random.default_rng(np.random.SeedSequence([int(seed), int(wid), int(tid)]))


def _bf16_bits_from_f32(a: np.ndarray) -> np.ndarray:
    """Input recipe: keep the upper 16 bits of fp32 samples (truncation).

    The layer never rounds with this; it only shapes the synthetic input
    distribution (N(0,1) values carried in bf16)."""
    return (np.ascontiguousarray(a, dtype=np.float32).view(np.uint32) >> 16).astype(np.uint16)


def make_x(w: Workload, seed: int = 0, T: Optional[int] = None, tid_offset: int = 0) -> np.ndarray:
    """Activations as bf16 bit patterns, uint16 [T, H], N(0,1)."""
    T = w.T if T is None else T
    g = rng_for(seed, w.wid, _TID_X + tid_offset * 100)
    return _bf16_bits_from_f32(g.standard_normal((T, w.H), dtype=np.float32))


def zipf_ranks(w: Workload, seed: int = 0) -> np.ndarray:
    """rank[e] in 1..E (1 = most popular), a seeded random permutation."""
    g = rng_for(seed, w.wid, _TID_RANK)
    return (g.permutation(w.E) + 1).astype(np.int64)


def hot_experts(w: Workload, seed: int = 0) -> np.ndarray:
    """Experts held as MXFP4 delta-cache entries: the n_hot of highest Zipf prior
    (rank 1..n_hot), independent of the batch.  Returns slot[e] (int32, -1 = not
    cached), slots numbered by rank."""
    slot = np.full(w.E, -1, dtype=np.int32)
    if w.n_hot:
        r = zipf_ranks(w, seed)
        hot = r <= w.n_hot
        slot[hot] = (r[hot] - 1).astype(np.int32)
    return slot


def make_logits(w: Workload, seed: int = 0, x_bits: Optional[np.ndarray] = None,
                T: Optional[int] = None, tid_offset: int = 0) -> np.ndarray:
    """Router logits fp32 [T, E].

    * router : logits = x . Wr^T with Wr ~ N(0,1)*0.1, fp64 accumulation rounded
               to fp32 (the router GEMM is outside the layer; both sides get the
               same logits).
    * uniform: U(0,1).
    * zipf   : U(0,1) + beta*ln(rank_e^-s) (a Zipf(s) popularity prior).
    """
    T = w.T if T is None else T
    if w.logits == "router":
        if x_bits is None:
            x_bits = make_x(w, seed, T, tid_offset)
        xf = (x_bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
        g = rng_for(seed, w.wid, _TID_ROUTER)
        wr = g.standard_normal((w.E, w.H)) * 0.1
        return (xf @ wr.T).astype(np.float32)
    g = rng_for(seed, w.wid, _TID_LOGITS + tid_offset * 100)
    u = g.random((T, w.E), dtype=np.float64)
    if w.logits == "uniform":
        return u.astype(np.float32)
    if w.logits == "zipf":
        r = zipf_ranks(w, seed).astype(np.float64)
        return (u - w.zipf_beta * w.zipf_s * np.log(r)[None, :]).astype(np.float32)
    raise ValueError(w.logits)


def _w2_matrix(g: np.random.Generator, rows: int, K: int, sigma: float):
    codes = g.integers(0, 256, size=(rows, K // 4), dtype=np.uint8)
    sc = np.abs(g.standard_normal((rows, K // 32), dtype=np.float32) * np.float32(sigma))
    return codes, sc.astype(np.float16)


def make_w2_expert(w: Workload, e: int, seed: int = 0, layer: int = 0):
    """One expert in the 2-bit codebook format.

    Returns (codes1 uint8 [2I, H/4], scales1 fp16 [2I, H/32],
             codes2 uint8 [H, I/4],  scales2 fp16 [H, I/32]).
    Codes are uniform over the four codebook entries (uniform bytes)."""
    g = rng_for(seed, w.wid, _TID_W2_BASE + layer * 4096 + e)
    c1, s1 = _w2_matrix(g, 2 * w.I, w.H, w.scale_sigma)
    c2, s2 = _w2_matrix(g, w.H, w.I, w.scale_sigma)
    return c1, s1, c2, s2


def make_w2_layer(w: Workload, seed: int = 0, layer: int = 0):
    """All experts stacked: codes1 [E,2I,H/4], scales1 [E,2I,H/32], codes2 [E,H,I/4],
    scales2 [E,H,I/32]."""
    E, H, I = w.E, w.H, w.I
    c1 = np.empty((E, 2 * I, H // 4), np.uint8)
    s1 = np.empty((E, 2 * I, H // 32), np.float16)
    c2 = np.empty((E, H, I // 4), np.uint8)
    s2 = np.empty((E, H, I // 32), np.float16)
    for e in range(E):
        c1[e], s1[e], c2[e], s2[e] = make_w2_expert(w, e, seed, layer)
    return c1, s1, c2, s2


def _mx_matrix(g: np.random.Generator, rows: int, K: int, lo: int, hi: int):
    q = g.integers(0, 256, size=(rows, K // 2), dtype=np.uint8)
    s = g.integers(lo, hi + 1, size=(rows, K // 32), dtype=np.uint8)
    return q, s


def make_mxfp4_expert(w: Workload, e: int, seed: int = 0, layer: int = 0):
    """One expert in MXFP4: (q1 uint8 [2I,H/2], s1 uint8 [2I,H/32], q2 [H,I/2], s2 [H,I/32]).
    E2M1 codes uniform over all 16; E8M0 bytes uniform in [e8m0_lo, e8m0_hi]."""
    g = rng_for(seed, w.wid, _TID_MX_BASE + layer * 4096 + e)
    q1, s1 = _mx_matrix(g, 2 * w.I, w.H, w.e8m0_lo, w.e8m0_hi)
    q2, s2 = _mx_matrix(g, w.H, w.I, w.e8m0_lo, w.e8m0_hi)
    return q1, s1, q2, s2


def make_mxfp4_layer(w: Workload, n: Optional[int] = None, seed: int = 0, layer: int = 0):
    """n experts (default E; for a delta cache: n_hot slots) stacked like make_w2_layer."""
    n = w.E if n is None else n
    E, H, I = n, w.H, w.I
    q1 = np.empty((E, 2 * I, H // 2), np.uint8)
    s1 = np.empty((E, 2 * I, H // 32), np.uint8)
    q2 = np.empty((E, H, I // 2), np.uint8)
    s2 = np.empty((E, H, I // 32), np.uint8)
    for e in range(E):
        q1[e], s1[e], q2[e], s2[e] = make_mxfp4_expert(w, e, seed, layer)
    return q1, s1, q2, s2
