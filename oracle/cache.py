"""The FP4 delta cache's management policy, written out step by step.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

The pages keep "the hottest experts" at FP4 precision as a quality layer
over the 2-bit experts (blog "这个项目我们能学到什么?" on vLLM-Moet, the FP4
delta-cache paragraph; vLLM-Moet README, line table: "2-bit experts ... an
FP4 delta cache") and treat the GPU as a cache of hot experts (the same blog,
"GPU作为专家缓存").  They do not say how hotness is measured or how slots are
reused; the readings taken here (parity unpinned against the pages: these are
conventions, pinned by invariants and hand-worked cases in
``tests/test_oracle_cache.py``):

1. Hotness is a running count of routed assignments per expert, an integer
   exponential moving average updated once per step from the step's group
   sizes:  c <- c - (c >> d) + n_e  (d = decay shift; d >= 31 keeps the plain
   cumulative count; additions saturate at 2^32 - 1).
2. The cached set is the S experts of largest count, ties to the lowest
   expert id (the routing tie rule).
3. Slots are stable: a cached expert that stays in the set keeps its slot.
   Experts leaving the set free their slots; experts entering it take the
   free slots in ascending slot order, in the order of the ranking
   (hottest first).  Every slot holds at most one expert.
"""
from __future__ import annotations

from typing import Tuple

import numpy as np

U32_MAX = 0xFFFFFFFF


def update_counts(counts: np.ndarray, group_sizes: np.ndarray, decay_shift: int) -> np.ndarray:
    """c <- c - (c >> d) + n (d >= 31: no decay), saturating at 2^32-1; uint32."""
    c = np.asarray(counts, dtype=np.uint64)
    n = np.asarray(group_sizes, dtype=np.uint64)
    if decay_shift < 31:
        c = c - (c >> np.uint64(decay_shift))
    return np.minimum(c + n, U32_MAX).astype(np.uint32)


def ranking(counts: np.ndarray) -> np.ndarray:
    """Expert ids ordered by (count descending, id ascending)."""
    c = np.asarray(counts, dtype=np.int64)
    E = c.size
    return np.array(sorted(range(E), key=lambda e: (-int(c[e]), e)), dtype=np.int64)


def select(counts: np.ndarray, S: int) -> np.ndarray:
    """The cached set: the first S experts of the ranking, in ranking order."""
    return ranking(counts)[:S]


def assign(expert_slot: np.ndarray, slot_expert: np.ndarray, hot: np.ndarray) -> Tuple[np.ndarray, np.ndarray, np.ndarray]:
    """New maps after the cached set becomes ``hot`` (in ranking order).

    Returns (expert_slot [E] int32, -1 = not cached; slot_expert [S] int32,
    -1 = empty; promoted [S] int32: the expert newly placed in slot s by this
    update, -1 where the slot kept its expert or stays empty)."""
    es = np.array(expert_slot, dtype=np.int32, copy=True)
    se = np.array(slot_expert, dtype=np.int32, copy=True)
    S = se.size
    hot_set = set(int(e) for e in hot)
    for s in range(S):                       # evict: experts that left the set
        e = int(se[s])
        if e >= 0 and e not in hot_set:
            es[e] = -1
            se[s] = -1
    free = [s for s in range(S) if se[s] < 0]
    promoted = np.full(S, -1, dtype=np.int32)
    fi = 0
    for e in hot:                            # promote: hottest first, lowest free slot first
        e = int(e)
        if es[e] < 0:
            s = free[fi]
            fi += 1
            es[e] = s
            se[s] = e
            promoted[s] = e
    return es, se, promoted


def step(counts, expert_slot, slot_expert, offsets, decay_shift):
    """One update from a step's grouping offsets [E+1]: counts, then the
    cached set, then the maps.  Returns (counts, expert_slot, slot_expert,
    promoted)."""
    sizes = np.diff(np.asarray(offsets, dtype=np.int64))
    c = update_counts(counts, sizes, decay_shift)
    hot = select(c, np.asarray(slot_expert).size)
    es, se, pr = assign(expert_slot, slot_expert, hot)
    return c, es, se, pr
