"""Pins for the oracle's FP4 delta-cache policy (no GPU).

  * a sequence worked by hand (tests/golden/cache_sequence.txt);
  * closed forms of the integer moving average (no decay = cumulative sum,
    decay shift 0 = the last step only, the fixed point 2^d * n of a constant
    input, saturation);
  * the ranking against numpy's lexsort (an independent sort);
  * invariants over random sequences: the cached set is the top-S set, the
    slot map is a bijection onto the cached set, a retained expert never
    moves, and promoted experts fill the freed slots in ascending order,
    hottest first.
"""
import os

import numpy as np
import pytest

from oracle import cache as K

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "cache_sequence.txt")


def _read_sequence():
    hdr, steps, cur = {}, [], None
    for ln in open(GOLDEN, encoding="utf-8"):
        ln = ln.strip()
        if not ln or ln.startswith("#"):
            continue
        key, *vals = ln.split()
        vals = [int(v) for v in vals]
        if key in ("E", "S", "decay"):
            hdr[key] = vals[0]
        elif key == "sizes":
            cur = {"sizes": np.array(vals)}
            steps.append(cur)
        else:
            cur[key] = np.array(vals)
    return hdr, steps


def test_hand_worked_sequence():
    hdr, steps = _read_sequence()
    E, S, d = hdr["E"], hdr["S"], hdr["decay"]
    counts = np.zeros(E, np.uint32)
    es = np.full(E, -1, np.int32)
    se = np.full(S, -1, np.int32)
    assert len(steps) == 5
    for st in steps:
        off = np.concatenate([[0], np.cumsum(st["sizes"])])
        counts, es, se, pr = K.step(counts, es, se, off, d)
        assert np.array_equal(es, st["expert_slot"])
        assert np.array_equal(se, st["slot_expert"])
        assert np.array_equal(pr, st["promoted"])


def test_counts_closed_forms():
    g = np.random.default_rng(3)
    seq = g.integers(0, 50, size=(20, 7))
    c = np.zeros(7, np.uint32)
    for n in seq:
        c = K.update_counts(c, n, 31)
    assert np.array_equal(c, seq.sum(axis=0))                  # no decay: cumulative
    c = np.zeros(7, np.uint32)
    for n in seq:
        c = K.update_counts(c, n, 0)
    assert np.array_equal(c, seq[-1])                          # shift 0: last step only
    for d in (1, 2, 3):                                        # fixed point of a constant input
        n = np.array([0, 1, 8, 40, 1000])
        c = (n << d).astype(np.uint32)
        assert np.array_equal(K.update_counts(c, n, d), c)
    big = np.array([0xFFFFFFF0, 5], np.uint32)
    assert np.array_equal(K.update_counts(big, np.array([100, 1]), 31), [0xFFFFFFFF, 6])


def test_ranking_against_lexsort():
    g = np.random.default_rng(4)
    for _ in range(50):
        E = int(g.integers(1, 60))
        c = g.integers(0, 6, size=E)               # many ties
        want = np.lexsort((np.arange(E), -c))
        assert np.array_equal(K.ranking(c), want)


@pytest.mark.parametrize("E,S,d", [(16, 4, 31), (40, 8, 2), (9, 9, 1), (30, 1, 31), (5, 8, 3)])
def test_random_sequences_keep_the_invariants(E, S, d):
    g = np.random.default_rng(E * 100 + S)
    counts = np.zeros(E, np.uint32)
    es = np.full(E, -1, np.int32)
    se = np.full(S, -1, np.int32)
    for _ in range(40):
        sizes = g.poisson(g.uniform(0, 5, size=E))
        off = np.concatenate([[0], np.cumsum(sizes)])
        prev_es, prev_se = es.copy(), se.copy()
        counts, es, se, pr = K.step(counts, es, se, off, d)
        hot = K.select(counts, S)
        cached = set(int(e) for e in np.nonzero(es >= 0)[0])
        assert cached == set(int(e) for e in hot)               # cached set = top-S
        for e in cached:                                          # bijection
            assert se[es[e]] == e
        assert sorted(int(s) for s in es[es >= 0]) == sorted(int(s) for s in np.nonzero(se >= 0)[0])
        for e in range(E):                                        # retained experts keep their slot
            if prev_es[e] >= 0 and es[e] >= 0:
                assert es[e] == prev_es[e]
        new = [int(e) for e in hot if prev_es[e] < 0]             # promotions, hottest first
        freed = sorted(s for s in range(S) if prev_se[s] < 0 or es[prev_se[s]] < 0)
        assert [int(es[e]) for e in new] == freed[:len(new)]
        assert sorted(int(e) for e in pr[pr >= 0]) == sorted(new)
        for s in range(S):
            assert pr[s] == (se[s] if se[s] >= 0 and prev_se[s] != se[s] else -1)
