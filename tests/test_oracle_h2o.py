"""Pins for the H2O / StreamingLLM selection oracle (CPU only)."""
import itertools

import numpy as np
import pytest

from oracle import h2o


def brute_topk(scores, k):
    """Selected iff fewer than k elements beat it under (score desc, index asc)."""
    n = len(scores)
    sel = []
    for i in range(n):
        beats = sum(1 for j in range(n)
                    if scores[j] > scores[i] or (scores[j] == scores[i] and j < i))
        if beats < k:
            sel.append(i)
    return np.array(sel, dtype=np.int64)


def test_hand_worked_select(golden):
    rows = list(golden("h2o_select.txt"))
    cum = np.array([float(x) for x in rows[0][1:]])
    for row in rows[1:]:
        budget = int(row[1])
        want = [int(x) for x in row[3:]]
        got = h2o.h2o_keep(cum, len(cum), budget, n_sink=2, window=2)
        assert got.tolist() == want, budget


@pytest.mark.parametrize("seed", range(40))
def test_topk_matches_brute_force_with_ties(seed):
    rng = np.random.default_rng(seed)
    n = int(rng.integers(1, 13))
    scores = rng.integers(0, 4, n).astype(np.float64)        # many ties
    for k in range(0, n + 2):
        assert h2o.topk_positions(scores, k).tolist() == brute_topk(scores, k).tolist()


def test_streaming_rules_from_handbook(golden):
    rows = list(golden("streaming_keep.txt"))
    # recent-only: sinks = 0, window = budget
    S, budget, sinks, lo, hi = (int(x) for x in rows[0][:5])
    keep = h2o.h2o_keep(np.random.rand(S), S, budget, n_sink=sinks, window=budget)
    assert keep.tolist() == list(range(lo, hi + 1))
    assert h2o.streaming_keep(S, budget, 0).tolist() == keep.tolist()
    # sinks + window: heavy hitters = 0, window = budget - sinks
    S, budget, sinks, lo, hi, lo2, hi2 = (int(x) for x in rows[1])
    want = list(range(lo, hi + 1)) + list(range(lo2, hi2 + 1))
    for cum in (np.random.rand(S), np.zeros(S), np.arange(S, 0, -1.0)):
        keep = h2o.h2o_keep(cum, S, budget, n_sink=sinks, window=budget - sinks)
        assert keep.tolist() == want
    assert h2o.streaming_keep(S, budget, sinks).tolist() == want


@pytest.mark.parametrize("seed", range(20))
def test_keep_invariants(seed):
    rng = np.random.default_rng(100 + seed)
    S = int(rng.integers(1, 300))
    n_sink = int(rng.integers(0, 6))
    window = int(rng.integers(0, 40))
    budget = n_sink + window + int(rng.integers(0, 60))
    cum = rng.random(S)
    keep = h2o.h2o_keep(cum, S, budget, n_sink, window)
    assert len(keep) == min(S, budget)
    assert np.all(np.diff(keep) > 0)
    if S > budget:
        assert set(range(n_sink)) <= set(keep.tolist())
        assert set(range(S - window, S)) <= set(keep.tolist())
        # every kept middle slot scores >= every evicted middle slot
        mid = set(range(n_sink, S - window))
        kept_mid = [j for j in keep if j in mid]
        lost_mid = [j for j in mid if j not in set(keep.tolist())]
        if kept_mid and lost_mid:
            assert min(cum[kept_mid]) >= max(cum[lost_mid])


def test_equal_scores_keep_lowest_candidates():
    keep = h2o.h2o_keep(np.ones(50), 50, budget=20, n_sink=4, window=6)
    assert keep.tolist() == list(range(4)) + list(range(4, 14)) + list(range(44, 50))


def test_sequence_scores_follow_tokens_through_eviction():
    # Book-keep, by ORIGINAL position, the attention each token received over
    # the steps it survived, and compare with the oracle's per-slot scores
    # after many evict+compact steps (catches scores not moving with K/V).
    rng = np.random.default_rng(7)
    Hq, Hkv, d, S0 = 4, 2, 8, 24
    budget, n_sink, window = 14, 2, 3
    seq = h2o.H2OSequence(rng.standard_normal((Hkv, S0, d)), rng.standard_normal((Hkv, S0, d)))
    ledger = [dict() for _ in range(Hkv)]
    for step in range(30):
        q = rng.standard_normal((Hq, d))
        pos_before = None
        o, p, keep = seq.step(q, rng.standard_normal((Hkv, d)), rng.standard_normal((Hkv, d)),
                              0.35, budget, n_sink, window, evict=False)
        for kvh in range(Hkv):
            for slot, pos in enumerate(seq.pos[kvh]):
                ledger[kvh][int(pos)] = ledger[kvh].get(int(pos), 0.0) + p[kvh * 2:(kvh + 1) * 2, slot].sum()
        if keep is not None:
            seq.apply_keep(keep)
        assert seq.S == min(S0 + step + 1, budget)
        for kvh in range(Hkv):
            pos = seq.pos[kvh]
            assert np.all(np.diff(pos) > 0)
            assert pos[:n_sink].tolist() == list(range(n_sink))
            assert pos[-window:].tolist() == list(range(seq.seen - window, seq.seen))
            for slot, ps in enumerate(pos):
                assert abs(seq.cum[kvh, slot] - ledger[kvh][int(ps)]) < 1e-12
