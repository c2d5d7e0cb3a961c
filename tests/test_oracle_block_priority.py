"""Pins for the block-priority oracle (CPU only)."""
import math
from fractions import Fraction

import numpy as np
import pytest

import workloads
from oracle import block_priority as BP


def test_hand_worked_blocks(golden):
    rows = list(golden("block_agg.txt"))
    for i in range(0, len(rows), 4):
        tok = np.array([float(x) for x in rows[i][1:]])
        want = {r[0]: float(r[1]) for r in rows[i + 1:i + 4]}
        assert BP.block_scores(tok, 16, BP.AGG_MAX)[0] == want["max"]
        assert abs(BP.block_scores(tok, 16, BP.AGG_MEAN)[0] - want["mean"]) < 1e-15
        assert abs(BP.block_scores(tok, 16, BP.AGG_TOPP, 0.10)[0] - want["topp"]) < 1e-15


def test_partial_last_block_uses_valid_tokens_only():
    tok = np.array([1.0] * 16 + [4.0, 2.0])
    assert BP.block_scores(tok, 16, BP.AGG_MEAN).tolist() == [1.0, 3.0]
    assert BP.block_scores(tok, 16, BP.AGG_MAX).tolist() == [1.0, 4.0]


def _correctly_rounded_f32(num, den):
    exact = Fraction(num, den)
    x = np.float32(float(exact))
    cands = [np.nextafter(x, np.float32(-1)), x, np.nextafter(x, np.float32(2))]
    return min(cands, key=lambda c: (abs(Fraction(float(c)) - exact), int(np.float32(c).view(np.uint32)) & 1))


@pytest.mark.parametrize("seed", range(15))
def test_percentile_is_rank_based_and_correctly_rounded(seed):
    rng = np.random.default_rng(seed)
    n = int(rng.integers(1, 40))
    s = rng.integers(0, 5, n).astype(np.float64)          # ties broken by block index
    pct = BP.percentiles(s)
    for i in range(n):
        r = sum(1 for j in range(n) if s[j] < s[i] or (s[j] == s[i] and j < i))
        assert pct[i] == _correctly_rounded_f32(2 * r + 1, 2 * n)


def test_evict_order_brute_force():
    rng = np.random.default_rng(1)
    reqs = [rng.integers(0, 3, int(rng.integers(1, 9))).astype(np.float64) for _ in range(6)]
    order = BP.evict_order(reqs, 0.4)
    allk = [(reqs[r][b], r, b) for r in range(6) for b in range(len(reqs[r]))]
    N = len(allk)
    assert len(order) == math.ceil(0.4 * N)
    for pos, code in enumerate(order):
        r, b = int(code >> 32), int(code & 0xFFFFFFFF)
        before = sum(1 for (s, r2, b2) in allk
                     if (s, r2, b2) < (reqs[r][b], r, b))
        assert before == pos


def test_uniform_scores_order_by_rank_then_request():
    reqs = [np.zeros(4) for _ in range(3)]
    pct = [BP.percentiles(s) for s in reqs]
    order = BP.evict_order(pct, 1.0)
    got = [(int(c >> 32), int(c & 0xFFFFFFFF)) for c in order]
    assert got == [(r, b) for b in range(4) for r in range(3)]


def test_evict_count_quarter():
    assert [BP.evict_count(n, 0.25) for n in (1, 3, 4, 5, 144_001)] == [1, 1, 1, 2, 36_001]


def test_topp_count_uses_fp32_product():
    assert BP.topp_count(16, 0.1) == 2
    assert BP.topp_count(64, 0.1) == 7
    assert BP.topp_count(256, 0.1) == 26
    assert BP.topp_count(30, 0.1) == 3      # fp64 0.1*30 would give ceil(3.0000000000000004) = 4
    assert BP.topp_count(5, 0.1) == 1


def test_dirichlet_decay_total_is_geometric():
    # Increments sum to 1 per request per step, so after T steps of
    # score <- 0.98 score + inc from zero, a request's total is (1-0.98^T)/(1-0.98).
    wl = workloads.block_priority(seed=3, R=4, steps=200, min_len=64, max_len=512)
    off = wl.offsets
    score = np.zeros(wl.total_tokens)
    for t in range(wl.steps):
        score = BP.decay_update(score, wl.increments(t), wl.decay)
    want = (1 - 0.98 ** 200) / (1 - 0.98)
    for r in range(wl.R):
        assert abs(score[off[r]:off[r + 1]].sum() - want) < 1e-4     # fp32 increments
    assert abs(want - 49.12060) < 1e-4      # 0.98^200 = 0.0175879...


def test_priority_pass_shapes():
    wl = workloads.block_priority(seed=3, R=5, steps=1, min_len=100, max_len=400)
    tok = wl.increments(0).astype(np.float64)
    blk, normed, order = BP.priority_pass(tok, wl.offsets, 16, BP.AGG_MAX, 0.1,
                                          BP.NORM_PERCENTILE, 0.25)
    N = sum(len(b) for b in blk)
    assert len(order) == math.ceil(0.25 * N)
    assert [len(b) for b in blk] == [int(-(-L // 16)) for L in wl.lengths]
