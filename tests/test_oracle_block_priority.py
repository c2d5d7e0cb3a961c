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


# --- temporal aggregation variants and block policies -----------------------


def test_window_sum_closed_forms():
    # constant attention c every step: the window holds min(steps, W) copies
    for W in range(1, 5):
        for steps in range(1, 9):
            got = BP.window_sum([np.full(3, 0.25)] * steps, W)
            np.testing.assert_array_equal(got, np.full(3, 0.25 * min(steps, W)))
    # hand example: increments 1, 2, 3, 4 -> last two sum to 7; a window longer
    # than the history sums everything
    seq = [np.array([float(x)]) for x in (1, 2, 3, 4)]
    assert BP.window_sum(seq, 2)[0] == 7.0
    assert BP.window_sum(seq, 10)[0] == 10.0
    assert BP.window_sum(seq, 1)[0] == 4.0


def test_window_ring_recurrence_equals_window_sum_exactly():
    # the kernel's update (score += inc - history[step % W]; history[...] = inc,
    # history and score starting at zero) reproduces the window sum; checked in
    # exact rational arithmetic on a random sequence
    rng = np.random.default_rng(7)
    W, steps = 3, 11
    incs = [rng.integers(0, 100, 5) for _ in range(steps)]
    score = [Fraction(0)] * 5
    hist = [[Fraction(0)] * 5 for _ in range(W)]
    for t, inc in enumerate(incs):
        for j in range(5):
            score[j] += Fraction(int(inc[j])) - hist[t % W][j]
            hist[t % W][j] = Fraction(int(inc[j]))
        want = BP.window_sum([x.astype(np.float64) for x in incs[:t + 1]], W)
        assert [float(x) for x in score] == list(want)


def test_max_update_keeps_the_peak():
    s = np.zeros(3)
    for inc in ([1.0, -2.0, 0.5], [5.0, -3.0, 0.25], [3.0, -1.0, 0.75]):
        s = BP.max_update(s, np.array(inc))
    np.testing.assert_array_equal(s, [5.0, 0.0, 0.75])   # the zero start stays the floor


def test_fraction_of_hot_tokens():
    blk = np.array([0.1, 0.5, 0.9, 0.5, 0.2])
    # block size 4: [0.1 .5 .9 .5] has 3 of 4 at >= 0.5; the partial block [0.2] has none
    np.testing.assert_array_equal(BP.block_scores(blk, 4, BP.AGG_FRAC_HOT, threshold=0.5), [0.75, 0.0])
    np.testing.assert_array_equal(BP.block_scores(blk, 4, BP.AGG_FRAC_HOT, threshold=-1.0), [1.0, 1.0])
    np.testing.assert_array_equal(BP.block_scores(blk, 4, BP.AGG_FRAC_HOT, threshold=2.0), [0.0, 0.0])
    # 1 of 3 is an fp32 division
    assert BP.block_scores(np.array([1.0, 0.0, 0.0]), 3, BP.AGG_FRAC_HOT, threshold=0.5)[0] == \
        np.float64(np.float32(1) / np.float32(3))


def test_all_cold_evicts_only_cold_blocks():
    # request 0 blocks (block size 2): maxes 0.2, 0.9, 0.1; request 1: 0.4, 0.6
    tok = np.array([0.2, 0.1, 0.9, 0.3, 0.0, 0.1, 0.4, 0.4, 0.6, 0.0])
    off = np.array([0, 6, 10])
    blocks, normed, order = BP.priority_pass(tok, off, 2, BP.AGG_ALL_COLD, 0.1, BP.NORM_NONE, 1.0,
                                             threshold=0.5)
    np.testing.assert_array_equal(blocks[0], [0.2, 0.9, 0.1])
    # cold blocks only, by max ascending: (0, 2) 0.1, (0, 0) 0.2, (1, 0) 0.4
    np.testing.assert_array_equal(order, [(0 << 32) | 2, (0 << 32) | 0, (1 << 32) | 0])
    # evict_frac 0.2 of N = 5 blocks -> ceil(1.0) = 1: the coldest only
    _, _, order = BP.priority_pass(tok, off, 2, BP.AGG_ALL_COLD, 0.1, BP.NORM_NONE, 0.2, threshold=0.5)
    np.testing.assert_array_equal(order, [(0 << 32) | 2])
    # a threshold below every score leaves nothing evictable
    _, _, order = BP.priority_pass(tok, off, 2, BP.AGG_ALL_COLD, 0.1, BP.NORM_NONE, 1.0, threshold=-1.0)
    assert order.shape == (0,)
