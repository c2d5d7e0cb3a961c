"""Pins for the SnapKV oracle (CPU only)."""
import math

import numpy as np
import pytest
import torch

import workloads
from oracle import snapkv
from oracle.attention import bf16_bits_to_f64


def test_maxpool_hand_worked(golden):
    rows = list(golden("maxpool_k7.txt"))
    for inp, out in zip(rows[0::2], rows[1::2]):
        x = np.array([float(v) for v in inp[1:]])
        want = [float(v) for v in out[1:]]
        assert snapkv.maxpool1d(x, 7).tolist() == want


def test_single_query_single_head_is_one_softmax_row():
    # W = 1, G = 1: the vote is the last query's softmax restricted to the prefix.
    rng = np.random.default_rng(5)
    S, d = 40, 16
    K = rng.standard_normal((1, S, d))
    q = rng.standard_normal((1, 1, d))
    vote = snapkv.snapkv_vote(q, K, 1 / math.sqrt(d))
    ref = torch.softmax(torch.from_numpy(K[0] @ q[0, 0]) / math.sqrt(d), dim=0).numpy()
    np.testing.assert_allclose(vote[0], ref[:S - 1], rtol=1e-12, atol=1e-15)


@pytest.mark.parametrize("t", [0, 1, 2, 3])
def test_window_queries_are_causal(t):
    # All window queries point along u.  Window key S-W+t is strongly
    # attractive, the other window keys strongly repulsive.  Query i sees the
    # attractive key only if i >= t, so the prefix collects ~t whole rows.
    d, W, P = 8, 4, 16
    S = P + W
    u = np.zeros(d)
    u[0] = 1.0
    rng = np.random.default_rng(9)
    K = np.zeros((1, S, d))
    K[0, :P] = 0.05 * rng.standard_normal((P, d))
    K[0, P:] = -60 * u
    K[0, P + t] = 60 * u
    q = np.tile(u, (1, W, 1))
    vote = snapkv.snapkv_vote(q, K, 1 / math.sqrt(d))
    assert abs(vote.sum() - t) < 1e-6


def test_votes_sum_over_the_query_group():
    # q heads 0,1 (kv 0) favour prefix key 2; q heads 2,3 (kv 1) favour key 6.
    d, W, P = 8, 3, 10
    S = P + W
    e = np.eye(d)
    K = np.zeros((2, S, d))
    K[:, P:] = -60 * (e[0] + e[1])
    K[0, 2] = 60 * e[0]
    K[1, 6] = 60 * e[1]
    q = np.stack([np.tile(e[0], (W, 1))] * 2 + [np.tile(e[1], (W, 1))] * 2)
    vote = snapkv.snapkv_vote(q, K, 1.0)
    assert abs(vote[0, 2] - 2 * W) < 1e-9 and abs(vote[1, 6] - 2 * W) < 1e-9
    assert abs(vote.sum() - 4 * W) < 1e-9


def test_keep_size_and_planted_keys_survive():
    wl = workloads.snapkv_custom(seed=21, L=1, Hq=8, Hkv=2, d=64, S=2048, W=16, keep_k=128,
                                 n_planted=8, plant_amp=16.0)
    lay = wl.layer(0)
    keep, vote, pooled = snapkv.snapkv_select(bf16_bits_to_f64(lay.q_obs), bf16_bits_to_f64(lay.K),
                                              wl.scale, wl.keep_k, 7)
    assert keep.shape == (wl.Hkv, wl.keep_k + wl.W)
    for h in range(wl.Hkv):
        assert np.all(np.diff(keep[h]) > 0)
        assert keep[h, -wl.W:].tolist() == list(range(wl.S - wl.W, wl.S))
        assert set(lay.planted[h].tolist()) <= set(keep[h].tolist())
        # pooling keeps the neighbours of a strong key with it
        assert pooled[h, lay.planted[h][0]] == vote[h, lay.planted[h][0]]


def test_short_prefix_keeps_everything():
    rng = np.random.default_rng(4)
    K = rng.standard_normal((1, 20, 8))
    q = rng.standard_normal((2, 4, 8))
    keep, _, _ = snapkv.snapkv_select(q, K, 0.3, keep_k=64)
    assert keep[0].tolist() == list(range(20))


# ---- cold-start seed ("prefill attention as the seed score") ----

def test_seed_of_each_group_sums_to_its_rows():
    # every observation row is one softmax over the keys it sees: G*W in total
    rng = np.random.default_rng(12)
    K = rng.standard_normal((2, 30, 8))
    q = rng.standard_normal((6, 5, 8))
    seed = snapkv.prefill_seed(q, K, 0.7)
    np.testing.assert_allclose(seed.sum(axis=1), [3 * 5, 3 * 5], rtol=1e-12)


def test_seed_with_zero_queries_is_harmonic():
    # q = 0: row i spreads 1 / (P + i + 1) over keys 0..P+i, so key j collects
    # G * sum_{i : P + i >= j} 1 / (P + i + 1)
    G, W, P, d = 3, 4, 9, 8
    S = P + W
    rng = np.random.default_rng(2)
    K = rng.standard_normal((1, S, d))
    seed = snapkv.prefill_seed(np.zeros((G, W, d)), K, 1.0)[0]
    want = [G * sum(1.0 / (P + i + 1) for i in range(W) if P + i >= j) for j in range(S)]
    np.testing.assert_allclose(seed, want, rtol=1e-12)


def test_seed_on_the_prefix_is_the_vote():
    # the row-by-row vote and the masked-matrix seed are separate code paths
    rng = np.random.default_rng(13)
    K = rng.standard_normal((2, 50, 16))
    q = rng.standard_normal((4, 7, 16))
    seed = snapkv.prefill_seed(q, K, 0.25)
    vote = snapkv.snapkv_vote(q, K, 0.25)
    np.testing.assert_allclose(seed[:, :43], vote, rtol=1e-12, atol=1e-15)


@pytest.mark.parametrize("t", [0, 2, 3])
def test_seed_of_a_window_key_counts_only_later_rows(t):
    # window key P+t is strongly attractive: rows i >= t put ~all their weight
    # on it, rows i < t cannot see it; two q heads share the kv head
    d, W, P = 8, 4, 16
    S = P + W
    u = np.zeros(d)
    u[0] = 1.0
    rng = np.random.default_rng(3)
    K = np.zeros((1, S, d))
    K[0, :P] = 0.05 * rng.standard_normal((P, d))
    K[0, P:] = -60 * u
    K[0, P + t] = 60 * u
    q = np.tile(u, (2, W, 1))
    seed = snapkv.prefill_seed(q, K, 1 / math.sqrt(d))[0]
    assert abs(seed[P + t] - 2 * (W - t)) < 1e-6
    assert abs(seed[:P].sum() - 2 * t) < 1e-6


# ---- GQA union of per-head picks ----

def test_per_head_votes_add_up_to_the_group_vote():
    rng = np.random.default_rng(14)
    K = rng.standard_normal((2, 40, 8))
    q = rng.standard_normal((8, 6, 8))
    vh = snapkv.snapkv_vote_per_head(q, K, 0.5)
    vg = snapkv.snapkv_vote(q, K, 0.5)
    np.testing.assert_allclose(vh.reshape(2, 4, -1).sum(axis=1), vg, rtol=1e-12)


def test_union_keeps_every_heads_favourite():
    # one kv head, two q heads: head 0 looks along e0 (key 3 answers), head 1
    # along e1 (key 11 answers, more strongly).  One pick per head: the summed
    # vote keeps only key 11, the union keeps both.
    d, W, P = 8, 2, 16
    S = P + W
    e = np.eye(d)
    K = np.zeros((1, S, d))
    K[0, 3] = 30 * e[0]
    K[0, 11] = 40 * e[1]
    K[0, P:] = -60 * (e[0] + e[1])
    q = np.stack([np.tile(e[0], (W, 1)), np.tile(e[1], (W, 1))])
    keep, vote, _ = snapkv.snapkv_select_union(q, K, 1.0, keep_k=1, kernel=1)
    assert keep[0].tolist() == [3, 11, P, P + 1]
    assert vote[0].argmax() == 3 and vote[1].argmax() == 11
    keep_sum, _, _ = snapkv.snapkv_select(q, K, 1.0, keep_k=1, kernel=1)
    assert keep_sum[0].tolist() == [11, P, P + 1]


def test_union_with_one_q_head_per_group_is_the_summed_selection():
    rng = np.random.default_rng(15)
    K = rng.standard_normal((3, 200, 16))
    q = rng.standard_normal((3, 8, 16))
    keep_u, _, _ = snapkv.snapkv_select_union(q, K, 0.4, keep_k=20)
    keep_s, _, _ = snapkv.snapkv_select(q, K, 0.4, keep_k=20)
    for h in range(3):
        assert keep_u[h].tolist() == keep_s[h].tolist()


def test_union_size_and_order():
    rng = np.random.default_rng(16)
    G, W, S, k = 4, 8, 300, 25
    K = rng.standard_normal((1, S, 16))
    q = rng.standard_normal((G, W, 16))
    keep, _, pooled = snapkv.snapkv_select_union(q, K, 0.4, keep_k=k)
    u = keep[0]
    assert np.all(np.diff(u) > 0)
    assert u[-W:].tolist() == list(range(S - W, S))
    assert k <= len(u) - W <= G * k
    for g in range(G):
        assert set(np.argsort(-pooled[g], kind="stable")[:k].tolist()) <= set(u.tolist())
