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
