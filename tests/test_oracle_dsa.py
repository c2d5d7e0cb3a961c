"""Pins for the DSA sparse-decode and Quest oracle (CPU only)."""
import math

import numpy as np
import torch

from oracle import dsa
from oracle.attention import decode_attention


def test_indexer_hand_worked(golden):
    rows = list(golden("indexer_d2.txt"))
    q = np.array([float(x) for x in rows[0][1:]]).reshape(2, 2)
    k = np.array([float(x) for x in rows[1][1:]]).reshape(-1, 2)
    for wrow, irow in zip(rows[2::2], rows[3::2]):
        w = np.array([float(x) for x in wrow[1:]])
        want = [float(x) for x in irow[1:]]
        assert dsa.indexer_scores(q, w, k).tolist() == want


def test_short_context_selects_everything_and_equals_dense():
    rng = np.random.default_rng(2)
    Hq, Hkv, S, d = 8, 2, 50, 16
    q, K, V = rng.standard_normal((Hq, d)), rng.standard_normal((Hkv, S, d)), rng.standard_normal((Hkv, S, d))
    o, sel, _ = dsa.sparse_decode_step(q, K, V, rng.standard_normal((4, 8)), rng.standard_normal(4),
                                       rng.standard_normal((S, 8)), top_k=64, scale=0.25)
    assert sel.tolist() == list(range(S))
    np.testing.assert_allclose(o, decode_attention(q, K, V, 0.25)[0], rtol=1e-13, atol=1e-14)


def test_exact_topk_logits_equal_masked_softmax():
    # Feeding the exact logits as the indexer (one head, G = 1) gives the
    # handbook's "exact top-k" selection: mask all but the k best logits to
    # -inf, softmax, multiply by V (checked with torch ops in fp64).
    rng = np.random.default_rng(3)
    S, d, k = 200, 16, 24
    q, K, V = rng.standard_normal((1, d)), rng.standard_normal((1, S, d)), rng.standard_normal((1, S, d))
    logits = K[0] @ q[0]
    sel = dsa.select_topk(logits, k)
    o = dsa.masked_attention(q, K, V, sel, 1 / math.sqrt(d))
    lt = torch.from_numpy(logits) / math.sqrt(d)
    mask = torch.zeros(S, dtype=torch.bool)
    mask[lt.topk(k).indices] = True
    ref = lt.masked_fill(~mask, float("-inf")).softmax(-1) @ torch.from_numpy(V[0])
    np.testing.assert_allclose(o[0], ref.numpy(), rtol=1e-12, atol=1e-14)


def test_quest_hand_worked_and_is_an_upper_bound(golden):
    rows = list(golden("quest_bound.txt"))
    q = np.array([float(x) for x in rows[0][1:]])
    K = np.array([float(x) for x in rows[1][1:]]).reshape(-1, 2)
    assert dsa.quest_page_bound(q, K, page=2).tolist() == [float(rows[2][1])]
    rng = np.random.default_rng(8)
    q, K = rng.standard_normal(32), rng.standard_normal((160, 32))
    ub = dsa.quest_page_bound(q, K, 16)
    true_max = (K @ q).reshape(10, 16).max(1)
    assert np.all(ub >= true_max - 1e-12)
