"""Pins for the DSA sparse-decode and Quest oracle (CPU only)."""
import math

import numpy as np
import pytest
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


# ---- Quest page selection in a decode step ----

def test_quest_decode_hand_worked(golden):
    rows = {r[0]: [float(x) for x in r[1:]] for r in golden("quest_decode.txt")}
    K = np.array(rows["k"]).reshape(1, 5, 2)
    q = np.array([rows["q0"], rows["q1"]])
    V = np.arange(10, dtype=np.float64).reshape(1, 5, 2)
    o, chosen, bounds = dsa.quest_decode_step(q, K, V, budget_pages=1, scale=0.5, page=2)
    assert bounds.tolist() == [rows["bounds0"], rows["bounds1"]]
    assert [c.tolist() for c in chosen] == [[0], [1]]
    for h in range(2):
        toks = np.array(rows[f"tokens{h}"], dtype=np.int64)
        w = np.exp(0.5 * (K[0, toks] @ q[h]))
        np.testing.assert_allclose(o[h], (w / w.sum()) @ V[0, toks], rtol=1e-12)


@pytest.mark.parametrize("S", [7, 16, 100, 160])
def test_quest_with_every_page_in_budget_is_full_attention(S):
    rng = np.random.default_rng(S)
    q = rng.standard_normal((4, 32))
    K, V = rng.standard_normal((2, S, 32)), rng.standard_normal((2, S, 32))
    o, chosen, _ = dsa.quest_decode_step(q, K, V, budget_pages=S // 16 + 1, scale=0.2)
    full, _ = decode_attention(q, K, V, 0.2)
    np.testing.assert_allclose(o, full, rtol=1e-12, atol=1e-14)
    assert all(c.tolist() == list(range(S // 16)) for c in chosen)


def test_quest_bound_is_tight_on_a_constant_page():
    rng = np.random.default_rng(3)
    k = rng.standard_normal(16)
    K = np.tile(k, (32, 1))
    K[16:] = rng.standard_normal((16, 16))
    q = rng.standard_normal(16)
    assert abs(dsa.quest_page_bound(q, K, 16)[0] - q @ k) < 1e-12


def test_page_minmax_attained_per_dimension():
    rng = np.random.default_rng(4)
    K = rng.standard_normal((37, 8))                  # two full pages and 5 tokens
    kmin, kmax = dsa.page_minmax(K, 16)
    assert kmin.shape == (3, 8)
    for p, (a, b) in enumerate([(0, 16), (16, 32), (32, 37)]):
        rows = K[a:b]
        assert np.all(rows >= kmin[p]) and np.all(rows <= kmax[p])
        for d in range(8):
            assert kmin[p, d] in rows[:, d] and kmax[p, d] in rows[:, d]


def test_quest_heads_choose_alone_and_keep_the_partial_page():
    # one kv head, two q heads looking along opposite directions: each keeps
    # the page its own direction favours; both keep the partial page
    d = 8
    e = np.eye(d)
    K = np.zeros((1, 16 * 4 + 3, d))
    K[0, 16 * 1 + 5] = 10 * e[0]
    K[0, 16 * 3 + 2] = -10 * e[0]
    q = np.stack([e[0], -e[0]])
    V = np.random.default_rng(5).standard_normal(K.shape)
    _, chosen, bounds = dsa.quest_decode_step(q, K, V, budget_pages=1, scale=1.0)
    assert chosen[0].tolist() == [1] and chosen[1].tolist() == [3]
    assert bounds.shape == (2, 4)
