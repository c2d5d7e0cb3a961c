"""Property checks of the oracle over random small shapes (CPU only).

Each property holds by the mathematics, independently of how the oracle
computes it, so a dropped term, a wrong mask or a reversed tie order fails
one of them.
"""
import math

import numpy as np
import pytest

hyp = pytest.importorskip("hypothesis")
from hypothesis import given, settings, strategies as st  # noqa: E402

from oracle import block_signal, dsa, snapkv  # noqa: E402
from oracle.attention import decode_attention  # noqa: E402
from oracle.h2o import topk_positions  # noqa: E402

SETTINGS = settings(max_examples=40, deadline=None)


@SETTINGS
@given(st.lists(st.integers(0, 4), min_size=1, max_size=40), st.integers(1, 45))
def test_topk_is_the_lexicographic_prefix(vals, k):
    # k largest by value, ties to the lower index, reported ascending
    x = np.array(vals, dtype=np.float64)
    want = sorted(sorted(range(len(x)), key=lambda i: (-x[i], i))[:k])
    assert topk_positions(x, k).tolist() == want


@SETTINGS
@given(st.lists(st.floats(-5, 5), min_size=1, max_size=30), st.sampled_from([1, 3, 5, 7]))
def test_maxpool_is_the_clipped_window_max(vals, kernel):
    x = np.array(vals)
    out = snapkv.maxpool1d(x, kernel)
    h = kernel // 2
    for j in range(len(x)):
        assert out[j] == max(x[max(0, j - h):j + h + 1])
        assert out[j] >= x[j]


@SETTINGS
@given(st.integers(0, 10_000), st.integers(1, 3), st.integers(1, 3), st.integers(1, 6), st.integers(1, 12))
def test_seed_and_votes_are_window_attention(seed, Hkv, G, W, P):
    rng = np.random.default_rng(seed)
    d = 8
    S = P + W
    K = rng.standard_normal((Hkv, S, d))
    q = rng.standard_normal((Hkv * G, W, d))
    sd = snapkv.prefill_seed(q, K, 0.7)
    vh = snapkv.snapkv_vote_per_head(q, K, 0.7)
    np.testing.assert_allclose(sd.sum(axis=1), G * W, rtol=1e-12)            # one softmax per row
    np.testing.assert_allclose(sd[:, :P], vh.reshape(Hkv, G, P).sum(axis=1), rtol=1e-10, atol=1e-15)
    assert np.all(sd >= 0)
    # window key P + i is seen by rows i..W-1 only: a bound by row count
    for i in range(W):
        assert np.all(sd[:, P + i] <= G * (W - i) + 1e-12)


@SETTINGS
@given(st.integers(0, 10_000), st.integers(1, 4), st.integers(1, 12), st.integers(1, 5))
def test_union_contains_each_heads_picks(seed, G, P, keep_k):
    rng = np.random.default_rng(seed)
    W, d = 3, 8
    K = rng.standard_normal((1, P + W, d))
    q = rng.standard_normal((G, W, d))
    keep, vote, pooled = snapkv.snapkv_select_union(q, K, 0.5, keep_k, kernel=3)
    u = keep[0]
    assert np.all(np.diff(u) > 0)
    assert u[-W:].tolist() == list(range(P, P + W))
    picks = set()
    for g in range(G):
        picks |= set(topk_positions(pooled[g], keep_k).tolist())
    assert set(u[:-W].tolist()) == picks
    assert min(keep_k, P) <= len(picks) <= min(G * keep_k, P)


@SETTINGS
@given(st.integers(0, 10_000), st.integers(1, 40), st.integers(1, 4))
def test_quest_bound_covers_every_logit_and_is_tight_on_one_key_pages(seed, n_pages, page):
    rng = np.random.default_rng(seed)
    d = 6
    q = rng.standard_normal(d)
    K = rng.standard_normal((n_pages * page, d))
    ub = dsa.quest_page_bound(q, K, page)
    logits = (K @ q).reshape(n_pages, page)
    assert np.all(ub >= logits.max(axis=1) - 1e-12)
    if page == 1:
        np.testing.assert_allclose(ub, logits[:, 0], rtol=1e-12, atol=1e-12)


@SETTINGS
@given(st.integers(0, 10_000), st.integers(1, 3), st.integers(1, 4), st.integers(1, 70), st.integers(1, 9))
def test_block_masses_split_the_heads_attention(seed, Hkv, G, S, k):
    rng = np.random.default_rng(seed)
    d = 8
    q = rng.standard_normal((Hkv * G, d))
    K, V = rng.standard_normal((Hkv, S, d)), rng.standard_normal((Hkv, S, d))
    _, p = decode_attention(q, K, V, 1 / math.sqrt(d))
    m = block_signal.block_masses(p)
    assert len(m) == -(-S // 16)
    assert abs(m.sum() - Hkv * G) < 1e-9
    chosen = block_signal.top_blocks(m, k)
    rest = np.setdiff1d(np.arange(len(m)), chosen)
    if len(rest):
        assert m[chosen].min() >= m[rest].max()
