"""DSA-style sparse decode and the Quest page bound (fp64).  Test only.

Follows "Long context, KV eviction and sparse attention":
  * DSA paragraph: a light indexer with few heads scores every past token;
    each query then runs full attention over only its 2048 best-scored
    tokens.  The indexer score read here is the ReLU-weighted dot
    I[s] = sum_j w_j * ReLU(q^I_j . k^I_s) over the indexer heads j, with
    one shared indexer key per token and one selected set per (sequence,
    step) shared by every q head; bf16 inputs, not FP8.
  * sparse-selection section: restricting a query to a selected set means
    masking every other logit to -inf before the softmax; "exact top-k" keeps
    each query's k largest logits; Quest bounds a page's logit by
    sum_d max(q_d * kmin_d, q_d * kmax_d) and keeps the best pages.
Ties in a top-k go to the lower position; the selected set is reported in
ascending order; with S <= k every position is selected.

Quest as a decode-time selector (the same section's listing, read for what it
computes): per q head, every full page of its kv head gets the bound; the
budget_pages pages with the largest bounds (ties to the lower page; every
full page when there are no more than that) are attended, together with the
trailing partial page, which is always attended; the query is the last
token, so every page is causally visible.  Page minima and maxima are
elementwise over the page's tokens (over its valid tokens for the partial
page, whose bound is never used).
"""
from __future__ import annotations

import numpy as np

from .attention import softmax
from .h2o import topk_positions


def indexer_scores(q_idx: np.ndarray, w: np.ndarray, k_idx: np.ndarray) -> np.ndarray:
    """I[s] = sum_j w[j] * max(0, q_idx[j] . k_idx[s]).  q_idx [Hi][Di], k_idx [S][Di]."""
    dots = k_idx @ q_idx.T                  # [S][Hi]
    return np.maximum(dots, 0.0) @ w


def select_topk(I: np.ndarray, k: int) -> np.ndarray:
    return topk_positions(I, k)


def masked_attention(q: np.ndarray, K: np.ndarray, V: np.ndarray, sel: np.ndarray, scale: float):
    """Attention of every q head over the selected positions only.

    q [Hq][d]; K, V [Hkv][S][d]; sel: ascending positions shared by all heads.
    Returns o [Hq][d].
    """
    Hq, d = q.shape
    Hkv = K.shape[0]
    G = Hq // Hkv
    o = np.zeros((Hq, d))
    for h in range(Hq):
        kvh = h // G
        p = softmax((K[kvh, sel] @ q[h]) * scale)
        o[h] = p @ V[kvh, sel]
    return o


def sparse_decode_step(q, K, V, q_idx, w, k_idx, top_k, scale):
    """Indexer scores -> top-k -> attention over the selection.  Returns (o, sel, I)."""
    I = indexer_scores(q_idx, w, k_idx)
    sel = select_topk(I, top_k)
    return masked_attention(q, K, V, sel, scale), sel, I


def quest_page_bound(q: np.ndarray, K: np.ndarray, page: int = 16) -> np.ndarray:
    """Upper bound of q.k over each full page of K [S][d].

    The sparse-selection section bounds a query's logit against any key of a
    page by taking, in every dimension, the larger of q_d times the page's
    smallest and q_d times its largest value of that dimension:
        bound[p] = sum_d max(q_d * min_t K[t, d], q_d * max_t K[t, d])
    over the page's tokens t.  Only full pages (S // page of them) get one.
    """
    S, d = K.shape
    bounds = np.zeros(S // page)
    for p in range(S // page):
        tokens = K[p * page:(p + 1) * page]          # the page's keys, [page][d]
        lo = tokens.min(axis=0)                      # per-dimension minimum
        hi = tokens.max(axis=0)                      # per-dimension maximum
        bounds[p] = np.sum(np.maximum(q * lo, q * hi))
    return bounds


def page_minmax(K: np.ndarray, page: int = 16):
    """Elementwise min and max over each page of K [S][d] -> (kmin, kmax), [ceil(S/page)][d] each."""
    S, d = K.shape
    n = -(-S // page)
    kmin = np.empty((n, d))
    kmax = np.empty((n, d))
    for p in range(n):
        rows = K[p * page:min(S, (p + 1) * page)]
        kmin[p] = rows.min(axis=0)
        kmax[p] = rows.max(axis=0)
    return kmin, kmax


def quest_select_pages(bounds: np.ndarray, budget_pages: int) -> np.ndarray:
    """Full pages attended by one q head: the budget_pages largest bounds, ascending."""
    return topk_positions(bounds, budget_pages)


def quest_decode_step(q, K, V, budget_pages, scale, page=16):
    """One decode step with Quest page selection per q head.

    q [Hq][d]; K, V [Hkv][S][d] (the new token included).  Returns (o [Hq][d],
    chosen pages per q head (list of ascending arrays), bounds [Hq][S // page]).
    """
    Hq, d = q.shape
    Hkv, S, _ = K.shape
    G = Hq // Hkv
    n_full = S // page
    o = np.zeros((Hq, d))
    chosen = []
    bounds = np.zeros((Hq, n_full))
    for h in range(Hq):
        kvh = h // G
        bounds[h] = quest_page_bound(q[h], K[kvh], page)
        pages = quest_select_pages(bounds[h], budget_pages)
        chosen.append(pages)
        tokens = np.concatenate([np.arange(p * page, (p + 1) * page) for p in pages] +
                                [np.arange(n_full * page, S)]).astype(np.int64)
        w = softmax((K[kvh, tokens] @ q[h]) * scale)
        o[h] = w @ V[kvh, tokens]
    return o, chosen, bounds
