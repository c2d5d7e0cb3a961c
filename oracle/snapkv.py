"""SnapKV prefill selection (fp64).  Test infrastructure only.

Follows "From sliding window to attention-guided eviction" §4.3, step by step:
  (2) take the attention weights of the last W prompt queries (the
      observation window) over the prefix positions;
  (3) per head, sum those weights over the W queries (the vote);
  (4) smooth the vote with a 1D max-pool of kernel 7;
  (5) keep each head's top-k voted positions plus the window itself.
With GQA the kept KV is shared by the q heads of a group; the reading used
here sums the votes of the G q heads of a kv head before pooling (the
per-kv-head "sum-pool"), so there is one keep-set per kv head.

Readings where the page is silent: window query i (0-based) sits at position
S - W + i and sees keys 0..S-W+i (causal); only prefix keys j < S - W get
votes; the pool has stride 1, is clipped at the prefix edges (as if padded
with -inf) and returns one value per prefix position; ties go to the lower
position.

Two variants from the same page:
  * GQA union (§4.3, "KV sharing under GQA"): each q head scores and picks its
    own top-k from its own (pooled) vote, and the kept KV of a kv head is the
    union of its G heads' picks, plus the window.
  * Cold-start seed (§2.3, the third option, "prefill attention as the seed
    score"): the reading used here seeds each kept key's accumulated score
    with the attention the observation window gave it -- summed over the G*W
    rows like the vote, but over every key, window keys included (causally).
    That is exactly the H2O accumulator the kv head would hold had the last W
    prompt tokens been decoded one at a time with the same queries.
"""
from __future__ import annotations

import numpy as np

from .attention import softmax
from .h2o import topk_positions


def snapkv_vote(q_obs: np.ndarray, K: np.ndarray, scale: float) -> np.ndarray:
    """Vote per kv head over the prefix.  q_obs: [Hq][W][d], K: [Hkv][S][d]."""
    Hq, W, _ = q_obs.shape
    Hkv, S, _ = K.shape
    G = Hq // Hkv
    P = S - W
    vote = np.zeros((Hkv, P))
    for h in range(Hq):
        kvh = h // G
        for i in range(W):
            qpos = P + i
            w = softmax((K[kvh, :qpos + 1] @ q_obs[h, i]) * scale)
            vote[kvh] += w[:P]
    return vote


def snapkv_vote_per_head(q_obs: np.ndarray, K: np.ndarray, scale: float) -> np.ndarray:
    """Vote of every q head over the prefix (no sum over the group).  -> [Hq][S-W]."""
    Hq, W, _ = q_obs.shape
    Hkv, S, _ = K.shape
    G = Hq // Hkv
    P = S - W
    vote = np.zeros((Hq, P))
    for h in range(Hq):
        for i in range(W):
            w = softmax((K[h // G, :P + i + 1] @ q_obs[h, i]) * scale)
            vote[h] += w[:P]
    return vote


def prefill_seed(q_obs: np.ndarray, K: np.ndarray, scale: float) -> np.ndarray:
    """Cold-start seed of every key 0..S-1 per kv head.  -> [Hkv][S].

    Written as a masked matrix (W x S causal logits per q head, one softmax
    per row, column sums) rather than row by row like the vote, so that the
    two can be checked against each other on the prefix.
    """
    Hq, W, _ = q_obs.shape
    Hkv, S, _ = K.shape
    G = Hq // Hkv
    P = S - W
    visible = np.arange(S)[None, :] <= (P + np.arange(W))[:, None]   # [W][S]
    seed = np.zeros((Hkv, S))
    for h in range(Hq):
        logits = np.where(visible, (q_obs[h] @ K[h // G].T) * scale, -np.inf)
        seed[h // G] += softmax(logits).sum(axis=0)
    return seed


def maxpool1d(x: np.ndarray, kernel: int = 7) -> np.ndarray:
    """Stride-1 max-pool, window [j - kernel//2, j + kernel//2] clipped to the array."""
    n = x.shape[-1]
    half = kernel // 2
    out = np.empty_like(x)
    for j in range(n):
        out[..., j] = np.max(x[..., max(0, j - half):min(n, j + half + 1)], axis=-1)
    return out


def snapkv_keep(pooled_row: np.ndarray, S: int, W: int, keep_k: int) -> np.ndarray:
    """Top-keep_k prefix positions by pooled vote, then the window (ascending)."""
    hh = topk_positions(pooled_row, keep_k)
    return np.concatenate([hh, np.arange(S - W, S)]).astype(np.int64)


def snapkv_select(q_obs, K, scale, keep_k, kernel=7):
    """Full per-layer selection: returns (keep [Hkv][n], vote [Hkv][S-W], pooled)."""
    Hkv, S, _ = K.shape
    W = q_obs.shape[1]
    vote = snapkv_vote(q_obs, K, scale)
    pooled = maxpool1d(vote, kernel)
    keep = np.stack([snapkv_keep(pooled[h], S, W, keep_k) for h in range(Hkv)])
    return keep, vote, pooled


def snapkv_union_keep(pooled_heads: np.ndarray, S: int, W: int, keep_k: int) -> np.ndarray:
    """Union of the top-keep_k picks of a group's q heads, then the window, ascending."""
    picks = set()
    for row in pooled_heads:
        picks.update(topk_positions(row, keep_k).tolist())
    return np.concatenate([np.array(sorted(picks), dtype=np.int64),
                           np.arange(S - W, S)]).astype(np.int64)


def snapkv_select_union(q_obs, K, scale, keep_k, kernel=7):
    """Per-head selection, union per kv head: (list of keep arrays, per-head vote, pooled)."""
    Hq, W, _ = q_obs.shape
    Hkv, S, _ = K.shape
    G = Hq // Hkv
    vote = snapkv_vote_per_head(q_obs, K, scale)
    pooled = maxpool1d(vote, kernel)
    keep = [snapkv_union_keep(pooled[h * G:(h + 1) * G], S, W, keep_k) for h in range(Hkv)]
    return keep, vote, pooled
