"""H2O heavy-hitter eviction with StreamingLLM sinks + window (fp64).  Test only.

Follows "From sliding window to attention-guided eviction":
  §4.1  StreamingLLM keeps the first 4 positions (sinks) and the most recent
        W positions, everything in between is dropped;
  §4.2  H2O keeps sinks + the top-(budget - sinks - window) tokens by
        cumulative attention among the non-locked middle + the recent window,
        and evicts the rest, every decode step (the pseudocode's loop body:
        accumulate, top-k over the middle slice, build the evict mask, evict).
and "Long context, KV eviction and sparse attention" (StreamingLLM section):
the recent-only rule keeps the last ``budget`` positions, the sink+window rule
keeps ``range(sinks)`` plus the last ``budget - sinks`` positions.

Readings where the pages are silent (all listed in the design notes):
  * the middle slice in the pseudocode returns slice-relative indices; the
    selected slots are those indices plus ``n_sink``;
  * ties at equal score go to the lower slot;
  * the new token is appended before attention and counts in the window;
  * eviction runs only when the live length exceeds the budget.
"""
from __future__ import annotations

import numpy as np

from .attention import decode_attention, h2o_accumulate


def topk_positions(scores: np.ndarray, k: int) -> np.ndarray:
    """Indices of the k largest scores, ties to the lower index, ascending order."""
    scores = np.asarray(scores)
    n = scores.shape[0]
    k = min(k, n)
    if k <= 0:
        return np.zeros(0, dtype=np.int64)
    idx = np.arange(n)
    order = np.lexsort((idx, -scores.astype(np.float64)))   # by score desc, then index asc
    return np.sort(order[:k])


def h2o_keep(cum_row: np.ndarray, S: int, budget: int, n_sink: int, window: int) -> np.ndarray:
    """Slots kept for one kv head of one sequence (ascending).

    If S <= budget nothing is evicted.  Otherwise keep = [0, n_sink) union
    HH union [S - window, S), where HH holds the (budget - n_sink - window)
    slots of [n_sink, S - window) with the largest cumulative score.
    """
    if S <= budget:
        return np.arange(S, dtype=np.int64)
    k = budget - n_sink - window
    if k < 0:
        raise ValueError("budget must cover sinks + window")
    middle = np.asarray(cum_row[n_sink:S - window])
    hh = topk_positions(middle, k) + n_sink
    keep = np.concatenate([np.arange(n_sink), hh, np.arange(S - window, S)]).astype(np.int64)
    return keep


def streaming_keep(S: int, budget: int, n_sink: int) -> np.ndarray:
    """StreamingLLM (§4.1 / handbook listing): sinks + the last budget - sinks slots."""
    if S <= budget:
        return np.arange(S, dtype=np.int64)
    return np.concatenate([np.arange(n_sink), np.arange(S - (budget - n_sink), S)]).astype(np.int64)


class H2OSequence:
    """One sequence's per-layer cache state, stepped literally as the pseudocode.

    K, V: [Hkv][S][d] fp64 in slot order; cum: [Hkv][S]; pos: [Hkv][S] the
    original token position held in each slot.  All kv heads always hold the
    same number of slots (the budget applies per kv head).
    """

    def __init__(self, K: np.ndarray, V: np.ndarray):
        self.K = np.array(K, dtype=np.float64)
        self.V = np.array(V, dtype=np.float64)
        Hkv, S, _ = self.K.shape
        self.cum = np.zeros((Hkv, S))
        self.pos = np.tile(np.arange(S, dtype=np.int64), (Hkv, 1))
        self.seen = S

    @property
    def S(self) -> int:
        return self.K.shape[1]

    def append(self, k_new: np.ndarray, v_new: np.ndarray) -> None:
        Hkv = self.K.shape[0]
        self.K = np.concatenate([self.K, k_new[:, None, :]], axis=1)
        self.V = np.concatenate([self.V, v_new[:, None, :]], axis=1)
        self.cum = np.concatenate([self.cum, np.zeros((Hkv, 1))], axis=1)
        self.pos = np.concatenate([self.pos, np.full((Hkv, 1), self.seen, dtype=np.int64)], axis=1)
        self.seen += 1

    def attend(self, q: np.ndarray, scale: float):
        o, p = decode_attention(q, self.K, self.V, scale)
        self.cum = h2o_accumulate(self.cum, p)
        return o, p

    def select(self, budget: int, n_sink: int, window: int) -> np.ndarray:
        """Kept slots per kv head, [Hkv][n_keep]."""
        return np.stack([h2o_keep(self.cum[h], self.S, budget, n_sink, window)
                         for h in range(self.K.shape[0])])

    def apply_keep(self, keep: np.ndarray) -> None:
        """Evict every slot not in ``keep`` (per kv head), preserving slot order."""
        Hkv = self.K.shape[0]
        self.K = np.stack([self.K[h, keep[h]] for h in range(Hkv)])
        self.V = np.stack([self.V[h, keep[h]] for h in range(Hkv)])
        self.cum = np.stack([self.cum[h, keep[h]] for h in range(Hkv)])
        self.pos = np.stack([self.pos[h, keep[h]] for h in range(Hkv)])

    def step(self, q, k_new, v_new, scale, budget, n_sink, window, evict=True):
        """Append, attend, accumulate, select and (optionally) evict.

        Returns (o, p, keep) where keep is the kept-slot array (pre-eviction
        slot indices) or None when nothing was evicted.
        """
        self.append(k_new, v_new)
        o, p = self.attend(q, scale)
        keep = None
        if self.S > budget:
            keep = self.select(budget, n_sink, window)
            if evict:
                self.apply_keep(keep)
        return o, p, keep
