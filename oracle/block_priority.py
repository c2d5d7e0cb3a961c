"""Block offload priority from token scores (fp64; fp32 where fixed).  Test only.

Follows "Sparse attention x KV-cache offloading: eight questions":
  §2.1  temporal aggregation - exponential decay: every step the old score is
        multiplied by the decay factor and the step's attention is added;
        max pooling over steps: the score is the largest attention any step
        gave the token; sliding-window average: the mean of the last W steps'
        attention (kept here as the window sum, which orders the same);
  §3.1  token -> block aggregation: the block's max, its mean, or its top-p%
        (read as: the mean of the ceil(p * n) largest token scores of the
        block's n valid tokens, with p * n evaluated as an fp32 product);
  §3.2  cross-request normalisation by each request's own percentile (read
        as: rank r of the block inside its request by (score asc, block asc),
        percentile = fp32(2r + 1) / fp32(2n), one correctly rounded fp32
        division) or no normalisation (raw block score);
  §5.1  an fp32 score accumulator per block.
"From sliding window to attention-guided eviction" §5.1 (block-level
degradation of token policies):
  - order blocks by their fraction of important tokens, lowest first (read
    as: the fraction of the block's valid tokens whose score is >= a
    threshold, fp32(count) / fp32(n));
  - evict only all-cold blocks (read as: a block may be evicted only when
    all its tokens score below the threshold, i.e. its max is below it; the
    evictable blocks keep the max-aggregation order and the evict count is
    capped by how many there are).
The global evict order sorts every block of every request by (normalised
score asc, request asc, block asc) and emits the first ceil(frac * N).
A partial last block aggregates its valid tokens only.
"""
from __future__ import annotations

import math

import numpy as np

AGG_MAX, AGG_MEAN, AGG_TOPP, AGG_FRAC_HOT, AGG_ALL_COLD = 0, 1, 2, 3, 4
NORM_NONE, NORM_PERCENTILE = 0, 1
UPDATE_DECAY, UPDATE_MAX, UPDATE_WINDOW = 0, 1, 2


def decay_update(score: np.ndarray, inc: np.ndarray, decay: float) -> np.ndarray:
    """score <- decay * score + inc (fp64)."""
    return decay * np.asarray(score, dtype=np.float64) + np.asarray(inc, dtype=np.float64)


def max_update(score: np.ndarray, inc: np.ndarray) -> np.ndarray:
    """Max pooling over steps: score <- max(score, inc) (fp64)."""
    return np.maximum(np.asarray(score, dtype=np.float64), np.asarray(inc, dtype=np.float64))


def window_sum(increments, window: int) -> np.ndarray:
    """Sliding window over steps: the sum of the last `window` increments
    (`increments` oldest first, one array per step)."""
    steps = [np.asarray(x, dtype=np.float64) for x in increments]
    total = np.zeros_like(steps[0])
    for x in steps[max(0, len(steps) - window):]:
        total = total + x
    return total


def topp_count(n: int, top_p: float) -> int:
    """ceil(p * n) with the product taken in fp32, at least 1."""
    prod = np.float32(top_p) * np.float32(n)
    return max(1, int(math.ceil(float(prod))))


def block_scores(tokens: np.ndarray, block_size: int, agg: int, top_p: float = 0.1,
                 threshold: float = 0.0) -> np.ndarray:
    """Fold one request's token scores into per-block scores."""
    tokens = np.asarray(tokens, dtype=np.float64)
    L = tokens.shape[0]
    nblk = (L + block_size - 1) // block_size
    out = np.empty(nblk)
    for i in range(nblk):
        blk = tokens[i * block_size:min((i + 1) * block_size, L)]
        if agg in (AGG_MAX, AGG_ALL_COLD):
            out[i] = blk.max()
        elif agg == AGG_FRAC_HOT:
            hot = int(np.count_nonzero(blk >= threshold))
            out[i] = np.float32(hot) / np.float32(blk.shape[0])
        elif agg == AGG_MEAN:
            out[i] = blk.mean()
        elif agg == AGG_TOPP:
            k = topp_count(blk.shape[0], top_p)
            out[i] = np.sort(blk)[::-1][:k].mean()
        else:
            raise ValueError("unknown aggregation")
    return out


def percentiles(scores: np.ndarray) -> np.ndarray:
    """Per-request percentile of each block: fp32((2r+1)/(2n)) with r the rank."""
    scores = np.asarray(scores, dtype=np.float64)
    n = scores.shape[0]
    order = np.lexsort((np.arange(n), scores))        # score asc, then block asc
    rank = np.empty(n, dtype=np.int64)
    rank[order] = np.arange(n)
    return (2 * rank + 1).astype(np.float32) / np.float32(2 * n)


def evict_count(n_blocks: int, frac: float) -> int:
    return int(math.ceil(frac * n_blocks))


def evict_order(norm_scores_per_request, frac: float, evictable_per_request=None) -> np.ndarray:
    """Global order [(req << 32) | blk] of the ceil(frac*N) lowest-priority blocks
    (N counts every block; with `evictable_per_request` only those blocks are
    ordered and the count is capped by their number)."""
    keys, total = [], 0
    for r, s in enumerate(norm_scores_per_request):
        s = np.asarray(s, dtype=np.float64)
        total += s.shape[0]
        for b in range(s.shape[0]):
            if evictable_per_request is None or evictable_per_request[r][b]:
                keys.append((s[b], r, b))
    keys.sort()
    n = min(evict_count(total, frac), len(keys))
    return np.array([(r << 32) | b for (_, r, b) in keys[:n]], dtype=np.int64)


def priority_pass(token_scores: np.ndarray, offsets: np.ndarray, block_size: int, agg: int,
                  top_p: float, norm: int, frac: float, threshold: float = 0.0):
    """Block scores, normalised scores and the global evict order for all requests."""
    R = offsets.shape[0] - 1
    blk = [block_scores(token_scores[offsets[r]:offsets[r + 1]], block_size, agg, top_p, threshold)
           for r in range(R)]
    if norm == NORM_PERCENTILE:
        normed = [percentiles(b).astype(np.float64) for b in blk]
    elif norm == NORM_NONE:
        normed = blk
    else:
        raise ValueError("unknown normalisation")
    evictable = [np.asarray(b) < threshold for b in blk] if agg == AGG_ALL_COLD else None
    return blk, normed, evict_order(normed, frac, evictable)
