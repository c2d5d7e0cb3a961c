"""Per-step top-k block signal from one decode step (fp64).  Test only.

Follows "Sparse attention x KV-cache offloading: eight questions" §5.1
(metadata cost): every KV block keeps an fp32 score accumulator and an int32
last-update step, and each decode step accumulates the scores of each
request's top-k blocks (k = 512 in the page's estimate).  The reading used
here, where the page leaves the score open: a block's score for the step is
the attention mass the step's query put on it, summed over every q head and
the block's valid keys; the request's top-k blocks by that mass (ties to the
lower block; every block when there are no more than k) add their mass to
their accumulator and take the step as their last update; the other blocks
are left as they were.  Blocks are the paged cache's pages (16 tokens, every
kv head), indexed by physical page through the block table.
"""
from __future__ import annotations

import numpy as np

from .h2o import topk_positions


def block_masses(p: np.ndarray, page: int = 16) -> np.ndarray:
    """Attention mass per block: p [Hq][S] (one step's probabilities) -> [ceil(S / page)]."""
    Hq, S = p.shape
    n = -(-S // page)
    out = np.zeros(n)
    for b in range(n):
        out[b] = p[:, b * page:min(S, (b + 1) * page)].sum()
    return out


def top_blocks(mass: np.ndarray, k: int) -> np.ndarray:
    """The k blocks with the largest mass (ties to the lower block), ascending."""
    return topk_positions(mass, k)


def apply_signal(acc: np.ndarray, last: np.ndarray, block_table_row: np.ndarray, blocks: np.ndarray,
                 mass: np.ndarray, step: int):
    """Accumulate the chosen blocks' mass into their physical block's metadata (copies returned)."""
    acc = acc.copy()
    last = last.copy()
    for blk in blocks:
        phys = block_table_row[blk]
        acc[phys] += mass[blk]
        last[phys] = step
    return acc, last
