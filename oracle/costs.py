"""Byte counts of the KV cache (closed forms).  Test infrastructure only.

"Long context, KV eviction and sparse attention", section on the cost of long
context: a token stores one K and one V vector per kv head per layer, so its
16-bit KV takes 2 * layers * kv_heads * head_dim * 2 bytes.  "Sparse attention
x KV offloading" §1: decode reads the whole KV once per step.
"""
from __future__ import annotations


def kv_bytes_per_token(layers: int, kv_heads: int, head_dim: int, elem_bytes: int = 2) -> int:
    return 2 * layers * kv_heads * head_dim * elem_bytes


def kv_bytes(layers: int, kv_heads: int, head_dim: int, tokens: int, elem_bytes: int = 2) -> int:
    return kv_bytes_per_token(layers, kv_heads, head_dim, elem_bytes) * tokens


def decode_read_seconds(layers, kv_heads, head_dim, tokens, hbm_bytes_per_s, elem_bytes=2):
    """Time to stream the whole KV once at a given HBM bandwidth."""
    return kv_bytes(layers, kv_heads, head_dim, tokens, elem_bytes) / hbm_bytes_per_s


# "Sparse attention x KV-cache offloading: eight questions" §5.1 (metadata
# cost): each KV block keeps an fp32 score accumulator and an int32
# last-update step, and each decode step writes one fp32 score per top-k
# block of every request.
BLOCK_META_BYTES = 4 + 4


def block_metadata_bytes(requests: int, blocks_per_request: int) -> int:
    """Bytes of per-block signal metadata for a whole batch."""
    return requests * blocks_per_request * BLOCK_META_BYTES


def signal_update_bytes(requests: int, topk_blocks: int, score_bytes: int = 4) -> int:
    """Score bytes one decode step writes for the batch's top-k blocks."""
    return requests * topk_blocks * score_bytes
