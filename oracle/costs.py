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
