"""Decode attention with per-key score emission (fp64).  Test infrastructure only.

Follows "From sliding window to attention-guided eviction" §3.1: a query's
weights are a softmax over its logits against every visible key, so they sum
to one; "Long context, KV eviction and sparse attention" (sparse-selection
section) fixes the logit scale as head_dim^-1/2 and maps q head h to kv head
h // (Hq/Hkv) (keys repeated per group).  Decode means one query per head
against the full cache ("Sparse attention x KV offloading" §1, §2.3).
"""
from __future__ import annotations

import numpy as np


def bf16_bits_to_f64(bits) -> np.ndarray:
    """Widen bf16 bit patterns (uint16) to fp64 exactly."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32).astype(np.float64)


def softmax(s: np.ndarray) -> np.ndarray:
    """Softmax along the last axis (max-subtracted; exact reformulation)."""
    m = np.max(s, axis=-1, keepdims=True)
    e = np.exp(s - m)
    return e / np.sum(e, axis=-1, keepdims=True)


def decode_attention(q: np.ndarray, K: np.ndarray, V: np.ndarray, scale: float):
    """One decode step of GQA attention for one sequence.

    q: [Hq][d]; K, V: [Hkv][S][d] (all live keys, the new token included).
    Returns (o [Hq][d], p [Hq][S]) with p_h = softmax(K_{h//G} q_h * scale)
    and o_h = p_h V_{h//G}.
    """
    Hq, d = q.shape
    Hkv, S, _ = K.shape
    G = Hq // Hkv
    o = np.zeros((Hq, d))
    p = np.zeros((Hq, S))
    for h in range(Hq):
        kvh = h // G
        s = (K[kvh] @ q[h]) * scale
        p[h] = softmax(s)
        o[h] = p[h] @ V[kvh]
    return o, p


def h2o_accumulate(cum: np.ndarray, p: np.ndarray) -> np.ndarray:
    """H2O cumulative score update ("...eviction" §4.2 step 1 and pseudocode).

    Every decode step adds each key's attention weight to that key's running
    total.  With GQA the score is kept per kv head and sums the G q heads that
    share it.  cum: [Hkv][S], p: [Hq][S]; returns the updated copy.
    """
    Hkv = cum.shape[0]
    G = p.shape[0] // Hkv
    out = cum.copy()
    for kvh in range(Hkv):
        out[kvh] += p[kvh * G:(kvh + 1) * G].sum(axis=0)
    return out
