"""Pins for the decode-attention oracle (CPU only).

The oracle's output is checked against things that do not come from the
oracle itself: PyTorch's own fp64 scaled-dot-product attention, closed forms
(one key, identical keys), the softmax-sums-to-one invariant of the H2O score,
a constructed GQA case, and the KV byte counts printed on the pages.
"""
import math

import numpy as np
import pytest
import torch

from oracle import attention as A
from oracle import costs
from oracle.h2o import H2OSequence


def _rand(rng, *shape):
    return rng.standard_normal(shape)


def test_matches_torch_sdpa_and_pins_probabilities():
    # S <= d, so V_kvh (S x d) has full row rank: o = p V fixes p uniquely.
    rng = np.random.default_rng(11)
    Hq, Hkv, S, d = 8, 2, 12, 16
    q, K, V = _rand(rng, Hq, d), _rand(rng, Hkv, S, d), _rand(rng, Hkv, S, d)
    scale = 1.0 / math.sqrt(d)
    o, p = A.decode_attention(q, K, V, scale)
    G = Hq // Hkv
    Kt = torch.from_numpy(K).repeat_interleave(G, 0)            # q head h -> kv head h // G
    Vt = torch.from_numpy(V).repeat_interleave(G, 0)
    ref = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(q)[:, None, :], Kt, Vt).squeeze(1).numpy()   # default scale d^-1/2
    np.testing.assert_allclose(o, ref, rtol=1e-12, atol=1e-12)
    for h in range(Hq):
        p_from_ref = np.linalg.lstsq(V[h // G].T, ref[h], rcond=None)[0]
        np.testing.assert_allclose(p[h], p_from_ref, rtol=1e-9, atol=1e-10)


def test_single_key_returns_value():
    rng = np.random.default_rng(1)
    q, K, V = _rand(rng, 4, 8), _rand(rng, 2, 1, 8), _rand(rng, 2, 1, 8)
    o, p = A.decode_attention(q, K, V, 0.3)
    np.testing.assert_array_equal(p, np.ones((4, 1)))
    np.testing.assert_allclose(o, np.repeat(V[:, 0], 2, axis=0), rtol=0, atol=1e-15)


def test_identical_keys_give_uniform_weights():
    rng = np.random.default_rng(2)
    S, d = 37, 8
    K = np.tile(_rand(rng, 1, 1, d), (1, S, 1))
    V = _rand(rng, 1, S, d)
    o, p = A.decode_attention(_rand(rng, 3, d), K, V, 1 / math.sqrt(d))
    np.testing.assert_allclose(p, np.full((3, S), 1.0 / S), rtol=1e-13)
    np.testing.assert_allclose(o, np.tile(V[0].mean(0), (3, 1)), rtol=1e-12, atol=1e-13)


def test_cumulative_score_totals_steps_times_heads():
    # Each softmax row sums to one, so with no eviction the H2O totals are
    # steps * Hq overall and steps * G per kv head.
    rng = np.random.default_rng(3)
    Hq, Hkv, d, S0, steps = 8, 4, 16, 30, 9
    seq = H2OSequence(_rand(rng, Hkv, S0, d), _rand(rng, Hkv, S0, d))
    for _ in range(steps):
        seq.step(_rand(rng, Hq, d), _rand(rng, Hkv, d), _rand(rng, Hkv, d), 0.25,
                 budget=10**9, n_sink=4, window=4)
    assert seq.S == S0 + steps
    np.testing.assert_allclose(seq.cum.sum(), steps * Hq, rtol=1e-13)
    np.testing.assert_allclose(seq.cum.sum(axis=1), np.full(Hkv, steps * Hq // Hkv), rtol=1e-13)


def test_cumulative_score_uses_the_query_group_of_each_kv_head():
    # q heads 0,1 share kv head 0 and stare at key 3; heads 2,3 share kv head 1
    # and stare at key 5.  A wrong group mapping (h % Hkv) moves the mass.
    d, S = 8, 9
    e = np.eye(d)
    K = np.zeros((2, S, d))
    K[0, 3] = 40 * e[0]
    K[1, 5] = 40 * e[1]
    q = np.stack([e[0], e[0], e[1], e[1]])
    _, p = A.decode_attention(q, K, np.zeros_like(K), 1.0)
    cum = A.h2o_accumulate(np.zeros((2, S)), p)
    assert cum[0, 3] > 1.999 and cum[1, 5] > 1.999
    np.testing.assert_allclose(cum.sum(axis=1), [2.0, 2.0], rtol=1e-14)


def test_bf16_widening_is_exact():
    bits = np.array([0x3F80, 0xBF80, 0x4049, 0x0000, 0x8000, 0x7F7F], dtype=np.uint16)
    want = [1.0, -1.0, 3.140625, 0.0, -0.0, 3.3895313892515355e38]
    np.testing.assert_array_equal(A.bf16_bits_to_f64(bits), want)


def test_kv_bytes_match_printed_values(golden):
    rows = list(golden("kv_cache_bytes.txt"))
    for model, L, H, d, T, val, unit in rows[:2]:
        got = costs.kv_bytes(int(L), int(H), int(d), int(T)) / 1e9
        assert f"{got:.1f}" == val, (model, got)
    model, L, H, d, T, gb, ms = rows[2]
    b = costs.kv_bytes(int(L), int(H), int(d), int(T))
    assert b == 10_737_418_240                      # exactly 10 GiB
    assert abs(b / 1e9 - float(gb)) / float(gb) < 0.08
    t_ms = costs.decode_read_seconds(int(L), int(H), int(d), int(T), 3.35e12) * 1e3
    assert abs(t_ms - float(ms)) / float(ms) < 0.08
