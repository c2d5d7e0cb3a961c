"""GPU parity of DSA-style sparse decode against the oracle.

* indexer scores within relative L2 2e-3 of the fp64 oracle;
* the selected positions bit-exact when the oracle's top-k routine gets the
  GPU's own fp32 scores;
* the output within relative L2 2e-3 of the oracle's masked attention over
  that selection (and equal to dense attention when S <= top_k).
"""
import numpy as np
import pytest
import torch

import workloads
from oracle import dsa
from oracle.attention import bf16_bits_to_f64, decode_attention
from _harness import Guards, bf16, rel_l2

import attention_guided_kv_gb300 as K

pytestmark = pytest.mark.gpu
TOL = 2e-3


class SparseState:
    def __init__(self, wl, out_f32=True):
        self.wl = wl
        dev = "cuda"
        self.kpool = bf16(workloads.paged_pool(wl.K, wl.block_table, wl.num_pages, wl.page))
        self.vpool = bf16(workloads.paged_pool(wl.V, wl.block_table, wl.num_pages, wl.page))
        self.kv = K.paged_kv(self.kpool, self.vpool, wl.Hq)
        self.bt = torch.from_numpy(wl.block_table).to(dev)
        self.seq = torch.full((wl.B,), wl.S0, dtype=torch.int32, device=dev)
        idx = np.zeros((wl.B, wl.max_len, wl.Di), dtype=np.uint16)
        idx[:, :wl.S0] = wl.k_idx
        self.idx_k = bf16(idx)
        self.guards = g = Guards()
        self.seq = g.like(self.seq)
        self.bt = g.like(self.bt)
        self.out = g.new((wl.B, wl.Hq, wl.d), torch.float32 if out_f32 else torch.bfloat16)
        self.topk = g.new((wl.B, wl.top_k), torch.int32, fill=-7)
        self.scores = g.new((wl.B, wl.max_len), torch.float32)
        self.ws = g.new((K.kvsel_sparse_decode_workspace(self.kv, wl.B, wl.max_len, wl.top_k, True),), torch.uint8)

    def step(self, t, append=True):
        wl = self.wl
        K.kvsel_sparse_decode(self.kv, self.bt, self.seq, bf16(wl.q[t]), bf16(wl.q_idx[t]),
                              torch.from_numpy(wl.w_idx[t]).cuda(), self.idx_k, self.out, self.ws,
                              top_k=wl.top_k, k_new=bf16(wl.k_new[t]) if append else None,
                              v_new=bf16(wl.v_new[t]) if append else None,
                              idx_k_new=bf16(wl.k_idx_new[t]) if append else None,
                              topk_out=self.topk, scores_out=self.scores)


def _logical(wl, b, t_done):
    """Oracle-side K, V [Hkv][S][d] and indexer keys [S][Di] after t_done appends."""
    Kb = bf16_bits_to_f64(wl.K[b])
    Vb = bf16_bits_to_f64(wl.V[b])
    ki = bf16_bits_to_f64(wl.k_idx[b])
    if t_done:
        Kb = np.concatenate([Kb, bf16_bits_to_f64(wl.k_new[:t_done, b]).transpose(1, 0, 2)], axis=1)
        Vb = np.concatenate([Vb, bf16_bits_to_f64(wl.v_new[:t_done, b]).transpose(1, 0, 2)], axis=1)
        ki = np.concatenate([ki, bf16_bits_to_f64(wl.k_idx_new[:t_done, b])], axis=0)
    return Kb, Vb, ki


def _check(st, t, heads=None):
    wl = st.wl
    torch.cuda.synchronize()
    st.guards.check()
    S = int(st.seq[0])
    scores = st.scores.cpu().numpy()
    topk = st.topk.cpu().numpy()
    out = st.out.double().cpu().numpy()
    for b in range(wl.B):
        Kb, Vb, ki = _logical(wl, b, t + 1)
        assert Kb.shape[1] == S
        I = dsa.indexer_scores(bf16_bits_to_f64(wl.q_idx[t, b]), wl.w_idx[t, b].astype(np.float64), ki)
        assert rel_l2(scores[b, :S], I) < TOL
        sel = dsa.select_topk(scores[b, :S].astype(np.float32), wl.top_k)     # same fp32 scores
        n = len(sel)
        np.testing.assert_array_equal(topk[b, :n], sel)
        assert (topk[b, n:] == -1).all()
        qb = bf16_bits_to_f64(wl.q[t, b])
        if heads is None:
            o = dsa.masked_attention(qb, Kb, Vb, sel, wl.scale)
            assert rel_l2(out[b], o) < TOL
        else:
            for h in heads:
                kvh = h // wl.G
                oh = dsa.masked_attention(qb[h:h + 1], Kb[kvh:kvh + 1], Vb[kvh:kvh + 1], sel, wl.scale)
                assert rel_l2(out[b, h], oh[0]) < TOL


def test_three_steps_multi_chunk():
    wl = workloads.sparse_decode(seed=14, B=2, S0=40000, steps=3, top_k=512)
    st = SparseState(wl)
    for t in range(3):
        st.step(t)
        _check(st, t)
    assert st.seq.cpu().tolist() == [40003, 40003]
    assert K.read_status(st.ws) == 0


@pytest.mark.parametrize("page", [64, 256])
def test_larger_pages_across_a_page_boundary(page):
    """Pool pages of 64 or 256 tokens: appends crossing into a new page, the selected rows resolved
    through the bigger pages (every kv head's row at its own offset in the page)."""
    wl = workloads.sparse_decode(seed=24, B=2, S0=20478, steps=3, top_k=700, page=page)
    st = SparseState(wl)
    for t in range(3):
        st.step(t)
        _check(st, t)
    assert st.seq.cpu().tolist() == [20481, 20481]
    assert K.read_status(st.ws) == 0


@pytest.mark.parametrize("S0", [140000, 250000])
def test_scores_all_at_most_zero_tie_thousands_at_zero(S0):
    """Every indexer weight negative: every score is <= 0 and thousands of keys tie at exactly 0
    (10.2K at 140K keys, 14.2K at 250K), all in one radix bin of the cluster select.  Ties go to
    the lower positions."""
    wl = workloads.sparse_decode(seed=25, B=1, S0=S0, steps=1, Hq=16, Hkv=2, top_k=2048)
    wl.w_idx = -np.abs(wl.w_idx)
    st = SparseState(wl)
    st.step(0)
    _check(st, 0)


def test_aligned_score_rows_across_the_select_cluster():
    """Rows whose length is a multiple of 4 (16-byte score copies in the cluster select), chunks
    of 2 rounds per warp, the last CTA of the cluster partly and the rest of the chunk empty."""
    wl = workloads.sparse_decode(seed=26, B=2, S0=65533, steps=3, top_k=2048)
    assert wl.max_len % 4 == 0
    st = SparseState(wl)
    for t in range(3):
        st.step(t)
        _check(st, t)
    assert K.read_status(st.ws) == 0


@pytest.mark.parametrize("negative", [False, True])
def test_rows_longer_than_the_select_cluster(negative):
    """270K positions: past the cluster select's 256K, the slice select with its final CTA (and,
    with every score <= 0, its whole-row fallback)."""
    wl = workloads.sparse_decode(seed=27, B=1, S0=270000, steps=1, Hq=8, Hkv=1, top_k=2048)
    if negative:
        wl.w_idx = -np.abs(wl.w_idx)
    st = SparseState(wl)
    st.step(0)
    _check(st, 0)
    assert K.read_status(st.ws) == 0


def test_mixed_lengths_in_one_batch():
    """Rows of different lengths in one call: below, at and just above top_k (the select-all path
    and the cluster select side by side), a short row and long ones; each row checked against the
    oracle on its own prefix."""
    wl = workloads.sparse_decode(seed=28, B=6, S0=9000, steps=1, Hq=16, Hkv=2, top_k=2048)
    lens = np.array([9000, 2046, 2047, 2048, 100, 5000])
    st = SparseState(wl)
    st.seq.copy_(torch.from_numpy(lens.astype(np.int32)))
    st.step(0)
    torch.cuda.synchronize()
    st.guards.check()
    assert st.seq.cpu().tolist() == (lens + 1).tolist()
    scores = st.scores.cpu().numpy()
    topk = st.topk.cpu().numpy()
    out = st.out.double().cpu().numpy()
    for b in range(wl.B):
        n0 = int(lens[b])
        S = n0 + 1
        Kb = np.concatenate([bf16_bits_to_f64(wl.K[b][:, :n0]), bf16_bits_to_f64(wl.k_new[0, b])[:, None]], axis=1)
        Vb = np.concatenate([bf16_bits_to_f64(wl.V[b][:, :n0]), bf16_bits_to_f64(wl.v_new[0, b])[:, None]], axis=1)
        ki = np.concatenate([bf16_bits_to_f64(wl.k_idx[b][:n0]), bf16_bits_to_f64(wl.k_idx_new[0, b])[None]], axis=0)
        I = dsa.indexer_scores(bf16_bits_to_f64(wl.q_idx[0, b]), wl.w_idx[0, b].astype(np.float64), ki)
        assert rel_l2(scores[b, :S], I) < TOL
        sel = dsa.select_topk(scores[b, :S].astype(np.float32), wl.top_k)
        np.testing.assert_array_equal(topk[b, :len(sel)], sel)
        assert (topk[b, len(sel):] == -1).all()
        o = dsa.masked_attention(bf16_bits_to_f64(wl.q[0, b]), Kb, Vb, sel, wl.scale)
        assert rel_l2(out[b], o) < TOL
    assert K.read_status(st.ws) == 0


def test_short_context_selects_all_and_matches_dense():
    wl = workloads.sparse_decode(seed=15, B=3, S0=300, steps=1, top_k=2048)
    st = SparseState(wl)
    st.step(0)
    _check(st, 0)
    out = st.out.double().cpu().numpy()
    for b in range(wl.B):
        Kb, Vb, _ = _logical(wl, b, 1)
        o, _ = decode_attention(bf16_bits_to_f64(wl.q[0, b]), Kb, Vb, wl.scale)
        assert rel_l2(out[b], o) < TOL
    assert (st.topk.cpu().numpy()[:, :301] == np.arange(301)).all()


def test_ties_resolve_to_lower_positions():
    wl = workloads.sparse_decode(seed=16, B=1, S0=20000, steps=1, top_k=300)
    # quantise the indexer keys hard so that many scores tie exactly
    kf = (bf16_bits_to_f64(wl.k_idx) > 0.8).astype(np.float32)
    wl.k_idx = workloads.f32_to_bf16_bits(kf)
    kn = (bf16_bits_to_f64(wl.k_idx_new) > 0.8).astype(np.float32)
    wl.k_idx_new = workloads.f32_to_bf16_bits(kn)
    st = SparseState(wl)
    st.step(0)
    _check(st, 0)


def test_large_top_k_single_stage():
    """top_k >= 16384: one CTA per row sweeps the whole row (rows longer than 32K stream)."""
    wl = workloads.sparse_decode(seed=19, B=2, S0=50001, steps=1, Hq=16, Hkv=2, top_k=20000)
    st = SparseState(wl)
    st.step(0)
    _check(st, 0)


@pytest.mark.parametrize("G", [1, 4, 8, 12, 16])
def test_group_sizes_and_bf16_output(G):
    wl = workloads.sparse_decode(seed=17 + G, B=2, S0=5000, steps=1, Hq=8 * G, Hkv=8, top_k=1000)
    st = SparseState(wl, out_f32=False)
    st.step(0)
    _check(st, 0)


def test_sixteen_heads_on_256_token_pages():
    """Both widenings at once: 16 q heads per kv head (heads g + 8 in the wide tile's rows 8..15)
    gathering rows out of 256-token pool pages, across an append that opens a new page."""
    wl = workloads.sparse_decode(seed=29, B=2, S0=4094, steps=3, Hq=32, Hkv=2, top_k=700, page=256)
    st = SparseState(wl)
    for t in range(3):
        st.step(t)
        _check(st, t)
    assert st.seq.cpu().tolist() == [4097, 4097]
    assert K.read_status(st.ws) == 0


@pytest.mark.slow
def test_full_size_70b_128k_sampled():
    """Batch 4 x 128K, 70B shape, indexer 4 x 64, top-2048: sampled heads vs the oracle."""
    wl = workloads.sparse_decode(steps=2)
    st = SparseState(wl)
    rng = np.random.default_rng(1)
    for t in range(2):
        st.step(t)
        _check(st, t, heads=sorted(rng.choice(wl.Hq, 6, replace=False).tolist()))
