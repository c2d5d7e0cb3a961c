"""GPU parity of Quest page selection in decode against the oracle.

* the page min / max built for a prompt, and kept current by the appends,
  bit-exact (min and max of bf16 values are bf16 values);
* the page bounds within relative L2 1e-5 of the fp64 oracle (fp32 sums of
  exact products);
* each head's pages bit-exact when the oracle's top-k routine gets the GPU's
  own fp32 bounds;
* the output within relative L2 2e-3 of the oracle's attention over those
  pages plus the partial page (dense attention when every page fits); a
  bf16 output is compared with the oracle rounded to bf16, since bf16's own
  rounding (relative 2^-9) would otherwise fill the whole bar.
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
BOUND_TOL = 1e-5
PAGE = 16


class QuestState:
    def __init__(self, wl, budget, out_f32=True):
        self.wl = wl
        self.budget = budget
        dev = "cuda"
        self.kpool = bf16(workloads.paged_pool(wl.K, wl.block_table, wl.num_pages, page=wl.page))
        self.vpool = bf16(workloads.paged_pool(wl.V, wl.block_table, wl.num_pages, page=wl.page))
        self.kv = K.paged_kv(self.kpool, self.vpool, wl.Hq)
        tiles = wl.page // PAGE       # Quest pages per pool page
        self.guards = g = Guards()
        self.bt = g.like(torch.from_numpy(wl.block_table).to(dev))
        self.seq = g.like(torch.full((wl.B,), wl.S0, dtype=torch.int32, device=dev))
        self.meta = g.new((wl.num_pages, wl.Hkv, tiles, 2, wl.d), torch.bfloat16)
        self.out = g.new((wl.B, wl.Hq, wl.d), torch.float32 if out_f32 else torch.bfloat16)
        self.pages = g.new((wl.B, wl.Hq, budget), torch.int32, fill=-7)
        self.bounds = g.new((wl.B, wl.Hq, wl.max_pages * tiles), torch.float32)
        self.ws = g.new((K.kvsel_quest_decode_workspace(self.kv, wl.B, wl.max_pages, budget, True, True),),
                        torch.uint8)
        K.kvsel_quest_page_meta(self.kv, self.bt, self.seq, self.meta, self.ws)

    def step(self, t, append=True):
        wl = self.wl
        K.kvsel_quest_decode(self.kv, self.bt, self.seq, bf16(wl.q[t]), self.meta, self.out, self.ws,
                             budget_pages=self.budget, k_new=bf16(wl.k_new[t]) if append else None,
                             v_new=bf16(wl.v_new[t]) if append else None, pages_out=self.pages,
                             bounds_out=self.bounds)
        torch.cuda.synchronize()
        assert K.read_status(self.ws) == 0
        self.guards.check()


def _logical(wl, b, appended):
    Kb = bf16_bits_to_f64(wl.K[b])
    Vb = bf16_bits_to_f64(wl.V[b])
    if appended:
        Kb = np.concatenate([Kb, bf16_bits_to_f64(wl.k_new[:appended, b]).transpose(1, 0, 2)], axis=1)
        Vb = np.concatenate([Vb, bf16_bits_to_f64(wl.v_new[:appended, b]).transpose(1, 0, 2)], axis=1)
    return Kb, Vb


def _check_meta(st, appended):
    wl = st.wl
    meta = st.meta.double().cpu().numpy()
    for b in range(wl.B):
        Kb, _ = _logical(wl, b, appended)
        S = Kb.shape[1]
        for kvh in range(wl.Hkv):
            kmin, kmax = dsa.page_minmax(Kb[kvh], PAGE)
            for p in range(-(-S // PAGE)):
                phys, j = wl.block_table[b, p * PAGE // wl.page], (p * PAGE % wl.page) // PAGE
                np.testing.assert_array_equal(meta[phys, kvh, j, 0], kmin[p])
                np.testing.assert_array_equal(meta[phys, kvh, j, 1], kmax[p])


def _check(st, t, appended, heads=None):
    wl = st.wl
    bounds = st.bounds.cpu().numpy()
    pages = st.pages.cpu().numpy()
    out = st.out.double().cpu().numpy()
    S = int(st.seq[0])
    n_full = S // PAGE
    for b in range(wl.B):
        Kb, Vb = _logical(wl, b, appended)
        assert Kb.shape[1] == S
        qb = bf16_bits_to_f64(wl.q[t, b])
        for h in (range(wl.Hq) if heads is None else heads):
            kvh = h // wl.G
            if n_full:
                ub = dsa.quest_page_bound(qb[h], Kb[kvh], PAGE)
                assert rel_l2(bounds[b, h, :n_full], ub) < BOUND_TOL, (b, h)
            sel = dsa.quest_select_pages(bounds[b, h, :n_full].astype(np.float64), st.budget)
            np.testing.assert_array_equal(pages[b, h, :len(sel)], sel)
            assert (pages[b, h, len(sel):] == -1).all()
            toks = np.concatenate([np.arange(p * PAGE, (p + 1) * PAGE) for p in sel] +
                                  [np.arange(n_full * PAGE, S)]).astype(np.int64)
            o = dsa.masked_attention(qb[h:h + 1], Kb[kvh:kvh + 1], Vb[kvh:kvh + 1], toks, wl.scale)[0]
            if st.out.dtype == torch.bfloat16:   # the bar is on the accumulated value: same output grid
                o = bf16_bits_to_f64(workloads.f32_to_bf16_bits(o.astype(np.float32)))
            assert rel_l2(out[b, h], o) < TOL, (b, h)


@pytest.mark.parametrize("S0", [1000, 1024, 5])
def test_page_meta_for_a_prompt(S0):
    wl = workloads.sparse_decode(seed=40 + S0, B=2, S0=S0, steps=1, Hq=8, Hkv=2)
    st = QuestState(wl, budget=4)
    torch.cuda.synchronize()
    assert K.read_status(st.ws) == 0
    _check_meta(st, 0)


def test_steps_across_a_page_boundary():
    # 2030 keys: the second append fills page 126, the third opens page 127
    wl = workloads.sparse_decode(seed=41, B=2, S0=2030, steps=4, Hq=16, Hkv=4)
    st = QuestState(wl, budget=16)
    for t in range(4):
        st.step(t)
        _check(st, t, t + 1)
    _check_meta(st, 4)
    assert st.seq.cpu().tolist() == [2034, 2034]


@pytest.mark.parametrize("page,S0", [(256, 2555), (64, 1000), (32, 5)])
def test_pool_pages_of_32_to_256_tokens(page, S0):
    """Quest pages stay 16 tokens inside larger pool pages: appends cross Quest-page and (at 256:
    the sixth append is token 2560) pool-page boundaries; meta, bounds, pages and output as at
    page 16."""
    wl = workloads.sparse_decode(seed=60 + page, B=2, S0=S0, steps=8, Hq=16, Hkv=2, page=page)
    st = QuestState(wl, budget=12)
    torch.cuda.synchronize()
    _check_meta(st, 0)
    for t in range(wl.steps):
        st.step(t)
        _check(st, t, t + 1)
    _check_meta(st, wl.steps)
    assert st.seq.cpu().tolist() == [S0 + wl.steps] * wl.B


def test_sixteen_heads_choose_their_own_pages_at_page_256():
    # a planted page per q head of a 16-head group: heads 8..15 run in the wide tile's second half
    wl = workloads.sparse_decode(seed=48, B=1, S0=4000, steps=1, Hq=16, Hkv=1, page=256)
    Kf = bf16_bits_to_f64(wl.K[0]).astype(np.float32)
    qf = bf16_bits_to_f64(wl.q[0, 0]).astype(np.float32)
    planted = {}
    for h in range(wl.Hq):
        p = 7 + 15 * h
        u = qf[h] / np.linalg.norm(qf[h])
        Kf[0, p * PAGE:(p + 1) * PAGE] += 6.0 * u
        planted[h] = p
    wl.K = workloads.f32_to_bf16_bits(Kf)[None]
    st = QuestState(wl, budget=3)
    st.step(0)
    _check(st, 0, 1)
    pages = st.pages.cpu().numpy()
    for h, p in planted.items():
        assert p in pages[0, h].tolist()


def test_without_append_and_with_every_page_in_budget():
    wl = workloads.sparse_decode(seed=42, B=3, S0=300, steps=1, Hq=16, Hkv=4)
    st = QuestState(wl, budget=32)
    st.step(0, append=False)
    _check(st, 0, 0)
    out = st.out.double().cpu().numpy()
    for b in range(wl.B):
        Kb, Vb = _logical(wl, b, 0)
        o, _ = decode_attention(bf16_bits_to_f64(wl.q[0, b]), Kb, Vb, wl.scale)
        assert rel_l2(out[b], o) < TOL
    assert st.seq.cpu().tolist() == [300] * 3


@pytest.mark.parametrize("S0", [4, 15, 31])
def test_short_contexts(S0):
    # no full page, or a single one, before the partial page
    wl = workloads.sparse_decode(seed=43 + S0, B=2, S0=S0, steps=2, Hq=8, Hkv=2)
    st = QuestState(wl, budget=1)
    for t in range(2):
        st.step(t)
        _check(st, t, t + 1)
    _check_meta(st, 2)


@pytest.mark.parametrize("G,budget", [(1, 3), (8, 20), (5, 64), (12, 40), (16, 20)])
def test_group_sizes_budgets_and_bf16_output(G, budget):
    wl = workloads.sparse_decode(seed=50 + G, B=2, S0=6000 + G, steps=1, Hq=4 * G, Hkv=4)
    st = QuestState(wl, budget=budget, out_f32=False)
    st.step(0)
    _check(st, 0, 1)


def test_heads_choose_their_own_pages():
    # plant, for every q head, one page whose keys answer that head strongly:
    # each head must keep its own planted page, and the kv head streams the union
    wl = workloads.sparse_decode(seed=44, B=1, S0=4000, steps=1, Hq=8, Hkv=2)
    Kf = bf16_bits_to_f64(wl.K[0]).astype(np.float32)
    qf = bf16_bits_to_f64(wl.q[0, 0]).astype(np.float32)
    planted = {}
    for h in range(wl.Hq):
        p = 10 + 23 * h
        u = qf[h] / np.linalg.norm(qf[h])
        Kf[h // wl.G, p * PAGE:(p + 1) * PAGE] += 6.0 * u
        planted[h] = p
    wl.K = workloads.f32_to_bf16_bits(Kf)[None]
    st = QuestState(wl, budget=2)
    st.step(0)
    _check(st, 0, 1)
    pages = st.pages.cpu().numpy()
    for h, p in planted.items():
        assert p in pages[0, h].tolist()


def test_long_page_lists_per_warp():
    # one kv head with a 10000-page budget over 12.5K pages: each attention warp
    # walks more than one 32-entry chunk of the page list
    wl = workloads.sparse_decode(seed=45, B=1, S0=200003, steps=1, Hq=1, Hkv=1)
    st = QuestState(wl, budget=10000)
    st.step(0)
    _check(st, 0, 1)


def test_equal_bounds_keep_the_lower_pages():
    # every full page holds the same 16 keys: all bounds tie exactly
    wl = workloads.sparse_decode(seed=46, B=2, S0=3000, steps=1, Hq=8, Hkv=2)
    K4 = wl.K.copy()
    for b in range(wl.B):
        for kvh in range(wl.Hkv):
            page = K4[b, kvh, :16].copy()
            for p in range(wl.S0 // 16):
                K4[b, kvh, 16 * p:16 * (p + 1)] = page
    wl.K = K4                      # the appended token lands in the partial page 187
    st = QuestState(wl, budget=40)
    st.step(0)
    _check(st, 0, 1)
    assert (st.pages.cpu().numpy() == np.arange(40)).all()


def test_rows_longer_than_the_register_select():
    # 18750 full pages: the per-head selection falls back to the row_topk path
    wl = workloads.sparse_decode(seed=47, B=1, S0=300003, steps=1, Hq=2, Hkv=1)
    st = QuestState(wl, budget=100)
    st.step(0)
    _check(st, 0, 1)


@pytest.mark.slow
def test_full_size_70b_128k_sampled():
    """Batch 4 x 128K, 64 q / 8 kv heads, 128 pages (2048 tokens) per head: sampled heads."""
    wl = workloads.sparse_decode(steps=2)
    st = QuestState(wl, budget=128)
    rng = np.random.default_rng(2)
    for t in range(2):
        st.step(t)
        _check(st, t, t + 1, heads=sorted(rng.choice(wl.Hq, 4, replace=False).tolist()))
