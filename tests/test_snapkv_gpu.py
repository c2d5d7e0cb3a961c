"""GPU parity of SnapKV prefill selection against the oracle.

* votes within relative L2 2e-3 of the fp64 oracle;
* keep-sets bit-exact when the oracle's max-pool + top-k get the GPU's own
  fp32 votes;
* the planted high-affinity keys survive at the full Qwen2.5-7B shape.
"""
import numpy as np
import pytest
import torch

import workloads
from oracle import snapkv
from oracle.attention import bf16_bits_to_f64
from _harness import Guards, bf16, rel_l2

import attention_guided_kv_gb300 as K

pytestmark = pytest.mark.gpu
TOL = 2e-3


class SnapState:
    """All layers of a SnapKV workload in one paged pool (layer l owns pages l*P .. l*P+P-1)."""

    def __init__(self, wl, layers):
        self.wl = wl
        self.layers = layers
        P = wl.pages
        pool = np.zeros((len(layers) * P, wl.Hkv, 16, wl.d), dtype=np.uint16)
        bts = np.zeros((len(layers), P), dtype=np.int32)
        q = np.zeros((len(layers), wl.Hq, wl.W, wl.d), dtype=np.uint16)
        for i, lay in enumerate(layers):
            pool[i * P:(i + 1) * P] = workloads.paged_pool(lay.K[None], lay.block_table[None], P)
            bts[i] = lay.block_table + i * P
            q[i] = lay.q_obs
        self.kpool = bf16(pool)
        self.kv = K.paged_kv(self.kpool, self.kpool, wl.Hq)
        self.bt = torch.from_numpy(bts).cuda()
        self.q = bf16(q)
        L = len(layers)
        self.guards = g = Guards()
        self.keep = g.new((L, wl.Hkv, wl.keep_k + wl.W), torch.int32, fill=-7)
        self.vote = g.new((L, wl.Hkv, max(wl.S - wl.W, 1)), torch.float32)
        self.ws = g.new((K.kvsel_snapkv_select_workspace(self.kv, L, wl.S, wl.W, True),), torch.uint8)

    def run(self):
        wl = self.wl
        K.kvsel_snapkv_select(self.kv, self.bt, self.q, self.keep, self.ws, seq_len=wl.S,
                              keep_k=wl.keep_k, pool_kernel=wl.pool_kernel, vote_out=self.vote)
        torch.cuda.synchronize()
        assert K.read_status(self.ws) == 0
        self.guards.check()


def _check(st, layer_ids=None, kv_heads=None):
    wl = st.wl
    keep = st.keep.cpu().numpy()
    vote = st.vote.cpu().numpy()
    P = wl.S - wl.W
    for i, lay in enumerate(st.layers):
        if layer_ids is not None and i not in layer_ids:
            continue
        for h in (range(wl.Hkv) if kv_heads is None else kv_heads):
            G = wl.G
            v = snapkv.snapkv_vote(bf16_bits_to_f64(lay.q_obs[h * G:(h + 1) * G]),
                                   bf16_bits_to_f64(lay.K[h:h + 1]), wl.scale)[0]
            assert rel_l2(vote[i, h, :P], v) < TOL, (i, h)
            pooled = snapkv.maxpool1d(vote[i, h, :P].astype(np.float64), wl.pool_kernel)
            want = snapkv.snapkv_keep(pooled, wl.S, wl.W, wl.keep_k)
            np.testing.assert_array_equal(keep[i, h, :len(want)], want)


def test_small_two_layers():
    wl = workloads.snapkv_custom(seed=31, L=2, Hq=8, Hkv=2, d=128, S=3000, W=16, keep_k=256,
                                 n_planted=8, plant_amp=16.0)
    layers = [wl.layer(l) for l in range(wl.L)]
    st = SnapState(wl, layers)
    st.run()
    _check(st)
    keep = st.keep.cpu().numpy()
    for i, lay in enumerate(layers):
        for h in range(wl.Hkv):
            assert set(lay.planted[h].tolist()) <= set(keep[i, h].tolist())


@pytest.mark.parametrize("S,W,keep_k,G", [(1000, 32, 2048, 7), (40, 40, 16, 2), (777, 5, 100, 1),
                                          (4099, 32, 1024, 7)])
def test_shapes_and_short_prompts(S, W, keep_k, G):
    wl = workloads.snapkv_custom(seed=S, L=1, Hq=4 * G, Hkv=4, d=128, S=S, W=W, keep_k=keep_k,
                                 n_planted=2)
    st = SnapState(wl, [wl.layer(0)])
    st.run()
    if S - W <= keep_k:
        keep = st.keep.cpu().numpy()
        for h in range(wl.Hkv):
            assert keep[0, h].tolist() == list(range(S)) + [-1] * (keep_k + W - S)
        if S > W:
            _check(st)
    else:
        _check(st)


@pytest.mark.slow
def test_full_size_qwen7b_sampled_layers():
    """28 layers x 32K prompt, 28 q / 4 kv heads, W=32, pool 7, keep 2048 (+32)."""
    wl = workloads.snapkv_qwen7b()
    layers = [wl.layer(l) for l in range(wl.L)]
    st = SnapState(wl, layers)
    st.run()
    _check(st, layer_ids=[0, 27], kv_heads=[0, 3])
    keep = st.keep.cpu().numpy()
    assert keep.shape == (28, 4, 2080)
    assert (np.diff(keep, axis=-1) > 0).all()
    kept = sum(len(set(lay.planted[h].tolist()) & set(keep[i, h].tolist()))
               for i, lay in enumerate(layers) for h in range(wl.Hkv))
    assert kept >= 0.99 * 28 * 4 * 64, kept


# ---- the union keep mode and cold-start seeds (kvsel_snapkv_select_ex) ----

def _run_ex(st, mode, head_pad=5, layer_pad=3):
    """Run the extended entry point; seeds go to strided rows padded with NaN sentinels."""
    wl = st.wl
    L = len(st.layers)
    G = wl.G if mode == K.KVSEL_SNAP_HEAD_UNION else 1
    cap = G * wl.keep_k + wl.W
    hs = cap + head_pad
    ls = wl.Hkv * hs + layer_pad
    g = Guards()
    seed = g.new((L * ls,), torch.float32, fill=float("nan"))
    keep = g.new((L, wl.Hkv, cap), torch.int32, fill=-7)
    count = g.new((L, wl.Hkv), torch.int32, fill=-7)
    vrows = wl.Hq if mode == K.KVSEL_SNAP_HEAD_UNION else wl.Hkv
    vote = g.new((L, vrows, max(wl.S - wl.W, 1)), torch.float32)
    ws = g.new((K.kvsel_snapkv_select_ex_workspace(st.kv, L, wl.S, wl.W, True, mode),), torch.uint8)
    K.kvsel_snapkv_select_ex(st.kv, st.bt, st.q, keep, ws, seq_len=wl.S, keep_k=wl.keep_k, mode=mode,
                             pool_kernel=wl.pool_kernel, vote_out=vote, keep_count=count, seed_out=seed,
                             seed_layer_stride=ls, seed_head_stride=hs)
    torch.cuda.synchronize()
    assert K.read_status(ws) == 0
    g.check()
    seed = seed.cpu().numpy()
    rows = np.stack([np.stack([seed[l * ls + h * hs:l * ls + h * hs + cap] for h in range(wl.Hkv)])
                     for l in range(L)])
    # nothing written between the rows
    for l in range(L):
        for h in range(wl.Hkv):
            assert np.isnan(seed[l * ls + h * hs + cap:l * ls + (h + 1) * hs]).all()
        assert np.isnan(seed[l * ls + wl.Hkv * hs:(l + 1) * ls]).all()
    return keep.cpu().numpy(), count.cpu().numpy(), vote.cpu().numpy(), rows


def _check_seeds(wl, lay, h, keep_row, n, seed_row):
    want = snapkv.prefill_seed(bf16_bits_to_f64(lay.q_obs[h * wl.G:(h + 1) * wl.G]),
                               bf16_bits_to_f64(lay.K[h:h + 1]), wl.scale)[0]
    assert rel_l2(seed_row[:n], want[keep_row[:n]]) < TOL
    assert (seed_row[n:] == 0).all()


@pytest.mark.parametrize("S,W,keep_k,G", [(3000, 16, 256, 4), (1000, 32, 2048, 7), (40, 40, 16, 2),
                                          (777, 5, 100, 1)])
def test_group_sum_seeds_and_counts(S, W, keep_k, G):
    wl = workloads.snapkv_custom(seed=S + 1, L=2, Hq=2 * G, Hkv=2, d=128, S=S, W=W, keep_k=keep_k,
                                 n_planted=4)
    st = SnapState(wl, [wl.layer(l) for l in range(wl.L)])
    keep, count, vote, seed = _run_ex(st, K.KVSEL_SNAP_GROUP_SUM)
    P = S - W
    for i, lay in enumerate(st.layers):
        for h in range(wl.Hkv):
            if P > keep_k:
                pooled = snapkv.maxpool1d(vote[i, h, :P].astype(np.float64), wl.pool_kernel)
                want = snapkv.snapkv_keep(pooled, S, W, keep_k)
            else:
                want = np.arange(S)
            n = len(want)
            assert count[i, h] == n
            np.testing.assert_array_equal(keep[i, h, :n], want)
            assert (keep[i, h, n:] == -1).all()
            _check_seeds(wl, lay, h, keep[i, h], n, seed[i, h])
            # a kept prefix key's seed is its raw vote
            pre = keep[i, h, :n] < P
            np.testing.assert_array_equal(seed[i, h, :n][pre], vote[i, h, keep[i, h, :n][pre]])


@pytest.mark.parametrize("S,W,keep_k,G", [(3000, 32, 128, 7), (4099, 5, 300, 2), (2000, 16, 64, 4),
                                          (777, 8, 100, 1), (300, 16, 512, 3)])
def test_union_of_per_head_picks(S, W, keep_k, G):
    wl = workloads.snapkv_custom(seed=S + 2, L=1, Hq=4 * G, Hkv=4, d=128, S=S, W=W, keep_k=keep_k,
                                 n_planted=4)
    st = SnapState(wl, [wl.layer(0)])
    keep, count, vote, seed = _run_ex(st, K.KVSEL_SNAP_HEAD_UNION)
    lay = st.layers[0]
    P = S - W
    want_vote = snapkv.snapkv_vote_per_head(bf16_bits_to_f64(lay.q_obs), bf16_bits_to_f64(lay.K), wl.scale)
    for qh in range(wl.Hq):
        assert rel_l2(vote[0, qh, :P], want_vote[qh]) < TOL, qh
    sizes = []
    for h in range(wl.Hkv):
        pooled = snapkv.maxpool1d(vote[0, h * G:(h + 1) * G, :P].astype(np.float64), wl.pool_kernel)
        want = snapkv.snapkv_union_keep(pooled, S, W, keep_k)
        n = len(want)
        assert count[0, h] == n
        np.testing.assert_array_equal(keep[0, h, :n], want)
        assert (keep[0, h, n:] == -1).all()
        _check_seeds(wl, lay, h, keep[0, h], n, seed[0, h])
        sizes.append(n - W)
    if P > keep_k and G > 1:
        assert max(sizes) > keep_k           # the heads disagree somewhere


@pytest.mark.slow
def test_full_size_qwen7b_union_with_seeds_sampled():
    """28 layers x 32K, 28 q / 4 kv heads, W=32, pool 7, keep 2048 per q head, union + seeds."""
    wl = workloads.snapkv_qwen7b()
    layers = [wl.layer(l) for l in range(wl.L)]
    st = SnapState(wl, layers)
    keep, count, vote, seed = _run_ex(st, K.KVSEL_SNAP_HEAD_UNION)
    P = wl.S - wl.W
    G = wl.G
    for i in (0, 27):
        lay = layers[i]
        for h in (0, 3):
            q = bf16_bits_to_f64(lay.q_obs[h * G:(h + 1) * G])
            k = bf16_bits_to_f64(lay.K[h:h + 1])
            want_vote = snapkv.snapkv_vote_per_head(q, k, wl.scale)
            for g in range(G):
                assert rel_l2(vote[i, h * G + g, :P], want_vote[g]) < TOL
            pooled = snapkv.maxpool1d(vote[i, h * G:(h + 1) * G, :P].astype(np.float64), wl.pool_kernel)
            want = snapkv.snapkv_union_keep(pooled, wl.S, wl.W, wl.keep_k)
            n = len(want)
            assert count[i, h] == n
            np.testing.assert_array_equal(keep[i, h, :n], want)
            _check_seeds(wl, lay, h, keep[i, h], n, seed[i, h])
    assert (count >= wl.keep_k + wl.W).all() and (count <= G * wl.keep_k + wl.W).all()
    kept = 0
    for i, lay in enumerate(layers):
        for h in range(wl.Hkv):
            row = keep[i, h, :count[i, h]]
            assert (np.diff(row) > 0).all()
            kept += len(set(lay.planted[h].tolist()) & set(row.tolist()))
    assert kept >= 0.99 * 28 * 4 * 64, kept


@pytest.mark.parametrize("pool_kernel", [1, 3, 9, 13, 33])
def test_pool_widths(pool_kernel):
    # the pool is taken while the select loads the votes: lane shuffles up to
    # a half-width of 4, a plain loop above
    wl = workloads.snapkv_custom(seed=pool_kernel, L=1, Hq=8, Hkv=2, d=128, S=5000, W=16, keep_k=300,
                                 pool_kernel=pool_kernel, n_planted=4)
    st = SnapState(wl, [wl.layer(0)])
    st.run()
    _check(st)
    keep, count, vote, _ = _run_ex(st, K.KVSEL_SNAP_HEAD_UNION)
    P = wl.S - wl.W
    for h in range(wl.Hkv):
        pooled = snapkv.maxpool1d(vote[0, h * wl.G:(h + 1) * wl.G, :P].astype(np.float64), pool_kernel)
        want = snapkv.snapkv_union_keep(pooled, wl.S, wl.W, wl.keep_k)
        np.testing.assert_array_equal(keep[0, h, :count[0, h]], want)


def test_prefix_longer_than_the_register_rows():
    # prefix > 32768: the select sweeps the row in parts and re-reads (and re-pools) the votes
    wl = workloads.snapkv_custom(seed=77, L=1, Hq=8, Hkv=2, d=128, S=40000, W=32, keep_k=1024, n_planted=8,
                                 plant_amp=16.0)
    st = SnapState(wl, [wl.layer(0)])
    st.run()
    _check(st)
    keep, count, vote, seed = _run_ex(st, K.KVSEL_SNAP_HEAD_UNION)
    P = wl.S - wl.W
    lay = st.layers[0]
    for h in range(wl.Hkv):
        pooled = snapkv.maxpool1d(vote[0, h * wl.G:(h + 1) * wl.G, :P].astype(np.float64), wl.pool_kernel)
        want = snapkv.snapkv_union_keep(pooled, wl.S, wl.W, wl.keep_k)
        n = len(want)
        np.testing.assert_array_equal(keep[0, h, :n], want)
        _check_seeds(wl, lay, h, keep[0, h], n, seed[0, h])
