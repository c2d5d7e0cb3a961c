"""GPU parity of keep-list compaction (kvsel_kv_compact) against the oracle.

The oracle's eviction step (``H2OSequence.apply_keep``: gather every kv head's
K, V, score and position rows by its keep list, in order) is run on the raw
bf16 bit patterns, so the comparison is byte-exact.  Covered: random keep
lists with permuted pages and ragged page tails, counts taken from the rows'
-1 padding, rejected lists (the sequence is left untouched, the others are
compacted), and SnapKV's keep lists on the Qwen2.5-7B shape, with the
cold-start seeds written straight into the compacted score rows.
"""
import numpy as np
import pytest
import torch

import workloads
from oracle.h2o import H2OSequence
from oracle import snapkv
from oracle.attention import bf16_bits_to_f64
from _harness import Guards, bf16, rel_l2

import attention_guided_kv_gb300 as K

pytestmark = pytest.mark.gpu
PAGE = 16


class PagedBatch:
    """A paged cache of random bf16 rows with permuted pages and spare pages."""

    def __init__(self, seed, S_list, Hkv, spare=3, max_len=None, page=PAGE):
        rng = np.random.default_rng(seed)
        self.rng = rng
        self.page = P = page
        self.S = list(S_list)
        self.B, self.Hkv = len(S_list), Hkv
        self.max_len = max_len or max(max(S_list), 1)
        self.max_pages = (self.max_len + P - 1) // P
        used = sum((s + P - 1) // P for s in S_list)
        self.num_pages = used + spare
        ids = rng.permutation(self.num_pages).astype(np.int32)
        self.bt = np.full((self.B, self.max_pages), -1, dtype=np.int32)
        o = 0
        for b, s in enumerate(S_list):
            n = (s + P - 1) // P
            self.bt[b, :n] = ids[o:o + n]
            o += n
        self.kbits = rng.integers(0, 1 << 16, (self.num_pages, Hkv, P, 128), dtype=np.uint16)
        self.vbits = rng.integers(0, 1 << 16, (self.num_pages, Hkv, P, 128), dtype=np.uint16)
        self.scores = rng.random((self.B, Hkv, self.max_len), dtype=np.float32)
        self.pos = rng.integers(0, 1 << 30, (self.B, Hkv, self.max_len), dtype=np.int32)

    def logical(self, pool, b, S, bt=None):
        bt = self.bt if bt is None else bt
        out = np.zeros((self.Hkv, S, 128), dtype=np.uint16)
        for t in range(S):
            out[:, t] = pool[bt[b, t // self.page], :, t % self.page]
        return out

    def upload(self, g):
        self.kpool = bf16(self.kbits)
        self.vpool = bf16(self.vbits)
        self.kv = K.paged_kv(self.kpool, self.vpool, self.Hkv)
        self.d_bt = g.like(torch.from_numpy(self.bt).cuda())
        self.d_seq = g.like(torch.tensor(self.S, dtype=torch.int32, device="cuda"))
        self.d_scores = g.like(torch.from_numpy(self.scores).cuda())
        self.d_pos = g.like(torch.from_numpy(self.pos).cuda())
        self.d_freed = g.new((self.B, self.max_pages), torch.int32, fill=-7)


def _expected(pb, b, keep_rows):
    """The oracle's eviction step on the bit patterns of sequence b."""
    S = pb.S[b]
    ref = H2OSequence(pb.logical(pb.kbits, b, S).astype(np.float64),
                      pb.logical(pb.vbits, b, S).astype(np.float64))
    ref.cum = pb.scores[b, :, :S].astype(np.float64)
    ref.pos = pb.pos[b, :, :S].astype(np.int64)
    ref.apply_keep(np.asarray(keep_rows, dtype=np.int64).reshape(pb.Hkv, -1))
    return ref


def _check_sequence(pb, b, keep_rows, kn, vn, bt_new, scores_new, pos_new, freed, seq_new):
    n = len(keep_rows[0])
    ref = _expected(pb, b, keep_rows)
    assert seq_new[b] == n
    got_k = pb.logical(kn, b, n, bt_new).astype(np.float64)
    got_v = pb.logical(vn, b, n, bt_new).astype(np.float64)
    np.testing.assert_array_equal(got_k, ref.K)
    np.testing.assert_array_equal(got_v, ref.V)
    np.testing.assert_array_equal(scores_new[b, :, :n].astype(np.float64), ref.cum)
    np.testing.assert_array_equal(pos_new[b, :, :n].astype(np.int64), ref.pos)
    P = pb.page
    old_p, new_p = (pb.S[b] + P - 1) // P, (n + P - 1) // P
    np.testing.assert_array_equal(bt_new[b, :new_p], pb.bt[b, :new_p])
    assert (bt_new[b, new_p:old_p] == -1).all()
    np.testing.assert_array_equal(bt_new[b, old_p:], pb.bt[b, old_p:])
    assert freed[b, :old_p - new_p].tolist() == pb.bt[b, new_p:old_p].tolist()
    assert (freed[b, old_p - new_p:] == -1).all()


def _random_rows(rng, S, n, Hkv, structured):
    rows = []
    for _ in range(Hkv):
        if structured and n >= 8 and S >= n + 8:   # sinks + window + a random middle, as H2O keeps
            mid = np.sort(rng.choice(np.arange(4, S - 4), n - 8, replace=False))
            rows.append(np.concatenate([np.arange(4), mid, np.arange(S - 4, S)]))
        else:
            rows.append(np.sort(rng.choice(S, n, replace=False)))
    return [r.astype(np.int32) for r in rows]


@pytest.mark.parametrize("with_count,page", [(True, 16), (False, 16), (True, 256), (False, 64)])
def test_random_keep_lists_move_bytes_exactly(with_count, page):
    # ragged tails, a whole page kept exactly, an empty keep, a 3-chunk row,
    # identity rows (nothing moves) and a zero-length sequence; pages of 16 to 256 tokens
    S_list = [700, 33, 1000, 5, 16, 0, 611]
    n_list = [300, 17, 999, 0, 16, 0, 611]
    Hkv = 4
    pb = PagedBatch(11 + with_count, S_list, Hkv, page=page)
    stride = max(n_list) + 5
    keep = np.full((pb.B, Hkv, stride), -1, dtype=np.int32)
    counts = np.zeros((pb.B, Hkv), dtype=np.int32)
    rows_by_seq = []
    for b, (S, n) in enumerate(zip(S_list, n_list)):
        rows = _random_rows(pb.rng, S, n, Hkv, structured=(b % 2 == 0))
        rows_by_seq.append(rows)
        for h in range(Hkv):
            keep[b, h, :n] = rows[h]
            counts[b, h] = n
    g = Guards()
    pb.upload(g)
    d_keep = torch.from_numpy(keep).cuda()
    d_count = g.like(torch.from_numpy(counts).cuda()) if with_count else None
    ws = g.new((K.kvsel_kv_compact_workspace(pb.B, Hkv),), torch.uint8)
    K.kvsel_kv_compact(pb.kv, pb.d_bt, pb.d_seq, d_keep, ws, keep_count=d_count, scores=pb.d_scores,
                       pos_map=pb.d_pos, freed_pages=pb.d_freed)
    assert K.read_status(ws) == 0
    g.check()
    kn = pb.kpool.view(torch.int16).cpu().numpy().view(np.uint16)
    vn = pb.vpool.view(torch.int16).cpu().numpy().view(np.uint16)
    args = (kn, vn, pb.d_bt.cpu().numpy(), pb.d_scores.cpu().numpy(), pb.d_pos.cpu().numpy(),
            pb.d_freed.cpu().numpy(), pb.d_seq.cpu().numpy())
    for b in range(pb.B):
        _check_sequence(pb, b, rows_by_seq[b], *args)


@pytest.mark.parametrize("fault", ["counts_differ", "not_ascending", "slot_beyond_length",
                                   "count_beyond_stride", "length_beyond_table"])
def test_rejected_sequence_is_left_untouched(fault):
    S_list = [500, 400]
    Hkv, n, stride = 2, 120, 130
    pb = PagedBatch(5, S_list, Hkv)
    keep = np.full((2, Hkv, stride), -1, dtype=np.int32)
    counts = np.full((2, Hkv), n, dtype=np.int32)
    rows_by_seq = [_random_rows(pb.rng, S, n, Hkv, True) for S in S_list]
    for b in range(2):
        for h in range(Hkv):
            keep[b, h, :n] = rows_by_seq[b][h]
    S_dev = list(S_list)
    if fault == "counts_differ":      # e.g. the union mode's per-head counts
        counts[1, 1] = n - 1
    elif fault == "not_ascending":
        keep[1, 0, 50], keep[1, 0, 51] = keep[1, 0, 51], keep[1, 0, 50]
    elif fault == "slot_beyond_length":
        keep[1, 1, n - 1] = S_list[1]
    elif fault == "count_beyond_stride":
        counts[1, :] = stride + 1
    elif fault == "length_beyond_table":
        S_dev[1] = pb.max_pages * PAGE + 1
    g = Guards()
    pb.upload(g)
    pb.d_seq.copy_(torch.tensor(S_dev, dtype=torch.int32))
    ws = K.workspace(K.kvsel_kv_compact_workspace(2, Hkv))
    K.kvsel_kv_compact(pb.kv, pb.d_bt, pb.d_seq, torch.from_numpy(keep).cuda(), ws,
                       keep_count=torch.from_numpy(counts).cuda(), scores=pb.d_scores, pos_map=pb.d_pos,
                       freed_pages=pb.d_freed)
    assert K.read_status(ws) == K.KVSEL_ERR_BAD_INDEX
    g.check()
    kn = pb.kpool.view(torch.int16).cpu().numpy().view(np.uint16)
    vn = pb.vpool.view(torch.int16).cpu().numpy().view(np.uint16)
    bt_new, seq_new = pb.d_bt.cpu().numpy(), pb.d_seq.cpu().numpy()
    freed = pb.d_freed.cpu().numpy()
    # the valid sequence is compacted ...
    _check_sequence(pb, 0, rows_by_seq[0], kn, vn, bt_new, pb.d_scores.cpu().numpy(), pb.d_pos.cpu().numpy(),
                    freed, seq_new)
    # ... the rejected one keeps its bytes, table, length, scores and positions
    S1 = S_list[1]
    np.testing.assert_array_equal(pb.logical(kn, 1, S1), pb.logical(pb.kbits, 1, S1))
    np.testing.assert_array_equal(pb.logical(vn, 1, S1), pb.logical(pb.vbits, 1, S1))
    np.testing.assert_array_equal(bt_new[1], pb.bt[1])
    assert seq_new[1] == S_dev[1]
    np.testing.assert_array_equal(pb.d_scores.cpu().numpy()[1], pb.scores[1])
    np.testing.assert_array_equal(pb.d_pos.cpu().numpy()[1], pb.pos[1])
    assert (freed[1] == -7).all()


class SnapCache:
    """SnapKV layers in one paged K and V pool (layer l owns pages l*P .. l*P+P-1)."""

    def __init__(self, wl, layer_ids, g):
        self.wl = wl
        self.layers = [wl.layer(l) for l in layer_ids]
        L, P = len(self.layers), wl.pages
        kpool = np.zeros((L * P, wl.Hkv, PAGE, wl.d), dtype=np.uint16)
        vpool = np.zeros_like(kpool)
        bts = np.zeros((L, P), dtype=np.int32)
        q = np.zeros((L, wl.Hq, wl.W, wl.d), dtype=np.uint16)
        for i, lay in enumerate(self.layers):
            kpool[i * P:(i + 1) * P] = workloads.paged_pool(lay.K[None], lay.block_table[None], P)
            vpool[i * P:(i + 1) * P] = workloads.paged_pool(lay.V[None], lay.block_table[None], P)
            bts[i] = lay.block_table + i * P
            q[i] = lay.q_obs
        self.bt_host = bts
        self.kpool, self.vpool = bf16(kpool), bf16(vpool)
        self.kv = K.paged_kv(self.kpool, self.vpool, wl.Hq)
        self.bt = g.like(torch.from_numpy(bts).cuda())
        self.q = bf16(q)
        self.seq = g.like(torch.full((L,), wl.S, dtype=torch.int32, device="cuda"))
        cap = wl.keep_k + wl.W
        self.keep = g.new((L, wl.Hkv, cap), torch.int32, fill=-7)
        self.count = g.new((L, wl.Hkv), torch.int32, fill=-7)
        self.row = max(wl.S, cap)        # score row: every seed row needs the keep capacity
        self.cum = g.new((L, wl.Hkv, self.row), torch.float32, fill=float("nan"))
        self.freed = g.new((L, P), torch.int32, fill=-7)

    def select_and_compact(self):
        wl, L = self.wl, len(self.layers)
        ws = K.workspace(K.kvsel_snapkv_select_ex_workspace(self.kv, L, wl.S, wl.W, False))
        K.kvsel_snapkv_select_ex(self.kv, self.bt, self.q, self.keep, ws, seq_len=wl.S, keep_k=wl.keep_k,
                                 pool_kernel=wl.pool_kernel, keep_count=self.count, seed_out=self.cum,
                                 seed_layer_stride=wl.Hkv * self.row, seed_head_stride=self.row)
        ws2 = K.workspace(K.kvsel_kv_compact_workspace(L, wl.Hkv))
        torch.cuda.synchronize()
        keep_before = self.keep.cpu().numpy().copy()
        K.kvsel_kv_compact(self.kv, self.bt, self.seq, self.keep, ws2, keep_count=self.count,
                           freed_pages=self.freed)
        torch.cuda.synchronize()
        assert K.read_status(ws) == 0 and K.read_status(ws2) == 0
        return keep_before


def _check_snap(sc, keep, layer_ids_checked):
    wl = sc.wl
    n = min(wl.S, wl.keep_k + wl.W)
    kn = sc.kpool.view(torch.int16).cpu().numpy().view(np.uint16)
    vn = sc.vpool.view(torch.int16).cpu().numpy().view(np.uint16)
    bt_new = sc.bt.cpu().numpy()
    freed = sc.freed.cpu().numpy()
    count = sc.count.cpu().numpy()
    cum = sc.cum.cpu().numpy()
    assert (sc.seq.cpu().numpy() == n).all()
    assert (count == n).all()
    P = wl.pages
    new_p = (n + PAGE - 1) // PAGE
    for i in layer_ids_checked:
        lay = sc.layers[i]
        for h in range(wl.Hkv):
            rows = keep[i, h, :n]
            assert (np.diff(rows) > 0).all() and rows[0] >= 0 and rows[-1] < wl.S
            ref = H2OSequence(lay.K[h:h + 1].astype(np.float64), lay.V[h:h + 1].astype(np.float64))
            ref.apply_keep(rows[None].astype(np.int64))
            gk = np.stack([kn[bt_new[i, t // PAGE], h, t % PAGE] for t in range(n)]).astype(np.float64)
            gv = np.stack([vn[bt_new[i, t // PAGE], h, t % PAGE] for t in range(n)]).astype(np.float64)
            np.testing.assert_array_equal(gk, ref.K[0])
            np.testing.assert_array_equal(gv, ref.V[0])
            cap = wl.keep_k + wl.W
            assert np.isfinite(cum[i, h, :n]).all() and (cum[i, h, n:cap] == 0).all()
            assert np.isnan(cum[i, h, cap:]).all()
        assert (bt_new[i, new_p:] == -1).all()
        assert freed[i, :P - new_p].tolist() == sc.bt_host[i, new_p:].tolist()
        assert (freed[i, P - new_p:] == -1).all()


def test_snapkv_keep_then_compact_two_layers():
    wl = workloads.snapkv_custom(seed=61, L=2, Hq=8, Hkv=2, d=128, S=3000, W=16, keep_k=256,
                                 n_planted=8, plant_amp=16.0)
    g = Guards()
    sc = SnapCache(wl, [0, 1], g)
    keep = sc.select_and_compact()
    g.check()
    _check_snap(sc, keep, [0, 1])
    # the kept rows are the oracle's SnapKV keep on the GPU's votes' pool order,
    # and the seeds at the compacted slots are the oracle's window attention
    for i, lay in enumerate(sc.layers):
        for h in range(wl.Hkv):
            Kf = bf16_bits_to_f64(lay.K[h:h + 1])
            seeds = snapkv.prefill_seed(bf16_bits_to_f64(lay.q_obs[h * wl.G:(h + 1) * wl.G]), Kf, wl.scale)[0]
            n = wl.keep_k + wl.W
            assert rel_l2(sc.cum.cpu().numpy()[i, h, :n], seeds[keep[i, h, :n]]) < 2e-3


def test_snapkv_short_prompt_keeps_everything():
    wl = workloads.snapkv_custom(seed=62, L=1, Hq=8, Hkv=2, d=128, S=1000, W=32, keep_k=2048, n_planted=2)
    g = Guards()
    sc = SnapCache(wl, [0], g)
    keep = sc.select_and_compact()
    g.check()
    assert keep[0, 0, :1000].tolist() == list(range(1000))
    _check_snap(sc, keep, [0])
    np.testing.assert_array_equal(sc.bt.cpu().numpy(), sc.bt_host)


@pytest.mark.slow
def test_snapkv_compact_full_qwen7b_shape():
    """28 layers x 32K prompt, keep 2048 + 32 per kv head, compacted in place."""
    wl = workloads.snapkv_qwen7b()
    g = Guards()
    sc = SnapCache(wl, range(wl.L), g)
    keep = sc.select_and_compact()
    g.check()
    _check_snap(sc, keep, [0, 13, 27])
