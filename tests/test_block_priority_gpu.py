"""GPU parity of block offload priority against the oracle.

* block scores (and the decayed token scores) within relative L2 2e-3 of the
  fp64 oracle;
* the eviction order bit-exact when the oracle's percentile / order routines
  are fed the GPU's own fp32 block scores (the selection is compared on
  identical inputs);
* with max aggregation and no update the block scores are exact, so the
  order must also equal the oracle's end to end.
"""
import math

import numpy as np
import pytest
import torch

import workloads
from oracle import block_priority as BP
from _harness import Guards, rel_l2

import attention_guided_kv_gb300 as K

pytestmark = pytest.mark.gpu
TOL = 2e-3


def _run(tok, offsets, bs, agg, norm, frac, inc=None, decay=1.0, top_p=0.1):
    dev = "cuda"
    R = len(offsets) - 1
    nblk = sum(int(-(-int(offsets[r + 1] - offsets[r]) // bs)) for r in range(R))
    maxb = max(nblk, 1)
    g = Guards()
    t_tok = g.like(torch.from_numpy(np.asarray(tok, dtype=np.float32)).to(dev))
    t_inc = None if inc is None else torch.from_numpy(np.asarray(inc, dtype=np.float32)).to(dev)
    t_off = torch.from_numpy(np.asarray(offsets, dtype=np.int64)).to(dev)
    bso = g.new((maxb,), torch.float32, fill=float("nan"))
    cap = max(1, math.ceil(frac * maxb))
    order = g.new((cap,), torch.int64, fill=-7)
    n_out = g.new((2,), torch.int64)
    ws = g.new((K.kvsel_block_priority_workspace(R, maxb),), torch.uint8)
    K.kvsel_block_priority(t_tok, t_off, order, n_out, ws, block_size=bs, agg=agg, norm=norm,
                           evict_frac=frac, increment=t_inc, decay=decay, top_p=top_p,
                           block_score_out=bso, max_total_blocks=maxb)
    assert K.read_status(ws) == 0
    g.check()
    n_ev, N = n_out.cpu().tolist()
    assert N == nblk
    return t_tok.cpu().numpy(), bso.cpu().numpy()[:nblk], order.cpu().numpy()[:n_ev], n_ev


def _split(blk, offsets, bs):
    out, g = [], 0
    for r in range(len(offsets) - 1):
        n = int(-(-int(offsets[r + 1] - offsets[r]) // bs))
        out.append(blk[g:g + n])
        g += n
    return out


def _expected_order(blocks_per_req, norm, frac):
    if norm == BP.NORM_PERCENTILE:
        keys = [BP.percentiles(b.astype(np.float64)).astype(np.float64) for b in blocks_per_req]
    else:
        keys = [b.astype(np.float64) for b in blocks_per_req]
    return BP.evict_order(keys, float(np.float32(frac)))


@pytest.mark.parametrize("bs", [16, 64, 256])
@pytest.mark.parametrize("agg", [BP.AGG_MAX, BP.AGG_MEAN, BP.AGG_TOPP])
def test_fold_and_order_small_workload(bs, agg):
    wl = workloads.block_priority(seed=7, R=9, steps=3, min_len=300, max_len=9000)
    off = wl.offsets
    tok = wl.increments(0)
    inc = wl.increments(1)
    new_tok, blk, order, n_ev = _run(tok, off, bs, agg, BP.NORM_PERCENTILE, 0.25, inc=inc, decay=0.98)
    want_tok = BP.decay_update(tok.astype(np.float64), inc.astype(np.float64), 0.98)
    assert rel_l2(new_tok, want_tok) < 1e-6
    want_blk = np.concatenate([BP.block_scores(want_tok[off[r]:off[r + 1]], bs, agg, 0.1)
                               for r in range(wl.R)])
    assert rel_l2(blk, want_blk) < TOL
    # same fp32 block scores into the oracle's normalisation + order: bit-exact
    want = _expected_order(_split(blk, off, bs), BP.NORM_PERCENTILE, 0.25)
    assert n_ev == len(want) == math.ceil(0.25 * len(blk))
    np.testing.assert_array_equal(order, want)


@pytest.mark.parametrize("norm", [BP.NORM_PERCENTILE, BP.NORM_NONE])
def test_max_aggregation_order_is_exact_end_to_end(norm):
    rng = np.random.default_rng(5)
    lens = rng.integers(1, 3000, 13)
    off = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
    tok = (rng.integers(0, 40, int(off[-1])) * 0.25).astype(np.float32)    # many ties
    _, blk, order, _ = _run(tok, off, 16, BP.AGG_MAX, norm, 0.4)
    blocks, normed, want = BP.priority_pass(tok.astype(np.float64), off, 16, BP.AGG_MAX, 0.1, norm, 0.4)
    np.testing.assert_array_equal(blk, np.concatenate(blocks).astype(np.float32))
    np.testing.assert_array_equal(order, want)


@pytest.mark.parametrize("nblocks", [8192, 8193, 12500, 16384, 16385, 24576, 40000])
def test_percentile_ranks_at_and_above_8192_blocks(nblocks):
    """Requests of up to 8192 blocks are ranked by the shared-memory radix sort, up to 16384 by
    the register bitonic sort and above that by the radix sort through the workspace (whole
    tiles, a ragged last tile): all must give the oracle's order."""
    rng = np.random.default_rng(nblocks)
    lens = np.array([nblocks * 16 - 7, 300, nblocks * 16], dtype=np.int64)
    off = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
    tok = (rng.integers(0, 500, int(off[-1])) * 0.125).astype(np.float32)   # ties across blocks
    _, blk, order, _ = _run(tok, off, 16, BP.AGG_MAX, BP.NORM_PERCENTILE, 0.3)
    blocks, normed, want = BP.priority_pass(tok.astype(np.float64), off, 16, BP.AGG_MAX, 0.1,
                                            BP.NORM_PERCENTILE, 0.3)
    np.testing.assert_array_equal(blk, np.concatenate(blocks).astype(np.float32))
    np.testing.assert_array_equal(order, want)


def test_edge_cases():
    # single-token requests, an empty request, frac 0 and 1
    off = np.array([0, 1, 1, 5, 37], dtype=np.int64)
    tok = np.linspace(1.0, 0.0, 37).astype(np.float32)
    for frac in (0.0, 1.0):
        _, blk, order, n_ev = _run(tok, off, 16, BP.AGG_MEAN, BP.NORM_PERCENTILE, frac)
        want = _expected_order(_split(blk, off, 16), BP.NORM_PERCENTILE, frac)
        assert n_ev == len(want)
        np.testing.assert_array_equal(order, want)
    _, blk, _, _ = _run(tok, off, 16, BP.AGG_TOPP, BP.NORM_NONE, 0.5, top_p=1.0)
    want = np.concatenate([BP.block_scores(tok[off[r]:off[r + 1]].astype(np.float64), 16, BP.AGG_TOPP, 1.0)
                           for r in range(4)])
    assert rel_l2(blk, want) < 1e-6


def test_dirichlet_decay_invariant_on_device():
    # increments sum to one per request per step: after T steps each request's
    # token scores sum to (1 - 0.98^T) / (1 - 0.98)
    wl = workloads.block_priority(seed=3, R=6, steps=40, min_len=4096, max_len=20000)
    off = wl.offsets
    tok = np.zeros(wl.total_tokens, dtype=np.float32)
    R = wl.R
    t_tok = torch.from_numpy(tok).cuda()
    t_off = torch.from_numpy(off).cuda()
    nblk = int(sum(-(-int(x) // 64) for x in wl.lengths))
    order = torch.zeros(nblk, dtype=torch.int64, device="cuda")
    n_out = torch.zeros(2, dtype=torch.int64, device="cuda")
    ws = K.workspace(K.kvsel_block_priority_workspace(R, nblk))
    for t in range(wl.steps):
        inc = torch.from_numpy(wl.increments(t)).cuda()
        K.kvsel_block_priority(t_tok, t_off, order, n_out, ws, block_size=64, agg=BP.AGG_MEAN,
                               norm=BP.NORM_PERCENTILE, evict_frac=0.25, increment=inc, decay=0.98,
                               max_total_blocks=nblk)
    sums = np.add.reduceat(t_tok.double().cpu().numpy(), off[:-1])
    np.testing.assert_allclose(sums, (1 - 0.98 ** 40) / (1 - 0.98), rtol=1e-4)
    assert K.read_status(ws) == 0


@pytest.mark.slow
def test_full_size_64_requests_all_variants():
    """64 requests, 4K..128K tokens: every block size / aggregation, order bit-exact."""
    wl = workloads.block_priority()
    off = wl.offsets
    tok = wl.increments(0)
    inc = wl.increments(1)
    want_tok = BP.decay_update(tok.astype(np.float64), inc.astype(np.float64), 0.98)
    for bs in (16, 64, 256):
        for agg in (BP.AGG_MAX, BP.AGG_MEAN, BP.AGG_TOPP):
            new_tok, blk, order, n_ev = _run(tok, off, bs, agg, BP.NORM_PERCENTILE, 0.25, inc=inc,
                                             decay=0.98)
            assert rel_l2(new_tok, want_tok) < 1e-6
            if agg == BP.AGG_MAX:
                want_blk = np.concatenate([BP.block_scores(new_tok[off[r]:off[r + 1]], bs, agg)
                                           for r in range(wl.R)])
                assert rel_l2(blk, want_blk) < TOL
            want = _expected_order(_split(blk, off, bs), BP.NORM_PERCENTILE, 0.25)
            np.testing.assert_array_equal(order, want)


# --- temporal aggregation variants and block policies -----------------------
def _run_ex(tok_dev, off, bs, agg, norm, frac, **kw):
    dev = "cuda"
    R = len(off) - 1
    nblk = sum(int(-(-int(off[r + 1] - off[r]) // bs)) for r in range(R))
    t_off = torch.from_numpy(np.asarray(off, dtype=np.int64)).to(dev)
    g = Guards()
    bso = g.new((nblk,), torch.float32, fill=float("nan"))
    order = g.new((max(1, math.ceil(frac * nblk)),), torch.int64, fill=-7)
    n_out = g.new((2,), torch.int64)
    ws = g.new((K.kvsel_block_priority_workspace(R, nblk),), torch.uint8)
    K.kvsel_block_priority(tok_dev, t_off, order, n_out, ws, block_size=bs, agg=agg, norm=norm,
                           evict_frac=frac, block_score_out=bso, max_total_blocks=nblk, **kw)
    assert K.read_status(ws) == 0
    g.check()
    n_ev, N = n_out.cpu().tolist()
    assert N == nblk
    return bso.cpu().numpy(), order.cpu().numpy()[:n_ev]


@pytest.mark.parametrize("update", [K.KVSEL_UPDATE_MAX, K.KVSEL_UPDATE_WINDOW])
def test_max_and_window_updates_over_steps(update):
    rng = np.random.default_rng(11 + update)
    lens = rng.integers(1, 900, 6)
    off = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
    T, W, steps = int(off[-1]), 3, 7
    tok = torch.zeros(T, device="cuda")
    hist = torch.zeros(W, T, device="cuda")
    incs = [rng.dirichlet(np.full(T, 0.5)).astype(np.float32) for _ in range(steps)]
    want = np.zeros(T)
    for t, inc in enumerate(incs):
        blk, order = _run_ex(tok, off, 16, BP.AGG_MAX, BP.NORM_PERCENTILE, 0.25,
                             increment=torch.from_numpy(inc).cuda(), update=update, history=hist,
                             window=W, step=t)
        if update == K.KVSEL_UPDATE_MAX:
            want = BP.max_update(want, inc)
        got = tok.cpu().numpy()
        if update == K.KVSEL_UPDATE_MAX:
            np.testing.assert_array_equal(got, want.astype(np.float32))       # max is exact
        else:
            assert rel_l2(got, BP.window_sum(incs[:t + 1], W)) < 1e-6
        # the order on the GPU's own scores is exact
        blocks, _, exp = BP.priority_pass(got.astype(np.float64), off, 16, BP.AGG_MAX, 0.1,
                                          BP.NORM_PERCENTILE, 0.25)
        np.testing.assert_array_equal(blk, np.concatenate(blocks).astype(np.float32))
        np.testing.assert_array_equal(order, exp)


@pytest.mark.parametrize("agg", [K.KVSEL_AGG_FRAC_HOT, K.KVSEL_AGG_ALL_COLD])
@pytest.mark.parametrize("norm", [BP.NORM_NONE, BP.NORM_PERCENTILE])
@pytest.mark.parametrize("bs", [16, 64])
def test_threshold_policies_exact(agg, norm, bs):
    rng = np.random.default_rng(3 + agg + 10 * norm + bs)
    lens = rng.integers(1, 4000, 9)
    off = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
    tok = (rng.integers(0, 64, int(off[-1])) * 0.015625).astype(np.float32)  # ties, exact in fp32
    thr = 0.75
    blk, order = _run_ex(torch.from_numpy(tok).cuda(), off, bs, agg, norm, 0.4, threshold=thr)
    blocks, _, want = BP.priority_pass(tok.astype(np.float64), off, bs, agg, 0.1, norm, 0.4, threshold=thr)
    np.testing.assert_array_equal(blk, np.concatenate(blocks).astype(np.float32))
    np.testing.assert_array_equal(order, want)


@pytest.mark.parametrize("agg", [BP.AGG_MAX, K.KVSEL_AGG_ALL_COLD])
def test_token_level_blocks_of_long_requests(agg):
    """Block size 1 turns every token into a block: requests of 100K and 70K tokens rank through
    the workspace sort (13 and 9 tiles), with thousands of tied scores, next to short ones."""
    rng = np.random.default_rng(17 + agg)
    lens = np.array([100000, 5, 70001, 0, 3000], dtype=np.int64)
    off = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
    tok = (rng.integers(0, 300, int(off[-1])) * 0.125).astype(np.float32)   # exact in fp32, tied
    kw = {"threshold": 30.0} if agg == K.KVSEL_AGG_ALL_COLD else {}
    blk, order = _run_ex(torch.from_numpy(tok).cuda(), off, 1, agg, BP.NORM_PERCENTILE, 0.3, **kw)
    blocks, _, want = BP.priority_pass(tok.astype(np.float64), off, 1, agg, 0.1, BP.NORM_PERCENTILE, 0.3, **kw)
    np.testing.assert_array_equal(blk, np.concatenate(blocks).astype(np.float32))
    np.testing.assert_array_equal(order, want)
