"""Failure detection on the GPU, without a fault: bounded waits that run out.

A short wait limit (kvsel_set_wait_limit) and a wait that nothing ends,
planted from the host in a freshly zeroed workspace:

* decode: one (sequence, kv head) pair's readiness counter is preset far
  above the count its owners bring it to, so their wait for each other's
  statistics never completes;
* block priority: the sort's grid-barrier counter is preset so that no CTA
  is ever the last to arrive.

Each call must return, the status read back must be KVSEL_ERR_TIMEOUT, the
guards around every output must be intact, and once the workspace is zeroed
again the next call on the same workspace must match the oracle.
"""
import math

import numpy as np
import pytest
import torch

import workloads
from oracle import block_priority as BP
from oracle.attention import bf16_bits_to_f64, decode_attention
from _harness import DecodeState, Guards, bf16, rel_l2

import attention_guided_kv_gb300 as K

pytestmark = pytest.mark.gpu
TOL = 2e-3
SHORT = 20000          # spins of ~64 ns: about a millisecond per expired wait
PAIR_COUNTERS = 256    # decode workspace: the per-pair readiness counters follow the 256-byte status block
BAR_COUNTER = 64       # block-priority workspace: the sort's grid-barrier arrival counter


def _decode_ok(st, wl):
    S = wl.S0 + 1
    for b in range(wl.B):
        Kb = np.concatenate([bf16_bits_to_f64(wl.K[b]), bf16_bits_to_f64(wl.k_new[0, b])[:, None]], axis=1)
        Vb = np.concatenate([bf16_bits_to_f64(wl.V[b]), bf16_bits_to_f64(wl.v_new[0, b])[:, None]], axis=1)
        o, p = decode_attention(bf16_bits_to_f64(wl.q[0, b]), Kb, Vb, wl.scale)
        assert rel_l2(st.out[b].double().cpu().numpy(), o) < TOL
        assert rel_l2(st.probs[b, :, :S].double().cpu().numpy(), p) < TOL


def test_decode_readiness_wait_times_out_and_recovers():
    wl = workloads.decode_custom(seed=21, B=2, Hq=16, Hkv=8, d=128, S0=700, steps=1, budget=64,
                                 n_sink=4, window=16, permute_pages=True)
    st = DecodeState(wl)
    K.set_wait_limit(st.ws, SHORT)
    st.ws[PAIR_COUNTERS:PAIR_COUNTERS + 4].view(torch.int32).fill_(1 << 20)   # pair 0: never its owner count
    st.decode(0)
    torch.cuda.synchronize()
    assert K.read_status(st.ws) == K.KVSEL_ERR_TIMEOUT
    st.guards.check()
    # the same workspace, zeroed again (which also restores the default limit), on a fresh cache
    ws = st.ws
    ws.zero_()
    st2 = DecodeState(wl)
    st2.ws = ws
    st2.decode(0)
    torch.cuda.synchronize()
    assert K.read_status(ws) == 0
    st.guards.check()
    st2.guards.check()
    _decode_ok(st2, wl)


def test_block_priority_barrier_times_out_and_recovers():
    wl = workloads.block_priority(seed=7, R=9, steps=2, min_len=300, max_len=9000)
    off = wl.offsets
    tok0 = wl.increments(0)
    bs = 16
    nblk = int(sum(-(-int(L) // bs) for L in wl.lengths))
    g = Guards()
    t_off = g.like(torch.from_numpy(off).cuda())
    cap = math.ceil(0.25 * nblk)
    order = g.new((cap,), torch.int64, fill=-7)
    n_out = g.new((2,), torch.int64)
    bso = g.new((nblk,), torch.float32)
    ws = g.new((K.kvsel_block_priority_workspace(wl.R, nblk),), torch.uint8)

    def run():
        tok = g.like(torch.from_numpy(tok0).cuda())
        K.kvsel_block_priority(tok, t_off, order, n_out, ws, block_size=bs, agg=K.KVSEL_AGG_MEAN,
                               norm=K.KVSEL_NORM_PERCENTILE, evict_frac=0.25, block_score_out=bso,
                               max_total_blocks=nblk)

    K.set_wait_limit(ws, SHORT)
    ws[BAR_COUNTER:BAR_COUNTER + 4].view(torch.int32).fill_(1 << 30)          # no CTA is ever the last
    run()
    torch.cuda.synchronize()
    assert K.read_status(ws) == K.KVSEL_ERR_TIMEOUT
    g.check()
    assert (order.cpu().numpy() == -7).all()       # the sort stopped before writing anything
    ws.zero_()
    run()
    assert K.read_status(ws) == 0
    g.check()
    blocks, normed, want = BP.priority_pass(tok0.astype(np.float64), off, bs, BP.AGG_MEAN, 0.1,
                                            BP.NORM_PERCENTILE, 0.25)
    gblk = bso.cpu().numpy()
    assert rel_l2(gblk, np.concatenate(blocks)) < 1e-6
    # the order is bit-exact on the GPU's own block scores (the oracle's ranking routine)
    per_req, base = [], 0
    for r in range(wl.R):
        n = len(blocks[r])
        per_req.append(BP.percentiles(gblk[base:base + n].astype(np.float64)).astype(np.float64))
        base += n
    np.testing.assert_array_equal(order.cpu().numpy()[:int(n_out[0])], BP.evict_order(per_req, 0.25))


def test_wait_limit_needs_an_aligned_workspace():
    ws = K.workspace(512)
    with pytest.raises(K.KvselError):
        K.set_wait_limit(ws[16:], 10)
    K.set_wait_limit(ws, 0)
    torch.cuda.synchronize()
    assert int(ws[32:36].view(torch.int32)[0]) == 0
