"""GPU parity of the per-step top-k block signal emitted by the decode launch.

* block masses within relative L2 2e-3 of the oracle's (fp64 probabilities
  summed over the q heads and each block's keys);
* the chosen blocks bit-exact when the oracle's top-k routine gets the GPU's
  own fp32 masses, and the per-block metadata exactly what the oracle's
  update gives on them (fp32 accumulation, the step stamped);
* O unchanged by the signal (within 2e-3 of the oracle).
"""
import numpy as np
import pytest
import torch

import workloads
from oracle import block_signal as bsig
from oracle.attention import bf16_bits_to_f64, decode_attention
from _harness import DecodeState, bf16, rel_l2

import attention_guided_kv_gb300 as K

pytestmark = pytest.mark.gpu
TOL = 2e-3


class SignalState(DecodeState):
    def __init__(self, wl, k, **kw):
        super().__init__(wl, **kw)
        self.k = k
        g = self.guards
        self.ws = g.new((K.kvsel_decode_attn_ex_workspace(self.kv, wl.B, wl.max_len, self.probs is not None,
                                                          True),), torch.uint8)
        n_pool = self.kpool.shape[0]
        self.score = g.new((n_pool,), torch.float32)
        self.last = g.new((n_pool,), torch.int32, fill=-1)
        self.topk = g.new((wl.B, k), torch.int32, fill=-7)
        self.mass = g.new((wl.B, -(-wl.max_len // 16)), torch.float32)

    def decode_signal(self, step):
        wl = self.wl
        self.ensure_append_page()
        K.kvsel_decode_attn(self.kv, self.bt, self.seq, bf16(wl.q[step]), self.out, self.ws,
                            k_new=bf16(wl.k_new[step]), v_new=bf16(wl.v_new[step]), pos_map=self.pos,
                            next_pos=self.next_pos, probs=self.probs, h2o_cum=self.cum, max_len=wl.max_len,
                            block_score=self.score, block_step=self.last, signal_topk=self.k,
                            signal_step=100 + step, signal_topk_out=self.topk, signal_mass_out=self.mass)
        self.S += 1


def _logical(wl, b, steps_done):
    Kb = bf16_bits_to_f64(wl.K[b])
    Vb = bf16_bits_to_f64(wl.V[b])
    Kb = np.concatenate([Kb, bf16_bits_to_f64(wl.k_new[:steps_done, b]).transpose(1, 0, 2)], axis=1)
    Vb = np.concatenate([Vb, bf16_bits_to_f64(wl.v_new[:steps_done, b]).transpose(1, 0, 2)], axis=1)
    return Kb, Vb


def _run_and_check(st, steps, seqs=None):
    wl = st.wl
    acc = st.score.cpu().numpy().astype(np.float32)
    last = st.last.cpu().numpy().astype(np.int64)
    for t in range(steps):
        st.decode_signal(t)
        torch.cuda.synchronize()
        assert K.read_status(st.ws) == 0
        st.guards.check()
        mass = st.mass.cpu().numpy()
        topk = st.topk.cpu().numpy()
        out = st.out.double().cpu().numpy()
        bt = st.bt_host
        for b in range(wl.B):
            S = int(st.S[b])
            n = -(-S // 16)
            m = mass[b, :n].astype(np.float64)
            if seqs is None or b in seqs:
                Kb, Vb = _logical(wl, b, t + 1)
                o, p = decode_attention(bf16_bits_to_f64(wl.q[t, b]), Kb, Vb, wl.scale)
                assert rel_l2(m, bsig.block_masses(p)) < TOL, (t, b)
                assert rel_l2(out[b], o) < TOL, (t, b)
            chosen = bsig.top_blocks(m, st.k)
            np.testing.assert_array_equal(topk[b, :len(chosen)], chosen)
            assert (topk[b, len(chosen):] == -1).all()
            for j in chosen:                      # fp32 accumulation, as on the GPU
                phys = bt[b, j]
                acc[phys] = np.float32(acc[phys] + np.float32(m[j]))
                last[phys] = 100 + t
        np.testing.assert_array_equal(st.score.cpu().numpy(), acc)
        np.testing.assert_array_equal(st.last.cpu().numpy().astype(np.int64), last)


def test_ragged_steps_group_of_four():
    wl = workloads.decode_custom(seed=61, B=3, Hq=16, Hkv=4, d=128, S0=3001, steps=3, budget=2048, n_sink=4,
                                 window=64)
    st = SignalState(wl, k=64, spare_pages=8)
    _run_and_check(st, 3)


def test_group_of_sixteen():
    """16 q heads per kv head: each block's mass sums all 16 heads' probabilities."""
    wl = workloads.decode_custom(seed=63, B=2, Hq=64, Hkv=4, d=128, S0=1500, steps=2, budget=1024, n_sink=4,
                                 window=64)
    st = SignalState(wl, k=40, spare_pages=8)
    _run_and_check(st, 2)


def test_every_block_when_k_covers_the_sequence():
    wl = workloads.decode_custom(seed=62, B=2, Hq=8, Hkv=8, d=128, S0=500, steps=2, budget=256, n_sink=4,
                                 window=64)
    st = SignalState(wl, k=512, spare_pages=4)
    _run_and_check(st, 2)


def test_ties_go_to_the_lower_blocks():
    # zero queries: every key gets the same weight, so every full block ties
    wl = workloads.decode_custom(seed=63, B=2, Hq=16, Hkv=2, d=128, S0=2000, steps=1, budget=1024, n_sink=4,
                                 window=64)
    wl.q[:] = 0
    st = SignalState(wl, k=37, spare_pages=4)
    _run_and_check(st, 1)
    top = st.topk.cpu().numpy()
    assert top[0].tolist() == list(range(37))


@pytest.mark.slow
def test_headline_shape_sampled():
    """Batch 8 x 32K, 64 q / 8 kv heads, top-512 blocks: sampled sequences against the oracle."""
    wl = workloads.decode_70b(steps=2)
    st = SignalState(wl, k=512, with_pos=False)
    _run_and_check(st, 2, seqs={0, 5})
