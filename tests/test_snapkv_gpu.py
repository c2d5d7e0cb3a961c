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
from _harness import bf16, rel_l2

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
        self.keep = torch.full((L, wl.Hkv, wl.keep_k + wl.W), -7, dtype=torch.int32, device="cuda")
        self.vote = torch.zeros(L, wl.Hkv, max(wl.S - wl.W, 1), device="cuda")
        self.ws = K.workspace(K.kvsel_snapkv_select_workspace(self.kv, L, wl.S, wl.W, True))

    def run(self):
        wl = self.wl
        K.kvsel_snapkv_select(self.kv, self.bt, self.q, self.keep, self.ws, seq_len=wl.S,
                              keep_k=wl.keep_k, pool_kernel=wl.pool_kernel, vote_out=self.vote)
        torch.cuda.synchronize()
        assert K.read_status(self.ws) == 0


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
