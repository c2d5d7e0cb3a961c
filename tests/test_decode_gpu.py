"""GPU parity of score-emitting decode attention against the fp64 oracle.

Bar: O, probabilities and H2O scores within relative L2 <= 2e-3 of the
oracle on the same seeded bf16 inputs (fp32 accumulation on the GPU).
"""
import numpy as np
import pytest
import torch

import workloads
from oracle.attention import bf16_bits_to_f64, decode_attention, h2o_accumulate
from _harness import DecodeState, bf16, rel_l2

import attention_guided_kv_gb300 as K

pytestmark = pytest.mark.gpu
TOL = 2e-3


def _oracle_step(wl, b, step, S_total):
    """Oracle O, p, cum for sequence b after appending step's token (cum from zero)."""
    Kb = bf16_bits_to_f64(wl.K[b])
    Vb = bf16_bits_to_f64(wl.V[b])
    Kb = np.concatenate([Kb, bf16_bits_to_f64(wl.k_new[step, b])[:, None]], axis=1)
    Vb = np.concatenate([Vb, bf16_bits_to_f64(wl.v_new[step, b])[:, None]], axis=1)
    assert Kb.shape[1] == S_total
    o, p = decode_attention(bf16_bits_to_f64(wl.q[step, b]), Kb, Vb, wl.scale)
    cum = h2o_accumulate(np.zeros((wl.Hkv, S_total)), p)
    return o, p, cum


def _check_step(st, wl, step=0, bs=None):
    S = wl.S0 + 1
    for b in (range(wl.B) if bs is None else bs):
        o, p, cum = _oracle_step(wl, b, step, S)
        assert rel_l2(st.out[b].double().cpu().numpy(), o) < TOL
        if st.probs is not None:
            assert rel_l2(st.probs[b, :, :S].double().cpu().numpy(), p) < TOL
        assert rel_l2(st.cum[b, :, :S].double().cpu().numpy(), cum) < TOL


def test_decode_small_config_one_step():
    wl = workloads.decode_small()
    st = DecodeState(wl)
    st.decode(0)
    torch.cuda.synchronize()
    assert st.status() == (0, 0)
    _check_step(st, wl)
    assert int(st.seq[0]) == wl.S0 + 1
    assert int(st.pos[0, 3, wl.S0]) == wl.S0 and int(st.next_pos[0]) == wl.S0 + 1


@pytest.mark.parametrize("ctas", [1, 2, 7, 16, 64, 151, 0])
def test_work_split_invariance(ctas):
    wl = workloads.decode_custom(seed=31, B=2, Hq=32, Hkv=4, d=128, S0=999, steps=1, budget=512,
                                 n_sink=4, window=64, permute_pages=True)
    st = DecodeState(wl)
    st.decode(0, num_ctas=ctas)
    torch.cuda.synchronize()
    assert st.status() == (0, 0)
    _check_step(st, wl)


@pytest.mark.parametrize("Hq,Hkv", [(8, 8), (16, 8), (16, 4), (64, 8), (12, 2),
                                    (128, 8), (24, 2), (36, 4), (16, 1)])
def test_group_sizes(Hq, Hkv):
    """1 to 16 q heads per kv head (16: e.g. 128 q / 8 kv heads; 9 and 12: ragged upper rows)."""
    wl = workloads.decode_custom(seed=40 + Hq, B=2, Hq=Hq, Hkv=Hkv, d=128, S0=257, steps=1,
                                 budget=128, n_sink=4, window=16, permute_pages=True)
    st = DecodeState(wl)
    st.decode(0)
    torch.cuda.synchronize()
    assert st.status() == (0, 0)
    _check_step(st, wl)


@pytest.mark.parametrize("S0", [0, 1, 15, 16, 17, 31, 33, 4095])
def test_ragged_lengths_and_page_tails(S0):
    wl = workloads.decode_custom(seed=50 + S0, B=1, Hq=16, Hkv=8, d=128, S0=S0, steps=1, budget=8,
                                 n_sink=0, window=8, permute_pages=True)
    st = DecodeState(wl)
    st.decode(0, num_ctas=3)
    torch.cuda.synchronize()
    assert st.status() == (0, 0)
    _check_step(st, wl)


@pytest.mark.parametrize("page", [32, 256])
@pytest.mark.parametrize("S0", [0, 255, 256, 1000])
def test_larger_pages(page, S0):
    """Pool pages of 32 or 256 tokens (PagedAttention's blocks are 16 or 256): the append lands in
    the right row of a big page, ragged tails, permuted pages, a split that cuts pages."""
    wl = workloads.decode_custom(seed=60 + S0, B=2, Hq=32, Hkv=4, d=128, S0=S0, steps=1, budget=8,
                                 n_sink=0, window=8, permute_pages=True, page=page)
    st = DecodeState(wl)
    st.decode(0, num_ctas=5)
    torch.cuda.synchronize()
    assert st.status() == (0, 0)
    _check_step(st, wl)
    assert st.seq.cpu().tolist() == [S0 + 1] * wl.B


def test_256_token_pages_across_a_page_boundary():
    """Several steps whose appends cross from one 256-token page into the next, 70B head groups."""
    wl = workloads.decode_custom(seed=71, B=2, Hq=64, Hkv=8, d=128, S0=8190, steps=4, budget=8,
                                 n_sink=0, window=8, permute_pages=True, page=256)
    st = DecodeState(wl)
    for t in range(wl.steps):
        st.decode(t)
        torch.cuda.synchronize()
        assert st.status() == (0, 0)
    S = wl.S0 + wl.steps
    for b in range(wl.B):
        Kb = np.concatenate([bf16_bits_to_f64(wl.K[b]), bf16_bits_to_f64(wl.k_new[:, b]).transpose(1, 0, 2)], axis=1)
        Vb = np.concatenate([bf16_bits_to_f64(wl.V[b]), bf16_bits_to_f64(wl.v_new[:, b]).transpose(1, 0, 2)], axis=1)
        assert Kb.shape[1] == S
        o, p = decode_attention(bf16_bits_to_f64(wl.q[wl.steps - 1, b]), Kb, Vb, wl.scale)
        assert rel_l2(st.out[b].double().cpu().numpy(), o) < TOL
        assert rel_l2(st.probs[b, :, :S].double().cpu().numpy(), p) < TOL


def test_single_token_returns_its_value():
    wl = workloads.decode_custom(seed=3, B=1, Hq=16, Hkv=8, d=128, S0=0, steps=1, budget=8,
                                 n_sink=0, window=8)
    st = DecodeState(wl)
    st.decode(0)
    torch.cuda.synchronize()
    assert st.status() == (0, 0)
    v = bf16_bits_to_f64(wl.v_new[0, 0])
    np.testing.assert_allclose(st.out[0].double().cpu().numpy(), np.repeat(v, 2, axis=0), rtol=1e-6)
    np.testing.assert_array_equal(st.probs[0, :, 0].cpu().numpy(), np.ones(16, dtype=np.float32))


def test_mixed_batch_lengths_without_append():
    wl = workloads.decode_custom(seed=8, B=3, Hq=64, Hkv=8, d=128, S0=700, steps=1, budget=8,
                                 n_sink=0, window=8, permute_pages=True)
    st = DecodeState(wl)
    lens = np.array([1, 350, 700])
    st.seq.copy_(torch.from_numpy(lens.astype(np.int32)))
    st.decode(0, append=False)
    torch.cuda.synchronize()
    assert st.status() == (0, 0)
    for b in range(3):
        S = int(lens[b])
        Kb = bf16_bits_to_f64(wl.K[b])[:, :S]
        Vb = bf16_bits_to_f64(wl.V[b])[:, :S]
        o, p = decode_attention(bf16_bits_to_f64(wl.q[0, b]), Kb, Vb, wl.scale)
        assert rel_l2(st.out[b].double().cpu().numpy(), o) < TOL
        assert rel_l2(st.probs[b, :, :S].double().cpu().numpy(), p) < TOL
    assert st.seq.cpu().tolist() == lens.tolist()


def test_group_of_16_bf16_output_no_probs_and_a_split_cutting_pages():
    wl = workloads.decode_custom(seed=19, B=3, Hq=128, Hkv=8, d=128, S0=3001, steps=1, budget=8,
                                 n_sink=0, window=8, permute_pages=True, page=64)
    st = DecodeState(wl, with_probs=False, out_f32=False)
    st.decode(0, num_ctas=37)
    torch.cuda.synchronize()
    assert st.status() == (0, 0)
    _check_step(st, wl)


def test_bf16_output_and_no_probs_buffer():
    wl = workloads.decode_custom(seed=9, B=2, Hq=64, Hkv=8, d=128, S0=2000, steps=1, budget=8,
                                 n_sink=0, window=8, permute_pages=True)
    st = DecodeState(wl, with_probs=False, out_f32=False)
    st.decode(0)
    torch.cuda.synchronize()
    assert st.status() == (0, 0)
    _check_step(st, wl)


def test_bad_block_table_entry_is_reported_not_faulted():
    wl = workloads.decode_custom(seed=10, B=1, Hq=16, Hkv=8, d=128, S0=100, steps=1, budget=8,
                                 n_sink=0, window=8)
    st = DecodeState(wl)
    st.bt[0, 2] = wl.num_pages + 5          # outside the pool: the kernel clamps and reports
    st.decode(0)
    assert K.read_status(st.ws) == K.KVSEL_ERR_BAD_INDEX
    assert K.read_status(st.ws) == 0        # cleared by the read
    st.guards.check()


@pytest.mark.slow
def test_full_size_70b_layer_sampled():
    """Batch 8 x 32K Llama-2-70B layer, permuted pages, default launch: oracle on sampled heads."""
    wl = workloads.decode_70b()
    st = DecodeState(wl)
    st.decode(0)
    torch.cuda.synchronize()
    assert st.status() == (0, 0)
    S = wl.S0 + 1
    rng = np.random.default_rng(0)
    for b in rng.choice(wl.B, 3, replace=False):
        kvh = int(rng.integers(wl.Hkv))
        Kb = np.concatenate([bf16_bits_to_f64(wl.K[b, kvh]),
                             bf16_bits_to_f64(wl.k_new[0, b, kvh])[None]], 0)[None]
        Vb = np.concatenate([bf16_bits_to_f64(wl.V[b, kvh]),
                             bf16_bits_to_f64(wl.v_new[0, b, kvh])[None]], 0)[None]
        hs = slice(kvh * wl.G, (kvh + 1) * wl.G)
        o, p = decode_attention(bf16_bits_to_f64(wl.q[0, b, hs]), Kb, Vb, wl.scale)
        assert rel_l2(st.out[b, hs].double().cpu().numpy(), o) < TOL
        assert rel_l2(st.probs[b, hs, :S].double().cpu().numpy(), p) < TOL
        assert rel_l2(st.cum[b, kvh, :S].double().cpu().numpy(), p.sum(0)) < TOL
    # softmax rows sum to one at any size: total H2O mass = Hq per sequence
    tot = st.cum[:, :, :S].double().sum(dim=(1, 2)).cpu().numpy()
    np.testing.assert_allclose(tot, np.full(wl.B, wl.Hq), rtol=1e-4)
