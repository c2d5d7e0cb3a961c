"""GPU parity of H2O selection and compaction against the oracle.

Selection is bit-exact: the GPU and the oracle get the same fp32 score
arrays and must return identical keep lists.  Compaction must move bytes
exactly.  The end-to-end decode+evict loop (the small config, evicting every
step) must keep identical sets except at near-ties (oracle score within
1e-5 relative of the k-th score), after which the oracle continues from the
GPU's keep-set.
"""
import numpy as np
import pytest
import torch

import workloads
from oracle.attention import bf16_bits_to_f64
from oracle.h2o import H2OSequence, h2o_keep
from _harness import DecodeState, Guards, bf16, rel_l2

import attention_guided_kv_gb300 as K

pytestmark = pytest.mark.gpu
TOL = 2e-3


def _run_select(cum_np, S_list, budget, n_sink, window, max_len, pos=None):
    B, Hkv, _ = cum_np.shape
    dev = "cuda"
    kpool = torch.zeros(1, Hkv, 16, 128, dtype=torch.bfloat16, device=dev)
    kv = K.paged_kv(kpool, kpool, Hkv)
    g = Guards()
    bt = g.new((B, (max_len + 15) // 16), torch.int32)
    seq = g.like(torch.tensor(S_list, dtype=torch.int32, device=dev))
    cum = g.like(torch.from_numpy(cum_np.astype(np.float32)).to(dev))
    keep = g.new((B, Hkv, budget), torch.int32, fill=-7)
    ws = g.new((K.kvsel_h2o_evict_workspace(kv, B, budget),), torch.uint8)
    K.kvsel_h2o_evict(kv, bt, seq, cum, ws, budget=budget, n_sink=n_sink, window=window,
                      compact=False, keep_out=keep,
                      pos_map=None if pos is None else g.like(torch.from_numpy(pos).to(dev)))
    assert K.read_status(ws) == 0
    g.check()
    return keep.cpu().numpy()


def _expect(cum_np, S_list, budget, n_sink, window, pos=None):
    B, Hkv, _ = cum_np.shape
    out = np.full((B, Hkv, budget), -1, dtype=np.int64)
    for b in range(B):
        for h in range(Hkv):
            k = h2o_keep(cum_np[b, h].astype(np.float32), S_list[b], budget, n_sink, window)
            out[b, h, :len(k)] = k if pos is None else pos[b, h, k]
    return out


@pytest.mark.parametrize("seed", range(6))
def test_select_bit_exact_with_ties(seed):
    rng = np.random.default_rng(seed)
    B, Hkv, max_len = 3, 4, 5000
    S_list = [int(x) for x in rng.integers(1, max_len + 1, B)]
    budget, n_sink, window = int(rng.integers(40, 900)), int(rng.integers(0, 5)), int(rng.integers(0, 40))
    # coarse quantisation -> many exact ties at the threshold
    cum = (rng.integers(0, 50, (B, Hkv, max_len)) * 0.125).astype(np.float32)
    got = _run_select(cum, S_list, budget, n_sink, window, max_len)
    np.testing.assert_array_equal(got, _expect(cum, S_list, budget, n_sink, window))


def test_select_bit_exact_continuous_scores_and_positions():
    rng = np.random.default_rng(17)
    B, Hkv, max_len = 2, 8, 32896
    S_list = [32769, 20000]
    cum = rng.random((B, Hkv, max_len), dtype=np.float32) * np.float32(3.0)
    pos = rng.permutation(B * Hkv * max_len).astype(np.int32).reshape(B, Hkv, max_len)
    got = _run_select(cum, S_list, 6553, 4, 1024, max_len, pos=pos)
    np.testing.assert_array_equal(got, _expect(cum, S_list, 6553, 4, 1024, pos=pos))


@pytest.mark.parametrize("max_len,S_list,budget", [
    (70001, [70001, 40000, 33000], 6553),   # rows longer than the register-resident size, odd stride
    (4999, [4999, 3001, 4000], 1000),       # row starts not 16-byte aligned
    (60000, [60000, 45000, 30000], 20000),  # k above the shared-memory upper-set capacity
])
def test_select_long_unaligned_and_large_k(max_len, S_list, budget):
    rng = np.random.default_rng(max_len)
    cum = rng.random((len(S_list), 2, max_len), dtype=np.float32)
    cum[1] = np.round(cum[1] * 64) / 64           # second kv head: many exact ties
    got = _run_select(cum, S_list, budget, 4, 256, max_len)
    np.testing.assert_array_equal(got, _expect(cum, S_list, budget, 4, 256))


def test_select_reuses_previous_threshold_across_calls():
    """Calls on one workspace start from the previous threshold: exact whether
    the scores grew (bound too low), shrank (bound too high) or were shuffled."""
    rng = np.random.default_rng(23)
    B, Hkv, max_len, budget = 2, 4, 32896, 6553
    S_list = [32896, 30000]
    dev = "cuda"
    kpool = torch.zeros(1, Hkv, 16, 128, dtype=torch.bfloat16, device=dev)
    kv = K.paged_kv(kpool, kpool, Hkv)
    bt = torch.zeros(B, max_len // 16 + 1, dtype=torch.int32, device=dev)
    seq = torch.tensor(S_list, dtype=torch.int32, device=dev)
    keep = torch.zeros((B, Hkv, budget), dtype=torch.int32, device=dev)
    ws = K.workspace(K.kvsel_h2o_evict_workspace(kv, B, budget))
    base = rng.random((B, Hkv, max_len), dtype=np.float32)
    variants = [base, base + np.float32(0.001) * rng.random(base.shape, dtype=np.float32),
                base * np.float32(0.25), base + np.float32(10.0), rng.permutation(base.ravel()).reshape(base.shape),
                np.round(base * 16) / 16]
    for cum_np in variants:
        cum_np = cum_np.astype(np.float32)
        K.kvsel_h2o_evict(kv, bt, seq, torch.from_numpy(cum_np).to(dev), ws, budget=budget, n_sink=4,
                          window=1024, keep_out=keep)
        assert K.read_status(ws) == 0
        np.testing.assert_array_equal(keep.cpu().numpy(), _expect(cum_np, S_list, budget, 4, 1024))


def test_streaming_and_sliding_window_special_cases():
    rng = np.random.default_rng(2)
    cum = rng.random((1, 2, 400), dtype=np.float32)
    got = _run_select(cum, [320], 256, 4, 252, 400)          # StreamingLLM: heavy = 0
    want = list(range(4)) + list(range(68, 320))
    assert got[0, 0].tolist() == want and got[0, 1].tolist() == want
    got = _run_select(cum, [320], 256, 0, 256, 400)          # sliding window
    assert got[0, 0].tolist() == list(range(64, 320))
    got = _run_select(cum, [100], 256, 4, 16, 400)           # short: nothing evicted
    assert got[0, 0].tolist() == list(range(100)) + [-1] * 156


def test_all_equal_scores_keep_lowest_candidates():
    cum = np.ones((1, 1, 64), dtype=np.float32)
    got = _run_select(cum, [50], 20, 4, 6, 64)
    assert got[0, 0].tolist() == list(range(14)) + list(range(44, 50))


@pytest.mark.parametrize("page", [16, 64, 256])
def test_compaction_moves_rows_exactly(page):
    wl = workloads.decode_custom(seed=12, B=2, Hq=16, Hkv=8, d=128, S0=700, steps=1, budget=300,
                                 n_sink=4, window=40, permute_pages=True, page=page)
    P = wl.page
    st = DecodeState(wl, spare_pages=4)
    rng = np.random.default_rng(3)
    cum = rng.random((wl.B, wl.Hkv, wl.max_len), dtype=np.float32)
    st.cum.copy_(torch.from_numpy(cum))
    k_before = st.kpool.view(torch.int16).cpu().numpy().copy()
    v_before = st.vpool.view(torch.int16).cpu().numpy().copy()
    bt_before = st.bt_host.copy()
    pos_before = st.pos.cpu().numpy().copy()
    st.evict(compact=True)
    assert st.status() == (0, 0)
    kn = st.kpool.view(torch.int16).cpu().numpy()
    vn = st.vpool.view(torch.int16).cpu().numpy()
    cn = st.cum.cpu().numpy()
    pn = st.pos.cpu().numpy()
    keep_out = st.keep.cpu().numpy()
    for b in range(wl.B):
        for h in range(wl.Hkv):
            keep = h2o_keep(cum[b, h], wl.S0, wl.budget, wl.n_sink, wl.window)
            assert keep_out[b, h].tolist() == pos_before[b, h, keep].tolist()
            for i, src in enumerate(keep):
                ps, pd = bt_before[b, src // P], st.bt_host[b, i // P]
                assert np.array_equal(kn[pd, h, i % P], k_before[ps, h, src % P])
                assert np.array_equal(vn[pd, h, i % P], v_before[ps, h, src % P])
            np.testing.assert_array_equal(cn[b, h, :wl.budget], cum[b, h, keep])
            np.testing.assert_array_equal(pn[b, h, :wl.budget], pos_before[b, h, keep])
    new_pages = (wl.budget + P - 1) // P
    old_pages = (wl.S0 + P - 1) // P
    assert (st.bt_host[:, new_pages:old_pages] == -1).all()
    fr = st.freed.cpu().numpy()
    for b in range(wl.B):
        assert fr[b, :old_pages - new_pages].tolist() == bt_before[b, new_pages:old_pages].tolist()
        assert (fr[b, old_pages - new_pages:] == -1).all()
    assert st.seq.cpu().tolist() == [wl.budget] * wl.B


def _run_mode_a(wl, steps, link=False, track=None):
    """Evict-every-step loop on GPU and oracle with teacher forcing at near-ties.

    The GPU steps every sequence of the batch; the oracle follows the
    sequences in ``track`` (all of them by default)."""
    track = list(range(wl.B)) if track is None else list(track)
    st = DecodeState(wl, spare_pages=8, link=link)
    refs = {b: H2OSequence(bf16_bits_to_f64(wl.K[b]), bf16_bits_to_f64(wl.V[b])) for b in track}
    swaps = 0
    for t in range(steps):
        st.decode(t)
        torch.cuda.synchronize()
        S = int(st.S[0])
        probs = dict(zip(track, st.probs[track, :, :S].double().cpu().numpy()))
        outs = dict(zip(track, st.out[track].double().cpu().numpy()))
        cum_gpu = dict(zip(track, st.cum[track, :, :S].double().cpu().numpy()))
        for b, ref in refs.items():
            ref.append(bf16_bits_to_f64(wl.k_new[t, b]), bf16_bits_to_f64(wl.v_new[t, b]))
            o, p = ref.attend(bf16_bits_to_f64(wl.q[t, b]), wl.scale)
            assert ref.S == S
            assert rel_l2(outs[b], o) < TOL, (t, b)
            assert rel_l2(probs[b], p) < TOL, (t, b)
            assert rel_l2(cum_gpu[b], ref.cum) < TOL, (t, b)
        st.evict(compact=True)
        torch.cuda.synchronize()
        assert st.status() == (0, 0)
        if S <= wl.budget:
            continue
        kept_pos = st.keep.cpu().numpy()
        for b, ref in refs.items():
            want = ref.select(wl.budget, wl.n_sink, wl.window)
            want_pos = np.stack([ref.pos[h, want[h]] for h in range(wl.Hkv)])
            if not np.array_equal(kept_pos[b], want_pos):
                for h in range(wl.Hkv):
                    diff = set(kept_pos[b, h].tolist()) ^ set(want_pos[h].tolist())
                    if not diff:
                        continue
                    k = wl.budget - wl.n_sink - wl.window
                    mid = ref.cum[h, wl.n_sink:S - wl.window]
                    kth = np.sort(mid)[::-1][k - 1]
                    slot = {int(p): i for i, p in enumerate(ref.pos[h])}
                    for p in diff:
                        assert abs(ref.cum[h, slot[p]] - kth) <= 1e-5 * kth, (t, b, h, p)
                    swaps += 1
                gpu_slots = []
                for h in range(wl.Hkv):
                    slot = {int(p): i for i, p in enumerate(ref.pos[h])}
                    gpu_slots.append([slot[int(x)] for x in kept_pos[b, h]])
                gpu_slots = np.array(gpu_slots, dtype=np.int64)
                ref.apply_keep(gpu_slots)
            else:
                ref.apply_keep(want)
    return swaps


def test_small_config_evict_every_step_end_to_end():
    wl = workloads.decode_small()
    swaps = _run_mode_a(wl, wl.steps)
    assert swaps <= 4


@pytest.mark.slow
def test_70b_shape_evict_every_step_end_to_end():
    """The 70B layer shape evicting every step: batch 8 x 32K, budget 6553 = 4 sinks + 1024
    window + 5525 heavy hitters, all 128 steps with the decode -> select hand-off; the oracle
    follows sequences 0 and 5 step by step (outputs, probabilities, scores, keep-sets)."""
    wl = workloads.decode_70b()
    swaps = _run_mode_a(wl, wl.steps, link=True, track=[0, 5])
    assert swaps <= 32, swaps


@pytest.mark.parametrize("link,page", [(False, 16), (True, 16), (True, 256), (False, 32)])
def test_custom_config_evict_every_step_permuted_pages(link, page):
    wl = workloads.decode_custom(seed=77, B=3, Hq=64, Hkv=8, d=128, S0=500, steps=12, budget=200,
                                 n_sink=4, window=33, permute_pages=True, page=page)
    _run_mode_a(wl, wl.steps, link=link)


def test_group_of_16_evict_every_step():
    """16 q heads per kv head: the H2O score sums all 16 heads' probabilities of a key."""
    wl = workloads.decode_custom(seed=78, B=2, Hq=64, Hkv=4, d=128, S0=400, steps=6, budget=150,
                                 n_sink=4, window=20, permute_pages=True)
    _run_mode_a(wl, wl.steps, link=True)


def test_link_reset_after_an_outside_score_write():
    """A caller lifts unlisted slots far above every score (a prefill seed, say) between a decode
    step and the select; after kvsel_h2o_link_reset the select keeps them: the exact top-k."""
    wl = workloads.decode_custom(seed=79, B=2, Hq=16, Hkv=4, d=128, S0=3000, steps=2, budget=500,
                                 n_sink=4, window=32, permute_pages=True)
    st = DecodeState(wl, spare_pages=8, link=True)
    st.decode(0)
    st.evict(compact=False)       # thresholds for the next decode's lists
    st.decode(1)
    torch.cuda.synchronize()
    assert (st.link_counts() > 0).all()
    cum = st.cum.cpu().numpy().copy()
    S = int(st.S[0])
    keep_before = st.keep.cpu().numpy().copy()
    pos0 = st.pos.cpu().numpy()
    lifted = []
    for b in range(wl.B):
        for h in range(wl.Hkv):
            kept = set(keep_before[b, h].tolist())
            j = next(x for x in range(wl.n_sink, S - wl.window) if int(pos0[b, h, x]) not in kept)
            cum[b, h, j] = cum[b, h, :S].max() * 4.0 + 1.0
            lifted.append((b, h, j))
    st.cum.copy_(torch.from_numpy(cum))
    K.kvsel_h2o_link_reset(st.ws_ev, wl.B, wl.Hkv)
    assert (st.link_counts() == 0).all()
    st.evict(compact=False)
    torch.cuda.synchronize()
    assert st.status() == (0, 0)
    keep = st.keep.cpu().numpy()
    pos = st.pos.cpu().numpy()
    for b in range(wl.B):
        for h in range(wl.Hkv):
            want = h2o_keep(cum[b, h].astype(np.float32), S, wl.budget, wl.n_sink, wl.window)
            np.testing.assert_array_equal(keep[b, h, :len(want)], pos[b, h, want])
    for b, h, j in lifted:
        assert pos[b, h, j] in keep[b, h]


def test_decode_hands_candidates_to_select():
    """With the hand-off, the select keeps exactly the top-k of the GPU's own
    scores (compacting on every other step), and each list is used once."""
    wl = workloads.decode_custom(seed=5, B=2, Hq=16, Hkv=4, d=128, S0=3000, steps=8, budget=1000,
                                 n_sink=4, window=64, permute_pages=True)
    st = DecodeState(wl, spare_pages=16, link=True)
    used = 0
    for t in range(wl.steps):
        st.decode(t)
        torch.cuda.synchronize()
        S = st.seq.cpu().numpy()
        cum = st.cum.cpu().numpy().copy()
        pos = st.pos.cpu().numpy().copy()
        counts = st.link_counts()
        if t > 0:   # a threshold exists from the previous select
            assert (counts >= wl.budget - wl.n_sink - wl.window).all() and (counts <= 16384).all(), counts
            used += 1
        st.evict(compact=(t % 2 == 0))
        torch.cuda.synchronize()
        assert st.status() == (0, 0)
        assert (st.link_counts() == 0).all()
        keep = st.keep.cpu().numpy()
        for b in range(wl.B):
            for h in range(wl.Hkv):
                want = h2o_keep(cum[b, h].astype(np.float32), int(S[b]), wl.budget, wl.n_sink, wl.window)
                np.testing.assert_array_equal(keep[b, h, :len(want)], pos[b, h, want])
    assert used == wl.steps - 1
