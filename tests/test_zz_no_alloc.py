"""The allocation-free decode entry point matches the workspace one.

kvsel_decode_attn_noalloc exists for callers that cannot allocate device
memory (no device allocator at hand, or allocation forbidden mid-step); it
runs the same decode kernel on the library's built-in scratch array instead
of a caller-provided workspace.  This test drives two identical caches, one
through each entry point, for two decode steps in a row (so the second call
runs on scratch the first one left behind) and compares outputs,
probabilities, H2O scores and lengths, and checks the outputs and
probabilities against the fp64 oracle as well.  It sits in a file of its own
that is collected last.
"""

import numpy as np
import pytest
import torch

import workloads
from oracle.attention import bf16_bits_to_f64, decode_attention
from _harness import DecodeState, bf16, rel_l2

import attention_guided_kv_gb300 as K

pytestmark = pytest.mark.gpu
TOL = 2e-3


def _noalloc_step(st, step):
    wl = st.wl
    K.kvsel_decode_attn_noalloc(st.kv, st.bt, st.seq, bf16(wl.q[step]), st.out,
                                k_new=bf16(wl.k_new[step]), v_new=bf16(wl.v_new[step]),
                                pos_map=st.pos, next_pos=st.next_pos, probs=st.probs,
                                h2o_cum=st.cum, max_len=wl.max_len)
    st.S += 1


def test_noalloc_matches_workspace_entry_point_two_calls():
    wl = workloads.decode_custom(seed=61, B=3, Hq=64, Hkv=8, d=128, S0=1500, steps=2, budget=512,
                                 n_sink=4, window=64, permute_pages=True)
    ref = DecodeState(wl)
    alt = DecodeState(wl)
    for step in range(2):
        ref.decode(step)
        _noalloc_step(alt, step)
        torch.cuda.synchronize()
        S = int(ref.S[0])
        assert rel_l2(alt.out.double().cpu().numpy(), ref.out.double().cpu().numpy()) < TOL
        assert rel_l2(alt.probs[:, :, :S].double().cpu().numpy(),
                      ref.probs[:, :, :S].double().cpu().numpy()) < TOL
        assert rel_l2(alt.cum[:, :, :S].double().cpu().numpy(),
                      ref.cum[:, :, :S].double().cpu().numpy()) < TOL
        assert alt.seq.cpu().tolist() == ref.seq.cpu().tolist() == [S] * wl.B
        assert alt.pos.cpu().tolist() == ref.pos.cpu().tolist()
        # and against the oracle directly: O and probabilities of every sequence at this step
        for b in range(wl.B):
            Kb = np.concatenate([bf16_bits_to_f64(wl.K[b]),
                                 bf16_bits_to_f64(wl.k_new[:step + 1, b]).transpose(1, 0, 2)], axis=1)
            Vb = np.concatenate([bf16_bits_to_f64(wl.V[b]),
                                 bf16_bits_to_f64(wl.v_new[:step + 1, b]).transpose(1, 0, 2)], axis=1)
            o, p = decode_attention(bf16_bits_to_f64(wl.q[step, b]), Kb, Vb, wl.scale)
            assert rel_l2(alt.out[b].double().cpu().numpy(), o) < TOL
            assert rel_l2(alt.probs[b, :, :S].double().cpu().numpy(), p) < TOL
    assert K.read_status(ref.ws) == 0


def test_noalloc_rejects_calls_beyond_its_scratch():
    wl = workloads.decode_custom(seed=62, B=1, Hq=64, Hkv=8, d=128, S0=100, steps=1, budget=64,
                                 n_sink=4, window=16)
    st = DecodeState(wl)
    # scores without a probability buffer need batch * Hq * max_len * 4 bytes of logits
    # scratch: 64 * 40000 * 4 B = 10 MB, more than the built-in 8 MiB
    cum = torch.zeros(1, wl.Hkv, 40000, device="cuda")
    with pytest.raises(K.KvselError) as e:
        K.kvsel_decode_attn_noalloc(st.kv, st.bt, st.seq, bf16(wl.q[0]), st.out, h2o_cum=cum,
                                    max_len=40000)
    assert e.value.code == K.KVSEL_ERR_INVALID_ARG
    assert b"built-in" in K.lib().kvsel_last_error_string()
