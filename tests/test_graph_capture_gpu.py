"""The decode step and the H2O select captured in a CUDA graph, with each step's input copies
from pinned host memory, and replayed, give what the same calls give when made eagerly from
the same state: the probabilities, the H2O scores, the keep lists, the pool rows and the
lengths bit for bit, and O (which the owners of a pair add atomically) to fp32 rounding."""
import numpy as np
import pytest
import torch

import workloads
from _harness import bf16, rel_l2

import attention_guided_kv_gb300 as K

pytestmark = pytest.mark.gpu


def _pinned(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).pin_memory()


class _Run:
    """One sequence of the small workload (16 q / 8 kv heads, 1600 keys, budget 256), n steps."""

    def __init__(self, wl, n, compact):
        dev = "cuda"
        self.wl, self.compact = wl, compact
        self.kpool = bf16(workloads.paged_pool(wl.K, wl.block_table, wl.num_pages, wl.page), dev)
        self.vpool = bf16(workloads.paged_pool(wl.V, wl.block_table, wl.num_pages, wl.page), dev)
        self.kv = K.paged_kv(self.kpool, self.vpool, wl.Hq)
        self.bt = torch.from_numpy(wl.block_table).to(dev)
        self.seq = torch.full((wl.B,), wl.S0, dtype=torch.int32, device=dev)
        self.cum = torch.zeros(wl.B, wl.Hkv, wl.max_len, device=dev)
        self.probs = torch.zeros(wl.B, wl.Hq, wl.max_len, device=dev)
        self.pos = torch.from_numpy(np.tile(np.arange(wl.max_len, dtype=np.int32), (wl.B, wl.Hkv, 1))).to(dev)
        self.nxt = torch.full((wl.B,), wl.S0, dtype=torch.int32, device=dev)
        self.out = torch.zeros(n, wl.B, wl.Hq, wl.d, device=dev)                 # every step's O
        self.keep = torch.full((n, wl.B, wl.Hkv, wl.budget), -1, dtype=torch.int32, device=dev)
        self.freed = torch.full((wl.B, wl.max_pages), -1, dtype=torch.int32, device=dev)
        self.ws = K.workspace(K.kvsel_decode_attn_workspace(self.kv, wl.B, wl.max_len, True))
        self.ws_ev = K.workspace(K.kvsel_h2o_evict_workspace(self.kv, wl.B, wl.budget))
        self.h = [_pinned(wl.q[:n]), _pinned(wl.k_new[:n]), _pinned(wl.v_new[:n])]
        self.d = [torch.empty_like(h[0], device=dev) for h in self.h]

    def steps(self, n):
        wl = self.wl
        for t in range(n):
            for h, d in zip(self.h, self.d):
                d.copy_(h[t], non_blocking=True)
            q, kn, vn = self.d
            K.kvsel_decode_attn(self.kv, self.bt, self.seq, q, self.out[t], self.ws, k_new=kn, v_new=vn,
                                pos_map=self.pos, next_pos=self.nxt, probs=self.probs, h2o_cum=self.cum,
                                max_len=wl.max_len, h2o_link=self.ws_ev)
            K.kvsel_h2o_evict(self.kv, self.bt, self.seq, self.cum, self.ws_ev, budget=wl.budget,
                              n_sink=wl.n_sink, window=wl.window, compact=self.compact, pos_map=self.pos,
                              keep_out=self.keep[t], freed_pages=self.freed if self.compact else None)
            if self.compact:  # the caller's allocator hands the first released page back for the next append
                self.bt[:, wl.budget // wl.page].copy_(self.freed[:, 0])

    def state(self):
        torch.cuda.synchronize()
        assert K.read_status(self.ws) == 0 and K.read_status(self.ws_ev) == 0
        return {name: getattr(self, name).cpu() for name in
                ("seq", "cum", "probs", "pos", "keep", "bt", "kpool", "vpool", "out")}


@pytest.mark.parametrize("compact", [False, True])
def test_decode_and_select_replayed_from_a_graph(compact):
    wl = workloads.decode_small()
    n = 8
    eager = _Run(wl, n, compact)
    eager.steps(n)
    want = eager.state()

    replayed = _Run(wl, n, compact)
    g = torch.cuda.CUDAGraph()
    torch.cuda.synchronize()
    with torch.cuda.graph(g):
        replayed.steps(n)
    g.replay()
    got = replayed.state()

    S_end = wl.budget if compact else wl.S0 + n     # every compacting select truncates to the budget
    assert got["seq"].tolist() == want["seq"].tolist() == [S_end] * wl.B
    for name in ("cum", "probs", "pos", "keep", "bt"):
        assert torch.equal(got[name], want[name]), name
    for name in ("kpool", "vpool"):
        assert torch.equal(got[name].view(torch.int16), want[name].view(torch.int16)), name
    assert rel_l2(got["out"].numpy(), want["out"].numpy()) < 1e-6
