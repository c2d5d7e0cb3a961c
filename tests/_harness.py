"""Helpers shared by the GPU tests: upload seeded workloads, drive the C ABI.

Nothing here computes the method: inputs come from ``workloads`` and
expected values from ``oracle``.
"""
from __future__ import annotations

import numpy as np
import torch

import attention_guided_kv_gb300 as K
import workloads


def bf16(bits, dev="cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(dev)


def rel_l2(x, ref) -> float:
    x = np.asarray(x, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    n = np.linalg.norm(ref)
    return float(np.linalg.norm(x - ref) / (n if n > 0 else 1.0))


GUARD_BYTES = 256
GUARD_BYTE = 0xA5


class Guards:
    """Output buffers with guard regions before and after each one.

    Every buffer is carved from a larger allocation whose first and last
    GUARD_BYTES bytes hold a fixed pattern; ``check()`` asserts that no call
    wrote outside the buffer it was given (the tail and padding paths of the
    kernels, without a sanitizer).
    """

    def __init__(self, dev="cuda"):
        self.dev = dev
        self._bufs = []

    def new(self, shape, dtype, fill=0):
        shape = tuple(int(s) for s in shape)
        n = int(np.prod(shape)) * torch.empty(0, dtype=dtype).element_size()
        body = (n + GUARD_BYTES - 1) // GUARD_BYTES * GUARD_BYTES
        raw = torch.full((2 * GUARD_BYTES + body,), GUARD_BYTE, dtype=torch.uint8, device=self.dev)
        t = raw[GUARD_BYTES:GUARD_BYTES + n].view(dtype).view(shape)
        t.fill_(fill)
        self._bufs.append((raw, n))
        return t

    def like(self, src, fill=None):
        t = self.new(src.shape, src.dtype)
        if fill is None:
            t.copy_(src)
        else:
            t.fill_(fill)
        return t

    def check(self):
        for i, (raw, n) in enumerate(self._bufs):
            head = raw[:GUARD_BYTES]
            tail = raw[GUARD_BYTES + n:]
            assert bool((head == GUARD_BYTE).all()), f"guard before buffer {i} was written"
            assert bool((tail == GUARD_BYTE).all()), f"guard after buffer {i} was written"


class DecodeState:
    """Device-side paged cache + bookkeeping for a DecodeWorkload."""

    def __init__(self, wl: workloads.DecodeWorkload, with_probs=True, with_pos=True,
                 out_f32=True, spare_pages=0, link=False, dev="cuda"):
        self.wl = wl
        self.link = link
        self.dev = dev
        npages = wl.num_pages + spare_pages
        self.kpool = bf16(workloads.paged_pool(wl.K, wl.block_table, npages, wl.page), dev)
        self.vpool = bf16(workloads.paged_pool(wl.V, wl.block_table, npages, wl.page), dev)
        self.kv = K.paged_kv(self.kpool, self.vpool, wl.Hq)
        self.bt_host = wl.block_table.copy()
        self.bt = torch.from_numpy(self.bt_host).to(dev)
        self.free = list(range(wl.num_pages, npages))
        self.S = np.full(wl.B, wl.S0, dtype=np.int64)
        # every buffer the calls write sits between guard regions (checked by status())
        self.guards = g = Guards(dev)
        self.bt = g.like(self.bt)
        self.seq = g.like(torch.from_numpy(self.S.astype(np.int32)).to(dev))
        self.cum = g.new((wl.B, wl.Hkv, wl.max_len), torch.float32)
        self.probs = g.new((wl.B, wl.Hq, wl.max_len), torch.float32) if with_probs else None
        if with_pos:
            pos = np.tile(np.arange(wl.max_len, dtype=np.int32), (wl.B, wl.Hkv, 1))
            self.pos = g.like(torch.from_numpy(pos).to(dev))
            self.next_pos = g.like(torch.full((wl.B,), wl.S0, dtype=torch.int32, device=dev))
        else:
            self.pos = self.next_pos = None
        self.out = g.new((wl.B, wl.Hq, wl.d), torch.float32 if out_f32 else torch.bfloat16)
        self.ws = g.new((max(256, K.kvsel_decode_attn_workspace(self.kv, wl.B, wl.max_len, with_probs)),),
                        torch.uint8)
        self.ws_ev = g.new((max(256, K.kvsel_h2o_evict_workspace(self.kv, wl.B, wl.budget)),), torch.uint8)
        self.keep = g.new((wl.B, wl.Hkv, wl.budget), torch.int32, fill=-1)
        self.freed = g.new((wl.B, self.bt_host.shape[1]), torch.int32, fill=-1)

    def ensure_append_page(self):
        """Give every sequence a page for its next slot (host-side allocator)."""
        changed = False
        for b in range(self.wl.B):
            p = int(self.S[b]) // self.wl.page
            if self.bt_host[b, p] < 0:
                self.bt_host[b, p] = self.free.pop()
                changed = True
        if changed:
            self.bt.copy_(torch.from_numpy(self.bt_host))

    def decode(self, step, num_ctas=0, append=True):
        wl = self.wl
        if append:
            self.ensure_append_page()
        K.kvsel_decode_attn(self.kv, self.bt, self.seq, bf16(wl.q[step], self.dev), self.out, self.ws,
                            k_new=bf16(wl.k_new[step], self.dev) if append else None,
                            v_new=bf16(wl.v_new[step], self.dev) if append else None,
                            pos_map=self.pos, next_pos=self.next_pos, probs=self.probs,
                            h2o_cum=self.cum, max_len=wl.max_len, num_ctas=num_ctas,
                            h2o_link=self.ws_ev if self.link else None)
        if append:
            self.S += 1

    def evict(self, compact=True):
        wl = self.wl
        K.kvsel_h2o_evict(self.kv, self.bt, self.seq, self.cum, self.ws_ev, budget=wl.budget,
                          n_sink=wl.n_sink, window=wl.window, compact=compact, pos_map=self.pos,
                          keep_out=self.keep, freed_pages=self.freed if compact else None)
        if compact:
            torch.cuda.synchronize()
            self.bt_host = self.bt.cpu().numpy().copy()
            fr = self.freed.cpu().numpy()
            self.free.extend(int(x) for x in fr.ravel() if x >= 0)
            self.S = np.minimum(self.S, wl.budget)

    def link_counts(self):
        """Candidate counts the decode step left for the select (white-box view)."""
        rows = self.wl.B * self.wl.Hkv
        off = 256 + (rows * 4 + 255) // 256 * 256
        return self.ws_ev[off:off + rows * 4].view(torch.int32).cpu().numpy().copy()

    def status(self):
        """Device status of both workspaces (read and cleared); asserts the guards are intact."""
        st = K.read_status(self.ws), K.read_status(self.ws_ev)
        self.guards.check()
        return st
