"""Seeded synthetic inputs for the attention-guided KV selection path.

This module is shared by the CPU oracle's tests, the GPU parity tests and the
benchmark.  It only *draws* data (numpy ``default_rng``) and lays it out; it
holds none of the method's arithmetic (no softmax, no scoring, no selection).

Every tensor is drawn in fp32 and rounded to bf16 with round-to-nearest-even,
and handed around as raw ``uint16`` bf16 bit patterns.  Consumers widen the
bits themselves (the oracle to fp64, the GPU path by reinterpreting the bytes).

The five workloads follow the shapes the pages use:

* ``decode_small``  - one sequence, 16 q / 8 kv heads, d=128, prompt 1600,
  64 decode steps, H2O budget 256 = 4 sinks + 64 window + 188 heavy hitters,
  key 0 pushed +4 along the mean query direction (a planted attention sink).
* ``decode_70b``    - Llama-2-70B layer shape (64 q / 8 kv heads, d=128),
  batch 8, 32K prompts, 16-token pages in a randomly permuted block table,
  128 decode steps, budget 20% of 32768 = 6553 = 4 + 1024 window + 5525.
* ``snapkv_qwen7b`` - Qwen2.5-7B shape (28 layers, 28 q / 4 kv heads), 32K
  prompt, 32 observation queries, 64 planted high-affinity keys per kv head.
* ``block_priority`` - 64 requests, lengths log-uniform in [4K, 128K],
  Dirichlet per-token increments (alpha 0.05 for even, 1.0 for odd requests).
* ``sparse_decode_70b`` - 70B attention shape, batch 4, 128K context,
  indexer of 4 heads x 64 dims, top-2048.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

PAGE = 16


# ----------------------------------------------------------------------------
# bf16 handling (data plumbing only)
# ----------------------------------------------------------------------------
def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round fp32 values to bf16 (nearest-even) and return the uint16 bits."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    lsb = (u >> 16) & np.uint32(1)
    return ((u + np.uint32(0x7FFF) + lsb) >> 16).astype(np.uint16)


def normal_bf16(rng: np.random.Generator, shape) -> np.ndarray:
    return f32_to_bf16_bits(rng.standard_normal(shape, dtype=np.float32))


def _bits_as_f32(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << 16).view(np.float32)


def _unit(v: np.ndarray) -> np.ndarray:
    return v / np.linalg.norm(v)


def paged_pool(logical: np.ndarray, block_table: np.ndarray, num_pages: int, page: int = PAGE) -> np.ndarray:
    """Scatter logical ``[B][Hkv][S][d]`` rows into a ``[pages][Hkv][page][d]`` pool.

    Token ``t`` of sequence ``b`` goes to page ``block_table[b][t // page]``,
    row ``t % page``.  Unused pool rows are zero.
    """
    B, Hkv, S, d = logical.shape
    pool = np.zeros((num_pages, Hkv, page, d), dtype=logical.dtype)
    npg = (S + page - 1) // page
    for b in range(B):
        full = np.zeros((Hkv, npg * page, d), dtype=logical.dtype)
        full[:, :S] = logical[b]
        pages = full.reshape(Hkv, npg, page, d).transpose(1, 0, 2, 3)
        pool[block_table[b, :npg]] = pages
    return pool


# ----------------------------------------------------------------------------
# decode + H2O workloads
# ----------------------------------------------------------------------------
@dataclass
class DecodeWorkload:
    name: str
    B: int
    Hq: int
    Hkv: int
    d: int
    S0: int
    steps: int
    budget: int
    n_sink: int
    window: int
    max_len: int
    max_pages: int
    num_pages: int
    block_table: np.ndarray          # int32 [B][max_pages]
    K: np.ndarray                    # bf16 bits [B][Hkv][S0][d] (logical order)
    V: np.ndarray
    q: np.ndarray                    # bf16 bits [steps][B][Hq][d]
    k_new: np.ndarray                # bf16 bits [steps][B][Hkv][d]
    v_new: np.ndarray
    seed: int = 0
    extra: dict = field(default_factory=dict)
    page: int = PAGE                 # tokens per pool page

    @property
    def G(self) -> int:
        return self.Hq // self.Hkv

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)


def _decode_workload(name, seed, B, Hq, Hkv, d, S0, steps, budget, n_sink, window,
                     permute_pages, plant_sink, page=PAGE):
    rng = np.random.default_rng(seed)
    max_len = S0 + steps
    max_pages = (max_len + page - 1) // page
    num_pages = B * max_pages
    if permute_pages:
        block_table = rng.permutation(num_pages).astype(np.int32).reshape(B, max_pages)
    else:
        block_table = np.arange(num_pages, dtype=np.int32).reshape(B, max_pages)
    K = np.empty((B, Hkv, S0, d), dtype=np.uint16)
    V = np.empty((B, Hkv, S0, d), dtype=np.uint16)
    Kf = [None] * B
    for b in range(B):
        kb = rng.standard_normal((Hkv, S0, d), dtype=np.float32)
        vb = rng.standard_normal((Hkv, S0, d), dtype=np.float32)
        Kf[b] = kb
        V[b] = f32_to_bf16_bits(vb)
    q = normal_bf16(rng, (steps, B, Hq, d))
    k_new = normal_bf16(rng, (steps, B, Hkv, d))
    v_new = normal_bf16(rng, (steps, B, Hkv, d))
    G = Hq // Hkv
    for b in range(B):
        if plant_sink:
            qf = _bits_as_f32(q[:, b])                      # [steps][Hq][d]
            for kvh in range(Hkv):
                u = _unit(qf[:, kvh * G:(kvh + 1) * G].reshape(-1, d).mean(0))
                Kf[b][kvh, 0] += np.float32(4.0) * u.astype(np.float32)
        K[b] = f32_to_bf16_bits(Kf[b])
        Kf[b] = None
    return DecodeWorkload(name, B, Hq, Hkv, d, S0, steps, budget, n_sink, window,
                          max_len, max_pages, num_pages, block_table, K, V, q,
                          k_new, v_new, seed, page=page)


def decode_small(seed: int = 0, S0: int = 1600, steps: int = 64) -> DecodeWorkload:
    """One sequence, 16 q / 8 kv heads, prompt 1600, 64 steps, budget 256 = 4+64+188."""
    return _decode_workload("decode_small", seed, B=1, Hq=16, Hkv=8, d=128, S0=S0,
                            steps=steps, budget=256, n_sink=4, window=64,
                            permute_pages=False, plant_sink=True)


def decode_70b(seed: int = 1, B: int = 8, S0: int = 32768, steps: int = 128) -> DecodeWorkload:
    """Llama-2-70B layer shape, batch 8 x 32K, permuted 16-token pages, 128 steps.

    Budget is 20% of the 32K prompt: floor(0.2 * 32768) = 6553 = 4 + 1024 + 5525.
    """
    budget = int(0.2 * 32768)
    return _decode_workload("decode_70b", seed, B=B, Hq=64, Hkv=8, d=128, S0=S0,
                            steps=steps, budget=budget, n_sink=4, window=1024,
                            permute_pages=True, plant_sink=False)


def decode_custom(seed, B, Hq, Hkv, d, S0, steps, budget, n_sink, window,
                  permute_pages=True, plant_sink=False, name="decode_custom", page=PAGE):
    return _decode_workload(name, seed, B, Hq, Hkv, d, S0, steps, budget, n_sink,
                            window, permute_pages, plant_sink, page)


# ----------------------------------------------------------------------------
# SnapKV workload
# ----------------------------------------------------------------------------
@dataclass
class SnapKVLayer:
    K: np.ndarray          # bf16 bits [Hkv][S][d]
    V: np.ndarray
    q_obs: np.ndarray      # bf16 bits [Hq][W][d]
    planted: np.ndarray    # int [Hkv][n_planted] prefix positions pushed toward q_obs
    block_table: np.ndarray  # int32 [max_pages] (random permutation of this layer's pages)


@dataclass
class SnapKVWorkload:
    name: str
    L: int
    Hq: int
    Hkv: int
    d: int
    S: int
    W: int
    keep_k: int
    pool_kernel: int
    n_planted: int
    seed: int
    plant_amp: float = 4.0

    @property
    def G(self) -> int:
        return self.Hq // self.Hkv

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)

    @property
    def pages(self) -> int:
        return (self.S + PAGE - 1) // PAGE

    def layer(self, l: int) -> SnapKVLayer:
        """Draw layer ``l`` (independent stream per layer, so layers can be drawn alone)."""
        rng = np.random.default_rng([self.seed, l])
        S, Hkv, Hq, d, W, G = self.S, self.Hkv, self.Hq, self.d, self.W, self.G
        bt = rng.permutation(self.pages).astype(np.int32)
        Kf = rng.standard_normal((Hkv, S, d), dtype=np.float32)
        V = normal_bf16(rng, (Hkv, S, d))
        q_obs = normal_bf16(rng, (Hq, W, d))
        qf = _bits_as_f32(q_obs)
        cells = max(0, (S - W) // 16)
        n_pl = min(self.n_planted, cells)          # a short prefix holds fewer planted keys
        planted = np.empty((Hkv, n_pl), dtype=np.int64)
        for kvh in range(Hkv):
            pos = 16 * rng.choice(cells, n_pl, replace=False) + rng.integers(0, 8, n_pl) if n_pl else \
                np.zeros(0, dtype=np.int64)
            pos.sort()
            planted[kvh] = pos
            u = _unit(qf[kvh * G:(kvh + 1) * G].reshape(-1, d).mean(0)).astype(np.float32)
            Kf[kvh, pos] += np.float32(self.plant_amp) * u
        return SnapKVLayer(f32_to_bf16_bits(Kf), V, q_obs, planted, bt)


def snapkv_qwen7b(seed: int = 2, L: int = 28, S: int = 32768) -> SnapKVWorkload:
    """Qwen2.5-7B shape; 64 planted keys per kv head pushed +16 along the unit mean query.

    (+16 gives each window query a logit boost of about 1.1 on average, so the
    planted keys collect about three times the background vote.)
    """
    return SnapKVWorkload("snapkv_qwen7b", L=L, Hq=28, Hkv=4, d=128, S=S, W=32,
                          keep_k=2048, pool_kernel=7, n_planted=64, seed=seed, plant_amp=16.0)


def snapkv_custom(seed, L, Hq, Hkv, d, S, W, keep_k, pool_kernel=7, n_planted=8, plant_amp=4.0):
    return SnapKVWorkload("snapkv_custom", L=L, Hq=Hq, Hkv=Hkv, d=d, S=S, W=W,
                          keep_k=keep_k, pool_kernel=pool_kernel, n_planted=n_planted, seed=seed,
                          plant_amp=plant_amp)


# ----------------------------------------------------------------------------
# block offload priority workload
# ----------------------------------------------------------------------------
@dataclass
class BlockPriorityWorkload:
    name: str
    R: int
    lengths: np.ndarray        # int64 [R]
    alphas: np.ndarray         # float64 [R]
    steps: int
    decay: float
    evict_frac: float
    seed: int

    @property
    def offsets(self) -> np.ndarray:
        off = np.zeros(self.R + 1, dtype=np.int64)
        off[1:] = np.cumsum(self.lengths)
        return off

    @property
    def total_tokens(self) -> int:
        return int(self.lengths.sum())

    def increments(self, step: int) -> np.ndarray:
        """Step ``step``'s per-token increments: Dirichlet(alpha_r * 1) per request, fp32.

        Each request's increments sum to 1 (up to fp32 rounding of the parts).
        Drawn from an independent stream per step so any step can be drawn alone.
        """
        rng = np.random.default_rng([self.seed, 1000 + step])
        out = np.empty(self.total_tokens, dtype=np.float32)
        off = self.offsets
        for r in range(self.R):
            g = rng.standard_gamma(self.alphas[r], int(self.lengths[r]))
            tot = g.sum()
            if tot <= 0.0:          # every gamma draw underflowed: put the mass on one token
                g = np.zeros_like(g)
                g[rng.integers(0, g.size)] = 1.0
                tot = 1.0
            out[off[r]:off[r + 1]] = (g / tot).astype(np.float32)
        return out


def block_priority(seed: int = 3, R: int = 64, steps: int = 200,
                   min_len: int = 4096, max_len: int = 131072) -> BlockPriorityWorkload:
    rng = np.random.default_rng(seed)
    lengths = np.round(np.exp(rng.uniform(math.log(min_len), math.log(max_len), R))).astype(np.int64)
    alphas = np.where(np.arange(R) % 2 == 0, 0.05, 1.0)
    return BlockPriorityWorkload("block_priority", R, lengths, alphas, steps, 0.98, 0.25, seed)


# ----------------------------------------------------------------------------
# DSA-style sparse decode workload
# ----------------------------------------------------------------------------
@dataclass
class SparseDecodeWorkload:
    name: str
    B: int
    Hq: int
    Hkv: int
    d: int
    S0: int
    steps: int
    Hi: int
    Di: int
    top_k: int
    max_len: int
    max_pages: int
    num_pages: int
    block_table: np.ndarray   # int32 [B][max_pages]
    K: np.ndarray             # bf16 bits [B][Hkv][S0][d]
    V: np.ndarray
    k_idx: np.ndarray         # bf16 bits [B][S0][Di]
    q: np.ndarray             # bf16 bits [steps][B][Hq][d]
    k_new: np.ndarray         # bf16 bits [steps][B][Hkv][d]
    v_new: np.ndarray
    q_idx: np.ndarray         # bf16 bits [steps][B][Hi][Di]
    w_idx: np.ndarray         # fp32 [steps][B][Hi]
    k_idx_new: np.ndarray     # bf16 bits [steps][B][Di]
    seed: int
    page: int = PAGE          # tokens per pool page

    @property
    def G(self) -> int:
        return self.Hq // self.Hkv

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)


def sparse_decode(seed: int = 4, B: int = 4, S0: int = 131072, steps: int = 64,
                  Hq: int = 64, Hkv: int = 8, d: int = 128, Hi: int = 4, Di: int = 64,
                  top_k: int = 2048, page: int = PAGE) -> SparseDecodeWorkload:
    rng = np.random.default_rng(seed)
    max_len = S0 + steps
    max_pages = (max_len + page - 1) // page
    num_pages = B * max_pages
    bt = rng.permutation(num_pages).astype(np.int32).reshape(B, max_pages)
    K = np.empty((B, Hkv, S0, d), dtype=np.uint16)
    V = np.empty((B, Hkv, S0, d), dtype=np.uint16)
    for b in range(B):
        K[b] = normal_bf16(rng, (Hkv, S0, d))
        V[b] = normal_bf16(rng, (Hkv, S0, d))
    k_idx = normal_bf16(rng, (B, S0, Di))
    q = normal_bf16(rng, (steps, B, Hq, d))
    k_new = normal_bf16(rng, (steps, B, Hkv, d))
    v_new = normal_bf16(rng, (steps, B, Hkv, d))
    q_idx = normal_bf16(rng, (steps, B, Hi, Di))
    w_idx = rng.standard_normal((steps, B, Hi), dtype=np.float32)
    k_idx_new = normal_bf16(rng, (steps, B, Di))
    return SparseDecodeWorkload("sparse_decode_70b", B, Hq, Hkv, d, S0, steps, Hi, Di, top_k,
                                max_len, max_pages, num_pages, bt, K, V, k_idx, q, k_new,
                                v_new, q_idx, w_idx, k_idx_new, seed, page=page)
