"""Python binding of libkvsel.so (attention-guided KV selection on GB300).

Argument marshalling only: every function takes torch CUDA tensors, checks
their dtype/device/contiguity, and hands raw device pointers and the current
stream to the C ABI declared in ``include/kvsel.h``.  Every step of the path
runs in the library's CUDA kernels; there is no CPU or PyTorch fallback.  If
the shared library is missing this module raises instead of degrading.
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libkvsel.so")

KVSEL_OK = 0
KVSEL_ERR_INVALID_ARG = 1
KVSEL_ERR_UNSUPPORTED = 2
KVSEL_ERR_CUDA = 3
KVSEL_ERR_TIMEOUT = 4
KVSEL_ERR_BAD_INDEX = 5
KVSEL_BF16 = 0
KVSEL_F32 = 1
KVSEL_AGG_MAX, KVSEL_AGG_MEAN, KVSEL_AGG_TOPP, KVSEL_AGG_FRAC_HOT, KVSEL_AGG_ALL_COLD = 0, 1, 2, 3, 4
KVSEL_NORM_NONE, KVSEL_NORM_PERCENTILE = 0, 1
KVSEL_UPDATE_DECAY, KVSEL_UPDATE_MAX, KVSEL_UPDATE_WINDOW = 0, 1, 2
KVSEL_SNAP_GROUP_SUM, KVSEL_SNAP_HEAD_UNION = 0, 1

_STATUS = {0: "OK", 1: "INVALID_ARG", 2: "UNSUPPORTED", 3: "CUDA", 4: "TIMEOUT", 5: "BAD_INDEX"}


class KvselError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"kvsel status {_STATUS.get(code, code)}: {msg}")
        self.code = code


class PagedKV(ctypes.Structure):
    _fields_ = [("k_pool", ctypes.c_void_p), ("v_pool", ctypes.c_void_p),
                ("num_pages", ctypes.c_int32), ("num_kv_heads", ctypes.c_int32),
                ("num_q_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("page_size", ctypes.c_int32)]


class BpOptions(ctypes.Structure):
    _fields_ = [("update", ctypes.c_int), ("history", ctypes.c_void_p), ("window", ctypes.c_int),
                ("step", ctypes.c_int64), ("history_tokens", ctypes.c_int64), ("threshold", ctypes.c_float)]


class BlockSignal(ctypes.Structure):
    _fields_ = [("topk_blocks", ctypes.c_int), ("step", ctypes.c_int32), ("block_score", ctypes.c_void_p),
                ("block_step", ctypes.c_void_p), ("topk_out", ctypes.c_void_p), ("mass_out", ctypes.c_void_p)]


class SnapOptions(ctypes.Structure):
    _fields_ = [("mode", ctypes.c_int), ("keep_count", ctypes.c_void_p), ("seed_out", ctypes.c_void_p),
                ("seed_layer_stride", ctypes.c_int64), ("seed_head_stride", ctypes.c_int64)]


_vp, _i, _f, _sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
_PKV = ctypes.POINTER(PagedKV)

# name -> (restype, argtypes)
_SIGS = {
    "kvsel_last_error_string": (ctypes.c_char_p, []),
    "kvsel_clear_status": (_i, [_vp, _vp]),
    "kvsel_read_status": (_i, [_vp, _vp]),
    "kvsel_set_wait_limit": (_i, [_vp, ctypes.c_uint, _vp]),
    "kvsel_trace_start": (_i, [ctypes.POINTER(ctypes.c_void_p), _i]),
    "kvsel_trace_stop": (_i, [ctypes.POINTER(ctypes.c_char_p), _i]),
    "kvsel_decode_attn_workspace": (_sz, [_PKV, _i, _i, _i]),
    "kvsel_decode_attn": (_i, [_PKV, _vp, _i, _vp, _i, _vp, _vp, _vp, _vp, _vp, _f, _vp, _i, _vp,
                               _vp, _i, _i, _vp, _sz, _vp, _sz, _vp]),
    "kvsel_decode_attn_noalloc": (_i, [_PKV, _vp, _i, _vp, _i, _vp, _vp, _vp, _vp, _vp, _f, _vp, _i,
                                       _vp, _vp, _i, _i, _vp]),
    "kvsel_h2o_evict_workspace": (_sz, [_PKV, _i, _i]),
    "kvsel_h2o_link_bytes": (_sz, [_i, _i]),
    "kvsel_h2o_link_reset": (_i, [_vp, _i, _i, _vp]),
    "kvsel_h2o_evict": (_i, [_PKV, _vp, _i, _vp, _i, _vp, _vp, _i, _i, _i, _i, _i, _vp, _vp, _vp,
                             _sz, _vp]),
    "kvsel_kv_compact_workspace": (_sz, [_i, _i]),
    "kvsel_kv_compact": (_i, [_PKV, _vp, _i, _vp, _i, _vp, _i, _vp, _vp, _vp, _i, _vp, _vp, _sz, _vp]),
    "kvsel_block_priority_workspace": (_sz, [_i, ctypes.c_int64]),
    "kvsel_block_priority": (_i, [_vp, _vp, _f, _vp, _i, _i, _i, _f, _i, _f, _vp, ctypes.c_int64, _vp,
                                  ctypes.c_int64, _vp, _vp, _sz, _vp]),
    "kvsel_block_priority_ex": (_i, [_vp, _vp, _f, _vp, _i, _i, _i, _f, _i, _f, _vp, ctypes.c_int64, _vp,
                                     ctypes.c_int64, _vp, _vp, _sz, ctypes.POINTER(BpOptions), _vp]),
    "kvsel_sparse_decode_workspace": (_sz, [_PKV, _i, _i, _i, _i]),
    "kvsel_sparse_decode": (_i, [_PKV, _vp, _i, _vp, _i, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i,
                                 _i, _f, _vp, _i, _vp, _vp, _vp, _sz, _vp]),
    "kvsel_snapkv_select_workspace": (_sz, [_PKV, _i, _i, _i, _i]),
    "kvsel_snapkv_select": (_i, [_PKV, _vp, _i, _i, _i, _vp, _i, _f, _i, _i, _vp, _vp, _vp, _sz, _vp]),
    "kvsel_snapkv_select_ex_workspace": (_sz, [_PKV, _i, _i, _i, _i, _i]),
    "kvsel_decode_attn_ex_workspace": (_sz, [_PKV, _i, _i, _i, _i]),
    "kvsel_decode_attn_ex": (_i, [_PKV, _vp, _i, _vp, _i, _vp, _vp, _vp, _vp, _vp, _f, _vp, _i, _vp, _vp, _i, _i,
                                  ctypes.POINTER(BlockSignal), _vp, _sz, _vp, _sz, _vp]),
    "kvsel_quest_page_meta": (_i, [_PKV, _vp, _i, _vp, _i, _vp, _vp, _vp]),
    "kvsel_quest_decode_workspace": (_sz, [_PKV, _i, _i, _i, _i, _i]),
    "kvsel_quest_decode": (_i, [_PKV, _vp, _i, _vp, _i, _vp, _vp, _vp, _vp, _i, _f, _vp, _i, _vp, _vp, _vp, _sz,
                                _vp]),
    "kvsel_snapkv_select_ex": (_i, [_PKV, _vp, _i, _i, _i, _vp, _i, _f, _i, _i, ctypes.POINTER(SnapOptions), _vp,
                                    _vp, _vp, _sz, _vp]),
}

_lib = None


def lib() -> ctypes.CDLL:
    """Load libkvsel.so once (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with __graft_entry__.build() "
                               "(nvcc, sm_103a); there is no fallback path")
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGS.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def exported_symbols():
    return list(_SIGS)


def _check(code: int):
    if code != KVSEL_OK:
        raise KvselError(code, lib().kvsel_last_error_string().decode())


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _need(t, dtype, name, allow_none=False):
    if t is None:
        if allow_none:
            return
        raise ValueError(f"{name} is required")
    if t.device.type != "cuda":
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _stream(stream):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def paged_kv(k_pool: torch.Tensor, v_pool: torch.Tensor, num_q_heads: int) -> PagedKV:
    """Descriptor of bf16 pools shaped [num_pages][num_kv_heads][page_size][head_dim]."""
    _need(k_pool, torch.bfloat16, "k_pool")
    _need(v_pool, torch.bfloat16, "v_pool")
    if k_pool.shape != v_pool.shape or k_pool.dim() != 4:
        raise ValueError("k_pool and v_pool must share one [pages][Hkv][page][d] shape")
    P, H, pg, d = k_pool.shape
    return PagedKV(k_pool.data_ptr(), v_pool.data_ptr(), P, H, num_q_heads, d, pg)


def clear_status(workspace: torch.Tensor, stream=None):
    _check(lib().kvsel_clear_status(_ptr(workspace), _stream(stream)))


def read_status(workspace: torch.Tensor, stream=None) -> int:
    """Synchronise and return (and clear) the device status word of a workspace."""
    return int(lib().kvsel_read_status(_ptr(workspace), _stream(stream)))


def set_wait_limit(workspace: torch.Tensor, spins: int, stream=None):
    """Bound the cross-CTA waits of kernels using this workspace (0 = the default of a few seconds)."""
    _check(lib().kvsel_set_wait_limit(_ptr(workspace), int(spins), _stream(stream)))


class LaunchTrace:
    """Record CUDA events around every library kernel launched by this thread.

    with LaunchTrace(capacity) as tr: ...   then tr.durations() -> [(name, ms)].
    """

    def __init__(self, capacity: int):
        self.capacity = capacity
        self.events = [torch.cuda.Event(enable_timing=True) for _ in range(2 * capacity)]
        for e in self.events:
            e.record()                       # materialise the cudaEvent_t handles
        self._handles = (ctypes.c_void_p * (2 * capacity))(*[e.cuda_event for e in self.events])
        self.names = []

    def __enter__(self):
        _check(lib().kvsel_trace_start(self._handles, self.capacity))
        return self

    def __exit__(self, *exc):
        buf = (ctypes.c_char_p * self.capacity)()
        n = lib().kvsel_trace_stop(buf, self.capacity)
        self.names = [buf[i].decode() for i in range(min(n, self.capacity))]
        return False

    def durations(self):
        torch.cuda.synchronize()
        return [(nm, self.events[2 * i].elapsed_time(self.events[2 * i + 1]))
                for i, nm in enumerate(self.names)]


# ----------------------------------------------------------------------------
# decode attention
# ----------------------------------------------------------------------------
def kvsel_decode_attn_workspace(kv: PagedKV, batch: int, max_len: int, with_probs: bool) -> int:
    return int(lib().kvsel_decode_attn_workspace(ctypes.byref(kv), batch, max_len, int(with_probs)))


def kvsel_decode_attn_ex_workspace(kv: PagedKV, batch: int, max_len: int, with_probs: bool,
                                   with_signal: bool) -> int:
    return int(lib().kvsel_decode_attn_ex_workspace(ctypes.byref(kv), batch, max_len, int(with_probs),
                                                    int(with_signal)))


def kvsel_decode_attn(kv: PagedKV, block_table, seq_lens, q, out, workspace, *, k_new=None,
                      v_new=None, pos_map=None, next_pos=None, scale=None, probs=None,
                      h2o_cum=None, max_len=None, num_ctas=0, h2o_link=None, block_score=None,
                      block_step=None, signal_topk=512, signal_step=0, signal_topk_out=None,
                      signal_mass_out=None, stream=None):
    """Append (optional) + decode attention + probabilities + H2O score update.

    h2o_link: the workspace of the kvsel_h2o_evict calls that follow (same
    batch); the step then hands them its heavy-hitter candidates.
    block_score / block_step (per physical block, fp32 / int32): given, the
    same launch also emits the step's top-k block signal (signal_topk blocks
    per sequence; optional outputs signal_topk_out [batch][signal_topk] and
    signal_mass_out [batch][ceil(max_len / 16)]); the workspace must then be
    sized by kvsel_decode_attn_ex_workspace(..., with_signal=True).
    """
    _need(block_table, torch.int32, "block_table")
    _need(seq_lens, torch.int32, "seq_lens")
    _need(q, torch.bfloat16, "q")
    _need(k_new, torch.bfloat16, "k_new", True)
    _need(v_new, torch.bfloat16, "v_new", True)
    _need(pos_map, torch.int32, "pos_map", True)
    _need(next_pos, torch.int32, "next_pos", True)
    _need(probs, torch.float32, "probs", True)
    _need(h2o_cum, torch.float32, "h2o_cum", True)
    _need(workspace, workspace.dtype, "workspace")
    if out.dtype not in (torch.bfloat16, torch.float32) or not out.is_contiguous():
        raise ValueError("out must be a contiguous bf16 or fp32 CUDA tensor")
    batch = seq_lens.shape[0]
    if max_len is None:
        for t in (probs, h2o_cum, pos_map):
            if t is not None:
                max_len = t.shape[-1]
                break
        else:
            max_len = block_table.shape[1] * kv.page_size
    if scale is None:
        scale = kv.head_dim ** -0.5
    odt = KVSEL_F32 if out.dtype == torch.float32 else KVSEL_BF16
    sig = None
    if block_score is not None or block_step is not None:
        _need(block_score, torch.float32, "block_score")
        _need(block_step, torch.int32, "block_step")
        _need(signal_topk_out, torch.int32, "signal_topk_out", True)
        _need(signal_mass_out, torch.float32, "signal_mass_out", True)
        sig = BlockSignal(int(signal_topk), int(signal_step), block_score.data_ptr(), block_step.data_ptr(),
                          signal_topk_out.data_ptr() if signal_topk_out is not None else None,
                          signal_mass_out.data_ptr() if signal_mass_out is not None else None)
    _check(lib().kvsel_decode_attn_ex(
        ctypes.byref(kv), _ptr(block_table), block_table.shape[1], _ptr(seq_lens), batch, _ptr(q),
        _ptr(k_new), _ptr(v_new), _ptr(pos_map), _ptr(next_pos), float(scale), _ptr(out), odt,
        _ptr(probs), _ptr(h2o_cum), int(max_len), int(num_ctas), ctypes.byref(sig) if sig is not None else None,
        _ptr(workspace), workspace.numel() * workspace.element_size(), _ptr(h2o_link),
        0 if h2o_link is None else h2o_link.numel() * h2o_link.element_size(), _stream(stream)))


def kvsel_decode_attn_noalloc(kv: PagedKV, block_table, seq_lens, q, out, *, k_new=None,
                              v_new=None, pos_map=None, next_pos=None, scale=None, probs=None,
                              h2o_cum=None, max_len=None, num_ctas=0, stream=None):
    """kvsel_decode_attn without a workspace, for callers that cannot allocate.

    The library's built-in 8 MiB device array serves as scratch; calls that
    need more are rejected, and calls that overlap on the GPU race.
    """
    for t, dt, nm, opt in ((block_table, torch.int32, "block_table", False),
                           (seq_lens, torch.int32, "seq_lens", False), (q, torch.bfloat16, "q", False),
                           (k_new, torch.bfloat16, "k_new", True), (v_new, torch.bfloat16, "v_new", True),
                           (pos_map, torch.int32, "pos_map", True), (next_pos, torch.int32, "next_pos", True),
                           (probs, torch.float32, "probs", True), (h2o_cum, torch.float32, "h2o_cum", True)):
        _need(t, dt, nm, opt)
    if out.dtype not in (torch.bfloat16, torch.float32) or not out.is_contiguous():
        raise ValueError("out must be a contiguous bf16 or fp32 CUDA tensor")
    if max_len is None:
        for t in (probs, h2o_cum, pos_map):
            if t is not None:
                max_len = t.shape[-1]
                break
        else:
            max_len = block_table.shape[1] * kv.page_size
    if scale is None:
        scale = kv.head_dim ** -0.5
    odt = KVSEL_F32 if out.dtype == torch.float32 else KVSEL_BF16
    _check(lib().kvsel_decode_attn_noalloc(
        ctypes.byref(kv), _ptr(block_table), block_table.shape[1], _ptr(seq_lens), seq_lens.shape[0],
        _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(pos_map), _ptr(next_pos), float(scale), _ptr(out), odt,
        _ptr(probs), _ptr(h2o_cum), int(max_len), int(num_ctas), _stream(stream)))


# ----------------------------------------------------------------------------
# H2O select / evict
# ----------------------------------------------------------------------------
def kvsel_h2o_link_reset(workspace, batch: int, num_kv_heads: int, stream=None):
    """Clear the decode -> select hand-off in an H2O evict workspace (after an outside write to h2o_cum)."""
    _check(lib().kvsel_h2o_link_reset(_ptr(workspace), int(batch), int(num_kv_heads), _stream(stream)))


def kvsel_h2o_evict_workspace(kv: PagedKV, batch: int, budget: int) -> int:
    return int(lib().kvsel_h2o_evict_workspace(ctypes.byref(kv), batch, budget))


def kvsel_h2o_evict(kv: PagedKV, block_table, seq_lens, h2o_cum, workspace, *, budget, n_sink,
                    window, compact=False, pos_map=None, keep_out=None, freed_pages=None,
                    stream=None):
    """H2O heavy hitters + StreamingLLM sinks/window; optional in-place compaction."""
    _need(block_table, torch.int32, "block_table")
    _need(seq_lens, torch.int32, "seq_lens")
    _need(h2o_cum, torch.float32, "h2o_cum")
    _need(pos_map, torch.int32, "pos_map", True)
    _need(keep_out, torch.int32, "keep_out", True)
    _need(freed_pages, torch.int32, "freed_pages", True)
    batch = seq_lens.shape[0]
    _check(lib().kvsel_h2o_evict(
        ctypes.byref(kv), _ptr(block_table), block_table.shape[1], _ptr(seq_lens), batch,
        _ptr(h2o_cum), _ptr(pos_map), h2o_cum.shape[-1], int(budget), int(n_sink), int(window),
        int(bool(compact)), _ptr(keep_out), _ptr(freed_pages), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _stream(stream)))


def kvsel_kv_compact_workspace(batch: int, num_kv_heads: int) -> int:
    return int(lib().kvsel_kv_compact_workspace(batch, num_kv_heads))


def kvsel_kv_compact(kv: PagedKV, block_table, seq_lens, keep, workspace, *, keep_count=None, scores=None,
                     pos_map=None, freed_pages=None, stream=None):
    """Move each row's kept slots (keep [batch][Hkv][stride], ascending) to the front, in place."""
    _need(block_table, torch.int32, "block_table")
    _need(seq_lens, torch.int32, "seq_lens")
    _need(keep, torch.int32, "keep")
    _need(keep_count, torch.int32, "keep_count", True)
    _need(scores, torch.float32, "scores", True)
    _need(pos_map, torch.int32, "pos_map", True)
    _need(freed_pages, torch.int32, "freed_pages", True)
    max_len = next((t.shape[-1] for t in (scores, pos_map) if t is not None), 0)
    _check(lib().kvsel_kv_compact(
        ctypes.byref(kv), _ptr(block_table), block_table.shape[-1], _ptr(seq_lens), seq_lens.shape[0],
        _ptr(keep), keep.shape[-1], _ptr(keep_count), _ptr(scores), _ptr(pos_map), int(max_len),
        _ptr(freed_pages), _ptr(workspace), workspace.numel() * workspace.element_size(), _stream(stream)))


def workspace(nbytes: int, device="cuda") -> torch.Tensor:
    """A zeroed, 256-byte aligned workspace buffer (status word cleared)."""
    return torch.zeros(max(int(nbytes), 256), dtype=torch.uint8, device=device)


# ----------------------------------------------------------------------------
# block offload priority
# ----------------------------------------------------------------------------
def kvsel_block_priority_workspace(num_requests: int, max_total_blocks: int) -> int:
    return int(lib().kvsel_block_priority_workspace(num_requests, max_total_blocks))


def kvsel_block_priority(token_scores, req_offsets, order_out, n_out, workspace, *, block_size, agg,
                         norm, evict_frac, increment=None, decay=1.0, top_p=0.1, block_score_out=None,
                         max_total_blocks=None, update=KVSEL_UPDATE_DECAY, history=None, window=1, step=0,
                         threshold=0.0, stream=None):
    """Score update (decay, max over steps or sliding-window sum) + token->block fold + per-request
    percentile + global evict order (kvsel_block_priority_ex)."""
    _need(token_scores, torch.float32, "token_scores")
    _need(increment, torch.float32, "increment", True)
    _need(history, torch.float32, "history", True)
    _need(req_offsets, torch.int64, "req_offsets")
    _need(order_out, torch.int64, "order_out")
    _need(n_out, torch.int64, "n_out")
    _need(block_score_out, torch.float32, "block_score_out", True)
    if max_total_blocks is None:
        max_total_blocks = block_score_out.numel() if block_score_out is not None else token_scores.numel()
    opt = BpOptions(int(update), _ptr(history), int(window), int(step),
                    (history.numel() // max(1, int(window))) if history is not None else 0, float(threshold))
    _check(lib().kvsel_block_priority_ex(
        _ptr(token_scores), _ptr(increment), float(decay), _ptr(req_offsets), req_offsets.numel() - 1,
        int(block_size), int(agg), float(top_p), int(norm), float(evict_frac), _ptr(block_score_out),
        int(max_total_blocks), _ptr(order_out), order_out.numel(), _ptr(n_out), _ptr(workspace),
        workspace.numel() * workspace.element_size(), ctypes.byref(opt), _stream(stream)))


# ----------------------------------------------------------------------------
# DSA-style sparse decode
# ----------------------------------------------------------------------------
def kvsel_sparse_decode_workspace(kv: PagedKV, batch: int, max_len: int, top_k: int,
                                  with_scores_out: bool) -> int:
    return int(lib().kvsel_sparse_decode_workspace(ctypes.byref(kv), batch, max_len, top_k,
                                                   int(with_scores_out)))


def kvsel_sparse_decode(kv: PagedKV, block_table, seq_lens, q, idx_q, idx_w, idx_k, out, workspace, *,
                        top_k=2048, k_new=None, v_new=None, idx_k_new=None, scale=None, topk_out=None,
                        scores_out=None, stream=None):
    """Indexer scores -> top-k positions -> attention over the selected keys."""
    for t, dt, nm, opt in ((block_table, torch.int32, "block_table", False),
                           (seq_lens, torch.int32, "seq_lens", False), (q, torch.bfloat16, "q", False),
                           (idx_q, torch.bfloat16, "idx_q", False), (idx_w, torch.float32, "idx_w", False),
                           (idx_k, torch.bfloat16, "idx_k", False), (k_new, torch.bfloat16, "k_new", True),
                           (v_new, torch.bfloat16, "v_new", True), (idx_k_new, torch.bfloat16, "idx_k_new", True),
                           (topk_out, torch.int32, "topk_out", True), (scores_out, torch.float32, "scores_out", True)):
        _need(t, dt, nm, opt)
    if out.dtype not in (torch.bfloat16, torch.float32) or not out.is_contiguous():
        raise ValueError("out must be a contiguous bf16 or fp32 CUDA tensor")
    B, Hi, Di = idx_q.shape
    max_len = idx_k.shape[1]
    if scale is None:
        scale = kv.head_dim ** -0.5
    odt = KVSEL_F32 if out.dtype == torch.float32 else KVSEL_BF16
    _check(lib().kvsel_sparse_decode(
        ctypes.byref(kv), _ptr(block_table), block_table.shape[1], _ptr(seq_lens), B, _ptr(q), _ptr(k_new),
        _ptr(v_new), _ptr(idx_q), _ptr(idx_w), _ptr(idx_k), _ptr(idx_k_new), Hi, Di, max_len, int(top_k),
        float(scale), _ptr(out), odt, _ptr(topk_out), _ptr(scores_out), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _stream(stream)))


# ----------------------------------------------------------------------------
# SnapKV prefill selection
# ----------------------------------------------------------------------------
def kvsel_snapkv_select_workspace(kv: PagedKV, num_layers: int, seq_len: int, obs_window: int,
                                  with_vote_out: bool) -> int:
    return int(lib().kvsel_snapkv_select_workspace(ctypes.byref(kv), num_layers, seq_len, obs_window,
                                                   int(with_vote_out)))


def kvsel_snapkv_select(kv: PagedKV, block_table, q_obs, keep_out, workspace, *, seq_len, keep_k,
                        pool_kernel=7, scale=None, vote_out=None, stream=None):
    """Observation-window votes, max-pool and top-k keep per layer and kv head."""
    _need(block_table, torch.int32, "block_table")
    _need(q_obs, torch.bfloat16, "q_obs")
    _need(keep_out, torch.int32, "keep_out")
    _need(vote_out, torch.float32, "vote_out", True)
    L, Hq, W, d = q_obs.shape
    if scale is None:
        scale = kv.head_dim ** -0.5
    _check(lib().kvsel_snapkv_select(
        ctypes.byref(kv), _ptr(block_table), block_table.shape[-1], L, int(seq_len), _ptr(q_obs), W,
        float(scale), int(pool_kernel), int(keep_k), _ptr(keep_out), _ptr(vote_out), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _stream(stream)))


def kvsel_snapkv_select_ex_workspace(kv: PagedKV, num_layers: int, seq_len: int, obs_window: int,
                                     with_vote_out: bool, mode: int = KVSEL_SNAP_GROUP_SUM) -> int:
    return int(lib().kvsel_snapkv_select_ex_workspace(ctypes.byref(kv), num_layers, seq_len, obs_window,
                                                      int(with_vote_out), int(mode)))


def kvsel_snapkv_select_ex(kv: PagedKV, block_table, q_obs, keep_out, workspace, *, seq_len, keep_k,
                           mode=KVSEL_SNAP_GROUP_SUM, pool_kernel=7, scale=None, vote_out=None,
                           keep_count=None, seed_out=None, seed_layer_stride=0, seed_head_stride=0,
                           stream=None):
    """SnapKV selection with the union keep mode, keep counts and cold-start seeds.

    seed_out is a float32 tensor (or a view into one) addressed with the given
    element strides: entry i of (layer l, kv head h) at l * seed_layer_stride +
    h * seed_head_stride + i from its first element.
    """
    _need(block_table, torch.int32, "block_table")
    _need(q_obs, torch.bfloat16, "q_obs")
    _need(keep_out, torch.int32, "keep_out")
    _need(vote_out, torch.float32, "vote_out", True)
    _need(keep_count, torch.int32, "keep_count", True)
    if seed_out is not None and (seed_out.dtype != torch.float32 or seed_out.device.type != "cuda"):
        raise ValueError("seed_out must be a CUDA float32 tensor")
    L, Hq, W, d = q_obs.shape
    if scale is None:
        scale = kv.head_dim ** -0.5
    opt = SnapOptions(int(mode), keep_count.data_ptr() if keep_count is not None else None,
                      seed_out.data_ptr() if seed_out is not None else None,
                      int(seed_layer_stride), int(seed_head_stride))
    _check(lib().kvsel_snapkv_select_ex(
        ctypes.byref(kv), _ptr(block_table), block_table.shape[-1], L, int(seq_len), _ptr(q_obs), W,
        float(scale), int(pool_kernel), int(keep_k), ctypes.byref(opt), _ptr(keep_out), _ptr(vote_out),
        _ptr(workspace), workspace.numel() * workspace.element_size(), _stream(stream)))


def kvsel_quest_page_meta(kv: PagedKV, block_table, seq_lens, page_meta, workspace, stream=None):
    """Per-page key min / max for every page of each sequence (status in the workspace's first word)."""
    _need(block_table, torch.int32, "block_table")
    _need(seq_lens, torch.int32, "seq_lens")
    _need(page_meta, torch.bfloat16, "page_meta")
    _check(lib().kvsel_quest_page_meta(ctypes.byref(kv), _ptr(block_table), block_table.shape[-1],
                                       _ptr(seq_lens), seq_lens.shape[0], _ptr(page_meta), _ptr(workspace),
                                       _stream(stream)))


def kvsel_quest_decode_workspace(kv: PagedKV, batch: int, max_pages: int, budget_pages: int,
                                 with_bounds_out: bool = False, with_pages_out: bool = False) -> int:
    return int(lib().kvsel_quest_decode_workspace(ctypes.byref(kv), batch, max_pages, budget_pages,
                                                  int(with_bounds_out), int(with_pages_out)))


def kvsel_quest_decode(kv: PagedKV, block_table, seq_lens, q, page_meta, out, workspace, *, budget_pages,
                       k_new=None, v_new=None, scale=None, pages_out=None, bounds_out=None, stream=None):
    """One decode step with Quest page selection per q head."""
    _need(block_table, torch.int32, "block_table")
    _need(seq_lens, torch.int32, "seq_lens")
    _need(q, torch.bfloat16, "q")
    _need(page_meta, torch.bfloat16, "page_meta")
    _need(k_new, torch.bfloat16, "k_new", True)
    _need(v_new, torch.bfloat16, "v_new", True)
    _need(pages_out, torch.int32, "pages_out", True)
    _need(bounds_out, torch.float32, "bounds_out", True)
    if out.dtype not in (torch.bfloat16, torch.float32):
        raise ValueError("out must be bfloat16 or float32")
    if scale is None:
        scale = kv.head_dim ** -0.5
    _check(lib().kvsel_quest_decode(
        ctypes.byref(kv), _ptr(block_table), block_table.shape[-1], _ptr(seq_lens), seq_lens.shape[0], _ptr(q),
        _ptr(k_new), _ptr(v_new), _ptr(page_meta), int(budget_pages), float(scale), _ptr(out),
        KVSEL_F32 if out.dtype == torch.float32 else KVSEL_BF16, _ptr(pages_out), _ptr(bounds_out),
        _ptr(workspace), workspace.numel() * workspace.element_size(), _stream(stream)))
