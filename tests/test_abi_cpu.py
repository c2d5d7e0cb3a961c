"""The C-ABI library builds, loads and exports every declared symbol (no GPU).

Only host-side argument checks are exercised here: they return before any
CUDA call, so they run on a machine without a GPU.
"""
import ctypes
import glob
import os
import re

import pytest

from conftest import ROOT

import attention_guided_kv_gb300 as K


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(K.LIB_PATH):
        from attention_guided_kv_gb300 import _build
        _build.build()
    return K.lib()


def declared_symbols():
    names = []
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        names += re.findall(r"KVSEL_API\s+[\w\s\*]*?\b(kvsel_\w+)\s*\(", text)
    return sorted(set(names))


def test_every_declared_symbol_is_exported(lib):
    names = declared_symbols()
    assert len(names) >= 7
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) == set(K.exported_symbols())


def test_binding_does_not_import_the_oracle():
    src = open(os.path.join(ROOT, "attention_guided_kv_gb300", "__init__.py")).read()
    assert "oracle" not in re.sub(r'""".*?"""', "", src, flags=re.S)
    for f in glob.glob(os.path.join(ROOT, "attention_guided_kv_gb300", "csrc", "*")):
        assert "oracle" not in open(f).read(), f


def _kv(**kw):
    d = dict(k_pool=16, v_pool=16, num_pages=10, num_kv_heads=8, num_q_heads=64, head_dim=128,
             page_size=16)
    d.update(kw)
    return K.PagedKV(**d)


def test_workspace_sizes(lib):
    kv = _kv()
    a = K.kvsel_decode_attn_workspace(kv, 8, 32896, True)
    b = K.kvsel_decode_attn_workspace(kv, 8, 32896, False)
    assert a > 0 and b - a >= 8 * 64 * 32896 * 4           # logits scratch when probs are not kept
    assert K.kvsel_decode_attn_workspace(kv, 8, 32896, True) < 8 << 20
    assert K.kvsel_h2o_evict_workspace(kv, 8, 6553) >= 8 * 8 * 6553 * 4
    # the decode hand-off sits at the start of every evict workspace
    assert K.kvsel_h2o_evict_workspace(kv, 8, 6553) >= K.lib().kvsel_h2o_link_bytes(8, 8) + 8 * 8 * 6553 * 4
    assert K.lib().kvsel_h2o_link_bytes(8, 8) >= 64 * 16384 * 8
    assert K.lib().kvsel_h2o_link_bytes(0, 8) == 0
    assert K.kvsel_decode_attn_workspace(_kv(num_q_heads=12), 1, 10, True) == 0


def _decode_status(lib, kv, **over):
    args = dict(block_table=16, max_pages=4, seq_lens=16, batch=1, q=16, k_new=None, v_new=None,
                pos_map=None, next_pos=None, scale=0.1, out=16, out_dtype=0, probs=None, cum=None,
                max_len=64, num_ctas=0, ws=256, ws_bytes=1 << 30, link=None, link_bytes=0, stream=None)
    args.update(over)
    return lib.kvsel_decode_attn(ctypes.byref(kv), args["block_table"], args["max_pages"],
                                 args["seq_lens"], args["batch"], args["q"], args["k_new"],
                                 args["v_new"], args["pos_map"], args["next_pos"], args["scale"],
                                 args["out"], args["out_dtype"], args["probs"], args["cum"],
                                 args["max_len"], args["num_ctas"], args["ws"], args["ws_bytes"],
                                 args["link"], args["link_bytes"], args["stream"])


def test_decode_host_validation(lib):
    assert _decode_status(lib, _kv(k_pool=None)) == K.KVSEL_ERR_INVALID_ARG
    assert _decode_status(lib, _kv(head_dim=64)) == K.KVSEL_ERR_UNSUPPORTED
    for bad_page in (8, 24, 48, 512):                           # 16, 32, 64, 128, 256 are accepted
        assert _decode_status(lib, _kv(page_size=bad_page)) == K.KVSEL_ERR_UNSUPPORTED
    assert _decode_status(lib, _kv(num_q_heads=160, num_kv_heads=8)) == K.KVSEL_ERR_UNSUPPORTED
    assert _decode_status(lib, _kv(num_q_heads=12)) == K.KVSEL_ERR_INVALID_ARG
    assert _decode_status(lib, _kv(), k_new=16) == K.KVSEL_ERR_INVALID_ARG
    assert _decode_status(lib, _kv(), pos_map=16) == K.KVSEL_ERR_INVALID_ARG
    assert _decode_status(lib, _kv(), out_dtype=7) == K.KVSEL_ERR_INVALID_ARG
    assert _decode_status(lib, _kv(), num_ctas=1025) == K.KVSEL_ERR_INVALID_ARG
    assert _decode_status(lib, _kv(), q=8) == K.KVSEL_ERR_INVALID_ARG          # misaligned
    assert _decode_status(lib, _kv(), ws_bytes=100) == K.KVSEL_ERR_INVALID_ARG
    assert _decode_status(lib, _kv(), ws=None) == K.KVSEL_ERR_INVALID_ARG
    assert b"workspace" in lib.kvsel_last_error_string()
    need = K.lib().kvsel_h2o_link_bytes(1, 8)
    assert _decode_status(lib, _kv(), link=512, link_bytes=need - 1) == K.KVSEL_ERR_INVALID_ARG
    assert _decode_status(lib, _kv(), link=512 + 16, link_bytes=need) == K.KVSEL_ERR_INVALID_ARG  # misaligned
    assert b"h2o_link" in lib.kvsel_last_error_string()


def test_evict_host_validation(lib):
    kv = _kv()

    def st(**over):
        a = dict(bt=16, max_pages=4, seq=16, batch=1, cum=16, pos=None, max_len=64, budget=10,
                 n_sink=4, window=4, compact=0, keep=None, freed=None, ws=256, ws_bytes=1 << 20)
        a.update(over)
        return lib.kvsel_h2o_evict(ctypes.byref(a.pop("kv", kv)), a["bt"], a["max_pages"], a["seq"],
                                   a["batch"], a["cum"], a["pos"], a["max_len"], a["budget"],
                                   a["n_sink"], a["window"], a["compact"], a["keep"], a["freed"],
                                   a["ws"], a["ws_bytes"], None)
    assert st(budget=7) == K.KVSEL_ERR_INVALID_ARG          # budget < sinks + window
    assert st(n_sink=-1) == K.KVSEL_ERR_INVALID_ARG
    assert st(cum=None) == K.KVSEL_ERR_INVALID_ARG
    assert st(ws_bytes=8) == K.KVSEL_ERR_INVALID_ARG
    assert st(kv=_kv(page_size=8)) == K.KVSEL_ERR_UNSUPPORTED
    assert st(compact=1, kv=_kv(k_pool=None)) == K.KVSEL_ERR_INVALID_ARG


def test_block_priority_host_validation(lib):
    def st(**over):
        a = dict(tok=16, inc=None, decay=0.98, off=16, R=4, bs=16, agg=0, top_p=0.1, norm=1,
                 frac=0.25, bso=None, maxb=100, order=16, cap=25, n_out=16, ws=256, ws_bytes=1 << 20)
        a.update(over)
        return lib.kvsel_block_priority(a["tok"], a["inc"], a["decay"], a["off"], a["R"], a["bs"],
                                        a["agg"], a["top_p"], a["norm"], a["frac"], a["bso"], a["maxb"],
                                        a["order"], a["cap"], a["n_out"], a["ws"], a["ws_bytes"], None)
    assert st(bs=0) == K.KVSEL_ERR_UNSUPPORTED
    assert st(bs=512) == K.KVSEL_ERR_UNSUPPORTED
    assert st(agg=3) == K.KVSEL_ERR_INVALID_ARG
    assert st(norm=2) == K.KVSEL_ERR_INVALID_ARG
    assert st(agg=2, top_p=0.0) == K.KVSEL_ERR_INVALID_ARG
    assert st(frac=1.5) == K.KVSEL_ERR_INVALID_ARG
    assert st(order=None) == K.KVSEL_ERR_INVALID_ARG
    assert st(tok=None) == K.KVSEL_ERR_INVALID_ARG
    assert st(ws_bytes=64) == K.KVSEL_ERR_INVALID_ARG
    assert K.kvsel_block_priority_workspace(64, 150000) > 150000 * 28


def test_sparse_decode_host_validation(lib):
    kv = _kv()

    def st(**over):
        a = dict(bt=16, max_pages=8200, seq=16, batch=4, q=16, kn=None, vn=None, iq=16, iw=16, ik=16,
                 ikn=None, Hi=4, Di=64, max_len=131136, top_k=2048, scale=0.1, out=16, odt=0,
                 topk=None, scores=None, ws=256, ws_bytes=1 << 30)
        a.update(over)
        return lib.kvsel_sparse_decode(ctypes.byref(a.pop("kv", kv)), a["bt"], a["max_pages"], a["seq"],
                                       a["batch"], a["q"], a["kn"], a["vn"], a["iq"], a["iw"], a["ik"],
                                       a["ikn"], a["Hi"], a["Di"], a["max_len"], a["top_k"], a["scale"],
                                       a["out"], a["odt"], a["topk"], a["scores"], a["ws"], a["ws_bytes"],
                                       None)
    assert st(Di=128) == K.KVSEL_ERR_UNSUPPORTED
    assert st(Hi=9) == K.KVSEL_ERR_UNSUPPORTED
    assert st(kn=16) == K.KVSEL_ERR_INVALID_ARG          # k_new without v_new / idx_k_new
    assert st(top_k=0) == K.KVSEL_ERR_INVALID_ARG
    assert st(max_len=(1 << 28) + 1) == K.KVSEL_ERR_UNSUPPORTED
    assert st(ws_bytes=100) == K.KVSEL_ERR_INVALID_ARG
    assert st(kv=_kv(num_q_heads=136)) == K.KVSEL_ERR_UNSUPPORTED     # 17 q heads per kv head


def test_snapkv_ex_host_validation(lib):
    kv = _kv(num_q_heads=32, num_kv_heads=4, num_pages=4096)   # G = 8

    def st(opt=None, **over):
        a = dict(bt=16, max_pages=4096, L=2, S=4096, q=16, W=32, scale=0.1, pool=7, keep_k=256,
                 keep=16, vote=None, ws=256, ws_bytes=1 << 30)
        a.update(over)
        return lib.kvsel_snapkv_select_ex(ctypes.byref(kv), a["bt"], a["max_pages"], a["L"], a["S"], a["q"],
                                          a["W"], a["scale"], a["pool"], a["keep_k"],
                                          ctypes.byref(opt) if opt is not None else None, a["keep"],
                                          a["vote"], a["ws"], a["ws_bytes"], None)
    assert st(K.SnapOptions(mode=2)) == K.KVSEL_ERR_INVALID_ARG
    # union capacity is G * keep_k + W = 2080: a seed row of 2079 elements is too short
    assert st(K.SnapOptions(mode=1, seed_out=16, seed_layer_stride=4 * 2080,
                            seed_head_stride=2079)) == K.KVSEL_ERR_INVALID_ARG
    assert b"seed strides" in lib.kvsel_last_error_string()
    # layers overlapping each other
    assert st(K.SnapOptions(mode=1, seed_out=16, seed_layer_stride=3 * 2080,
                            seed_head_stride=2080)) == K.KVSEL_ERR_INVALID_ARG
    # group sum: capacity keep_k + W = 288
    assert st(K.SnapOptions(mode=0, seed_out=16, seed_layer_stride=4 * 287,
                            seed_head_stride=287)) == K.KVSEL_ERR_INVALID_ARG
    need = K.kvsel_snapkv_select_ex_workspace(kv, 2, 4096, 32, False, K.KVSEL_SNAP_HEAD_UNION)
    assert st(K.SnapOptions(mode=1), ws_bytes=need - 1) == K.KVSEL_ERR_INVALID_ARG
    # the union keeps per-q-head votes and picks: more workspace than the group sum
    assert need > K.kvsel_snapkv_select_ex_workspace(kv, 2, 4096, 32, False, K.KVSEL_SNAP_GROUP_SUM)
    assert need >= 2 * 2 * 32 * (4096 - 32) * 4        # per-head votes and picks
    assert K.kvsel_snapkv_select_ex_workspace(kv, 2, 4096, 32, False, 5) == 0
    assert (K.kvsel_snapkv_select_workspace(kv, 2, 4096, 32, True) ==
            K.kvsel_snapkv_select_ex_workspace(kv, 2, 4096, 32, True, K.KVSEL_SNAP_GROUP_SUM))


def test_decode_block_signal_host_validation(lib):
    kv = _kv()
    need = K.kvsel_decode_attn_ex_workspace(kv, 1, 64, True, True)
    assert need > K.kvsel_decode_attn_workspace(kv, 1, 64, True)
    assert K.kvsel_decode_attn_ex_workspace(kv, 1, 64, True, False) == K.kvsel_decode_attn_workspace(kv, 1, 64,
                                                                                                      True)

    def st(sig, ws_bytes=1 << 30):
        return lib.kvsel_decode_attn_ex(ctypes.byref(kv), 16, 4, 16, 1, 16, None, None, None, None, 0.1, 16, 0,
                                        16, None, 64, 0, ctypes.byref(sig) if sig is not None else None, 256,
                                        ws_bytes, None, 0, None)
    assert st(K.BlockSignal(topk_blocks=0, step=1, block_score=16, block_step=16)) == K.KVSEL_ERR_INVALID_ARG
    assert b"block signal" in lib.kvsel_last_error_string()
    assert st(K.BlockSignal(topk_blocks=8, step=1, block_score=None, block_step=16)) == K.KVSEL_ERR_INVALID_ARG
    # the signal's scratch comes on top of the plain decode's workspace
    base = K.kvsel_decode_attn_workspace(kv, 1, 64, True)
    assert st(K.BlockSignal(topk_blocks=8, step=1, block_score=16, block_step=16),
              ws_bytes=base) == K.KVSEL_ERR_INVALID_ARG
    assert b"workspace too small" in lib.kvsel_last_error_string()


def test_quest_host_validation(lib):
    kv = _kv(num_pages=64)

    def st(kv_=kv, **over):
        a = dict(bt=16, max_pages=64, seq=16, B=2, q=16, kn=None, vn=None, meta=16, budget=8, scale=0.1, out=16,
                 odt=0, pages=None, bounds=None, ws=256, ws_bytes=1 << 30)
        a.update(over)
        return lib.kvsel_quest_decode(ctypes.byref(kv_), a["bt"], a["max_pages"], a["seq"], a["B"], a["q"], a["kn"],
                                      a["vn"], a["meta"], a["budget"], a["scale"], a["out"], a["odt"], a["pages"],
                                      a["bounds"], a["ws"], a["ws_bytes"], None)
    assert st(kv_=_kv(num_q_heads=136, num_pages=64)) == K.KVSEL_ERR_UNSUPPORTED   # G = 17
    assert st(kv_=_kv(page_size=512, num_pages=64)) == K.KVSEL_ERR_UNSUPPORTED
    assert st(kv_=_kv(page_size=48, num_pages=64)) == K.KVSEL_ERR_UNSUPPORTED
    assert lib.kvsel_quest_page_meta(ctypes.byref(_kv(page_size=512)), 16, 64, 16, 2, 16, 256,
                                     None) == K.KVSEL_ERR_UNSUPPORTED
    # 256-token pool pages hold 16 Quest pages each: per-page buffers grow 16-fold with max_pages fixed
    w16 = K.kvsel_quest_decode_workspace(kv, 2, 64, 8, True, True)
    w256 = K.kvsel_quest_decode_workspace(_kv(page_size=256, num_pages=64), 2, 64, 8, True, True)
    assert w256 - w16 >= 15 * 4 * (2 * 8 * 64 * 4)
    assert K.kvsel_quest_decode_workspace(_kv(page_size=48, num_pages=64), 2, 64, 8) == 0
    assert st(kn=16) == K.KVSEL_ERR_INVALID_ARG                                   # k_new without v_new
    assert st(budget=0) == K.KVSEL_ERR_INVALID_ARG
    assert st(meta=None) == K.KVSEL_ERR_INVALID_ARG
    assert st(meta=8) == K.KVSEL_ERR_INVALID_ARG                                  # misaligned
    assert st(odt=5) == K.KVSEL_ERR_INVALID_ARG
    need = K.kvsel_quest_decode_workspace(kv, 2, 64, 8)
    assert st(ws_bytes=need - 1) == K.KVSEL_ERR_INVALID_ARG
    # taking the bounds and pages out of the workspace shrinks it by their size
    assert need - K.kvsel_quest_decode_workspace(kv, 2, 64, 8, True, True) >= 2 * 64 * 64 * 4 + 2 * 64 * 8 * 4
    assert lib.kvsel_quest_page_meta(ctypes.byref(kv), 16, 64, 16, 2, None, 256, None) == K.KVSEL_ERR_INVALID_ARG


def test_link_reset_host_validation(lib):
    # every check happens on the host, before anything is enqueued
    assert lib.kvsel_h2o_link_reset(None, 2, 8, None) == K.KVSEL_ERR_INVALID_ARG
    assert lib.kvsel_h2o_link_reset(256 + 16, 2, 8, None) == K.KVSEL_ERR_INVALID_ARG    # misaligned
    assert b"256-byte aligned" in lib.kvsel_last_error_string()
    assert lib.kvsel_h2o_link_reset(256, 0, 8, None) == K.KVSEL_ERR_INVALID_ARG
    assert lib.kvsel_h2o_link_reset(256, 2, 0, None) == K.KVSEL_ERR_INVALID_ARG


def test_wait_limit_host_validation(lib):
    assert lib.kvsel_set_wait_limit(None, 100, None) == K.KVSEL_ERR_INVALID_ARG
    assert lib.kvsel_set_wait_limit(16, 100, None) == K.KVSEL_ERR_INVALID_ARG     # misaligned workspace
    assert b"aligned" in lib.kvsel_last_error_string()


def test_kv_compact_host_validation(lib):
    def st(kv_=None, **over):
        a = dict(bt=16, max_pages=64, seq=16, B=2, keep=16, stride=100, count=None, scores=None, pos=None,
                 max_len=0, freed=None, ws=256, ws_bytes=1 << 20)
        a.update(over)
        return lib.kvsel_kv_compact(ctypes.byref(kv_ or _kv()), a["bt"], a["max_pages"], a["seq"], a["B"],
                                    a["keep"], a["stride"], a["count"], a["scores"], a["pos"], a["max_len"],
                                    a["freed"], a["ws"], a["ws_bytes"], None)
    assert st(kv_=_kv(v_pool=None)) == K.KVSEL_ERR_INVALID_ARG
    assert st(kv_=_kv(k_pool=8)) == K.KVSEL_ERR_INVALID_ARG          # misaligned pool
    assert st(kv_=_kv(page_size=512)) == K.KVSEL_ERR_UNSUPPORTED
    assert st(kv_=_kv(page_size=48)) == K.KVSEL_ERR_UNSUPPORTED
    assert st(keep=None) == K.KVSEL_ERR_INVALID_ARG
    assert st(stride=0) == K.KVSEL_ERR_INVALID_ARG
    assert st(scores=16) == K.KVSEL_ERR_INVALID_ARG                  # scores without max_len
    assert st(ws=128) == K.KVSEL_ERR_INVALID_ARG                     # misaligned workspace
    need = K.kvsel_kv_compact_workspace(2, 8)
    assert need >= 256 + 2 * 4 + 2 * 8 * 4
    assert st(ws_bytes=need - 1) == K.KVSEL_ERR_INVALID_ARG
    assert b"workspace too small" in lib.kvsel_last_error_string()
    assert K.kvsel_kv_compact_workspace(0, 8) == 0


def test_header_compiles_as_plain_c(tmp_path):
    # the boundary is a C ABI: the header must stand alone in C99 (every struct and enum named)
    import shutil
    import subprocess
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    src = tmp_path / "use.c"
    src.write_text('#include "kvsel.h"\n'
                   'int main(void) {\n'
                   '  kvsel_block_signal s; kvsel_snap_options o; kvsel_bp_options b; kvsel_paged_kv kv;\n'
                   '  (void)s; (void)o; (void)b; (void)kv;\n'
                   '  return (int)KVSEL_SNAP_HEAD_UNION + (int)KVSEL_UPDATE_WINDOW;\n'
                   '}\n')
    r = subprocess.run([cc, "-std=c99", "-Wall", "-Werror", "-pedantic", "-I", os.path.join(ROOT, "include"),
                        "-c", str(src), "-o", str(tmp_path / "use.o")], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
