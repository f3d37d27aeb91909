"""The C-ABI library loads, exports every entry point of include/sel.h, and rejects
bad arguments on the host before touching a GPU (no GPU needed)."""

import ctypes as C
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _header_functions():
    src = open(os.path.join(ROOT, "include", "sel.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(sel_[a-z_]+)\s*\(", src)))


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__
    path = __graft_entry__._builder().build()
    return C.CDLL(path)


def test_header_declares_the_boundary():
    names = _header_functions()
    for n in ("sel_score_paged", "sel_topk_expand", "sel_remap_global", "sel_select",
              "sel_workspace_bytes", "sel_error_string"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    missing = [n for n in _header_functions() if not hasattr(lib, n)]
    assert not missing, missing


def test_package_binding_has_the_same_names():
    import sparse_attention_kv_device_gb300 as pkg
    from sparse_attention_kv_device_gb300 import sel
    for n in _header_functions():
        assert n in sel.EXPORTS and hasattr(pkg, n), n


def test_error_strings(lib):
    lib.sel_error_string.restype = C.c_char_p
    for code in (0, -1, -2, -3, -4, -99):
        assert lib.sel_error_string(code)
    assert lib.sel_version() == 102


def test_wait_limit_hook_validates_and_restores(lib):
    f = lib.sel_debug_wait_limit
    f.argtypes = [C.c_int32, C.c_int64]
    assert f(-2, 10**9) == -1        # no such tile
    assert f(3, 10) == -1            # a limit below a microsecond is refused
    assert f(5, 10**6) == 0
    assert f(-1, 10**9) == 0         # normal operation again


def _problem(**kw):
    from sparse_attention_kv_device_gb300.sel import sel_problem
    p = sel_problem()
    p.num_reqs, p.num_rows, p.max_context = 1, 1, 4096
    p.num_heads, p.head_dim, p.key_page_size = 4, 128, 64
    p.index_topk, p.kpool, p.block_size, p.block_stride_rows = 2048, 4, 64, 64
    p.key_page_stride, p.num_key_pages, p.num_kv_blocks = 64 * 128, 16, 64
    p.max_key_pages_per_req, p.max_blocks_per_req, p.kpt_ld, p.bt_ld = 16, 64, 16, 64
    p.q_row_stride = 512
    fake = 0x10000  # never dereferenced: every case below fails validation first
    p.query_start_loc = p.positions = p.q = p.key_cache = p.key_page_table = p.block_table = fake
    for k, v in kw.items():
        setattr(p, k, v)
    return p


@pytest.mark.parametrize("field,value,code", [
    ("num_heads", 8, -2), ("head_dim", 64, -2), ("key_page_size", 32, -2),
    ("kpool", 0, -1), ("index_topk", 2047, -1), ("block_stride_rows", 32, -1),
    ("key_page_stride", 100, -1), ("q_row_stride", 256, -1), ("q_row_stride", 516, -2),
    ("num_rows", -1, -1), ("max_key_pages_per_req", 17, -1), ("max_blocks_per_req", 65, -1),
    ("segment_rows", 65, -1), ("max_context", 70000, -1), ("num_kv_blocks", 1 << 30, -1),
    ("q", 0, -1), ("q", 0x10008, -2),
])
def test_select_rejects_bad_problem(lib, field, value, code):
    lib.sel_select.argtypes = [C.c_void_p, C.c_void_p, C.c_int32, C.c_void_p, C.c_void_p, C.c_void_p,
                               C.c_void_p, C.c_size_t, C.c_void_p]
    lib.sel_workspace_bytes.restype = C.c_size_t
    p = _problem(**{field: value})
    assert lib.sel_select(C.byref(p), C.c_void_p(0x20000), 2052, None, None, None, C.c_void_p(0x30000),
                          1 << 30, None) == code
    assert lib.sel_workspace_bytes(C.byref(p)) == 0


def test_remap_rejects_bad_arguments(lib):
    f = lib.sel_remap_global
    f.argtypes = [C.c_void_p, C.c_int32, C.c_void_p, C.c_int64, C.c_int32, C.c_int32, C.c_void_p,
                  C.c_int32, C.c_int32, C.c_int32, C.c_int64, C.c_void_p, C.c_void_p, C.c_void_p]
    good = dict(req=0x1000, nreq=1, bt=0x2000, ld=8, mb=8, nkv=8, tok=0x3000, rows=2, width=8, bs=64,
                stride=64, slots=0x4000)

    def call(**kw):
        a = dict(good, **kw)
        return f(a["req"], a["nreq"], a["bt"], a["ld"], a["mb"], a["nkv"], a["tok"], a["rows"], a["width"],
                 a["bs"], a["stride"], a["slots"], None, None)

    assert call(width=6) == -1                 # not a multiple of 4
    assert call(stride=32) == -1               # stride below the block size
    assert call(mb=9) == -1                    # more valid columns than the row holds
    assert call(tok=0x3004) == -2              # not 16-byte aligned
    assert call(slots=None) == -1
    assert call(nkv=1 << 26) == -1             # slots would overflow int32
    assert call(rows=0, tok=None, slots=None) == 0   # empty batch: nothing to do


def test_workspace_remap_rejects_bad_arguments(lib):
    f = lib.sel_remap_workspace
    f.argtypes = [C.c_void_p, C.c_int32, C.c_void_p, C.c_int64, C.c_int32, C.c_int32, C.c_void_p, C.c_void_p,
                  C.c_int32, C.c_void_p, C.c_int32, C.c_int32, C.c_int32, C.c_int64, C.c_void_p, C.c_void_p,
                  C.c_void_p]
    good = dict(req=0x1000, nreq=1, bt=0x2000, ld=8, mb=8, nkv=8, wsr=0x5000, wss=0x6000, npf=2, tok=0x3000,
                rows=2, width=8, bs=64, stride=64, slots=0x4000)

    def call(**kw):
        a = dict(good, **kw)
        return f(a["req"], a["nreq"], a["bt"], a["ld"], a["mb"], a["nkv"], a["wsr"], a["wss"], a["npf"], a["tok"],
                 a["rows"], a["width"], a["bs"], a["stride"], a["slots"], None, None)

    assert call(wsr=None) == -1                # no workspace request ids
    assert call(wss=None) == -1                # prefill requests without starts
    assert call(npf=-1) == -1
    assert call(width=6) == -1
    assert call(tok=0x3004) == -2
    assert call(rows=0, tok=None, slots=None, wsr=None) == 0


def test_dcp_remap_rejects_bad_arguments(lib):
    f = lib.sel_remap_dcp
    f.argtypes = [C.c_void_p, C.c_int32, C.c_void_p, C.c_int64, C.c_int32, C.c_int32, C.c_void_p, C.c_int32,
                  C.c_int32, C.c_int32, C.c_int32, C.c_int32, C.c_int32, C.c_int32, C.c_void_p, C.c_void_p,
                  C.c_void_p]
    good = dict(req=0x1000, nreq=1, bt=0x2000, ld=8, mb=8, nkv=8, tok=0x3000, rows=2, width=8, bs=64, size=2,
                rank=1, inter=4, compact=1, slots=0x4000)

    def call(**kw):
        a = dict(good, **kw)
        return f(a["req"], a["nreq"], a["bt"], a["ld"], a["mb"], a["nkv"], a["tok"], a["rows"], a["width"], a["bs"],
                 a["size"], a["rank"], a["inter"], a["compact"], a["slots"], None, None)

    assert call(size=0) == -1
    assert call(rank=2) == -1                  # rank outside [0, dcp_size)
    assert call(rank=-1) == -1
    assert call(inter=0) == -1
    assert call(inter=48) == -1                # an interleave group would straddle a block
    assert call(width=6) == -1
    assert call(slots=0x4004) == -2
    assert call(rows=0, tok=None, slots=None) == 0


def test_topk_rejects_bad_arguments(lib):
    f = lib.sel_topk_expand
    f.argtypes = [C.c_void_p, C.c_int64, C.c_void_p, C.c_int32, C.c_int32, C.c_int32, C.c_void_p,
                  C.c_int32, C.c_void_p, C.c_void_p, C.c_void_p]
    assert f(0x1000, 512, 0x2000, 4, 2048, 4, 0x3000, 2048, None, None, None) == -1   # width < topk+kpool-1
    assert f(0x1000, 512, 0x2000, 4, 2048, 3, 0x3000, 2052, None, None, None) == -1   # kpool does not divide
    assert f(0x1000, 514, 0x2000, 4, 2048, 4, 0x3000, 2052, None, None, None) == -1   # ld not a multiple of 4
    assert f(0x1004, 512, 0x2000, 4, 2048, 4, 0x3000, 2052, None, None, None) == -2   # misaligned scores
    assert f(None, 512, None, 0, 2048, 4, None, 2052, None, None, None) == 0          # empty batch


def test_maxsim_rejects_bad_arguments(lib):
    f = lib.sel_maxsim_rerank
    f.argtypes = [C.c_void_p, C.c_int32, C.c_int32, C.c_int64, C.c_void_p, C.c_int64, C.c_int64, C.c_void_p,
                  C.c_void_p, C.c_int32, C.c_void_p, C.c_void_p, C.c_void_p, C.c_size_t, C.c_void_p]
    lib.sel_maxsim_workspace_bytes.restype = C.c_size_t
    wsb = lib.sel_maxsim_workspace_bytes()
    good = dict(q=0x1000, lq=32, d=128, qs=128, docs=0x2000, tot=1000, ds=128, off=0x3000, ln=0x4000, nd=10,
                sc=0x5000, ws=0x6000, wsb=wsb)

    def call(**kw):
        a = dict(good, **kw)
        return f(a["q"], a["lq"], a["d"], a["qs"], a["docs"], a["tot"], a["ds"], a["off"], a["ln"], a["nd"],
                 a["sc"], None, a["ws"], a["wsb"], None)

    assert call(lq=-1) == -1
    assert call(d=0) == -1
    assert call(nd=-1) == -1
    assert call(nd=0, q=None, docs=None, off=None, ln=None, sc=None) == 0   # empty batch: nothing queued
    assert call(sc=None) == -1
    assert call(docs=None) == -1
    assert call(ws=None) == -1
    assert call(qs=64) == -1                  # row stride below d
    assert call(tot=0) == -1
    assert call(d=2048, qs=2048, ds=2048) == -2
    assert call(qs=132) == -2                 # row stride not a multiple of 8
    assert call(docs=0x2008) == -2            # misaligned
    assert call(tot=1 << 31) == -2
    assert call(wsb=wsb - 1) == -4
    lib.sel_maxsim_launch_count.restype = C.c_int32
    assert lib.sel_maxsim_launch_count(32, 128) == 1
    assert lib.sel_maxsim_launch_count(300, 128) == 3
    assert lib.sel_maxsim_launch_count(128, 256) == 1
    assert lib.sel_maxsim_launch_count(128, 512) == 2
    assert lib.sel_maxsim_launch_count(32, 1024) == 1
    assert lib.sel_maxsim_launch_count(0, 128) == 1
