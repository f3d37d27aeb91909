"""CPU oracle for sparse-attention token selection (TEST INFRASTRUCTURE).

A thin ctypes wrapper around ``sel_oracle.c``, the plain C definition of the
selection path (scoring, top-k pools, expansion with the trailing incomplete pool,
block-table remap, valid counts). Only the tests, ``__graft_entry__.smoke()`` and
the CPU-baseline leg of ``bench.py`` may use it; the library never imports it, and
it imports nothing from the library. Inputs are numpy arrays (or any object
carrying the workload fields as attributes); nothing here moves data to a GPU.
"""

from __future__ import annotations

import ctypes as C
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "sel_oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_SO = os.path.join(_OUT_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None

ST_KEYPAGE_OOB = 1
ST_CTX_OVER_BOUND = 2
ST_BAD_QSL = 8


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (no fast-math, no FMA contraction)."""
    if not force and os.path.exists(_SO) and os.path.getmtime(_SO) >= os.path.getmtime(_SRC):
        return _SO
    os.makedirs(_OUT_DIR, exist_ok=True)
    tmp = _SO + f".tmp{os.getpid()}"
    subprocess.run(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math",
                    "-fPIC", "-shared", "-pthread", _SRC, "-o", tmp, "-lm"], check=True)
    os.replace(tmp, _SO)
    return _SO


class _Problem(C.Structure):
    _fields_ = [
        ("num_reqs", C.c_int32), ("num_rows", C.c_int32),
        ("qsl", C.c_void_p), ("positions", C.c_void_p),
        ("q", C.c_void_p), ("q_row_stride", C.c_int64),
        ("key_cache", C.c_void_p), ("key_page_stride", C.c_int64),
        ("num_key_pages", C.c_int32),
        ("key_page_table", C.c_void_p), ("kpt_ld", C.c_int64),
        ("max_key_pages_per_req", C.c_int32),
        ("block_table", C.c_void_p), ("bt_ld", C.c_int64),
        ("max_blocks_per_req", C.c_int32), ("num_kv_blocks", C.c_int32),
        ("block_size", C.c_int32), ("block_stride_rows", C.c_int64),
        ("heads", C.c_int32), ("dim", C.c_int32), ("key_page_size", C.c_int32),
        ("index_topk", C.c_int32), ("kpool", C.c_int32), ("out_width", C.c_int32),
        ("max_context", C.c_int64),
    ]


def _load(path: str):
    L = C.CDLL(path)
    P, I32, I64 = C.c_void_p, C.c_int32, C.c_int64
    L.orc_half_to_float_array.argtypes = [P, P, I64]
    L.orc_pool_score.argtypes = [P, P, C.c_int, C.c_int, P]
    L.orc_pool_score.restype = C.c_float
    L.orc_topk_pools.argtypes = [P, I32, I32, P]
    L.orc_topk_pools.restype = C.c_int
    L.orc_expand.argtypes = [I64, I32, I32, P, I32, I32, P]
    L.orc_expand.restype = C.c_int
    L.orc_remap_token.argtypes = [I32, P, I32, I32, I32, I64]
    L.orc_remap_token.restype = I64
    L.orc_remap_rows.argtypes = [P, I32, P, I64, I32, I32, P, I32, I32, I32, I64, P, P]
    L.orc_remap_ws_rows.argtypes = [P, I32, P, I64, I32, I32, P, P, I32, P, I32, I32, I32, I64, P, P]
    L.orc_dcp_local_index.argtypes = [I32, I32, I32, I32]
    L.orc_dcp_local_index.restype = I64
    L.orc_remap_dcp_rows.argtypes = [P, I32, P, I64, I32, I32, P, I32, I32, I32, I32, I32, I32, I32, P, P]
    L.orc_maxsim.argtypes = [P, I32, I32, P, I64, I64, P, P, I32, P, P]
    L.orc_bf16_to_double.argtypes = [C.c_uint16]
    L.orc_bf16_to_double.restype = C.c_double
    L.orc_mla_decode.argtypes = [P, P, I32, I32, I32, I32, P, I64, P, I64, I64, P, I32, P, C.c_double, P, P]
    L.orc_select.argtypes = [C.POINTER(_Problem), P, I32, I32, P, P, P, P, P, I64]
    L.orc_select.restype = I32
    L.orc_score_rows.argtypes = [C.POINTER(_Problem), P, I32, P, P, I64]
    L.orc_score_rows.restype = I32
    L.orc_topk_expand_rows.argtypes = [P, I64, P, I32, I32, I32, I32, P, P]
    L.orc_topk_expand_rows.restype = I32
    return L


def lib():
    global _lib
    with _lock:
        if _lib is None:
            _lib = _load(build())
        return _lib


def _p(a: np.ndarray):
    return a.ctypes.data_as(C.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def half_to_float(bits: np.ndarray) -> np.ndarray:
    """fp16 bit patterns (uint16) -> float32, decoded from the binary16 definition."""
    b = _c(bits, np.uint16).ravel()
    out = np.empty(b.shape, dtype=np.float32)
    lib().orc_half_to_float_array(_p(b), _p(out), b.size)
    return out.reshape(np.shape(bits))


def pool_score(q_row: np.ndarray, key: np.ndarray) -> tuple[float, float]:
    """(fp32 score, fp64 sum |q*k|) of one pool key [D] against one query row [H, D]."""
    qb = _c(q_row, np.float16).view(np.uint16)
    kb = _c(key, np.float16).view(np.uint16)
    a = C.c_double(0.0)
    s = lib().orc_pool_score(_p(qb), _p(kb), qb.shape[0], qb.shape[1], C.byref(a))
    return float(np.float32(s)), a.value


def topk_pools(scores: np.ndarray, K: int) -> np.ndarray:
    """The K best pools (score desc, index asc), in ascending index order."""
    s = _c(scores, np.float32)
    out = np.empty(max(K, 1), dtype=np.int32)
    n = lib().orc_topk_pools(_p(s), s.size, K, _p(out))
    if n < 0:
        raise MemoryError("oracle top-k allocation failed")
    return out[:n].copy()


def expand(ctx: int, topk: int, kpool: int, pools: np.ndarray, W: int) -> tuple[np.ndarray, int]:
    """Tokens of the kept pools plus the trailing incomplete pool, -1 padded to W."""
    pl = _c(pools, np.int32)
    out = np.empty(W, dtype=np.int32)
    n = lib().orc_expand(int(ctx), topk, kpool, _p(pl), pl.size, W, _p(out))
    if n < 0:
        raise ValueError("tokens do not fit in the output width")
    return out, n


def remap_token(t: int, bt_row: np.ndarray, max_blocks: int, num_kv_blocks: int,
                block_size: int, block_stride_rows: int) -> int:
    b = _c(bt_row, np.int32)
    return int(lib().orc_remap_token(int(t), _p(b), max_blocks, num_kv_blocks, block_size,
                                     int(block_stride_rows)))


def remap_rows(req_id, num_reqs, block_table, max_blocks, num_kv_blocks, token_idx,
               block_size, block_stride_rows):
    """Remap whole rows; returns (slots int64 [rows, width], counts int32 [rows])."""
    rq = _c(req_id, np.int32)
    bt = _c(block_table, np.int32)
    ti = _c(token_idx, np.int32)
    rows, width = ti.shape
    slots = np.empty((rows, width), dtype=np.int64)
    counts = np.empty(rows, dtype=np.int32)
    lib().orc_remap_rows(_p(rq), num_reqs, _p(bt), bt.shape[1], max_blocks, num_kv_blocks,
                         _p(ti), rows, width, block_size, int(block_stride_rows),
                         _p(slots), _p(counts))
    return slots, counts


def remap_ws_rows(req_id, num_reqs, block_table, max_blocks, num_kv_blocks, ws_req, ws_starts,
                  token_idx, block_size, block_stride_rows):
    """Remap with a prefill workspace: rows with ws_req >= 0 map t to ws_starts[ws_req] + t;
    returns (slots int64 [rows, width], counts int32 [rows])."""
    rq, bt, wr, ws, ti = (_c(req_id, np.int32), _c(block_table, np.int32), _c(ws_req, np.int32),
                          _c(ws_starts, np.int32), _c(token_idx, np.int32))
    rows, width = ti.shape
    slots = np.empty((rows, width), dtype=np.int64)
    counts = np.empty(rows, dtype=np.int32)
    lib().orc_remap_ws_rows(_p(rq), num_reqs, _p(bt), bt.shape[1], max_blocks, num_kv_blocks, _p(wr),
                            _p(ws), ws.size, _p(ti), rows, width, block_size, int(block_stride_rows),
                            _p(slots), _p(counts))
    return slots, counts


def dcp_local_index(t: int, dcp_size: int, dcp_rank: int, interleave: int) -> int:
    """Local index of token t on rank dcp_rank, or -1 when another rank owns it."""
    return int(lib().orc_dcp_local_index(int(t), dcp_size, dcp_rank, interleave))


def remap_dcp_rows(req_id, num_reqs, block_table, max_blocks, num_kv_blocks, token_idx, block_size,
                   dcp_size, dcp_rank, interleave, compact):
    """One decode-context-parallel rank's slots; returns (slots int64, counts int32)."""
    rq, bt, ti = _c(req_id, np.int32), _c(block_table, np.int32), _c(token_idx, np.int32)
    rows, width = ti.shape
    slots = np.empty((rows, width), dtype=np.int64)
    counts = np.empty(rows, dtype=np.int32)
    lib().orc_remap_dcp_rows(_p(rq), num_reqs, _p(bt), bt.shape[1], max_blocks, num_kv_blocks, _p(ti),
                             rows, width, block_size, dcp_size, dcp_rank, interleave, int(bool(compact)),
                             _p(slots), _p(counts))
    return slots, counts


def maxsim(q, docs, offsets, lengths):
    """MaxSim scores of query q [lq, d] (fp16) against the documents (offsets[i], lengths[i])
    of the packed fp16 tensor docs [total_tokens, >= d] (vLLM page "flash_maxsim_rerank",
    _maxsim_rerank_kernel). Returns (scores float32 [B], abs_bound float64 [B])."""
    qb = _c(q, np.float16).view(np.uint16)
    db = _c(docs, np.float16).view(np.uint16)
    of, ln = _c(offsets, np.int32), _c(lengths, np.int32)
    lq, d = qb.shape
    scores = np.empty(of.size, dtype=np.float32)
    bound = np.empty(of.size, dtype=np.float64)
    lib().orc_maxsim(_p(qb), lq, d, _p(db), db.shape[1], db.shape[0], _p(of), _p(ln), of.size, _p(scores), _p(bound))
    return scores, bound


def bf16_to_double(bits) -> np.ndarray:
    """bfloat16 bit patterns (uint16) -> float64, decoded by the oracle's C routine."""
    b = _c(bits, np.uint16).ravel()
    return np.array([lib().orc_bf16_to_double(int(x)) for x in b], dtype=np.float64).reshape(np.shape(bits))


def mla_decode(q_nope, q_pe, ckv, kpe, slots, kv_len, sm_scale):
    """Sparse MLA decode attention over selected slots (vLLM page "flashinfer_mla_sparse_sm90",
    _SM90State). bf16 inputs as uint16 bit patterns: q_nope [rows, heads, dc], q_pe
    [rows, heads, dr] (dr may be 0), ckv [num_slots, >= dc], kpe [num_slots, >= dr],
    slots int32 [rows, width], kv_len int32 [rows]. Returns (out float64 [rows, heads, dc],
    lse float64 [rows, heads])."""
    qn = _c(q_nope, np.uint16)
    qp = _c(q_pe, np.uint16)
    ck = _c(ckv, np.uint16)
    kp = _c(kpe, np.uint16)
    sl = _c(slots, np.int32)
    kl = _c(kv_len, np.int32)
    rows, heads, dc = qn.shape
    dr = qp.shape[2]
    out = np.empty((rows, heads, dc), dtype=np.float64)
    lse = np.empty((rows, heads), dtype=np.float64)
    lib().orc_mla_decode(_p(qn), _p(qp), rows, heads, dc, dr, _p(ck), ck.shape[1], _p(kp),
                         kp.shape[1] if kp.ndim == 2 else 0, ck.shape[0], _p(sl), sl.shape[1], _p(kl),
                         float(sm_scale), _p(out), _p(lse))
    return out, lse


class _Held:
    """Keeps the contiguous arrays a _Problem points into alive."""

    def __init__(self, w):
        self.qsl = _c(w.qsl, np.int32)
        self.positions = _c(w.positions, np.int32)
        self.q = _c(w.q, np.float16).view(np.uint16)
        self.key_cache = _c(w.key_cache, np.float16).view(np.uint16)
        self.kpt = _c(w.key_page_table, np.int32)
        self.bt = _c(w.block_table, np.int32)
        pr = _Problem()
        pr.num_reqs, pr.num_rows = int(w.num_reqs), int(w.num_rows)
        pr.qsl, pr.positions = _p(self.qsl), _p(self.positions)
        pr.q = _p(self.q)
        pr.q_row_stride = int(self.q.shape[1] * self.q.shape[2])
        pr.key_cache, pr.key_page_stride = _p(self.key_cache), int(w.key_page_stride)
        pr.num_key_pages = int(w.num_key_pages)
        pr.key_page_table, pr.kpt_ld = _p(self.kpt), int(self.kpt.shape[1])
        pr.max_key_pages_per_req = int(w.max_key_pages_per_req)
        pr.block_table, pr.bt_ld = _p(self.bt), int(self.bt.shape[1])
        pr.max_blocks_per_req = int(w.max_blocks_per_req)
        pr.num_kv_blocks = int(w.num_kv_blocks)
        pr.block_size = int(w.block_size)
        pr.block_stride_rows = int(w.block_stride_rows)
        pr.heads, pr.dim = int(self.q.shape[1]), int(self.q.shape[2])
        pr.key_page_size = 64
        pr.index_topk, pr.kpool = int(w.index_topk), int(w.kpool)
        pr.out_width = int(w.out_width)
        pr.max_context = int(w.max_context)
        if pr.kpool <= 0 or pr.index_topk % pr.kpool:
            raise ValueError("index_topk must be a positive multiple of kpool")
        self.problem = pr


def select(w, rows=None, nthreads: int | None = None, want_scores: bool = False,
           scores_ld: int | None = None) -> dict:
    """The whole selection for ``rows`` (default: every row) of workload ``w``.

    Returns dict(rows, slots int64 [n, W], counts int32 [n], token_idx int32 [n, W],
    status int, and with ``want_scores`` scores float32 [n, scores_ld] and
    abs_terms float64 [n, scores_ld], filled for j < ctx/kpool of rows with
    ctx > index_topk).
    """
    h = _Held(w)
    rows = np.arange(w.num_rows, dtype=np.int32) if rows is None else _c(rows, np.int32)
    n, W = rows.size, int(w.out_width)
    slots = np.empty((n, W), dtype=np.int64)
    counts = np.empty(n, dtype=np.int32)
    tok = np.empty((n, W), dtype=np.int32)
    sc = ab = None
    ld = 0
    if want_scores:
        ld = int(scores_ld if scores_ld is not None else max(1, int(w.max_context) // int(w.kpool)))
        sc = np.full((n, ld), np.nan, dtype=np.float32)
        ab = np.zeros((n, ld), dtype=np.float64)
    nt = nthreads if nthreads is not None else (os.cpu_count() or 1)
    st = lib().orc_select(C.byref(h.problem), _p(rows), n, nt, _p(slots), _p(counts), _p(tok),
                          _p(sc) if sc is not None else None,
                          _p(ab) if ab is not None else None, ld)
    if st < 0:
        raise ValueError("oracle: output width too small for the selected tokens")
    out = dict(rows=rows, slots=slots, counts=counts, token_idx=tok, status=int(st))
    if want_scores:
        out["scores"], out["abs_terms"] = sc, ab
    return out


def score_rows(w, rows=None, scores_ld: int | None = None):
    """Scores of every complete pool of each listed row: (scores, abs_terms, status)."""
    h = _Held(w)
    rows = np.arange(w.num_rows, dtype=np.int32) if rows is None else _c(rows, np.int32)
    ld = int(scores_ld if scores_ld is not None else max(1, int(w.max_context) // int(w.kpool)))
    sc = np.full((rows.size, ld), np.nan, dtype=np.float32)
    ab = np.zeros((rows.size, ld), dtype=np.float64)
    st = lib().orc_score_rows(C.byref(h.problem), _p(rows), rows.size, _p(sc), _p(ab), ld)
    return sc, ab, int(st)


def topk_expand_rows(scores: np.ndarray, ctx: np.ndarray, topk: int, kpool: int, W: int):
    """Top-k + expansion on given score rows: (token_idx int32 [n, W], counts int32 [n])."""
    s = _c(scores, np.float32)
    cx = _c(ctx, np.int64)
    n = cx.size
    tok = np.empty((n, W), dtype=np.int32)
    cnt = np.empty(n, dtype=np.int32)
    if lib().orc_topk_expand_rows(_p(s), s.shape[1], _p(cx), n, topk, kpool, W, _p(tok), _p(cnt)) < 0:
        raise ValueError("oracle: output width too small")
    return tok, cnt


def build_variant(replacements, tag: str) -> str:
    """Compile a copy of the oracle source with textual replacements applied.

    Used only by the tests that plant a mistake in the oracle and check that the
    pins catch it. Each ``(old, new)`` pair must occur in the source.
    """
    with open(_SRC) as f:
        src = f.read()
    for old, new in replacements:
        if old not in src:
            raise ValueError(f"mutation target not found: {old!r}")
        src = src.replace(old, new)
    os.makedirs(_OUT_DIR, exist_ok=True)
    c_path = os.path.join(_OUT_DIR, f"variant_{tag}.c")
    so_path = os.path.join(_OUT_DIR, f"variant_{tag}.so")
    with open(c_path, "w") as f:
        f.write(src)
    subprocess.run(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared",
                    "-pthread", c_path, "-o", so_path, "-lm"], check=True)
    return so_path


class using_library:
    """Context manager: route every oracle call through another build of the source."""

    def __init__(self, so_path: str):
        self.path = so_path
        self.saved = None

    def __enter__(self):
        global _lib
        with _lock:
            self.saved = _lib
            _lib = _load(self.path)
        return self

    def __exit__(self, *exc):
        global _lib
        with _lock:
            _lib = self.saved
        return False
