"""Python binding of libsel (include/sel.h): argument marshalling only.

Every function here has the name of a C entry point, checks that the tensors it is
given are on the right device with the right dtype and layout, turns them into raw
pointers and calls the library. All computation happens in the library's CUDA
kernels; there is no fallback of any kind: if libsel.so is missing or fails to load,
importing this module raises.
"""

from __future__ import annotations

import ctypes as C
import os

import torch

from . import build as _build

# SEL_LIBRARY selects another build of the same library (e.g. a diagnostics build)
_LIB_PATH = os.environ.get("SEL_LIBRARY", _build.LIB)

SEL_OK = 0
SEL_EINVAL = -1
SEL_EUNSUPPORTED = -2
SEL_ECUDA = -3
SEL_EWORKSPACE = -4

ST_KEYPAGE_OOB = 1
ST_CTX_OVER_BOUND = 2
ST_TIMEOUT = 4
ST_BAD_QSL = 8


class SelError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {sel_error_string(code)} (code {code})")


class sel_problem(C.Structure):
    _fields_ = [
        ("num_reqs", C.c_int32), ("num_rows", C.c_int32), ("max_context", C.c_int32),
        ("max_q_len", C.c_int32), ("num_heads", C.c_int32), ("head_dim", C.c_int32),
        ("index_topk", C.c_int32), ("kpool", C.c_int32), ("key_page_size", C.c_int32),
        ("block_size", C.c_int32), ("block_stride_rows", C.c_int64),
        ("key_page_stride", C.c_int64), ("num_key_pages", C.c_int32),
        ("num_kv_blocks", C.c_int32), ("max_key_pages_per_req", C.c_int32),
        ("max_blocks_per_req", C.c_int32), ("kpt_ld", C.c_int64), ("bt_ld", C.c_int64),
        ("q_row_stride", C.c_int64), ("segment_rows", C.c_int32), ("chunk_rows", C.c_int32),
        ("query_start_loc", C.c_void_p), ("positions", C.c_void_p), ("q", C.c_void_p),
        ("key_cache", C.c_void_p), ("key_page_table", C.c_void_p), ("block_table", C.c_void_p),
    ]


def _load():
    if not os.path.exists(_LIB_PATH):
        raise ImportError(f"libsel.so is not built ({_LIB_PATH}); run "
                          "sparse_attention_kv_device_gb300.build.build() or __graft_entry__.build()")
    lib = C.CDLL(_LIB_PATH)
    P, I32, I64, SZ = C.c_void_p, C.c_int32, C.c_int64, C.c_size_t
    PP = C.POINTER(sel_problem)
    lib.sel_error_string.argtypes = [C.c_int]
    lib.sel_error_string.restype = C.c_char_p
    lib.sel_version.restype = C.c_int
    lib.sel_workspace_bytes.argtypes = [PP]
    lib.sel_workspace_bytes.restype = SZ
    lib.sel_score_workspace_bytes.argtypes = [PP]
    lib.sel_score_workspace_bytes.restype = SZ
    lib.sel_score_paged.argtypes = [PP, P, I64, P, P, SZ, P]
    lib.sel_topk_expand.argtypes = [P, I64, P, I32, I32, I32, P, I32, P, P, P]
    lib.sel_remap_global.argtypes = [P, I32, P, I64, I32, I32, P, I32, I32, I32, I64, P, P, P]
    lib.sel_remap_workspace.argtypes = [P, I32, P, I64, I32, I32, P, P, I32, P, I32, I32, I32, I64, P, P, P]
    lib.sel_remap_dcp.argtypes = [P, I32, P, I64, I32, I32, P, I32, I32, I32, I32, I32, I32, I32, P, P, P]
    lib.sel_select.argtypes = [PP, P, I32, P, P, P, P, SZ, P]
    lib.sel_select_static.argtypes = [PP, P, I32, P, P, P, P]
    lib.sel_host_stage_bytes.argtypes = [PP, I32]
    lib.sel_host_stage_bytes.restype = SZ
    lib.sel_select_host.argtypes = [PP, P, I32, P, P, P, SZ, P, SZ, P]
    lib.sel_set_trace_events.argtypes = [C.POINTER(C.c_void_p), I32]
    lib.sel_debug_wait_limit.argtypes = [I32, I64]
    lib.sel_select_launch_count.argtypes = [PP]
    lib.sel_select_launch_count.restype = I32
    lib.sel_maxsim_workspace_bytes.argtypes = []
    lib.sel_maxsim_workspace_bytes.restype = SZ
    lib.sel_maxsim_rerank.argtypes = [P, I32, I32, I64, P, I64, I64, P, P, I32, P, P, P, SZ, P]
    lib.sel_maxsim_launch_count.argtypes = [I32, I32]
    lib.sel_mla_workspace_bytes.argtypes = [I32, I32]
    lib.sel_mla_workspace_bytes.restype = SZ
    lib.sel_mla_decode.argtypes = [P, I64, I64, P, I64, I64, I32, I32, I32, I32, P, I64, P, I64, I64, P, I32, P,
                                   C.c_float, P, P, P, P, SZ, P]
    lib.sel_mla_launch_count.argtypes = [I32]
    lib.sel_maxsim_launch_count.restype = I32
    for f in ("sel_score_paged", "sel_topk_expand", "sel_remap_global", "sel_remap_workspace", "sel_remap_dcp",
              "sel_select",
              "sel_select_static", "sel_select_host", "sel_set_trace_events", "sel_debug_wait_limit",
              "sel_maxsim_rerank"):
        getattr(lib, f).restype = C.c_int
    return lib


_lib = _load()

EXPORTS = ["sel_error_string", "sel_version", "sel_workspace_bytes", "sel_score_workspace_bytes",
           "sel_score_paged", "sel_topk_expand", "sel_remap_global", "sel_remap_workspace", "sel_remap_dcp",
           "sel_select",
           "sel_select_static", "sel_host_stage_bytes", "sel_select_host", "sel_set_trace_events",
           "sel_debug_wait_limit",
           "sel_select_launch_count", "sel_maxsim_workspace_bytes", "sel_maxsim_rerank", "sel_maxsim_launch_count",
           "sel_mla_workspace_bytes", "sel_mla_decode", "sel_mla_launch_count"]


def library_path() -> str:
    return _LIB_PATH


def sel_error_string(code: int) -> str:
    return _lib.sel_error_string(int(code)).decode()


def sel_version() -> int:
    return int(_lib.sel_version())


def _ptr(t):
    return None if t is None else C.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return C.c_void_p(stream.cuda_stream)


def _check(rc: int, where: str):
    if rc != SEL_OK:
        raise SelError(rc, where)


def _dev(t, dtype, name):
    if t is None:
        return
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")


class Problem:
    """A sel_problem plus the device tensors it points into (kept alive here).

    Tensors: query_start_loc int32 [num_reqs+1], positions int32 [num_rows],
    q fp16 [num_rows, 4, 128] (row stride may exceed 512), key_cache fp16 (any shape,
    contiguous, physical page p at element p * key_page_stride), key_page_table int32
    [num_reqs, kpt_ld], block_table int32 [num_reqs, bt_ld].
    """

    def __init__(self, *, query_start_loc, positions, q, key_cache, key_page_table, block_table,
                 index_topk, kpool, max_context, key_page_stride, num_key_pages, num_kv_blocks,
                 block_size=64, block_stride_rows=None, max_key_pages_per_req=None,
                 max_blocks_per_req=None, max_q_len=0, segment_rows=0, chunk_rows=0,
                 num_rows=None, host_inputs=False):
        # host_inputs: the per-step inputs (everything but key_cache) are host tensors,
        # for sel_select_host; the key cache always lives on the device.
        _dev(key_cache, torch.float16, "key_cache")
        for t, dt, n in ((query_start_loc, torch.int32, "query_start_loc"),
                         (positions, torch.int32, "positions"), (q, torch.float16, "q"),
                         (key_page_table, torch.int32, "key_page_table"),
                         (block_table, torch.int32, "block_table")):
            if host_inputs:
                if t.is_cuda or t.dtype != dt:
                    raise ValueError(f"{n} must be a host {dt} tensor")
            else:
                _dev(t, dt, n)
        if q.dim() != 3 or q.shape[1] != 4 or q.shape[2] != 128 or q.stride(2) != 1 or q.stride(1) != 128:
            raise ValueError("q must be [rows, 4, 128] with contiguous heads")
        if not (key_cache.is_contiguous() and key_page_table.is_contiguous() and block_table.is_contiguous()
                and positions.is_contiguous() and query_start_loc.is_contiguous()):
            raise ValueError("tables, positions and the key cache must be contiguous")
        self.tensors = (query_start_loc, positions, q, key_cache, key_page_table, block_table)
        p = sel_problem()
        p.num_reqs = int(query_start_loc.numel() - 1)
        p.num_rows = int(positions.numel() if num_rows is None else num_rows)
        p.max_context = int(max_context)
        p.max_q_len = int(max_q_len)
        p.num_heads, p.head_dim = 4, 128
        p.index_topk, p.kpool = int(index_topk), int(kpool)
        p.key_page_size = 64
        p.block_size = int(block_size)
        p.block_stride_rows = int(block_size if block_stride_rows is None else block_stride_rows)
        p.key_page_stride = int(key_page_stride)
        p.num_key_pages = int(num_key_pages)
        p.num_kv_blocks = int(num_kv_blocks)
        p.kpt_ld = int(key_page_table.shape[1])
        p.bt_ld = int(block_table.shape[1])
        p.max_key_pages_per_req = int(p.kpt_ld if max_key_pages_per_req is None else max_key_pages_per_req)
        p.max_blocks_per_req = int(p.bt_ld if max_blocks_per_req is None else max_blocks_per_req)
        p.q_row_stride = int(q.stride(0))
        p.segment_rows = int(segment_rows)
        p.chunk_rows = int(chunk_rows)
        p.query_start_loc = query_start_loc.data_ptr()
        p.positions = positions.data_ptr()
        p.q = q.data_ptr()
        p.key_cache = key_cache.data_ptr()
        p.key_page_table = key_page_table.data_ptr()
        p.block_table = block_table.data_ptr()
        self.c = p

    @property
    def num_rows(self):
        return int(self.c.num_rows)

    def byref(self):
        return C.byref(self.c)


def problem_from_workload(w, device="cuda", **overrides) -> Problem:
    """Copy a workload (any object with the workload fields) to the device as a Problem."""
    dev = torch.device(device)
    kw = dict(
        query_start_loc=torch.from_numpy(w.qsl).to(dev),
        positions=torch.from_numpy(w.positions).to(dev),
        q=torch.from_numpy(w.q).to(dev),
        key_cache=torch.from_numpy(w.key_cache).to(dev),
        key_page_table=torch.from_numpy(w.key_page_table).to(dev),
        block_table=torch.from_numpy(w.block_table).to(dev),
        index_topk=w.index_topk, kpool=w.kpool, max_context=w.max_context,
        key_page_stride=w.key_page_stride, num_key_pages=w.num_key_pages,
        num_kv_blocks=w.num_kv_blocks, block_size=w.block_size,
        block_stride_rows=w.block_stride_rows, max_key_pages_per_req=w.max_key_pages_per_req,
        max_blocks_per_req=w.max_blocks_per_req, max_q_len=w.max_q_len, chunk_rows=w.chunk_rows)
    kw.update(overrides)
    return Problem(**kw)


def sel_workspace_bytes(problem: Problem) -> int:
    n = int(_lib.sel_workspace_bytes(problem.byref()))
    if n == 0:
        raise SelError(SEL_EINVAL, "sel_workspace_bytes")
    return n


def sel_score_workspace_bytes(problem: Problem) -> int:
    n = int(_lib.sel_score_workspace_bytes(problem.byref()))
    if n == 0:
        raise SelError(SEL_EINVAL, "sel_score_workspace_bytes")
    return n


def new_workspace(nbytes, device):
    """A zero-filled device workspace of nbytes (the MaxSim workspace must start zero-filled;
    the selection's needs no initialisation, and zeros do no harm)."""
    return torch.zeros(max(int(nbytes), 1), dtype=torch.uint8, device=device)


def _workspace(ws, nbytes, device):
    if ws is None:
        ws = new_workspace(nbytes, device)
    elif ws.numel() * ws.element_size() < nbytes:
        raise SelError(SEL_EWORKSPACE, "workspace")
    return ws


def _on_current_device(where, *tensors):
    """The library queues work on the current CUDA device: every tensor must live there."""
    cur = torch.cuda.current_device()
    for t in tensors:
        if t is not None and t.is_cuda and t.device.index != cur:
            raise ValueError(f"{where}: tensor on {t.device}, but the current device is cuda:{cur}")


def sel_score_paged(problem: Problem, scores, status=None, ws=None, stream=None):
    """scores: fp32 [num_rows, scores_ld] on the device (row stride = scores.stride(0))."""
    _dev(scores, torch.float32, "scores")
    _dev(status, torch.int32, "status")
    if scores.stride(1) != 1:
        raise ValueError("scores rows must be contiguous")
    _on_current_device("sel_score_paged", scores, status, ws, *problem.tensors)
    ws = _workspace(ws, sel_score_workspace_bytes(problem), scores.device)
    _check(_lib.sel_score_paged(problem.byref(), _ptr(scores), scores.stride(0), _ptr(status), _ptr(ws),
                                ws.numel() * ws.element_size(), _stream(stream)), "sel_score_paged")
    return scores


def sel_topk_expand(scores, positions, index_topk, kpool, token_idx, valid_counts=None, status=None,
                    stream=None):
    """scores fp32 [rows, ld]; positions int32 [rows]; token_idx int32 [rows, out_width]."""
    _dev(scores, torch.float32, "scores")
    _dev(positions, torch.int32, "positions")
    _dev(token_idx, torch.int32, "token_idx")
    _dev(valid_counts, torch.int32, "valid_counts")
    _dev(status, torch.int32, "status")
    if scores.stride(1) != 1 or not token_idx.is_contiguous():
        raise ValueError("scores rows and token_idx must be contiguous")
    rows = int(positions.numel())
    _check(_lib.sel_topk_expand(_ptr(scores), scores.stride(0), _ptr(positions), rows, int(index_topk),
                                int(kpool), _ptr(token_idx), int(token_idx.shape[1]), _ptr(valid_counts),
                                _ptr(status), _stream(stream)), "sel_topk_expand")
    return token_idx, valid_counts


def sel_remap_global(req_id, block_table, token_idx, slots, *, num_kv_blocks, block_size=64,
                     block_stride_rows=None, max_blocks_per_req=None, valid_counts=None, stream=None):
    """req_id int32 [rows]; block_table int32 [num_reqs, bt_ld]; token_idx, slots int32 [rows, width]."""
    for t, n in ((req_id, "req_id"), (block_table, "block_table"), (token_idx, "token_idx"),
                 (slots, "slots"), (valid_counts, "valid_counts")):
        _dev(t, torch.int32, n)
    if not (token_idx.is_contiguous() and slots.is_contiguous() and block_table.is_contiguous()):
        raise ValueError("token_idx, slots and block_table must be contiguous")
    rows, width = token_idx.shape
    mb = block_table.shape[1] if max_blocks_per_req is None else max_blocks_per_req
    stride = block_size if block_stride_rows is None else block_stride_rows
    _check(_lib.sel_remap_global(_ptr(req_id), int(block_table.shape[0]), _ptr(block_table),
                                 int(block_table.shape[1]), int(mb), int(num_kv_blocks), _ptr(token_idx),
                                 int(rows), int(width), int(block_size), int(stride), _ptr(slots),
                                 _ptr(valid_counts), _stream(stream)), "sel_remap_global")
    return slots, valid_counts


def sel_remap_workspace(req_id, block_table, ws_req, ws_starts, token_idx, slots, *, num_kv_blocks, block_size=64,
                        block_stride_rows=None, max_blocks_per_req=None, valid_counts=None, stream=None):
    """sel_remap_global, with rows of prefill requests (ws_req >= 0) mapped to ws_starts[ws_req] + t."""
    for t, n in ((req_id, "req_id"), (block_table, "block_table"), (ws_req, "ws_req"), (ws_starts, "ws_starts"),
                 (token_idx, "token_idx"), (slots, "slots"), (valid_counts, "valid_counts")):
        _dev(t, torch.int32, n)
    if not (token_idx.is_contiguous() and slots.is_contiguous() and block_table.is_contiguous()):
        raise ValueError("token_idx, slots and block_table must be contiguous")
    rows, width = token_idx.shape
    mb = block_table.shape[1] if max_blocks_per_req is None else max_blocks_per_req
    stride = block_size if block_stride_rows is None else block_stride_rows
    _check(_lib.sel_remap_workspace(_ptr(req_id), int(block_table.shape[0]), _ptr(block_table),
                                    int(block_table.shape[1]), int(mb), int(num_kv_blocks), _ptr(ws_req),
                                    _ptr(ws_starts), int(ws_starts.numel()), _ptr(token_idx), int(rows), int(width),
                                    int(block_size), int(stride), _ptr(slots), _ptr(valid_counts), _stream(stream)),
           "sel_remap_workspace")
    return slots, valid_counts


def sel_remap_dcp(req_id, block_table, token_idx, slots, *, num_kv_blocks, dcp_size, dcp_rank, interleave=1,
                  compact=True, block_size=64, max_blocks_per_req=None, valid_counts=None, stream=None):
    """One decode-context-parallel rank's slots (its dense block table), optionally compacted to the front."""
    for t, n in ((req_id, "req_id"), (block_table, "block_table"), (token_idx, "token_idx"),
                 (slots, "slots"), (valid_counts, "valid_counts")):
        _dev(t, torch.int32, n)
    if not (token_idx.is_contiguous() and slots.is_contiguous() and block_table.is_contiguous()):
        raise ValueError("token_idx, slots and block_table must be contiguous")
    rows, width = token_idx.shape
    mb = block_table.shape[1] if max_blocks_per_req is None else max_blocks_per_req
    _check(_lib.sel_remap_dcp(_ptr(req_id), int(block_table.shape[0]), _ptr(block_table), int(block_table.shape[1]),
                              int(mb), int(num_kv_blocks), _ptr(token_idx), int(rows), int(width), int(block_size),
                              int(dcp_size), int(dcp_rank), int(interleave), int(bool(compact)), _ptr(slots),
                              _ptr(valid_counts), _stream(stream)), "sel_remap_dcp")
    return slots, valid_counts


def sel_select(problem: Problem, slots, valid_counts, token_idx=None, status=None, ws=None, stream=None):
    """slots int32 [num_rows, out_width]; valid_counts int32 [num_rows]."""
    for t, n in ((slots, "slots"), (valid_counts, "valid_counts"), (token_idx, "token_idx"),
                 (status, "status")):
        _dev(t, torch.int32, n)
    if not slots.is_contiguous() or (token_idx is not None and not token_idx.is_contiguous()):
        raise ValueError("slots and token_idx must be contiguous")
    _on_current_device("sel_select", slots, valid_counts, token_idx, status, ws, *problem.tensors)
    ws = _workspace(ws, sel_workspace_bytes(problem), slots.device)
    _check(_lib.sel_select(problem.byref(), _ptr(slots), int(slots.shape[1]), _ptr(valid_counts),
                           _ptr(token_idx), _ptr(status), _ptr(ws), ws.numel() * ws.element_size(),
                           _stream(stream)), "sel_select")
    return slots, valid_counts


def sel_select_static(problem: Problem, slots, valid_counts, token_idx=None, status=None, stream=None):
    """sel_select with the library's fixed device scratch array instead of a workspace.

    For callers that cannot allocate device memory per call; this binding allocates
    nothing either. Calls on one device must not overlap on the GPU (they share the
    array). Raises SelError(SEL_EWORKSPACE) when the problem needs more scratch than
    SEL_STATIC_WS_MAX_BYTES."""
    for t, n in ((slots, "slots"), (valid_counts, "valid_counts"), (token_idx, "token_idx"),
                 (status, "status")):
        _dev(t, torch.int32, n)
    if not slots.is_contiguous() or (token_idx is not None and not token_idx.is_contiguous()):
        raise ValueError("slots and token_idx must be contiguous")
    _on_current_device("sel_select_static", slots, valid_counts, token_idx, status, *problem.tensors)
    _check(_lib.sel_select_static(problem.byref(), _ptr(slots), int(slots.shape[1]), _ptr(valid_counts),
                                  _ptr(token_idx), _ptr(status), _stream(stream)), "sel_select_static")
    return slots, valid_counts


def sel_host_stage_bytes(problem: Problem, out_width: int) -> int:
    return int(_lib.sel_host_stage_bytes(problem.byref(), int(out_width)))


def sel_select_host(problem: Problem, slots_host, counts_host, stage, ws, status=None, stream=None):
    """problem's per-step inputs are HOST tensors (pinned); key_cache is on the device."""
    _dev(stage, torch.uint8, "stage")
    _dev(ws, torch.uint8, "ws")
    _check(_lib.sel_select_host(problem.byref(), _ptr(slots_host), int(slots_host.shape[1]),
                                _ptr(counts_host), _ptr(status), _ptr(stage), stage.numel(), _ptr(ws),
                                ws.numel(), _stream(stream)), "sel_select_host")
    return slots_host, counts_host


def sel_set_trace_events(events) -> None:
    """events: four torch.cuda.Event(enable_timing=True), or None to switch tracing off."""
    if not events:
        _check(_lib.sel_set_trace_events(None, 0), "sel_set_trace_events")
        return
    for e in events:
        if not e.cuda_event:   # torch creates the CUDA event on its first record
            e.record()
    arr = (C.c_void_p * len(events))(*[e.cuda_event for e in events])
    _check(_lib.sel_set_trace_events(arr, len(events)), "sel_set_trace_events")


def sel_debug_wait_limit(fault_tile: int = -1, wait_ns: int = 1_000_000_000) -> None:
    """Failure-detection test hook: later launches give every bounded wait wait_ns and
    (fault_tile >= 0) never load that tile, so the waits on it expire. The defaults restore
    normal operation."""
    _check(_lib.sel_debug_wait_limit(int(fault_tile), int(wait_ns)), "sel_debug_wait_limit")


def sel_select_launch_count(problem: Problem) -> int:
    return int(_lib.sel_select_launch_count(problem.byref()))


def sel_maxsim_workspace_bytes() -> int:
    return int(_lib.sel_maxsim_workspace_bytes())


def sel_maxsim_rerank(q, docs, doc_offsets, doc_lengths, scores=None, status=None, ws=None, stream=None):
    """MaxSim scores of one query against documents packed in one tensor.

    q fp16 [lq, d]; docs fp16 [total_tokens, d] (the packed tensor, read in place; a row
    stride above d is allowed); doc_offsets, doc_lengths int32 [B]. Row strides must be
    multiples of 8 elements. Returns scores fp32 [B]: per query row the best dot product
    over the document's rows, summed over the query rows (-inf for an empty document).
    ws (optional): a uint8 device tensor of sel_maxsim_workspace_bytes(), zero-filled before
    its first use (new_workspace); the kernel leaves it zero-filled, so it can be kept across calls."""
    _dev(q, torch.float16, "q")
    _dev(docs, torch.float16, "docs")
    _dev(doc_offsets, torch.int32, "doc_offsets")
    _dev(doc_lengths, torch.int32, "doc_lengths")
    _dev(status, torch.int32, "status")
    if q.dim() != 2 or docs.dim() != 2 or q.shape[1] != docs.shape[1]:
        raise ValueError("q [lq, d] and docs [total_tokens, d] must share d")
    if q.stride(1) != 1 or docs.stride(1) != 1 or not doc_offsets.is_contiguous() or not doc_lengths.is_contiguous():
        raise ValueError("q and docs need unit column stride; offsets and lengths must be contiguous")
    if doc_offsets.numel() != doc_lengths.numel():
        raise ValueError("doc_offsets and doc_lengths differ in length")
    num_docs = doc_offsets.numel()
    if scores is None:
        scores = torch.empty(num_docs, dtype=torch.float32, device=docs.device)
    _dev(scores, torch.float32, "scores")
    if ws is None:  # the workspace must start zero-filled (the kernel leaves it so)
        ws = new_workspace(sel_maxsim_workspace_bytes(), docs.device)
    _dev(ws, torch.uint8, "ws")
    lq, d = q.shape
    _check(_lib.sel_maxsim_rerank(_ptr(q), int(lq), int(d), int(q.stride(0)), _ptr(docs), int(docs.shape[0]),
                                  int(docs.stride(0)), _ptr(doc_offsets), _ptr(doc_lengths), int(num_docs),
                                  _ptr(scores), _ptr(status), _ptr(ws), ws.numel() * ws.element_size(),
                                  _stream(stream)), "sel_maxsim_rerank")
    return scores


def sel_maxsim_launch_count(lq: int, d: int) -> int:
    return int(_lib.sel_maxsim_launch_count(int(lq), int(d)))


def sel_mla_workspace_bytes(rows: int, width: int) -> int:
    return int(_lib.sel_mla_workspace_bytes(int(rows), int(width)))


def sel_mla_decode(q_nope, q_pe, ckv, kpe, slots, kv_len, sm_scale, out=None, lse=None, status=None, ws=None,
                   stream=None):
    """Sparse MLA decode attention over the selected slots.

    q_nope bf16 [rows, 16, 512]; q_pe bf16 [rows, 16, dr] with dr 0 or 64 (None for 0);
    ckv bf16 [num_slots, >= 512] (row stride a multiple of 8); kpe bf16 [num_slots, >= dr]
    (None for dr 0; may be a column slice of the same cache tensor); slots int32 [rows, width];
    kv_len int32 [rows]. Returns (out fp32 [rows, 16, 512], lse fp32 [rows, 16])."""
    _dev(q_nope, torch.bfloat16, "q_nope")
    _dev(q_pe, torch.bfloat16, "q_pe")
    _dev(ckv, torch.bfloat16, "ckv")
    _dev(kpe, torch.bfloat16, "kpe")
    _dev(slots, torch.int32, "slots")
    _dev(kv_len, torch.int32, "kv_len")
    _dev(status, torch.int32, "status")
    _on_current_device("sel_mla_decode", q_nope, q_pe, ckv, kpe, slots, kv_len, out, lse, status, ws)
    if q_nope.dim() != 3 or q_nope.stride(2) != 1:
        raise ValueError("q_nope must be [rows, heads, dc] with unit dim stride")
    rows, heads, dc = q_nope.shape
    dr = 0 if q_pe is None else int(q_pe.shape[2])
    if q_pe is not None and (q_pe.dim() != 3 or q_pe.shape[:2] != q_nope.shape[:2] or q_pe.stride(2) != 1):
        raise ValueError("q_pe must be [rows, heads, dr] with unit dim stride")
    if ckv.dim() != 2 or ckv.stride(1) != 1 or (kpe is not None and (kpe.dim() != 2 or kpe.stride(1) != 1)):
        raise ValueError("ckv / kpe must be [num_slots, dims] with unit column stride")
    if (dr > 0) != (kpe is not None):
        raise ValueError("kpe is needed exactly when q_pe has rotary dims")
    if slots.dim() != 2 or slots.shape[0] != rows or not slots.is_contiguous() or not kv_len.is_contiguous():
        raise ValueError("slots must be contiguous [rows, width]; kv_len contiguous [rows]")
    width = int(slots.shape[1])
    if out is None:
        out = torch.empty((rows, heads, dc), dtype=torch.float32, device=q_nope.device)
    if lse is None:
        lse = torch.empty((rows, heads), dtype=torch.float32, device=q_nope.device)
    _dev(out, torch.float32, "out")
    _dev(lse, torch.float32, "lse")
    if not out.is_contiguous() or not lse.is_contiguous():
        raise ValueError("out and lse must be contiguous")
    ws = _workspace(ws, sel_mla_workspace_bytes(rows, width), q_nope.device)
    _check(_lib.sel_mla_decode(_ptr(q_nope), int(q_nope.stride(0)), int(q_nope.stride(1)), _ptr(q_pe),
                               int(q_pe.stride(0)) if q_pe is not None else 0,
                               int(q_pe.stride(1)) if q_pe is not None else 0, int(rows), int(heads), int(dc),
                               int(dr), _ptr(ckv), int(ckv.stride(0)), _ptr(kpe),
                               int(kpe.stride(0)) if kpe is not None else 0, int(ckv.shape[0]), _ptr(slots), width,
                               _ptr(kv_len), float(sm_scale), _ptr(out), _ptr(lse), _ptr(status), _ptr(ws),
                               ws.numel() * ws.element_size(), _stream(stream)), "sel_mla_decode")
    return out, lse


def sel_mla_launch_count(rows: int) -> int:
    return int(_lib.sel_mla_launch_count(int(rows)))
