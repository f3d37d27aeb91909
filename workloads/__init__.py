"""Seeded synthetic inputs for sparse-attention token selection over a paged KV cache.

This module only draws random numbers and lays out tables: it holds none of the
selection arithmetic (no scoring, no top-k, no expansion, no remap), so both the
CPU oracle and the CUDA path can consume what it produces without sharing code.

Every workload is a batch of query rows grouped by request (``qsl`` = request start
offsets, ``positions`` = token position of each row, so a row sees ``position + 1``
tokens), a compressed key cache in 64-key pages placed through a per-request key
page table, and a 64-token-block KV block table, as described on the vLLM pages
"sparse_utils" (triton_convert_req_index_to_global_index, flat_kv_row_view) and
PR #59 of the ReVolta vLLM fork (request-segmented QSA scorer).

Recipe (all seeded; ``numpy.random.SeedSequence(seed).spawn(4)`` gives independent
streams for queries, keys, key-page placement and block placement):

* q ``[rows, 4, 128]`` fp16 and compressed keys ``[pools, 128]`` fp16, either
  integer-valued uniform in {-3..3} (exact fp32 dot products) or N(0,1)/sqrt(128).
* Each request owns ``ctx_max // kpool`` compressed keys (complete pools of its
  longest row) in ``ceil(pools / 64)`` key pages and ``ceil(ctx_max / 64)`` KV blocks.
* The physical key-page pool and KV-block pool hold 1.25x the pages/blocks needed
  (rounded up), and a seeded random permutation places the logical pages/blocks.
* Never-read memory is poisoned: unused physical key pages (and, with a page stride
  above one page, the interleaved pages of "other layers") hold fp16 NaN; key rows
  past a request's last complete pool inside its last page hold +3, which would win
  the selection if a kernel ever scored them.
* The KV cache itself is not materialised: selection only produces slot numbers.
"""

from __future__ import annotations

import dataclasses
import math
from typing import Sequence

import numpy as np

HEADS = 4
HEAD_DIM = 128
KEY_PAGE = 64      # compressed keys per key page
BLOCK = 64         # tokens per KV block


@dataclasses.dataclass
class Workload:
    name: str
    integer_mode: bool
    num_reqs: int
    num_rows: int                 # rows >= qsl[-1] are graph padding rows
    qsl: np.ndarray               # int32 [num_reqs + 1]
    positions: np.ndarray         # int32 [num_rows]
    q: np.ndarray                 # float16 [num_rows, 4, 128]
    key_cache: np.ndarray         # float16 flat, page p at p * key_page_stride
    key_page_stride: int          # elements between consecutive physical key pages
    num_key_pages: int
    key_page_table: np.ndarray    # int32 [num_reqs, kpt_ld]
    max_key_pages_per_req: int
    block_table: np.ndarray       # int32 [num_reqs, bt_ld]
    max_blocks_per_req: int
    num_kv_blocks: int
    block_size: int
    block_stride_rows: int
    index_topk: int
    kpool: int
    out_width: int
    max_context: int
    max_q_len: int
    chunk_rows: int = 256
    oob_entries: tuple = ()        # (req, logical block, value) written over the table

    @property
    def kpt_ld(self) -> int:
        return int(self.key_page_table.shape[1])

    @property
    def bt_ld(self) -> int:
        return int(self.block_table.shape[1])

    def row_contexts(self) -> np.ndarray:
        return self.positions.astype(np.int64) + 1


def _ceil_div(a: int, b: int) -> int:
    return -(-a // b)


def build_workload(requests: Sequence[Sequence[int]], *, name: str, seed: int,
                   integer_mode: bool, index_topk: int = 2048, kpool: int = 4,
                   key_page_stride_pages: int = 1, block_stride_rows: int | None = None,
                   oob_blocks: Sequence[tuple[int, int, int]] = (),
                   pad_rows: int = 0, chunk_rows: int = 256,
                   out_width: int | None = None, pool_factor: float = 1.25,
                   max_context: int | None = None, block_size: int = BLOCK) -> Workload:
    """Lay out one batch.

    ``requests[i]`` lists the context length (position + 1) of each query row of
    request i, in row order. ``oob_blocks`` entries ``(req, logical_block, value)``
    overwrite block-table entries (value is the physical id written; a negative
    ``value`` is written as is, a value >= 0 is added to ``num_kv_blocks`` so that
    it lands past the physical pool). ``block_size`` is the KV block size in tokens
    (``block_stride_rows`` defaults to it).
    """
    if block_stride_rows is None:
        block_stride_rows = block_size
    ss = np.random.SeedSequence(seed)
    rng_q, rng_k, rng_kp, rng_bt = (np.random.default_rng(s) for s in ss.spawn(4))

    num_reqs = len(requests)
    lens = [len(r) for r in requests]
    qsl = np.zeros(num_reqs + 1, dtype=np.int32)
    qsl[1:] = np.cumsum(lens)
    real_rows = int(qsl[-1])
    num_rows = real_rows + pad_rows
    positions = np.zeros(num_rows, dtype=np.int32)
    ctx_rows = [c for r in requests for c in r]
    positions[:real_rows] = np.asarray(ctx_rows, dtype=np.int64) - 1
    if pad_rows:
        positions[real_rows:] = 0

    def draw(rng, shape):
        if integer_mode:
            return rng.integers(-3, 4, size=shape).astype(np.float16)
        x = rng.standard_normal(size=shape, dtype=np.float32) / np.float32(math.sqrt(HEAD_DIM))
        return x.astype(np.float16)

    q = draw(rng_q, (num_rows, HEADS, HEAD_DIM))

    ctx_max = [max(r) if len(r) else 0 for r in requests]
    pools = [c // kpool for c in ctx_max]
    kpages = [_ceil_div(p, KEY_PAGE) for p in pools]
    blocks = [_ceil_div(c, block_size) for c in ctx_max]

    # key pages: physical pool = 1.25x needed, seeded placement
    num_key_pages = max(1, math.ceil(sum(kpages) * pool_factor))
    kp_perm = rng_kp.permutation(num_key_pages).astype(np.int32)
    kpt_ld = max(1, max(kpages) if kpages else 1)
    key_page_table = np.full((num_reqs, kpt_ld), -1, dtype=np.int32)
    nxt = 0
    for i in range(num_reqs):
        key_page_table[i, :kpages[i]] = kp_perm[nxt:nxt + kpages[i]]
        nxt += kpages[i]

    page_elems = KEY_PAGE * HEAD_DIM
    key_page_stride = key_page_stride_pages * page_elems
    key_cache = np.full(num_key_pages * key_page_stride, np.nan, dtype=np.float16)
    kc_pages = key_cache.reshape(num_key_pages, key_page_stride_pages, KEY_PAGE, HEAD_DIM)
    for i in range(num_reqs):
        if pools[i] == 0:
            continue
        keys = draw(rng_k, (pools[i], HEAD_DIM))
        padded = np.full((kpages[i] * KEY_PAGE, HEAD_DIM), 3.0, dtype=np.float16)
        padded[:pools[i]] = keys
        kc_pages[key_page_table[i, :kpages[i]], 0] = padded.reshape(kpages[i], KEY_PAGE, HEAD_DIM)

    # KV blocks: physical pool = 1.25x needed, seeded placement
    num_kv_blocks = max(1, math.ceil(sum(blocks) * pool_factor))
    bt_perm = rng_bt.permutation(num_kv_blocks).astype(np.int32)
    bt_ld = max(1, max(blocks) if blocks else 1)
    block_table = np.full((num_reqs, bt_ld), -1, dtype=np.int32)
    nxt = 0
    for i in range(num_reqs):
        block_table[i, :blocks[i]] = bt_perm[nxt:nxt + blocks[i]]
        nxt += blocks[i]
    applied = []
    for (req, lb, val) in oob_blocks:
        v = val if val < 0 else num_kv_blocks + val
        block_table[req, lb] = v
        applied.append((req, lb, v))

    if out_width is None:
        out_width = index_topk + kpool
    return Workload(
        name=name, integer_mode=integer_mode, num_reqs=num_reqs, num_rows=num_rows,
        qsl=qsl, positions=positions, q=q, key_cache=key_cache,
        key_page_stride=key_page_stride, num_key_pages=num_key_pages,
        key_page_table=key_page_table, max_key_pages_per_req=kpt_ld,
        block_table=block_table, max_blocks_per_req=bt_ld, num_kv_blocks=num_kv_blocks,
        block_size=block_size, block_stride_rows=block_stride_rows, index_topk=index_topk,
        kpool=kpool, out_width=out_width,
        max_context=max_context if max_context is not None else max([0] + ctx_rows),
        max_q_len=max([1] + lens), chunk_rows=chunk_rows, oob_entries=tuple(applied))


def _run(lo: int, hi: int) -> list[int]:
    return list(range(lo, hi + 1))


# The five workloads the selection path is measured and checked on, plus the
# ragged variant whose last request is short enough (<= index_topk) to select
# every token.
CONFIGS = {
    # 2 requests x 2 decode rows; contexts 999, 1000 / 2999, 3000; topk 256 (64 pools)
    "tiny": dict(requests=[[999, 1000], [2999, 3000]], integer_mode=True, index_topk=256),
    # 4 requests x 4 rows, positions 32,765..32,768 (contexts 32,766..32,769)
    "decode32k": dict(requests=[_run(32766, 32769)] * 4, integer_mode=True),
    # 8 requests x 5 rows at 128K; blocks and key pages interleaved with other layers
    "decode128k": dict(requests=[_run(131068, 131072)] * 8, integer_mode=False,
                       block_stride_rows=2 * BLOCK, key_page_stride_pages=2),
    # ragged decode with out-of-range block-table entries
    "ragged": dict(requests=[[262144], _run(199999, 200001), _run(131071, 131074),
                             _run(3994, 4000)], integer_mode=False,
                   oob_blocks=[(1, 0, 0), (1, 1500, 5), (1, 3125, 1 << 20), (2, 100, -2)]),
    "ragged_b": dict(requests=[[262144], _run(199999, 200001), _run(131071, 131074),
                               _run(1994, 2000)], integer_mode=False,
                     oob_blocks=[(1, 0, 0), (1, 1500, 5), (1, 3125, 1 << 20), (2, 100, -2)]),
    # 16 one-row decode requests at 128K, then one 4,096-row prefill chunk
    "mixed": dict(requests=[[131072]] * 16 + [_run(60001, 64096)], integer_mode=False),
}

CONFIG_SEEDS = {"tiny": 1001, "decode32k": 1002, "decode128k": 1003, "ragged": 1004,
                "ragged_b": 1014, "mixed": 1005}


def make_workload(name: str, seed: int | None = None, **overrides) -> Workload:
    """One of the named workloads (``CONFIGS``), seeded with ``1000 + config number``."""
    spec = dict(CONFIGS[name])
    spec.update(overrides)
    return build_workload(name=name, seed=CONFIG_SEEDS[name] if seed is None else seed, **spec)


def random_scores(rows: int, pools: int, *, seed: int, ties: str = "none") -> np.ndarray:
    """fp32 score rows for exercising a top-k on its own.

    ``ties``: "none" (continuous normal values), "coarse" (values on a grid of 16
    levels, so many exact ties), "zeros" (all 0, with a few -0.0 mixed in), or
    "inf" (normal values with some -inf entries, as pools on unreadable pages get).
    """
    rng = np.random.default_rng(seed)
    if ties == "zeros":
        s = np.zeros((rows, pools), dtype=np.float32)
        s[rng.random((rows, pools)) < 0.3] = -0.0
        return s
    s = rng.standard_normal((rows, pools), dtype=np.float32)
    if ties == "coarse":
        s = np.round(s * 4.0).astype(np.float32) / np.float32(4.0)
        s[s == 0] = np.where(rng.random(int((s == 0).sum())) < 0.5, 0.0, -0.0).astype(np.float32)
    elif ties == "inf":
        s[rng.random((rows, pools)) < 0.05] = -np.inf
    return s


def random_token_indices(rows: int, width: int, max_token: int, *, seed: int,
                         minus_one_frac: float = 0.1) -> np.ndarray:
    """int32 token indices in [0, max_token) with a fraction of -1 entries."""
    rng = np.random.default_rng(seed)
    t = rng.integers(0, max(1, max_token), size=(rows, width)).astype(np.int32)
    t[rng.random((rows, width)) < minus_one_frac] = -1
    return t


def selection_token_indices(contexts, width: int, *, topk: int = 2048, kpool: int = 4, seed: int) -> np.ndarray:
    """int32 token rows shaped like the selection's output for the given contexts: for
    ctx <= topk the tokens 0..ctx-1; otherwise topk / kpool distinct complete pools drawn at
    random, expanded to their kpool tokens, plus the trailing incomplete pool, ascending;
    then -1 up to width. (Random pools stand in for the scored top pools; the remap only
    sees the token order and density.)"""
    rng = np.random.default_rng(seed)
    ctx = np.asarray(contexts, dtype=np.int64)
    out = np.full((ctx.size, width), -1, dtype=np.int32)
    for r, c in enumerate(ctx):
        if c <= topk:
            toks = np.arange(c, dtype=np.int64)
        else:
            pools = c // kpool
            pick = np.sort(rng.choice(pools, size=topk // kpool, replace=False))
            toks = (pick[:, None] * kpool + np.arange(kpool)[None, :]).ravel()
            toks = np.concatenate([toks, np.arange(pools * kpool, c)])
        n = min(toks.size, width)
        out[r, :n] = toks[:n]
    return out
