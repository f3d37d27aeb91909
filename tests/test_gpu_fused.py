"""The fused selection (sel_select) on shapes and call patterns the named workloads do not
reach, through the C ABI, against the CPU oracle on the same seeded inputs.

* kpool 1, 3 and 8 with KV blocks of 16 and 48 tokens (powers of two and not, so both
  the shift and the division forms of the expansion and the remap run), index_topk of
  about 64 and about 2,048, and block strides above the block size: integer-valued
  inputs, so every output is bit exact.
* CUDA-graph replay after the request runs (query_start_loc: another split of the same
  rows, with an empty request and trailing padding rows) and the key page table change
  in place, as well as queries, keys, positions and the block table: the replays of
  ReVolta PR #59 ("Validation": graphs replayed after queries, keys, page tables,
  positions, lengths and request runs change).
* Every row of the full mixed step (16 decode rows at 128K and 4,096 prefill rows, 17
  chunks of 256 rows) under the parity rule, with repeated calls giving identical outputs.
"""

import numpy as np
import pytest
import torch

import workloads
from _gpu import DEV, assert_select_bitexact, assert_select_parity, lib, oracle_select, run_select

pytestmark = pytest.mark.gpu


def _width(topk, kpool):
    return ((topk + kpool - 1) + 3) // 4 * 4


# (kpool, block_size, index_topk, block stride in blocks, contexts per request)
VARIANTS = [
    (1, 16, 64, 1, [[3000, 3001, 3002], [65, 64, 63], [1000]]),
    (1, 48, 2048, 2, [[9000, 9001], [2049, 2048], [20000]]),
    (3, 16, 63, 3, [[3001, 3002, 3003], [64, 66], [700]]),
    (3, 48, 2046, 2, [[20001, 20002, 20003], [5000], [2047, 2049]]),
    (8, 16, 2048, 2, [[40000, 40007, 40003], [2049, 2055]]),
    (8, 48, 64, 1, [[5003, 5004], [60, 71, 72, 73]]),
]


@pytest.mark.parametrize("case", range(len(VARIANTS)))
def test_select_kpool_and_block_variants(case):
    kpool, bs, topk, stride_blocks, reqs = VARIANTS[case]
    w = workloads.build_workload(reqs, name=f"var{case}", seed=300 + case, integer_mode=True,
                                 index_topk=topk, kpool=kpool, block_size=bs,
                                 block_stride_rows=stride_blocks * bs, out_width=_width(topk, kpool))
    out = run_select(w)
    ref = oracle_select(w)
    assert out["status"] == ref["status"] == 0
    assert_select_bitexact(w, out, ref, np.arange(w.num_rows))


def test_graph_replay_after_request_runs_and_page_tables_change():
    """Capture once; before each replay rewrite query_start_loc (another split of the 16
    rows, an empty request, padding rows), permute the key page table's entries, and change
    queries, keys, positions and the block table; each replay is bit exact."""
    sel = lib()
    w = workloads.make_workload("decode32k")
    prob = sel.problem_from_workload(w, DEV)
    qsl_d, pos_d, q_d, kc_d, kpt_d, bt_d = prob.tensors
    slots = torch.empty((w.num_rows, w.out_width), dtype=torch.int32, device=DEV)
    counts = torch.empty(w.num_rows, dtype=torch.int32, device=DEV)
    tok = torch.empty_like(slots)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    ws = torch.zeros(sel.sel_workspace_bytes(prob), dtype=torch.uint8, device=DEV)
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        sel.sel_select(prob, slots, counts, token_idx=tok, status=status, ws=ws)  # warm-up outside capture
    stream.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        sel.sel_select(prob, slots, counts, token_idx=tok, status=status, ws=ws)
    rng = np.random.default_rng(123)
    splits = [[0, 3, 3, 9, 14], [0, 7, 8, 8, 16], [0, 0, 5, 11, 12], [0, 4, 8, 12, 16]]
    for step, split in enumerate(splits):
        w.qsl[:] = np.asarray(split, dtype=np.int32)
        w.q[:] = rng.integers(-3, 4, size=w.q.shape).astype(np.float16)
        kcv = w.key_cache.reshape(w.num_key_pages, 64, 128)
        live_mask = w.key_page_table >= 0
        live = w.key_page_table[live_mask]
        kcv[live[: len(live) // 3]] = rng.integers(-3, 4, size=(len(live) // 3, 64, 128)).astype(np.float16)
        w.key_page_table[live_mask] = rng.permutation(live)     # the same pages, other places
        w.positions[:] = 32768 - rng.integers(0, 6000, size=w.num_rows).astype(np.int32)
        perm = rng.permutation(w.num_kv_blocks).astype(np.int32)
        valid = w.block_table >= 0
        w.block_table[valid] = perm[w.block_table[valid]]
        for dst, src in ((qsl_d, w.qsl), (q_d, w.q), (kc_d, w.key_cache), (kpt_d, w.key_page_table),
                         (pos_d, w.positions), (bt_d, w.block_table)):
            dst.copy_(torch.from_numpy(src))
        status.zero_()
        g.replay()
        torch.cuda.synchronize()
        ref = oracle_select(w)
        out = dict(slots=slots.cpu().numpy(), counts=counts.cpu().numpy(), token_idx=tok.cpu().numpy())
        assert int(status.item()) == ref["status"] == 0, step
        assert_select_bitexact(w, out, ref, np.arange(w.num_rows))
        padding = np.arange(w.num_rows) >= split[-1]
        assert (out["slots"][padding] == -1).all() and (out["counts"][padding] == 0).all()


def test_select_mixed_every_row_and_repeat_calls():
    """All 4,112 rows of the mixed step (17 chunks of 256 rows, and again in the library's
    default chunks) under the parity rule, compared against the oracle in batches of rows;
    repeated calls are identical."""
    w = workloads.make_workload("mixed")
    first = run_select(w)
    assert first["status"] == 0
    wide = run_select(w, chunk_rows=0)
    assert wide["status"] == 0
    differing = [0, 0]
    for lo in range(0, w.num_rows, 512):
        rows = np.arange(lo, min(w.num_rows, lo + 512), dtype=np.int32)
        ref = oracle_select(w, rows=rows, want_scores=True)
        differing[0] += assert_select_parity(w, first, ref, rows)
        differing[1] += assert_select_parity(w, wide, ref, rows)
    assert max(differing) <= w.num_rows // 50, differing
    for _ in range(2):
        again = run_select(w)
        for k in ("slots", "counts", "token_idx"):
            np.testing.assert_array_equal(again[k], first[k])
