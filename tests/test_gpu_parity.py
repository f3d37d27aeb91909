"""GPU path (through the C ABI) against the CPU oracle on the same seeded inputs.

Integer-valued workloads and every integer/index step are compared bit for bit;
normal-valued workloads follow the tolerance rule of the selection (scores within
1e-4 * sum|q*k| of the oracle, kept sets equal up to swaps of near-tied pools)."""

import numpy as np
import pytest
import torch

import oracle
import workloads
from _golden import ints, load
from _gpu import (DEV, TOL, assert_select_bitexact, assert_select_parity, lib, oracle_select, run_scores,
                  run_select, sample_rows)

pytestmark = pytest.mark.gpu


# ---------------------------------------------------------------- remap (K-d)
@pytest.mark.parametrize("rows,width,stride", [(1, 4, 64), (37, 2052, 128), (300, 260, 64), (5, 8, 192)])
def test_remap_matches_oracle(rows, width, stride):
    sel = lib()
    rng = np.random.default_rng(rows * 7 + width)
    nreq, nb = 6, 40
    nkv = 300
    bt = rng.permutation(nkv)[:nreq * nb].reshape(nreq, nb).astype(np.int32)
    bt[0, 3] = -2
    bt[1, 5] = nkv + 7
    req = rng.integers(-1, nreq + 1, size=rows).astype(np.int32)   # includes invalid ids
    tok = workloads.random_token_indices(rows, width, (nb + 2) * 64, seed=rows + width)
    mb = nb - 1
    ref_slots, ref_counts = oracle.remap_rows(req, nreq, bt, mb, nkv, tok, 64, stride)
    t = lambda a: torch.from_numpy(a).to(DEV)
    slots = torch.full((rows, width), -7, dtype=torch.int32, device=DEV)
    counts = torch.full((rows,), -7, dtype=torch.int32, device=DEV)
    sel.sel_remap_global(t(req), t(bt), t(tok), slots, num_kv_blocks=nkv, block_size=64,
                         block_stride_rows=stride, max_blocks_per_req=mb, valid_counts=counts)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(slots.cpu().numpy().astype(np.int64), ref_slots)
    np.testing.assert_array_equal(counts.cpu().numpy(), ref_counts)


@pytest.mark.parametrize("mode", ["global", "workspace", "dcp", "dcp_compact"])
@pytest.mark.parametrize("block_size,kpool", [(64, 4), (6, 4), (16, 3), (5, 4)])
def test_remap_modes_on_selection_shaped_tokens(mode, block_size, kpool):
    """Runs of consecutive tokens (the selection's pools): an int4 of four consecutive tokens in
    one block takes one block-table load in the kernel; runs that cross a block, a short pool
    (kpool 3) and tokens past the guarded blocks go token by token. Bit exact in every mode."""
    sel = lib()
    rows, width, nreq, nkv = 61, 2052, 5, 4000
    rng = np.random.default_rng(block_size * 31 + kpool + len(mode))
    nb = 3000 // block_size + 4
    bt = rng.permutation(nkv)[:nreq * nb].reshape(nreq, nb).astype(np.int32) if nreq * nb <= nkv else \
        rng.integers(0, nkv, size=(nreq, nb)).astype(np.int32)
    bt[1, 3] = -1
    bt[2, 7] = nkv + 3
    mb = nb - 2                                   # the last blocks are past max_blocks_per_req
    ctx = rng.integers(1, nb * block_size + 3 * block_size, size=rows)
    ctx[:3] = [1, 2048, nb * block_size]          # a short row, a row at topk, a full table
    tok = workloads.selection_token_indices(ctx, width, topk=kpool * 256, kpool=kpool, seed=block_size + kpool)
    req = rng.integers(-1, nreq + 1, size=rows).astype(np.int32)
    req[:8] = np.arange(8) % nreq
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(DEV)
    slots = torch.full((rows, width), -7, dtype=torch.int32, device=DEV)
    counts = torch.full((rows,), -7, dtype=torch.int32, device=DEV)
    if mode == "global":
        ref_slots, ref_counts = oracle.remap_rows(req, nreq, bt, mb, nkv, tok, block_size, 2 * block_size)
        sel.sel_remap_global(t(req), t(bt), t(tok), slots, num_kv_blocks=nkv, block_size=block_size,
                             block_stride_rows=2 * block_size, max_blocks_per_req=mb, valid_counts=counts)
    elif mode == "workspace":
        wsr = rng.choice(np.array([-1, -1, -1, 0, 1, 5], np.int32), size=rows)
        starts = np.array([0, 90000], np.int32)
        ref_slots, ref_counts = oracle.remap_ws_rows(req, nreq, bt, mb, nkv, wsr, starts, tok, block_size,
                                                     2 * block_size)
        sel.sel_remap_workspace(t(req), t(bt), t(wsr), t(starts), t(tok), slots, num_kv_blocks=nkv,
                                block_size=block_size, block_stride_rows=2 * block_size, max_blocks_per_req=mb,
                                valid_counts=counts)
    else:
        compact = mode == "dcp_compact"
        dcp, rank = 2, 1
        inter = {64: 16, 6: 6, 16: 8, 5: 5}[block_size]   # block_size % interleave == 0 (sel.h)
        ref_slots, ref_counts = oracle.remap_dcp_rows(req, nreq, bt, mb, nkv, tok, block_size, dcp, rank, inter,
                                                      compact)
        sel.sel_remap_dcp(t(req), t(bt), t(tok), slots, num_kv_blocks=nkv, dcp_size=dcp, dcp_rank=rank,
                          interleave=inter, compact=compact, block_size=block_size, max_blocks_per_req=mb,
                          valid_counts=counts)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(slots.cpu().numpy().astype(np.int64), ref_slots)
    np.testing.assert_array_equal(counts.cpu().numpy(), ref_counts)


@pytest.mark.parametrize("dcp,inter,rank", [(4, 4, 3), (3, 4, 1), (8, 64, 5), (4, 16, 1)])
@pytest.mark.parametrize("compact", [False, True])
def test_dcp_remap_on_selection_shaped_tokens(dcp, inter, rank, compact):
    """Pools of four consecutive tokens under DCP: with power-of-two sizes and an interleave of 4
    or more the kernel maps an aligned pool with one ownership test and one table load; a rank
    count of 3 takes the division path. Guarded blocks included; bit exact against the oracle."""
    sel = lib()
    rows, width, nreq, nkv, bs = 67, 2052, 5, 6000, 64
    rng = np.random.default_rng(dcp * 100 + inter + rank)
    nb = 1100
    bt = rng.integers(0, nkv, size=(nreq, nb)).astype(np.int32)
    bt[1, 3] = -1
    bt[2, 7] = nkv + 3
    mb = nb - 2
    ctx = rng.integers(1, nb * bs * dcp, size=rows)
    ctx[:3] = [1, 2048, nb * bs * dcp]
    tok = workloads.selection_token_indices(ctx, width, topk=2048, kpool=4, seed=dcp + inter)
    req = rng.integers(-1, nreq + 1, size=rows).astype(np.int32)
    req[:8] = np.arange(8) % nreq
    ref_slots, ref_counts = oracle.remap_dcp_rows(req, nreq, bt, mb, nkv, tok, bs, dcp, rank, inter, compact)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(DEV)
    slots = torch.full((rows, width), -7, dtype=torch.int32, device=DEV)
    counts = torch.full((rows,), -7, dtype=torch.int32, device=DEV)
    sel.sel_remap_dcp(t(req), t(bt), t(tok), slots, num_kv_blocks=nkv, dcp_size=dcp, dcp_rank=rank,
                      interleave=inter, compact=compact, block_size=bs, max_blocks_per_req=mb,
                      valid_counts=counts)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(slots.cpu().numpy().astype(np.int64), ref_slots)
    np.testing.assert_array_equal(counts.cpu().numpy(), ref_counts)


@pytest.mark.parametrize("width", [3000, 5124])
@pytest.mark.parametrize("compact", [False, True])
@pytest.mark.parametrize("shape", ["selection", "random"])
def test_dcp_remap_rows_of_several_rounds(width, compact, shape):
    """Rows wider than one round of the kernel (2,560 tokens): the compaction's warp totals
    alternate between two buffers by round, and past 4,096 columns the compacted row goes
    straight to global memory instead of through shared memory. Bit exact against the oracle."""
    sel = lib()
    rows, nreq, nkv, bs, dcp, inter, rank = 37, 4, 9000, 64, 4, 16, 1
    rng = np.random.default_rng(width + compact + len(shape))
    nb = 2100
    bt = rng.integers(0, nkv, size=(nreq, nb)).astype(np.int32)
    bt[0, 5] = -1
    bt[3, 11] = nkv + 2
    mb = nb - 2
    if shape == "selection":
        ctx = rng.integers(1, nb * bs * dcp, size=rows)
        ctx[:2] = [nb * bs * dcp, 3 * width]
        tok = workloads.selection_token_indices(ctx, width, topk=4 * ((width - 4) // 4), kpool=4, seed=width)
    else:
        tok = workloads.random_token_indices(rows, width, nb * bs * dcp + 100, seed=width)
    req = rng.integers(-1, nreq + 1, size=rows).astype(np.int32)
    req[:6] = np.arange(6) % nreq
    ref_slots, ref_counts = oracle.remap_dcp_rows(req, nreq, bt, mb, nkv, tok, bs, dcp, rank, inter, compact)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(DEV)
    slots = torch.full((rows, width), -7, dtype=torch.int32, device=DEV)
    counts = torch.full((rows,), -7, dtype=torch.int32, device=DEV)
    sel.sel_remap_dcp(t(req), t(bt), t(tok), slots, num_kv_blocks=nkv, dcp_size=dcp, dcp_rank=rank,
                      interleave=inter, compact=compact, block_size=bs, max_blocks_per_req=mb,
                      valid_counts=counts)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(slots.cpu().numpy().astype(np.int64), ref_slots)
    np.testing.assert_array_equal(counts.cpu().numpy(), ref_counts)


def test_remap_golden_worked_example():
    sel = lib()
    g = load("remap_worked_example.txt")
    bt = np.stack([ints(g, "block_table_row0"), ints(g, "block_table_row1")]).astype(np.int32)
    tok = np.stack([ints(g, "tokens_row0"), ints(g, "tokens_row1")]).astype(np.int32)
    tok = np.concatenate([tok, np.full((2, 3), -1, np.int32)], axis=1)   # width 8 (multiple of 4)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(DEV)
    for key, stride in (("slots", int(g["stride"][0])), ("slots_b", int(g["stride_b"][0]))):
        slots = torch.empty((2, 8), dtype=torch.int32, device=DEV)
        counts = torch.empty(2, dtype=torch.int32, device=DEV)
        sel.sel_remap_global(t(ints(g, "req_id").astype(np.int32)), t(bt), t(tok), slots,
                             num_kv_blocks=int(g["num_kv_blocks"][0]), block_size=int(g["block_size"][0]),
                             block_stride_rows=stride, max_blocks_per_req=int(g["max_blocks"][0]),
                             valid_counts=counts)
        torch.cuda.synchronize()
        got = slots.cpu().numpy()
        np.testing.assert_array_equal(got[0, :5], ints(g, f"{key}_row0"))
        np.testing.assert_array_equal(got[1, :5], ints(g, f"{key}_row1"))
        np.testing.assert_array_equal(counts.cpu().numpy(), ints(g, "counts"))


@pytest.mark.parametrize("rows,width", [(1, 4), (37, 2052), (300, 260), (4112, 2052)])
def test_workspace_remap_matches_oracle(rows, width):
    """Decode rows, prefill rows of 3 requests and rows with a bad prefill id, bit exact."""
    sel = lib()
    rng = np.random.default_rng(rows * 11 + width)
    nreq, nb, nkv = 6, 40, 300
    bt = rng.permutation(nkv)[:nreq * nb].reshape(nreq, nb).astype(np.int32)
    bt[2, 7] = -5
    req = rng.integers(-1, nreq + 1, size=rows).astype(np.int32)
    wsr = rng.choice(np.array([-1, -1, 0, 1, 2, 3, -2], np.int32), size=rows)   # 3 and -2: out of range
    starts = np.array([0, 70000, 140000], np.int32)
    tok = workloads.random_token_indices(rows, width, (nb + 2) * 64, seed=rows + 3 * width)
    ref_slots, ref_counts = oracle.remap_ws_rows(req, nreq, bt, nb - 1, nkv, wsr, starts, tok, 64, 128)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(DEV)
    slots = torch.full((rows, width), -7, dtype=torch.int32, device=DEV)
    counts = torch.full((rows,), -7, dtype=torch.int32, device=DEV)
    sel.sel_remap_workspace(t(req), t(bt), t(wsr), t(starts), t(tok), slots, num_kv_blocks=nkv, block_size=64,
                            block_stride_rows=128, max_blocks_per_req=nb - 1, valid_counts=counts)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(slots.cpu().numpy().astype(np.int64), ref_slots)
    np.testing.assert_array_equal(counts.cpu().numpy(), ref_counts)


def test_workspace_remap_golden_worked_example():
    sel = lib()
    g = load("workspace_worked_example.txt")
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(DEV)
    tok = np.stack([ints(g, f"tokens_row{r}") for r in range(4)])
    slots = torch.empty((4, 4), dtype=torch.int32, device=DEV)
    counts = torch.empty(4, dtype=torch.int32, device=DEV)
    sel.sel_remap_workspace(t(ints(g, "req_id")), t(ints(g, "block_table_row0")[None, :]), t(ints(g, "ws_req")),
                            t(ints(g, "ws_starts")), t(tok), slots, num_kv_blocks=int(g["num_kv_blocks"][0]),
                            block_size=int(g["block_size"][0]), block_stride_rows=int(g["stride"][0]),
                            max_blocks_per_req=int(g["max_blocks"][0]), valid_counts=counts)
    torch.cuda.synchronize()
    for r in range(4):
        np.testing.assert_array_equal(slots.cpu().numpy()[r], ints(g, f"slots_row{r}"))
    np.testing.assert_array_equal(counts.cpu().numpy(), ints(g, "counts"))


@pytest.mark.parametrize("dcp,inter,rank", [(1, 1, 0), (2, 1, 1), (2, 4, 0), (4, 16, 3), (8, 64, 5)])
@pytest.mark.parametrize("compact", [False, True])
@pytest.mark.parametrize("rows,width", [(7, 260), (4112, 2052)])
def test_dcp_remap_matches_oracle(dcp, inter, rank, compact, rows, width):
    """One DCP rank's filtered (and compacted) slots, bit exact, with guarded blocks."""
    sel = lib()
    rng = np.random.default_rng(dcp * 1000 + inter * 10 + rank + rows)
    nreq, nb, nkv = 5, 48, 400
    bt = rng.permutation(nkv)[:nreq * nb].reshape(nreq, nb).astype(np.int32)
    bt[1, 2] = -1
    bt[3, 9] = nkv + 1
    req = rng.integers(-1, nreq + 1, size=rows).astype(np.int32)
    tok = workloads.random_token_indices(rows, width, nb * 64 * dcp + 200, seed=rows + dcp + inter)
    ref_slots, ref_counts = oracle.remap_dcp_rows(req, nreq, bt, nb - 2, nkv, tok, 64, dcp, rank, inter, compact)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(DEV)
    slots = torch.full((rows, width), -7, dtype=torch.int32, device=DEV)
    counts = torch.full((rows,), -7, dtype=torch.int32, device=DEV)
    sel.sel_remap_dcp(t(req), t(bt), t(tok), slots, num_kv_blocks=nkv, dcp_size=dcp, dcp_rank=rank,
                      interleave=inter, compact=compact, block_size=64, max_blocks_per_req=nb - 2,
                      valid_counts=counts)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(slots.cpu().numpy().astype(np.int64), ref_slots)
    np.testing.assert_array_equal(counts.cpu().numpy(), ref_counts)


def test_dcp_remap_golden_worked_example():
    sel = lib()
    g = load("dcp_worked_example.txt")
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(DEV)
    tok = np.stack([ints(g, f"tokens_row{r}") for r in range(3)])
    bt = np.stack([ints(g, "block_table_row0"), ints(g, "block_table_row1")])
    kw = dict(num_kv_blocks=int(g["num_kv_blocks"][0]), dcp_size=int(g["dcp_size"][0]),
              interleave=int(g["interleave"][0]), block_size=int(g["block_size"][0]),
              max_blocks_per_req=int(g["max_blocks"][0]))
    for rank, compact, key in ((0, False, "rank0_row"), (1, False, "rank1_row"), (0, True, "rank0_compact_row")):
        slots = torch.empty((3, 8), dtype=torch.int32, device=DEV)
        counts = torch.empty(3, dtype=torch.int32, device=DEV)
        sel.sel_remap_dcp(t(ints(g, "req_id")), t(bt), t(tok), slots, dcp_rank=rank, compact=compact,
                          valid_counts=counts, **kw)
        torch.cuda.synchronize()
        for r in range(3):
            np.testing.assert_array_equal(slots.cpu().numpy()[r], ints(g, f"{key}{r}"), err_msg=key)
        np.testing.assert_array_equal(counts.cpu().numpy(), ints(g, f"rank{rank}_counts"))


# ---------------------------------------------------------------- top-k + expansion (K-c)
TOPK_CASES = [
    # (topk, kpool, contexts)                          exercises
    (256, 4, [1, 7, 255, 256, 257, 258, 259, 1000, 3001]),        # short rows, trailing pools
    (2048, 4, [2049, 4096, 32765, 32768, 32769]),                 # one CTA per row
    (2048, 4, [131068, 131069, 131070, 131071, 131072]),         # 128K rows
    (2048, 4, [262144, 200001, 4000, 2000, 0]),                   # 256K rows, ragged
    (2048, 4, [400003]),                                          # 100,000 pools in one row
    (60, 3, [59, 60, 61, 62, 1000, 5000]),                        # kpool 3 (scalar stores)
    (16, 1, [16, 17, 50, 20000]),                                 # kpool 1: a plain top-k
]


@pytest.mark.parametrize("ties", ["none", "coarse", "zeros", "inf"])
@pytest.mark.parametrize("case", range(len(TOPK_CASES)))
def test_topk_expand_matches_oracle(case, ties):
    sel = lib()
    topk, kpool, ctxs = TOPK_CASES[case]
    ctx = np.array(ctxs, dtype=np.int64)
    W = ((topk + kpool - 1) + 3) // 4 * 4
    ld = max(4, (int(ctx.max()) // kpool + 3) // 4 * 4)
    scores = workloads.random_scores(len(ctx), ld, seed=100 * case + len(ties), ties=ties)
    ref_tok, ref_cnt = oracle.topk_expand_rows(scores, ctx, topk, kpool, W)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(DEV)
    tok = torch.full((len(ctx), W), -7, dtype=torch.int32, device=DEV)
    cnt = torch.full((len(ctx),), -7, dtype=torch.int32, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    sel.sel_topk_expand(t(scores), t((ctx - 1).astype(np.int32)), topk, kpool, tok, cnt, status=status)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(tok.cpu().numpy(), ref_tok)
    np.testing.assert_array_equal(cnt.cpu().numpy(), ref_cnt)
    assert int(status.item()) == 0


def test_topk_rows_beyond_scores_are_out_of_bound():
    sel = lib()
    scores = workloads.random_scores(2, 1024, seed=3)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(DEV)
    tok = torch.full((2, 260), -7, dtype=torch.int32, device=DEV)
    cnt = torch.full((2,), -7, dtype=torch.int32, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    # ctx 4,101 has 1,025 complete pools: one more than the 1,024 score columns
    sel.sel_topk_expand(t(scores), t(np.array([4095, 4100], np.int32)), 256, 4, tok, cnt, status=status)
    torch.cuda.synchronize()
    got = tok.cpu().numpy()
    assert (got[1] == -1).all() and int(cnt[1].item()) == 0
    assert int(status.item()) & 2
    ref, _ = oracle.topk_expand_rows(scores[:1], np.array([4096]), 256, 4, 260)
    np.testing.assert_array_equal(got[0], ref[0])


# ---------------------------------------------------------------- scorer (K-b)
@pytest.mark.parametrize("name", ["tiny", "decode32k"])
def test_scores_integer_exact(name):
    w = workloads.make_workload(name)
    gs, st = run_scores(w)
    os_, _, ost = oracle.score_rows(w, scores_ld=gs.shape[1])
    assert st == ost == 0
    for r in range(w.num_rows):
        P = (int(w.positions[r]) + 1) // w.kpool
        np.testing.assert_array_equal(gs[r, :P], os_[r, :P])


@pytest.mark.parametrize("name", ["decode128k", "ragged", "mixed"])
def test_scores_normal_within_tolerance(name):
    w = workloads.make_workload(name)
    rows = sample_rows(w, per_request=1)
    gs, st = run_scores(w)
    os_, ab, _ = oracle.score_rows(w, rows=rows, scores_ld=gs.shape[1])
    for k, r in enumerate(rows):
        P = (int(w.positions[r]) + 1) // w.kpool
        err = np.abs(gs[r, :P].astype(np.float64) - os_[k, :P].astype(np.float64))
        assert (err <= TOL * ab[k, :P]).all(), (name, r, float((err / np.maximum(ab[k, :P], 1e-30)).max()))


# ---------------------------------------------------------------- the fused path
@pytest.mark.parametrize("name", ["tiny", "decode32k"])
def test_select_integer_bitexact(name):
    w = workloads.make_workload(name)
    out = run_select(w)
    ref = oracle_select(w)
    assert out["status"] == ref["status"] == 0
    assert_select_bitexact(w, out, ref, np.arange(w.num_rows))


@pytest.mark.parametrize("name", ["decode128k", "ragged", "ragged_b", "mixed"])
def test_select_normal_parity(name):
    w = workloads.make_workload(name)
    out = run_select(w)
    rows = np.arange(w.num_rows, dtype=np.int32) if w.num_rows <= 64 else sample_rows(w)
    ref = oracle_select(w, rows=rows, want_scores=True)
    assert out["status"] == ref["status"]
    differing = assert_select_parity(w, out, ref, rows)
    assert differing <= max(1, len(rows) // 4), differing
    if name == "ragged":
        # the guarded blocks are -1 in place; counts follow the non -1 slots
        assert (out["counts"] <= w.index_topk + w.kpool - 1).all()


@pytest.mark.parametrize("name", ["decode128k", "mixed_head"])
def test_select_every_row_and_repeat_calls(name):
    """Every row (not a sample) follows the parity rule, and repeated calls in one process
    give identical outputs: a race inside a tail kernel shows up as rows that change."""
    if name == "mixed_head":   # the first 256 rows of the mixed workload as one chunk
        w = workloads.build_workload([[131072]] * 16 + [list(range(60001, 60241))], name=name, seed=1005,
                                     integer_mode=False)
    else:
        w = workloads.make_workload(name)
    rows = np.arange(w.num_rows, dtype=np.int32)
    ref = oracle_select(w, rows=rows, want_scores=True)
    first = run_select(w)
    differing = assert_select_parity(w, first, ref, rows)
    assert differing <= max(1, len(rows) // 50), differing
    for _ in range(3):
        again = run_select(w)
        for k in ("slots", "counts", "token_idx"):
            np.testing.assert_array_equal(again[k], first[k])


def test_select_long_rows():
    """300K context: rows of 75,000 pools, more than the row kernel stages in shared memory
    (the rest is read from L2); integer mode, bit exact."""
    w = workloads.build_workload([[300000, 300003], [40000], [2100]], name="long", seed=21, integer_mode=True)
    assert w.max_context // w.kpool > 32768
    out = run_select(w)
    ref = oracle_select(w)
    assert out["status"] == ref["status"] == 0
    assert_select_bitexact(w, out, ref, np.arange(w.num_rows))


@pytest.mark.parametrize("long_rows", [False, True])
def test_select_all_scores_tied(long_rows):
    """q = 0 makes every score 0.0: the lowest-index K pools are kept (staged and L2 rows)."""
    ctx = 300001 if long_rows else 40001
    w = workloads.build_workload([[ctx - 1], [ctx - 2, ctx - 1]], name="ties", seed=22, integer_mode=True)
    w.q[:] = 0
    out = run_select(w)
    ref = oracle_select(w)
    assert_select_bitexact(w, out, ref, np.arange(w.num_rows))
    K = w.index_topk // w.kpool
    assert (out["token_idx"][:, :K * w.kpool] == np.arange(K * w.kpool)).all()


@pytest.mark.parametrize("seg_rows,chunk_rows", [(1, 0), (2, 0), (3, 5), (4, 1), (64, 3), (0, 7)])
def test_segmentation_invariance(seg_rows, chunk_rows):
    """Integer mode: outputs do not depend on how rows are cut into segments or chunks."""
    w = workloads.make_workload("decode32k")
    ref = oracle_select(w)
    out = run_select(w, segment_rows=seg_rows, chunk_rows=chunk_rows)
    assert_select_bitexact(w, out, ref, np.arange(w.num_rows))


@pytest.mark.parametrize("case", ["chunk_of_1100_rows", "2100_requests"])
def test_select_large_first_chunk_waits_for_the_builder(case):
    """A first chunk of more than 1,024 rows, or a call with more than 2,048 requests, is too
    large for the scorer to plan itself: it takes the builder's plan. Later chunks read their
    plans while the previous chunk's select runs. Integer mode, every row bit exact."""
    if case == "chunk_of_1100_rows":
        w = workloads.build_workload([list(range(3000, 4100))], name=case, seed=31, integer_mode=True,
                                     index_topk=256)
        out = run_select(w, chunk_rows=2048)
    else:
        rng = np.random.default_rng(32)
        w = workloads.build_workload([[int(c)] for c in rng.integers(200, 1200, size=2100)], name=case, seed=32,
                                     integer_mode=True, index_topk=256)
        out = run_select(w)
    ref = oracle_select(w)
    assert out["status"] == ref["status"] == 0
    assert_select_bitexact(w, out, ref, np.arange(w.num_rows))


def test_select_rows_longer_than_the_stage_bit_exact():
    """Rows with more pools than the row select stages in shared memory (32,768 keys): 200K and
    256K rows and a 400K row (100,000 pools), whose keys past the stage are read from global
    memory in every phase. Integer mode (many equal scores, so the lowest-index rule decides at
    the threshold): every row bit exact."""
    w = workloads.build_workload([[262144], [200001, 200003], [400003]], name="long", seed=77,
                                 integer_mode=True, index_topk=2048)
    out = run_select(w)
    ref = oracle_select(w)
    assert out["status"] == ref["status"] == 0
    assert_select_bitexact(w, out, ref, np.arange(w.num_rows))


def test_batching_invariance():
    """A request selected alone or inside a batch gives the same rows."""
    full = workloads.build_workload([list(range(5000, 5005)), [9000, 9001], [300]], name="b", seed=8,
                                    integer_mode=True, index_topk=256)
    out = run_select(full)
    for i in range(full.num_reqs):
        lo, hi = int(full.qsl[i]), int(full.qsl[i + 1])
        ref = oracle_select(full, rows=np.arange(lo, hi, dtype=np.int32))
        np.testing.assert_array_equal(out["token_idx"][lo:hi], ref["token_idx"])
        np.testing.assert_array_equal(out["slots"][lo:hi].astype(np.int64), ref["slots"])


def test_padding_rows_and_empty_batch():
    w = workloads.build_workload([[3000], [100, 101]], name="pad", seed=5, integer_mode=True,
                                 index_topk=256, pad_rows=3)
    out = run_select(w)
    ref = oracle_select(w)
    assert_select_bitexact(w, out, ref, np.arange(w.num_rows))
    assert (out["slots"][3:] == -1).all() and (out["counts"][3:] == 0).all()
    sel = lib()
    prob = sel.problem_from_workload(w, DEV, num_rows=0)
    e = torch.empty((0, w.out_width), dtype=torch.int32, device=DEV)
    sel.sel_select(prob, e, torch.empty(0, dtype=torch.int32, device=DEV))


def test_status_bits_and_guards():
    w = workloads.build_workload([[3000, 3001], [2500]], name="st", seed=4, integer_mode=True,
                                 index_topk=256, kpool=4, max_context=3000)
    w.key_page_table[0, 5] = w.num_key_pages + 3
    out = run_select(w)
    ref = oracle_select(w)
    assert out["status"] == ref["status"] == 3
    assert_select_bitexact(w, out, ref, np.arange(w.num_rows))
    gs, st = run_scores(w)
    assert st & 1 and np.isneginf(gs[0, 5 * 64:6 * 64]).all()
    w.qsl[1] = 5
    out2 = run_select(w)
    assert out2["status"] & 8
    assert (out2["slots"] == -1).all() and (out2["counts"] == 0).all()


def test_output_guard_canaries():
    """Outputs embedded in larger buffers: nothing is written outside them."""
    sel = lib()
    w = workloads.make_workload("tiny")
    prob = sel.problem_from_workload(w, DEV)
    G = 1024
    canary = 0x5A5A5A5A
    n = w.num_rows * w.out_width
    big = torch.full((n + 2 * G,), canary, dtype=torch.int32, device=DEV)
    bigc = torch.full((w.num_rows + 2 * G,), canary, dtype=torch.int32, device=DEV)
    bigt = torch.full((n + 2 * G,), canary, dtype=torch.int32, device=DEV)
    ws_n = sel.sel_workspace_bytes(prob)
    ws = torch.full((ws_n + 2 * 4096,), 0x3C, dtype=torch.uint8, device=DEV)
    ws[4096:4096 + ws_n] = 0   # the workspace itself starts zero-filled
    slots = big[G:G + n].view(w.num_rows, w.out_width)
    tok = bigt[G:G + n].view(w.num_rows, w.out_width)
    sel.sel_select(prob, slots, bigc[G:G + w.num_rows], token_idx=tok, ws=ws[4096:4096 + ws_n])
    torch.cuda.synchronize()
    for b in (big, bigc, bigt):
        h = b.cpu().numpy()
        assert (h[:G] == canary).all() and (h[-G:] == canary).all()
    wsh = ws.cpu().numpy()
    assert (wsh[:4096] == 0x3C).all() and (wsh[-4096:] == 0x3C).all()
    ref = oracle_select(w)
    np.testing.assert_array_equal(slots.cpu().numpy().astype(np.int64), ref["slots"])


def test_graph_replay_after_inplace_changes():
    """Capture once, change queries, keys, positions and tables in place, replay."""
    sel = lib()
    w = workloads.make_workload("decode32k")
    prob = sel.problem_from_workload(w, DEV)
    qsl_d, pos_d, q_d, kc_d, kpt_d, bt_d = prob.tensors
    slots = torch.empty((w.num_rows, w.out_width), dtype=torch.int32, device=DEV)
    counts = torch.empty(w.num_rows, dtype=torch.int32, device=DEV)
    tok = torch.empty_like(slots)
    ws = sel.new_workspace(sel.sel_workspace_bytes(prob), DEV)
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        sel.sel_select(prob, slots, counts, token_idx=tok, ws=ws)   # warm-up outside capture
    stream.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        sel.sel_select(prob, slots, counts, token_idx=tok, ws=ws)
    rng = np.random.default_rng(99)
    for step in range(3):
        w.q[:] = rng.integers(-3, 4, size=w.q.shape).astype(np.float16)
        kcv = w.key_cache.reshape(w.num_key_pages, 64, 128)
        live = np.unique(w.key_page_table[w.key_page_table >= 0])
        kcv[live[: len(live) // 2]] = rng.integers(-3, 4, size=(len(live) // 2, 64, 128)).astype(np.float16)
        w.positions[:] = w.positions - step   # contexts shrink: 32,766-step ..
        perm = rng.permutation(w.num_kv_blocks).astype(np.int32)
        valid = w.block_table >= 0
        w.block_table[valid] = perm[w.block_table[valid]]
        q_d.copy_(torch.from_numpy(w.q))
        kc_d.copy_(torch.from_numpy(w.key_cache))
        pos_d.copy_(torch.from_numpy(w.positions))
        bt_d.copy_(torch.from_numpy(w.block_table))
        g.replay()
        torch.cuda.synchronize()
        ref = oracle_select(w)
        out = dict(slots=slots.cpu().numpy(), counts=counts.cpu().numpy(), token_idx=tok.cpu().numpy())
        assert_select_bitexact(w, out, ref, np.arange(w.num_rows))


@pytest.mark.parametrize("pinned", [True, False])
def test_select_host_path_matches_device(pinned):
    """Pinned host buffers go through one staging kernel each way; pageable ones through the
    copy engine. Both give the oracle's slots and counts."""
    sel = lib()
    w = workloads.make_workload("tiny")
    dprob = sel.problem_from_workload(w, DEV)
    if pinned:
        hp = lambda a: torch.from_numpy(np.ascontiguousarray(a)).pin_memory()
    else:
        hp = lambda a: torch.from_numpy(np.ascontiguousarray(a).copy())
    hprob = sel.Problem(query_start_loc=hp(w.qsl), positions=hp(w.positions), q=hp(w.q),
                        key_cache=dprob.tensors[3], key_page_table=hp(w.key_page_table),
                        block_table=hp(w.block_table), index_topk=w.index_topk, kpool=w.kpool,
                        max_context=w.max_context, key_page_stride=w.key_page_stride,
                        num_key_pages=w.num_key_pages, num_kv_blocks=w.num_kv_blocks,
                        block_stride_rows=w.block_stride_rows, max_q_len=w.max_q_len,
                        host_inputs=True)
    slots_h = torch.empty((w.num_rows, w.out_width), dtype=torch.int32)
    counts_h = torch.empty(w.num_rows, dtype=torch.int32)
    if pinned:
        slots_h, counts_h = slots_h.pin_memory(), counts_h.pin_memory()
    stage = torch.empty(sel.sel_host_stage_bytes(hprob, w.out_width), dtype=torch.uint8, device=DEV)
    ws = sel.new_workspace(sel.sel_workspace_bytes(dprob), DEV)
    sel.sel_select_host(hprob, slots_h, counts_h, stage, ws)
    torch.cuda.synchronize()
    ref = oracle_select(w)
    np.testing.assert_array_equal(slots_h.numpy().astype(np.int64), ref["slots"])
    np.testing.assert_array_equal(counts_h.numpy(), ref["counts"])


def test_trace_events_time_the_kernels():
    sel = lib()
    w = workloads.make_workload("decode32k")
    prob = sel.problem_from_workload(w, DEV)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
    slots = torch.empty((w.num_rows, w.out_width), dtype=torch.int32, device=DEV)
    counts = torch.empty(w.num_rows, dtype=torch.int32, device=DEV)
    sel.sel_set_trace_events(ev)
    try:
        sel.sel_select(prob, slots, counts)
    finally:
        sel.sel_set_trace_events(None)
    torch.cuda.synchronize()
    assert all(ev[i].elapsed_time(ev[i + 1]) > 0 for i in range(3))


def test_launch_count_one_builder_then_two_per_chunk():
    sel = lib()
    for name, chunks in (("decode128k", 1), ("tiny", 1), ("mixed", 17)):
        w = workloads.make_workload(name)
        assert sel.sel_select_launch_count(sel.problem_from_workload(w, DEV)) == 1 + 2 * chunks, name
    # the library's own chunking (chunk_rows 0): four times the SM count here, fewer chunks
    sms = torch.cuda.get_device_properties(DEV).multi_processor_count
    w = workloads.make_workload("mixed")
    wide = sel.problem_from_workload(w, DEV, chunk_rows=0)
    assert sel.sel_select_launch_count(wide) == 1 + 2 * -(-w.num_rows // (4 * sms))


@pytest.mark.parametrize("fill", ["ones", "one_word", "random"])
def test_select_workspace_needs_no_initialisation(fill):
    """The workspace needs no initialisation: the builder rewrites each chunk's plan header and
    tile counter before any scorer draws from it. A workspace of any prior content (all bits
    set; one repeated word; random bytes) gives bit-exact rows on the first call and on the
    calls after it, in one chunk or three."""
    sel = lib()
    w = workloads.build_workload([list(range(20000, 20005)), [9000, 9001, 9002], [70000], [4100, 4101]],
                                 name="ws", seed=41, integer_mode=True, index_topk=512)
    ref = oracle_select(w)
    for chunk_rows in (0, 4):
        prob = sel.problem_from_workload(w, DEV, chunk_rows=chunk_rows)
        n = sel.sel_workspace_bytes(prob)
        if fill == "ones":
            ws = torch.full((n,), 0xFF, dtype=torch.uint8, device=DEV)
        elif fill == "one_word":
            ws = torch.full(((n + 3) // 4,), 0x6A09E667, dtype=torch.int32, device=DEV).view(torch.uint8)
        else:
            g = torch.Generator(device="cpu").manual_seed(43)
            ws = torch.randint(0, 256, (n,), dtype=torch.uint8, generator=g).to(DEV)
        for _ in range(3):
            slots = torch.full((w.num_rows, w.out_width), -7, dtype=torch.int32, device=DEV)
            counts = torch.full((w.num_rows,), -7, dtype=torch.int32, device=DEV)
            tok = torch.full_like(slots, -7)
            status = torch.zeros(1, dtype=torch.int32, device=DEV)
            sel.sel_select(prob, slots, counts, token_idx=tok, status=status, ws=ws)
            torch.cuda.synchronize()
            out = dict(slots=slots.cpu().numpy(), counts=counts.cpu().numpy(), token_idx=tok.cpu().numpy(),
                       status=int(status.item()))
            assert out["status"] == 0
            assert_select_bitexact(w, out, ref, np.arange(w.num_rows))


def test_select_refuses_a_misaligned_workspace():
    """The plan records are read as 16-byte vectors: a workspace that is not 16-B aligned is
    refused with SEL_EUNSUPPORTED before anything is queued, by both entry points that take one."""
    sel = lib()
    w = workloads.make_workload("tiny")
    prob = sel.problem_from_workload(w, DEV)
    n = sel.sel_workspace_bytes(prob)
    base = torch.zeros(n + 64, dtype=torch.uint8, device=DEV)
    slots = torch.full((w.num_rows, w.out_width), -7, dtype=torch.int32, device=DEV)
    counts = torch.full((w.num_rows,), -7, dtype=torch.int32, device=DEV)
    with pytest.raises(sel.SelError) as e:
        sel.sel_select(prob, slots, counts, ws=base[8:8 + n])
    assert e.value.code == -2  # SEL_EUNSUPPORTED
    torch.cuda.synchronize()
    assert (slots == -7).all() and (counts == -7).all()
    ld = max(4, ((int(w.max_context) // int(w.kpool)) + 3) // 4 * 4)
    scores = torch.zeros((w.num_rows, ld), dtype=torch.float32, device=DEV)
    ns = sel.sel_score_workspace_bytes(prob)
    with pytest.raises(sel.SelError) as e:
        sel.sel_score_paged(prob, scores, ws=base[4:4 + ns])
    assert e.value.code == -2  # SEL_EUNSUPPORTED
    # the host-buffer entry point: a misaligned staging area or workspace is refused before
    # any input is copied or any output written
    hp = lambda x: torch.from_numpy(np.ascontiguousarray(x)).pin_memory()
    hprob = sel.Problem(query_start_loc=hp(w.qsl), positions=hp(w.positions), q=hp(w.q),
                        key_cache=prob.tensors[3], key_page_table=hp(w.key_page_table),
                        block_table=hp(w.block_table), index_topk=w.index_topk, kpool=w.kpool,
                        max_context=w.max_context, key_page_stride=w.key_page_stride,
                        num_key_pages=w.num_key_pages, num_kv_blocks=w.num_kv_blocks,
                        block_stride_rows=w.block_stride_rows, max_q_len=w.max_q_len,
                        host_inputs=True)
    slots_h = torch.full((w.num_rows, w.out_width), -7, dtype=torch.int32).pin_memory()
    counts_h = torch.full((w.num_rows,), -7, dtype=torch.int32).pin_memory()
    nst = sel.sel_host_stage_bytes(hprob, w.out_width)
    stage_base = torch.zeros(nst + 64, dtype=torch.uint8, device=DEV)
    for stage, ws in ((stage_base[4:4 + nst], base[:n]), (stage_base[:nst], base[8:8 + n])):
        with pytest.raises(sel.SelError) as e:
            sel.sel_select_host(hprob, slots_h, counts_h, stage, ws)
        assert e.value.code == -2  # SEL_EUNSUPPORTED
    torch.cuda.synchronize()
    assert (slots_h == -7).all() and (counts_h == -7).all()
