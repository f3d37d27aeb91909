"""Helpers for the GPU tests: run the library through its binding and compare with
the oracle under the parity rules."""

from __future__ import annotations

import numpy as np
import torch

import oracle

DEV = "cuda:0"
TOL = 1e-4   # |gpu score - oracle score| <= TOL * sum |q*k terms| (the selection's stated tolerance)


def lib():
    import sparse_attention_kv_device_gb300 as sel
    return sel


def run_select(w, want_tokens=True, **overrides):
    sel = lib()
    prob = sel.problem_from_workload(w, DEV, **overrides)
    slots = torch.full((w.num_rows, w.out_width), -7, dtype=torch.int32, device=DEV)
    counts = torch.full((w.num_rows,), -7, dtype=torch.int32, device=DEV)
    tok = torch.full_like(slots, -7) if want_tokens else None
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    sel.sel_select(prob, slots, counts, token_idx=tok, status=status)
    torch.cuda.synchronize()
    out = dict(slots=slots.cpu().numpy(), counts=counts.cpu().numpy(), status=int(status.item()))
    if want_tokens:
        out["token_idx"] = tok.cpu().numpy()
    return out


def run_scores(w, rows=None, **overrides):
    sel = lib()
    prob = sel.problem_from_workload(w, DEV, **overrides)
    ld = max(4, ((int(w.max_context) // int(w.kpool)) + 3) // 4 * 4)
    scores = torch.full((w.num_rows, ld), float("nan"), dtype=torch.float32, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    sel.sel_score_paged(prob, scores, status=status)
    torch.cuda.synchronize()
    s = scores.cpu().numpy()
    return (s if rows is None else s[rows]), int(status.item())


def request_of(w, r):
    return int(np.searchsorted(w.qsl, r, side="right") - 1)


def assert_select_bitexact(w, out, ref, rows):
    np.testing.assert_array_equal(out["counts"][rows], ref["counts"])
    np.testing.assert_array_equal(out["token_idx"][rows], ref["token_idx"])
    np.testing.assert_array_equal(out["slots"][rows].astype(np.int64), ref["slots"])


def _slot_of(w, req, t):
    """Validity check of one slot: the block-table formula written out for the test."""
    if t < 0:
        return -1
    b = t // w.block_size
    if b >= w.max_blocks_per_req:
        return -1
    ph = int(w.block_table[req, b])
    if ph < 0 or ph >= w.num_kv_blocks:
        return -1
    return ph * w.block_stride_rows + t % w.block_size


def assert_select_parity(w, out, ref, rows):
    """Normal-valued inputs: rows may differ only by swaps among near-tied pools.

    (a) equal token counts and trailing tokens; (b) every pool in the symmetric
    difference of kept sets lies within B_j + B_K of the K-th oracle score
    (B = TOL * sum |terms|); (c) slots of tokens both sides keep equal the oracle's,
    the others follow the block table; (d) count == non -1 slots.
    Returns the number of rows that differ from the oracle at all.
    """
    K = w.index_topk // w.kpool
    differing = 0
    for k, r in enumerate(rows):
        g_tok, o_tok = out["token_idx"][r], ref["token_idx"][k]
        g_sl, o_sl = out["slots"][r].astype(np.int64), ref["slots"][k]
        assert out["counts"][r] == int((g_sl != -1).sum()), r
        if np.array_equal(g_tok, o_tok):
            np.testing.assert_array_equal(g_sl, o_sl)
            np.testing.assert_array_equal(out["counts"][r], ref["counts"][k])
            continue
        differing += 1
        ctx = int(w.positions[r]) + 1
        assert ctx > w.index_topk, f"row {r}: short rows must match exactly"
        P = ctx // w.kpool
        n_tok = w.index_topk + ctx % w.kpool
        assert (g_tok[:n_tok] >= 0).all() and (g_tok[n_tok:] == -1).all()
        np.testing.assert_array_equal(g_tok[K * w.kpool:n_tok], o_tok[K * w.kpool:n_tok])
        g_pools = set((g_tok[:K * w.kpool:w.kpool] // w.kpool).tolist())
        o_pools = set((o_tok[:K * w.kpool:w.kpool] // w.kpool).tolist())
        assert len(g_pools) == K and max(g_pools) < P
        s, B = ref["scores"][k], TOL * ref["abs_terms"][k]
        kth = min(o_pools, key=lambda j: (s[j], -j))
        for j in g_pools ^ o_pools:
            assert abs(float(s[j]) - float(s[kth])) <= B[j] + B[kth], (r, j, s[j], s[kth])
        req = request_of(w, r)
        o_map = dict(zip(o_tok.tolist(), o_sl.tolist()))
        for t, sl in zip(g_tok.tolist(), g_sl.tolist()):
            want = o_map[t] if t in o_map else _slot_of(w, req, t)
            assert sl == want, (r, t, sl, want)
    return differing


def sample_rows(w, per_request=2, extra=()):
    """First and last rows of every request (and of every 256-row chunk), plus extras."""
    rows = set()
    for i in range(w.num_reqs):
        lo, hi = int(w.qsl[i]), int(w.qsl[i + 1])
        if hi > lo:
            rows.update(range(lo, min(hi, lo + per_request)))
            rows.update(range(max(lo, hi - per_request), hi))
    for c in range(0, w.num_rows, 256):
        rows.update({c, min(w.num_rows - 1, c + 255)})
    rows.update(extra)
    return np.array(sorted(r for r in rows if r < w.num_rows), dtype=np.int32)


def oracle_select(w, rows=None, want_scores=False):
    return oracle.select(w, rows=rows, want_scores=want_scores)
