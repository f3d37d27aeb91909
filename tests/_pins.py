"""Pins for the CPU oracle: checks against facts the pages and the mathematics fix.

Each function takes the oracle module (or a stand-in loaded from a mutated build)
and raises AssertionError when the oracle disagrees with an independent fact:
an exact integer computation, an IEEE decoding done by numpy, a library sort, a
closed form from the pages, or an invariant of the remap.
"""

from __future__ import annotations

import numpy as np

import workloads


def pin_half_decode(orc):
    """fp16 decoding of all 65,536 bit patterns equals numpy's binary16 conversion."""
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    got = orc.half_to_float(bits)
    ref = bits.view(np.float16).astype(np.float32)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan].view(np.uint32), ref[~nan].view(np.uint32))


def pin_score_integer_exact(orc, seed=7, n=64):
    """Integer-valued q, k: the fp32 score equals the exact int64 dot product
    sum_h sum_d q[h,d] k[d] (|score| <= 4*128*9 < 2^24, so fp32 is exact)."""
    rng = np.random.default_rng(seed)
    for i in range(n):
        qi = rng.integers(-3, 4, size=(4, 128))
        ki = rng.integers(-3, 4, size=128)
        if i == 0:   # extreme: every term +9
            qi = np.full((4, 128), 3)
            ki = np.full(128, 3)
        if i == 1:   # head-dependent signs: a dropped or repeated head shows
            qi = np.stack([np.full(128, 3), np.full(128, -1), np.full(128, 2), np.full(128, 1)])
            ki = rng.integers(1, 4, size=128)
        exact = int((qi.astype(np.int64) * ki.astype(np.int64)[None, :]).sum())
        s, a = orc.pool_score(qi.astype(np.float16), ki.astype(np.float16))
        assert s == float(exact), (i, s, exact)
        assert a == float(np.abs(qi * ki[None, :]).sum())


def pin_score_normal_bound(orc, seed=11, n=32):
    """Normal values: |s32 - exact| <= (n-1) u sum|terms| (sequential fp32 bound,
    u = 2^-24, n = 512 terms), well inside the 1e-4 sum|terms| tolerance; and the
    reported sum |q*k| equals the fp64 value."""
    rng = np.random.default_rng(seed)
    for _ in range(n):
        q = (rng.standard_normal((4, 128)) / np.sqrt(128)).astype(np.float16)
        k = (rng.standard_normal(128) / np.sqrt(128)).astype(np.float16)
        terms = q.astype(np.float64) * k.astype(np.float64)[None, :]
        exact = terms.sum()
        absum = np.abs(terms).sum()
        s, a = orc.pool_score(q, k)
        assert abs(s - exact) <= 511 * 2.0 ** -24 * absum + 1e-30
        assert abs(a - absum) <= 1e-12 * absum


def _check_topk_characterisation(scores, K, got):
    P = scores.size
    got = np.asarray(got)
    assert got.size == min(K, P)
    assert np.all(np.diff(got) > 0), "ascending, distinct"
    assert got.size == 0 or (got[0] >= 0 and got[-1] < P)
    chosen = np.zeros(P, dtype=bool)
    chosen[got] = True
    s_in = scores[chosen]
    i_in = np.nonzero(chosen)[0]
    s_out = scores[~chosen]
    i_out = np.nonzero(~chosen)[0]
    if s_in.size and s_out.size:
        # every kept pool beats every dropped one: higher score, or equal and lower index
        better = (s_in[:, None] > s_out[None, :]) | (
            (s_in[:, None] == s_out[None, :]) & (i_in[:, None] < i_out[None, :]))
        assert better.all()


def pin_topk_bruteforce(orc, seed=3, trials=300):
    """Tiny inputs: the kept set beats every dropped pool under (score desc, index asc)."""
    rng = np.random.default_rng(seed)
    for t in range(trials):
        P = int(rng.integers(1, 48))
        K = int(rng.integers(1, P + 1))
        mode = t % 4
        if mode == 0:
            s = rng.standard_normal(P).astype(np.float32)
        elif mode == 1:
            s = rng.integers(-2, 3, size=P).astype(np.float32)      # many exact ties
        elif mode == 2:
            s = rng.standard_normal(P).astype(np.float32)
            s[rng.random(P) < 0.3] = -np.inf
        else:
            s = np.where(rng.random(P) < 0.5, 0.0, -0.0).astype(np.float32)
        _check_topk_characterisation(s, K, orc.topk_pools(s, K))


def pin_topk_all_zero(orc):
    """All scores zero (with -0.0 mixed in): the K lowest pool indices win."""
    s = np.zeros(1000, dtype=np.float32)
    s[::3] = -0.0
    assert np.array_equal(orc.topk_pools(s, 64), np.arange(64, dtype=np.int32))


def pin_topk_stable_argsort(orc, seed=5):
    """A plain top-k equals numpy's stable argsort of -score (ties: lower index first)."""
    rng = np.random.default_rng(seed)
    for ties in ("none", "coarse", "inf"):
        s = workloads.random_scores(1, 4099, seed=seed, ties=ties)[0]
        for K in (1, 7, 512, 4099):
            ref = np.sort(np.argsort(-s, kind="stable")[:K])
            assert np.array_equal(orc.topk_pools(s, K), ref), (ties, K)


def pin_expand_closed_form(orc, seed=9):
    """Expansion: valid count == ctx if ctx <= topk else topk + ctx % kpool (the
    closed form of _kv_lens_host), strictly increasing tokens below ctx, kpool
    consecutive tokens per kept pool, the trailing tokens present, identity below topk."""
    rng = np.random.default_rng(seed)
    for topk, kpool in ((256, 4), (2048, 4), (60, 3), (16, 1), (64, 8)):
        W = topk + kpool
        K = topk // kpool
        for ctx in list(range(1, topk + 2 * kpool + 2)) + list(rng.integers(topk, 50 * topk, 40)):
            ctx = int(ctx)
            P = ctx // kpool
            pools = np.sort(rng.choice(P, size=min(K, P), replace=False)).astype(np.int32) \
                if ctx > topk else np.zeros(0, np.int32)
            tok, n = orc.expand(ctx, topk, kpool, pools, W)
            want = ctx if ctx <= topk else topk + ctx % kpool
            assert n == want, (topk, kpool, ctx, n, want)
            v = tok[:n]
            assert np.all(tok[n:] == -1)
            assert np.all(np.diff(v) > 0) and (n == 0 or (v[0] >= 0 and v[-1] < ctx))
            if ctx <= topk:
                assert np.array_equal(v, np.arange(ctx))
            else:
                body = v[:K * kpool].reshape(K, kpool)
                assert np.array_equal(body[:, 0] // kpool, pools)
                assert np.array_equal(body - body[:, :1], np.tile(np.arange(kpool), (K, 1)))
                assert np.array_equal(v[K * kpool:], np.arange(P * kpool, ctx))


def pin_remap_identity(orc):
    """Identity block table with stride == block size: slot == token; -1 stays -1."""
    bs = 64
    bt = np.arange(100, dtype=np.int32)
    for t in list(range(-1, 300)) + [100 * bs - 1]:
        s = orc.remap_token(t, bt, 100, 100, bs, bs)
        assert s == (t if t >= 0 else -1)
    assert orc.remap_token(100 * bs, bt, 100, 100, bs, bs) == -1   # block 100 out of bounds


def pin_remap_inverse(orc, seed=13):
    """Shuffled table and a row stride above the block size (other layers' pages in
    between): the slot decodes back to its token through the inverse permutation,
    and never lands in the rows between blocks."""
    rng = np.random.default_rng(seed)
    bs, stride, nb = 64, 192, 500
    perm = rng.permutation(nb).astype(np.int32)
    inv = np.argsort(perm)
    toks = rng.integers(0, nb * bs, size=2000).astype(np.int32)
    toks[::17] = -1
    req = np.zeros(toks.size, dtype=np.int32)
    slots, counts = orc.remap_rows(req, 1, perm[None, :], nb, nb, toks[:, None], bs, stride)
    slots = slots[:, 0]
    assert np.array_equal(slots == -1, toks == -1)
    ok = toks != -1
    assert np.all(slots[ok] % stride < bs)
    assert np.array_equal(inv[slots[ok] // stride] * bs + slots[ok] % stride, toks[ok])
    assert np.array_equal(counts, (toks != -1).astype(np.int32))


def pin_remap_guards(orc):
    """-1 for t == -1, a logical block past max_blocks, and a physical id outside
    [0, num_kv_blocks); in range, the formula block*stride + offset."""
    bt = np.array([5, -2, 7, 9, 3], dtype=np.int32)
    nkv = 8
    assert orc.remap_token(-1, bt, 5, nkv, 4, 4) == -1
    assert orc.remap_token(0, bt, 5, nkv, 4, 4) == 5 * 4 + 0
    assert orc.remap_token(3, bt, 5, nkv, 4, 10) == 5 * 10 + 3
    assert orc.remap_token(4, bt, 5, nkv, 4, 4) == -1      # physical -2
    assert orc.remap_token(9, bt, 5, nkv, 4, 4) == 7 * 4 + 1
    assert orc.remap_token(13, bt, 5, nkv, 4, 4) == -1     # physical 9 >= 8
    assert orc.remap_token(17, bt, 5, nkv, 4, 4) == 3 * 4 + 1
    assert orc.remap_token(17, bt, 4, nkv, 4, 4) == -1     # block 4 >= max_blocks 4
    assert orc.remap_token(20, bt, 5, nkv, 4, 4) == -1     # block 5 past the row


def pin_planted_winners(orc, seed=21):
    """Keys equal to 3*sign(sum_h q_h) reach the largest score any key in {-3..3}
    can reach, so K planted pools are exactly the kept set of their row."""
    w = workloads.build_workload([[2000]], name="planted", seed=seed, integer_mode=True,
                                 index_topk=256, kpool=4)
    K = 64
    P = 2000 // 4
    rng = np.random.default_rng(seed)
    planted = np.sort(rng.choice(P, size=K, replace=False))
    Q = w.q[0].astype(np.int64).sum(axis=0)
    best = (3 * np.sign(Q)).astype(np.float16)
    kc = w.key_cache.reshape(w.num_key_pages, -1, 64, 128)
    for j in planted:
        kc[w.key_page_table[0, j // 64], 0, j % 64] = best
    out = orc.select(w)
    tok = out["token_idx"][0]
    want = np.concatenate([(planted[:, None] * 4 + np.arange(4)[None, :]).ravel(),
                           np.arange(P * 4, 2000)])
    assert np.array_equal(tok[:want.size], want)
    assert np.all(tok[want.size:] == -1)


def pin_pipeline_counts(orc):
    """Whole selection on the tiny and 32K workloads: valid counts follow the closed
    form, token rows are ascending, and every slot lies inside its request's blocks."""
    for name in ("tiny", "decode32k"):
        w = workloads.make_workload(name)
        out = orc.select(w)
        ctx = w.row_contexts()
        want = np.where(ctx <= w.index_topk, ctx, w.index_topk + ctx % w.kpool)
        assert np.array_equal(out["counts"], want.astype(np.int32))
        for r in range(w.num_rows):
            req = int(np.searchsorted(w.qsl, r, side="right") - 1)
            n = out["counts"][r]
            tok = out["token_idx"][r]
            assert np.all(np.diff(tok[:n]) > 0) and np.all(tok[n:] == -1)
            allowed = set()
            nblk = -(-int(ctx[r]) // 64)
            for b in range(nblk):
                base = int(w.block_table[req, b]) * w.block_stride_rows
                allowed.update(range(base, base + 64))
            sl = out["slots"][r][:n]
            assert all(int(s) in allowed for s in sl)
            assert np.all(out["slots"][r][n:] == -1)


def pin_integer_scores_match_exact(orc):
    """Scores of the tiny workload equal exact int64 dot products through the tables."""
    w = workloads.make_workload("tiny")
    sc, ab, st = orc.score_rows(w)
    assert st == 0
    qi = w.q.astype(np.int64)
    kc = w.key_cache.reshape(w.num_key_pages, -1, 64, 128)[:, 0]
    for r in range(w.num_rows):
        req = int(np.searchsorted(w.qsl, r, side="right") - 1)
        P = int(w.positions[r] + 1) // w.kpool
        keys = kc[w.key_page_table[req, :(P + 63) // 64]].reshape(-1, 128)[:P].astype(np.int64)
        exact = keys @ qi[r].sum(axis=0)
        assert np.array_equal(sc[r, :P], exact.astype(np.float32))


def _golden(name):
    import _golden
    return _golden.load(name), _golden.ints


def pin_workspace_worked_example(orc):
    """Hand-worked prefill-workspace fixture (tests/golden/workspace_worked_example.txt)."""
    d, ints = _golden("workspace_worked_example.txt")
    toks = np.stack([ints(d, f"tokens_row{r}") for r in range(4)]).astype(np.int32)
    slots, counts = orc.remap_ws_rows(ints(d, "req_id"), 1, ints(d, "block_table_row0")[None, :],
                                      int(d["max_blocks"][0]), int(d["num_kv_blocks"][0]), ints(d, "ws_req"),
                                      ints(d, "ws_starts"), toks, int(d["block_size"][0]), int(d["stride"][0]))
    for r in range(4):
        assert np.array_equal(slots[r], ints(d, f"slots_row{r}")), r
    assert np.array_equal(counts, ints(d, "counts"))


def pin_workspace_decode_rows_are_remap(orc, seed=31):
    """Rows without a prefill request (-1) take exactly the global remap."""
    rng = np.random.default_rng(seed)
    bt = rng.permutation(64).astype(np.int32)[:48].reshape(3, 16)
    toks = rng.integers(-1, 16 * 8, size=(9, 12)).astype(np.int32)
    req = rng.integers(0, 3, size=9).astype(np.int32)
    ref = orc.remap_rows(req, 3, bt, 16, 64, toks, 8, 24)
    got = orc.remap_ws_rows(req, 3, bt, 16, 64, np.full(9, -1, np.int32), np.array([7], np.int32), toks, 8, 24)
    assert np.array_equal(got[0], ref[0]) and np.array_equal(got[1], ref[1])


def pin_dcp_worked_example(orc):
    """Hand-worked decode-context-parallel fixture (tests/golden/dcp_worked_example.txt), both
    ranks, with and without compaction."""
    d, ints = _golden("dcp_worked_example.txt")
    toks = np.stack([ints(d, f"tokens_row{r}") for r in range(3)]).astype(np.int32)
    bt = np.stack([ints(d, "block_table_row0"), ints(d, "block_table_row1")]).astype(np.int32)
    D, I, B = int(d["dcp_size"][0]), int(d["interleave"][0]), int(d["block_size"][0])
    mb, nkv = int(d["max_blocks"][0]), int(d["num_kv_blocks"][0])
    for rank in (0, 1):
        slots, counts = orc.remap_dcp_rows(ints(d, "req_id"), 2, bt, mb, nkv, toks, B, D, rank, I, False)
        for r in range(3):
            assert np.array_equal(slots[r], ints(d, f"rank{rank}_row{r}")), (rank, r)
        assert np.array_equal(counts, ints(d, f"rank{rank}_counts")), rank
    slots, counts = orc.remap_dcp_rows(ints(d, "req_id"), 2, bt, mb, nkv, toks, B, D, 0, I, True)
    for r in range(3):
        assert np.array_equal(slots[r], ints(d, f"rank0_compact_row{r}")), r


def pin_dcp_single_rank_is_remap(orc, seed=33):
    """One rank owns every token: the filter is the global remap with a dense table."""
    rng = np.random.default_rng(seed)
    bt = rng.permutation(80).astype(np.int32)[:60].reshape(3, 20)
    bt[1, 4] = -3
    toks = rng.integers(-1, 20 * 16 + 40, size=(10, 16)).astype(np.int32)
    req = rng.integers(0, 3, size=10).astype(np.int32)
    ref = orc.remap_rows(req, 3, bt, 20, 70, toks, 16, 16)
    for inter in (1, 2, 4, 16):
        got = orc.remap_dcp_rows(req, 3, bt, 20, 70, toks, 16, 1, 0, inter, False)
        assert np.array_equal(got[0], ref[0]) and np.array_equal(got[1], ref[1]), inter


def pin_dcp_interleave_partition(orc):
    """The ranks partition a request's tokens: every token has exactly one owner; a group of
    `interleave` consecutive tokens shares its owner and any dcp_size consecutive groups have
    distinct owners (round robin); on each rank the owned tokens, in increasing order, get
    the local indices 0, 1, 2, ... with no gap."""
    for D, I in ((2, 1), (2, 2), (3, 4), (4, 8), (8, 2)):
        n = D * I * 7 + 5
        owners = np.full(n, -1)
        local = np.full(n, -1)
        for rank in range(D):
            for t in range(n):
                l = orc.dcp_local_index(t, D, rank, I)
                if l >= 0:
                    assert owners[t] == -1, (D, I, t)
                    owners[t], local[t] = rank, l
        assert (owners >= 0).all()
        grp = owners[: (n // I) * I].reshape(-1, I)
        assert (grp == grp[:, :1]).all()
        g0 = grp[:, 0]
        for k in range(len(g0) - D + 1):
            assert len(set(g0[k:k + D].tolist())) == D
        for rank in range(D):
            assert np.array_equal(local[owners == rank], np.arange(int((owners == rank).sum())))
        assert orc.dcp_local_index(-1, D, 0, I) == -1


def pin_dcp_compaction(orc, seed=35):
    """Compaction moves exactly the non -1 slots of the uncompacted row, in column order, to the
    front and fills the rest with -1; the counts are unchanged."""
    rng = np.random.default_rng(seed)
    bt = rng.permutation(200).astype(np.int32)[:160].reshape(4, 40)
    toks = rng.integers(-1, 40 * 8 * 2, size=(12, 24)).astype(np.int32)
    req = rng.integers(0, 4, size=12).astype(np.int32)
    for D, I, rank in ((2, 4, 1), (4, 2, 3), (3, 8, 0)):
        a, ca = orc.remap_dcp_rows(req, 4, bt, 40, 200, toks, 8, D, rank, I, False)
        b, cb = orc.remap_dcp_rows(req, 4, bt, 40, 200, toks, 8, D, rank, I, True)
        assert np.array_equal(ca, cb)
        for r in range(12):
            kept = a[r][a[r] != -1]
            assert np.array_equal(b[r][:ca[r]], kept) and (b[r][ca[r]:] == -1).all()



# ---------------------------------------------------------------- MaxSim rerank
def _maxsim_exact(q, rows, offsets, lengths):
    """Brute force with integer arithmetic: numpy's int64 matmul, max over each doc's
    rows, sum over the query rows (integer-valued inputs only)."""
    qi = q.astype(np.int64)
    out = []
    for o, n in zip(offsets, lengths):
        idx = np.arange(o, o + max(n, 0))
        if idx.size == 0:
            out.append(-np.inf if qi.shape[0] else 0.0)
            continue
        r = np.zeros((idx.size, qi.shape[1]), dtype=np.int64)
        inside = (idx >= 0) & (idx < rows.shape[0])
        r[inside] = rows[idx[inside], :qi.shape[1]].astype(np.int64)
        out.append(float((qi @ r.T).max(axis=1).sum()))
    return np.array(out)


def pin_maxsim_worked_example(orc):
    """Hand-worked MaxSim fixture (tests/golden/maxsim_worked_example.txt): scattered and
    overlapping docs, an empty doc, a single-row doc."""
    import _golden
    d = _golden.load("maxsim_worked_example.txt")
    lq, dim = int(d["lq"][0]), int(d["d"][0])
    q = _golden.ints(d, "q").reshape(lq, dim).astype(np.float16)
    rows = _golden.ints(d, "rows").reshape(-1, dim).astype(np.float16)
    s, _ = orc.maxsim(q, rows, _golden.ints(d, "offsets"), _golden.ints(d, "lengths"))
    assert np.array_equal(s, _golden.floats(d, "scores")), s


def pin_maxsim_integer_exact(orc, seed=41):
    """Integer-valued fp16 inputs (|score| < 2^24, so every step is exact): the oracle equals
    the int64 brute force, over random scattered docs in a tensor wider than d."""
    rng = np.random.default_rng(seed)
    for lq, dim, width in ((3, 8, 8), (5, 16, 24), (1, 40, 48), (7, 4, 8)):
        total = 57
        rows = rng.integers(-3, 4, size=(total, width)).astype(np.float16)
        q = rng.integers(-3, 4, size=(lq, dim)).astype(np.float16)
        lengths = rng.integers(0, 9, size=11).astype(np.int32)
        offsets = rng.integers(0, total - 8, size=11).astype(np.int32)
        s, _ = orc.maxsim(q, rows, offsets, lengths)
        ref = _maxsim_exact(q, rows, offsets, lengths)
        assert np.array_equal(s.astype(np.float64), ref), (lq, dim, s, ref)


def pin_maxsim_single_row_closed_form(orc, seed=43):
    """A one-row doc has no max to take: its score is (sum_a q_a) . row, computed here in
    float64 from the column sums of q."""
    rng = np.random.default_rng(seed)
    q = (rng.standard_normal((9, 32)) / 4).astype(np.float16)
    rows = (rng.standard_normal((20, 32)) / 4).astype(np.float16)
    offs = np.arange(20, dtype=np.int32)
    s, _ = orc.maxsim(q, rows, offs, np.ones(20, np.int32))
    ref = rows.astype(np.float64) @ q.astype(np.float64).sum(axis=0)
    assert np.allclose(s, ref, rtol=1e-6, atol=1e-6), (s, ref)


def pin_maxsim_order_invariance(orc, seed=45):
    """The score is a function of the doc's set of rows: permuting the rows, or repeating
    one, leaves it unchanged (bit for bit, as each dot product is computed alone)."""
    rng = np.random.default_rng(seed)
    q = (rng.standard_normal((6, 16))).astype(np.float16)
    base = (rng.standard_normal((10, 16))).astype(np.float16)
    perm = base[rng.permutation(10)]
    dup = np.concatenate([base, base[3:4]])
    rows = np.concatenate([base, perm, dup])
    s, _ = orc.maxsim(q, rows, np.array([0, 10, 20], np.int32), np.array([10, 10, 11], np.int32))
    assert s[0] == s[1] == s[2], s


def pin_maxsim_degenerate(orc):
    """The page's masking: an empty (or negative-length) doc scores -inf, no query rows
    score 0; rows outside the tensor read as zero vectors."""
    q = np.array([[1, -2], [3, 1]], np.float16)
    rows = np.array([[-1, -1], [2, 0]], np.float16)
    s, _ = orc.maxsim(q, rows, np.array([0, 1, 0, 1, -3], np.int32), np.array([0, -2, 1, 5, 2], np.int32))
    # doc 2 = row 0: (-1+2) + (-3-1) = -3; doc 3 = row 1 and 4 zero rows: max(2,0) + max(6,0) = 8;
    # doc 4 = two rows before the tensor: 0 + 0
    assert s[0] == -np.inf and s[1] == -np.inf and s[2] == -3.0 and s[3] == 8.0 and s[4] == 0.0, s
    s, _ = orc.maxsim(np.zeros((0, 2), np.float16), rows, np.array([0, 0], np.int32), np.array([2, 0], np.int32))
    assert np.array_equal(s, np.zeros(2, np.float32)), s


def pin_maxsim_normal_bound(orc, seed=47):
    """Normal values: the oracle's score is within one fp32 rounding of the float64 brute
    force (numpy matmul, max, sum), and abs_bound equals sum_a max_j sum_k |q_ak t_jk|."""
    rng = np.random.default_rng(seed)
    q = (rng.standard_normal((32, 128)) / np.sqrt(128)).astype(np.float16)
    rows = rng.standard_normal((300, 128)).astype(np.float16)
    offs = np.array([0, 17, 100, 250], np.int32)
    lens = np.array([17, 83, 150, 50], np.int32)
    s, b = orc.maxsim(q, rows, offs, lens)
    q64, r64 = q.astype(np.float64), rows.astype(np.float64)
    for i, (o, n) in enumerate(zip(offs, lens)):
        sims = q64 @ r64[o:o + n].T
        ref = sims.max(axis=1).sum()
        absb = (np.abs(q64)[:, None, :] * np.abs(r64[o:o + n])[None, :, :]).sum(axis=2).max(axis=1).sum()
        assert abs(s[i] - ref) <= 2.0 ** -23 * abs(ref) + 1e-12 * absb, (i, s[i], ref)
        assert abs(b[i] - absb) <= 1e-12 * absb, (i, b[i], absb)


# ---------------------------------------------------------------- sparse MLA decode attention
def _bf(x):
    """float values that are exact in bfloat16 -> their bit patterns."""
    return (np.ascontiguousarray(x, dtype=np.float32).view(np.uint32) >> 16).astype(np.uint16)


def pin_bf16_decode(orc):
    """bfloat16 decoding of all 65,536 bit patterns equals torch's bfloat16 -> float64."""
    import torch
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    got = orc.bf16_to_double(bits)
    ref = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).to(torch.float64).numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])


def pin_mla_worked_example(orc):
    """Hand-worked fixture (tests/golden/mla_worked_example.txt): weights 1 : 2 : 4 from
    sm_scale = ln 2, a -1 inside kv_len, an entry past kv_len, an empty row, one entry."""
    import _golden
    d = _golden.load("mla_worked_example.txt")
    qn = _bf(_golden.floats(d, "q_nope").reshape(3, 1, 2))
    qp = _bf(_golden.floats(d, "q_pe").reshape(3, 1, 1))
    ckv = _bf(_golden.floats(d, "ckv").reshape(8, 2))
    kpe = _bf(_golden.floats(d, "kpe").reshape(8, 1))
    slots = np.stack([_golden.ints(d, f"slots_row{r}") for r in range(3)]).astype(np.int32)
    out, lse = orc.mla_decode(qn, qp, ckv, kpe, slots, _golden.ints(d, "kv_len"), float(d["sm_scale"][0]))
    for r in range(3):
        assert np.allclose(out[r, 0], _golden.floats(d, f"out_row{r}").astype(np.float64), rtol=1e-7, atol=1e-7), r
    want = np.array([float(x) for x in d["lse"]])
    assert np.array_equal(np.isinf(lse[:, 0]), np.isinf(want))
    fin = ~np.isinf(want)
    assert np.allclose(lse[fin, 0], want[fin], rtol=1e-12, atol=1e-12), lse


def _mla_int_inputs(rng, rows, heads, dc, dr, num_slots, lo=-3, hi=4):
    qn = rng.integers(lo, hi, size=(rows, heads, dc)).astype(np.float32)
    qp = rng.integers(lo, hi, size=(rows, heads, dr)).astype(np.float32)
    ckv = rng.integers(lo, hi, size=(num_slots, dc)).astype(np.float32)
    kpe = rng.integers(lo, hi, size=(num_slots, dr)).astype(np.float32)
    return qn, qp, ckv, kpe


def pin_mla_single_entry(orc, seed=51):
    """One valid entry: the softmax is 1, so out is that slot's ckv row exactly and lse is its
    logit, sm_scale times the exact int64 dot product (numpy)."""
    rng = np.random.default_rng(seed)
    qn, qp, ckv, kpe = _mla_int_inputs(rng, 4, 3, 16, 4, 10)
    slots = np.array([[7, -1], [0, 3], [9, 9], [-1, 2]], np.int32)
    kv_len = np.array([1, 1, 1, 2], np.int32)
    scale = 0.125
    out, lse = orc.mla_decode(_bf(qn), _bf(qp), _bf(ckv), _bf(kpe), slots, kv_len, scale)
    for r, s_ in enumerate([7, 0, 9, 2]):
        for h in range(3):
            assert np.array_equal(out[r, h], ckv[s_].astype(np.float64)), (r, h)
            dot = int(qn[r, h].astype(np.int64) @ ckv[s_].astype(np.int64) + qp[r, h].astype(np.int64) @ kpe[s_].astype(np.int64))
            assert lse[r, h] == scale * dot, (r, h, lse[r, h], scale * dot)


def pin_mla_uniform(orc, seed=53):
    """Zero queries: every logit is 0, so out is the plain mean of the row's valid ckv rows
    and lse = log(number of valid entries)."""
    rng = np.random.default_rng(seed)
    _, _, ckv, kpe = _mla_int_inputs(rng, 1, 1, 8, 2, 30)
    qn = np.zeros((2, 2, 8), np.float32)
    qp = np.zeros((2, 2, 2), np.float32)
    slots = np.array([[3, 11, -1, 29, 4, 40], [5, 6, 7, 8, 9, 10]], np.int32)
    kv_len = np.array([6, 4], np.int32)
    out, lse = orc.mla_decode(_bf(qn), _bf(qp), _bf(ckv), _bf(kpe), slots, kv_len, 0.3)
    for r, valid in enumerate([[3, 11, 29, 4], [5, 6, 7, 8]]):   # slot 40 is past num_slots = 30
        ref = ckv[valid].astype(np.float64).mean(axis=0)
        for h in range(2):
            assert np.allclose(out[r, h], ref, rtol=1e-14, atol=1e-14), (r, h)
            assert abs(lse[r, h] - np.log(len(valid))) < 1e-14


def pin_mla_entry_set(orc, seed=55):
    """The result depends only on the set of valid entries inside kv_len: permuting them, adding
    -1 or out-of-range slots inside kv_len, or valid slots past kv_len changes nothing."""
    rng = np.random.default_rng(seed)
    qn, qp, ckv, kpe = _mla_int_inputs(rng, 1, 4, 32, 8, 64)
    qn, qp = qn / 8, qp / 8
    base = rng.choice(64, size=12, replace=False).astype(np.int32)
    a = np.concatenate([base, np.full(4, -1, np.int32)])[None, :]
    perm = rng.permutation(base)
    b = np.concatenate([perm[:5], [-1, 70, -1], perm[5:], [0, 1, 2, 3, 5]]).astype(np.int32)[None, :]
    out_a, lse_a = orc.mla_decode(_bf(qn), _bf(qp), _bf(ckv), _bf(kpe), a, np.array([12], np.int32), 0.25)
    out_b, lse_b = orc.mla_decode(_bf(qn), _bf(qp), _bf(ckv), _bf(kpe), b, np.array([15], np.int32), 0.25)
    assert np.allclose(out_a, out_b, rtol=1e-12, atol=1e-12)
    assert np.allclose(lse_a, lse_b, rtol=1e-12, atol=1e-12)


def pin_mla_shift(orc, seed=57):
    """A constant added to every logit (a rotary key shared by all slots) leaves out unchanged
    and moves lse by that constant."""
    rng = np.random.default_rng(seed)
    qn, _, ckv, _ = _mla_int_inputs(rng, 2, 2, 16, 4, 20)
    kpe = np.ones((20, 4), np.float32)
    qp0 = np.zeros((2, 2, 4), np.float32)
    qp1 = np.full((2, 2, 4), 1.5, np.float32)        # q_pe . kpe = 6 for every slot
    slots = rng.permutation(20)[:10].astype(np.int32).reshape(2, 5)
    kv_len = np.array([5, 3], np.int32)
    o0, l0 = orc.mla_decode(_bf(qn), _bf(qp0), _bf(ckv), _bf(kpe), slots, kv_len, 0.5)
    o1, l1 = orc.mla_decode(_bf(qn), _bf(qp1), _bf(ckv), _bf(kpe), slots, kv_len, 0.5)
    assert np.allclose(o0, o1, rtol=1e-12, atol=1e-12)
    assert np.allclose(l1 - l0, 3.0, rtol=0, atol=1e-12)


def pin_mla_large_logits(orc):
    """Logits in the thousands (no overflow): a slot whose logit exceeds the others by 1000
    takes all the weight, so out is its ckv row and lse its logit, exactly."""
    ckv = np.array([[1, 2], [3, -4], [5, 6]], np.float32)
    kpe = np.array([[0], [0], [0]], np.float32)
    qn = np.array([[[1000, 1000]]], np.float32)        # dots 3000, -1000, 11000
    qp = np.zeros((1, 1, 1), np.float32)
    out, lse = orc.mla_decode(_bf(qn), _bf(qp), _bf(ckv), _bf(kpe), np.array([[0, 1, 2]], np.int32),
                              np.array([3], np.int32), 1.0)
    assert np.array_equal(out[0, 0], [5.0, 6.0]) and lse[0, 0] == 11000.0, (out, lse)


def pin_mla_duplicate_slot(orc):
    """A slot listed twice counts twice: with logits 0, 0, ln 2 the weights are 1 : 1 : 2."""
    ckv = np.array([[2, 0], [0, 8]], np.float32)
    kpe = np.array([[0], [1]], np.float32)
    qn = np.zeros((1, 1, 2), np.float32)
    qp = np.ones((1, 1, 1), np.float32)
    out, lse = orc.mla_decode(_bf(qn), _bf(qp), _bf(ckv), _bf(kpe), np.array([[0, 0, 1]], np.int32),
                              np.array([3], np.int32), float(np.log(2.0)))
    assert np.allclose(out[0, 0], [1.0, 4.0], rtol=1e-14, atol=1e-14), out
    assert abs(lse[0, 0] - np.log(4.0)) < 1e-14

ALL_PINS = [pin_half_decode, pin_score_integer_exact, pin_score_normal_bound,
            pin_topk_bruteforce, pin_topk_all_zero, pin_topk_stable_argsort,
            pin_expand_closed_form, pin_remap_identity, pin_remap_inverse, pin_remap_guards,
            pin_planted_winners, pin_pipeline_counts, pin_integer_scores_match_exact,
            pin_workspace_worked_example, pin_workspace_decode_rows_are_remap, pin_dcp_worked_example,
            pin_dcp_single_rank_is_remap, pin_dcp_interleave_partition, pin_dcp_compaction,
            pin_maxsim_worked_example, pin_maxsim_integer_exact, pin_maxsim_single_row_closed_form,
            pin_maxsim_order_invariance, pin_maxsim_degenerate, pin_maxsim_normal_bound,
            pin_bf16_decode, pin_mla_worked_example, pin_mla_single_entry, pin_mla_uniform,
            pin_mla_entry_set, pin_mla_shift, pin_mla_large_logits, pin_mla_duplicate_slot]
