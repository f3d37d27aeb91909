"""The CPU oracle against facts fixed by the pages and by mathematics (no GPU)."""

import numpy as np
import pytest

import oracle
import workloads
from _golden import floats, ints, load
from _pins import ALL_PINS


@pytest.mark.parametrize("pin", ALL_PINS, ids=lambda f: f.__name__)
def test_pin(pin):
    pin(oracle)


def test_golden_remap_worked_example():
    g = load("remap_worked_example.txt")
    bt = np.stack([ints(g, "block_table_row0"), ints(g, "block_table_row1")]).astype(np.int32)
    tok = np.stack([ints(g, "tokens_row0"), ints(g, "tokens_row1")]).astype(np.int32)
    args = (ints(g, "req_id"), 2, bt, int(g["max_blocks"][0]), int(g["num_kv_blocks"][0]), tok,
            int(g["block_size"][0]))
    slots, counts = oracle.remap_rows(*args, int(g["stride"][0]))
    assert np.array_equal(slots, np.stack([ints(g, "slots_row0"), ints(g, "slots_row1")]))
    assert np.array_equal(counts, ints(g, "counts"))
    slots_b, _ = oracle.remap_rows(*args, int(g["stride_b"][0]))
    assert np.array_equal(slots_b, np.stack([ints(g, "slots_b_row0"), ints(g, "slots_b_row1")]))


@pytest.mark.parametrize("case", ["a", "b", "c", "d"])
def test_golden_expand_worked_example(case):
    g = load("expand_worked_example.txt")
    topk, kpool, W = int(g["topk"][0]), int(g["kpool"][0]), int(g["width"][0])
    ctx = int(g[f"{case}_ctx"][0])
    s = floats(g, f"{case}_scores") if g[f"{case}_scores"] else np.zeros(0, np.float32)
    if ctx > topk:
        s = s.copy()
        s[np.signbit(s) & (s == 0)] = -0.0
        pools = oracle.topk_pools(s, topk // kpool)
    else:
        pools = np.zeros(0, np.int32)
    tok, n = oracle.expand(ctx, topk, kpool, pools, W)
    assert np.array_equal(tok, ints(g, f"{case}_tokens"))
    assert n == int(g[f"{case}_count"][0])
    # the same through the batched entry point
    sc = np.zeros((1, max(1, s.size)), np.float32)
    sc[0, :s.size] = s
    tok2, cnt2 = oracle.topk_expand_rows(sc, np.array([ctx]), topk, kpool, W)
    assert np.array_equal(tok2[0], tok) and cnt2[0] == n


def test_status_bits_and_guard_rows():
    w = workloads.build_workload([[3000, 3001], [2500]], name="st", seed=4, integer_mode=True,
                                 index_topk=256, kpool=4, max_context=3000)
    # request 0's logical key page 5 points outside the physical pool
    w.key_page_table[0, 5] = w.num_key_pages + 3
    out = oracle.select(w, want_scores=True)
    assert out["status"] & oracle.ST_KEYPAGE_OOB
    assert out["status"] & oracle.ST_CTX_OVER_BOUND        # row 1 has ctx 3001 > 3000
    assert np.all(np.isneginf(out["scores"][0, 5 * 64:6 * 64]))
    assert np.all(np.isfinite(out["scores"][0, :5 * 64]))
    sel_pools = set((out["token_idx"][0][:256] // 4).tolist())
    assert not (sel_pools & set(range(5 * 64, 6 * 64)))   # -inf pools never beat finite ones
    assert np.all(out["slots"][1] == -1) and out["counts"][1] == 0
    assert out["counts"][2] == 256 + 2500 % 4
    # a malformed request table empties every row
    w.qsl[1] = 5
    out2 = oracle.select(w)
    assert out2["status"] & oracle.ST_BAD_QSL
    assert np.all(out2["slots"] == -1) and np.all(out2["counts"] == 0)


def test_padding_rows_are_empty():
    w = workloads.build_workload([[3000], [100, 101]], name="pad", seed=5, integer_mode=True,
                                 index_topk=256, pad_rows=3)
    out = oracle.select(w)
    assert np.all(out["slots"][3:] == -1) and np.all(out["counts"][3:] == 0)
    assert list(out["counts"][:3]) == [256, 100, 101]


@pytest.mark.parametrize("name", ["decode128k", "ragged", "ragged_b"])
def test_config_counts_closed_form(name):
    """Sampled rows: count == closed form minus the tokens that land in guarded blocks."""
    w = workloads.make_workload(name)
    rows = np.unique(np.concatenate([w.qsl[1:] - 1, w.qsl[:-1]])).astype(np.int32)
    rows = rows[rows < w.qsl[-1]]
    out = oracle.select(w, rows=rows)
    guarded = {}
    for (req, lb, _v) in w.oob_entries:
        guarded.setdefault(req, set()).add(lb)
    for k, r in enumerate(rows):
        ctx = int(w.positions[r]) + 1
        req = int(np.searchsorted(w.qsl, r, side="right") - 1)
        want = ctx if ctx <= w.index_topk else w.index_topk + ctx % w.kpool
        tok = out["token_idx"][k][:want]
        hits = sum(1 for t in tok if (t // 64) in guarded.get(req, ()))
        assert out["counts"][k] == want - hits, (name, r)
    if name == "ragged":
        # request 1's trailing block 3125 is guarded: its trailing tokens never map to a slot
        r = int(w.qsl[2] - 1)
        k = int(np.nonzero(rows == r)[0][0])
        n_tok = w.index_topk + (int(w.positions[r]) + 1) % w.kpool
        assert np.all(out["slots"][k][n_tok - 1:n_tok] == -1)
