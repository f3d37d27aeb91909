"""The seeded input generators follow their stated recipes (CPU only): the selection
workloads' valid counts match _kv_lens_host's closed form, the MaxSim batch is scattered
with poisoned gaps, and the MLA decode inputs carry sorted distinct slots and the exact
kv_len of each row."""

import numpy as np

import workloads
from workloads.maxsim import build_maxsim, make_maxsim
from workloads.mla import make_mla


def _closed_form(ctx, topk, kpool):
    return np.where(ctx <= topk, ctx, topk + ctx % kpool)


def test_selection_rows_have_the_stated_contexts():
    w = workloads.make_workload("decode128k")
    ctx = w.positions.astype(np.int64) + 1
    assert ctx.min() == 131068 and ctx.max() == 131072
    counts = _closed_form(ctx, 2048, 4)
    assert set(counts.tolist()) == {2048, 2049, 2050, 2051}


def test_maxsim_recipe():
    w = make_maxsim("maxsim_small")
    lq, d = w.q.shape
    assert (lq, d) == (32, 128)
    fixed = [0, 1, 2, 31, 32, 33, 64, 65, 127, 128, 129, 513, -3]
    assert w.lengths[:len(fixed)].tolist() == fixed
    # the 40 generated documents do not overlap, and every row outside them is the poison row
    covered = np.zeros(w.docs.shape[0], bool)
    for o, n in zip(w.offsets[:40], w.lengths[:40]):
        if n > 0:
            assert not covered[o:o + n].any()
            covered[o:o + n] = True
    poison = (60.0 * np.sign(w.q[0].astype(np.float32) + 1e-3)).astype(np.float16)
    assert (w.docs[~covered] == poison).all()
    # scattered: document order in the tensor differs from index order
    starts = w.offsets[:40][w.lengths[:40] > 0]
    assert not np.all(np.diff(starts) > 0)
    big = make_maxsim("maxsim_rerank4k")
    assert big.num_docs == 4096 and big.lengths.min() >= 1 and big.lengths.max() <= 512
    assert big.doc_rows == int(big.lengths.sum()) and big.docs.nbytes > 129 * (1 << 20)


def test_maxsim_integer_values_are_exact_small_integers():
    w = build_maxsim(name="t", lq=4, d=16, num_docs=5, len_lo=1, len_hi=9, seed=3, values="int")
    assert np.array_equal(w.q, np.round(w.q)) and np.abs(w.q).max() <= 3


def test_mla_recipe():
    w = make_mla("mla_small")
    ctx = np.array([1, 7, 2047, 2048, 2049, 131072])
    assert np.array_equal(w.kv_len, _closed_form(ctx, 2048, 4))
    assert w.slots.shape[1] % 4 == 0 and w.slots.shape[1] >= 2048 + 4 - 1
    for r, n in enumerate(w.kv_len):
        row = w.slots[r]
        assert (row[n:] == -1).all()                      # the -1 tail past kv_len
        inside = row[:n]
        ok = inside[(inside >= 0) & (inside < w.cache.shape[0])]
        assert np.all(np.diff(ok) > 0)                     # distinct, ascending
    assert w.cache.shape[1] == w.dc + w.dr == 576
    assert abs(w.sm_scale - 192 ** -0.5) < 1e-12
    # holes: some -1 and out-of-range slots inside kv_len (mla_small only)
    inside = np.concatenate([w.slots[r, :n] for r, n in enumerate(w.kv_len)])
    assert (inside == -1).any() and (inside >= w.cache.shape[0]).any()


def test_generators_are_deterministic():
    a, b = make_mla("mla_small"), make_mla("mla_small")
    assert np.array_equal(a.slots, b.slots) and np.array_equal(a.q_nope, b.q_nope)
    m1, m2 = make_maxsim("maxsim_small"), make_maxsim("maxsim_small")
    assert np.array_equal(m1.offsets, m2.offsets) and np.array_equal(m1.docs, m2.docs)


def test_selection_token_indices_shape_and_order():
    t = workloads.selection_token_indices([131072, 60003, 1000, 2048], 2052, seed=3)
    assert t.shape == (4, 2052) and t.dtype == np.int32
    np.testing.assert_array_equal((t >= 0).sum(1), [2048, 2051, 1000, 2048])   # topk + ctx % kpool
    for r in range(4):
        v = t[r][t[r] >= 0]
        assert np.all(np.diff(v) > 0)                                  # ascending, distinct
        assert np.all(t[r][v.size:] == -1)                             # -1 tail
    pools = t[0][t[0] >= 0].reshape(-1, 4)
    assert np.all(pools[:, 0] % 4 == 0) and np.all(np.diff(pools, axis=1) == 1)   # whole pools
    np.testing.assert_array_equal(t[1][2048:2051], [60000, 60001, 60002])         # trailing pool
    np.testing.assert_array_equal(t[2][:1000], np.arange(1000))                   # ctx <= topk
