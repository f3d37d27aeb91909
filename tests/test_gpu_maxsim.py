"""MaxSim rerank on the GPU (through the C ABI) against the CPU oracle.

Integer-valued inputs make every dot product, maximum and sum exact in fp32, so those
cases compare bit for bit. Normal-valued inputs use the bound of an fp32 computation:
each dot product of d fp16 x fp16 products accumulated in fp32 is within d * 2^-23 *
sum|terms| of the exact value, a maximum moves by at most the largest error of its
candidates, and the sum of lq maxima adds lq * 2^-23 * sum|max|; the oracle's abs_bound
(sum over query rows of the largest sum|terms| over the document's rows) bounds both, so
|gpu - exact| <= (d + lq + 2) * 2^-23 * abs_bound."""

import numpy as np
import pytest
import torch

import oracle
from workloads.maxsim import build_maxsim, make_maxsim
from _gpu import DEV, lib

pytestmark = pytest.mark.gpu


def _t(a):
    return torch.from_numpy(np.ascontiguousarray(a)).to(DEV)


def run_maxsim(w, docs=None):
    sel = lib()
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    d = _t(w.docs) if docs is None else docs
    scores = sel.sel_maxsim_rerank(_t(w.q), d, _t(w.offsets), _t(w.lengths), status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0, "a bounded wait expired"
    return scores.cpu().numpy()


def tolerance(w, bound):
    lq, d = w.q.shape
    return (d + lq + 2) * 2.0 ** -23 * bound + 1e-30


def assert_close(w, got, idx=None):
    off, ln = (w.offsets, w.lengths) if idx is None else (w.offsets[idx], w.lengths[idx])
    ref, bound = oracle.maxsim(w.q, w.docs, off, ln)
    g = got if idx is None else got[idx]
    inf = np.isinf(ref)
    np.testing.assert_array_equal(np.isinf(g), inf)
    np.testing.assert_array_equal(g[inf], ref[inf])
    err = np.abs(g[~inf].astype(np.float64) - ref[~inf].astype(np.float64))
    tol = tolerance(w, bound[~inf])
    bad = np.nonzero(err > tol)[0]
    assert bad.size == 0, f"{bad.size} documents outside tolerance, first {bad[:5]}: err {err[bad[:5]]} tol {tol[bad[:5]]}"


def test_maxsim_small_int_bitexact():
    w = make_maxsim("maxsim_small", values="int")
    got = run_maxsim(w)
    ref, _ = oracle.maxsim(w.q, w.docs, w.offsets, w.lengths)
    np.testing.assert_array_equal(got, ref)


def test_maxsim_small_normal():
    w = make_maxsim("maxsim_small")
    assert_close(w, run_maxsim(w))


@pytest.mark.parametrize("lq,d,num_docs,len_hi", [
    (1, 128, 30, 200), (7, 64, 30, 200), (32, 96, 25, 150), (33, 128, 20, 150), (100, 200, 12, 120),
    (256, 128, 10, 100), (300, 128, 8, 90), (40, 1024, 6, 70), (70, 1024, 5, 40), (16, 8, 30, 80)])
def test_maxsim_shapes(lq, d, num_docs, len_hi):
    for values in ("int", "normal"):
        w = build_maxsim(name="shape", lq=lq, d=d, num_docs=num_docs, len_lo=0, len_hi=len_hi,
                         seed=lq * 1000 + d, values=values, extra_docs=True)
        got = run_maxsim(w)
        if values == "int":
            ref, _ = oracle.maxsim(w.q, w.docs, w.offsets, w.lengths)
            np.testing.assert_array_equal(got, ref)
        else:
            assert_close(w, got)


def test_maxsim_many_tiny_documents():
    """Mean length 4 rows: grabs of many documents, most tiles mixing four documents."""
    w = build_maxsim(name="tiny", lq=32, d=64, num_docs=6000, len_lo=0, len_hi=8, seed=5, gap_hi=3, values="int")
    got = run_maxsim(w)
    ref, _ = oracle.maxsim(w.q, w.docs, w.offsets, w.lengths)
    np.testing.assert_array_equal(got, ref)


def test_maxsim_strided_tensor():
    """The packed tensor is a column slice of a wider one (row stride 192 > d = 128)."""
    w = make_maxsim("maxsim_small")
    wide = np.zeros((w.docs.shape[0], 192), np.float16)
    wide[:, :128] = w.docs
    wide[:, 128:] = np.float16(50.0)
    dw = _t(wide)
    got = run_maxsim(w, docs=dw[:, :128])
    assert_close(w, got)


def test_maxsim_degenerate():
    sel = lib()
    w = make_maxsim("maxsim_small")
    # no query rows: every document scores 0
    sc = sel.sel_maxsim_rerank(_t(w.q[:0]), _t(w.docs), _t(w.offsets), _t(w.lengths))
    torch.cuda.synchronize()
    np.testing.assert_array_equal(sc.cpu().numpy(), np.zeros(w.num_docs, np.float32))
    # no documents: nothing to do
    sc = sel.sel_maxsim_rerank(_t(w.q), _t(w.docs), _t(w.offsets[:0]), _t(w.lengths[:0]))
    torch.cuda.synchronize()
    assert sc.numel() == 0
    # every document empty
    got = run_maxsim(build_maxsim(name="empty", lq=8, d=64, num_docs=50, len_lo=-2, len_hi=0, seed=3))
    assert np.all(np.isneginf(got))
    # one document covering the whole tensor
    w1 = build_maxsim(name="one", lq=32, d=128, num_docs=1, len_lo=3000, len_hi=3000, seed=9, gap_hi=0)
    assert_close(w1, run_maxsim(w1))


def test_maxsim_repeat_calls_and_graph():
    """Results do not depend on which CTA took which document: repeated calls and a CUDA
    graph replay give identical bits."""
    sel = lib()
    w = build_maxsim(name="rep", lq=32, d=128, num_docs=700, len_lo=1, len_hi=400, seed=77)
    q, docs, off, ln = _t(w.q), _t(w.docs), _t(w.offsets), _t(w.lengths)
    ws = torch.zeros(sel.sel_maxsim_workspace_bytes(), dtype=torch.uint8, device=DEV)
    first = sel.sel_maxsim_rerank(q, docs, off, ln, ws=ws).clone()
    second = sel.sel_maxsim_rerank(q, docs, off, ln, ws=ws)
    out = torch.empty_like(first)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        sel.sel_maxsim_rerank(q, docs, off, ln, scores=out, ws=ws, stream=s)
    out.fill_(7.0)
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(first, second) and torch.equal(first, out)
    assert_close(w, first.cpu().numpy())
    assert int(ws.sum().item()) == 0, "the kernel leaves its workspace counters at zero"


def test_maxsim_workspace_left_zero_across_query_blocks():
    """300 query rows run as three launches on one workspace; each leaves it zero-filled,
    and a second call on the same workspace gives the same bits."""
    sel = lib()
    w = build_maxsim(name="blocks", lq=300, d=128, num_docs=40, len_lo=0, len_hi=120, seed=12, values="int")
    ws = torch.zeros(sel.sel_maxsim_workspace_bytes(), dtype=torch.uint8, device=DEV)
    q, docs, off, ln = _t(w.q), _t(w.docs), _t(w.offsets), _t(w.lengths)
    a = sel.sel_maxsim_rerank(q, docs, off, ln, ws=ws).clone()
    assert int(ws.sum().item()) == 0
    b = sel.sel_maxsim_rerank(q, docs, off, ln, ws=ws)
    torch.cuda.synchronize()
    assert torch.equal(a, b)
    ref, _ = oracle.maxsim(w.q, w.docs, w.offsets, w.lengths)
    np.testing.assert_array_equal(a.cpu().numpy(), ref)


@pytest.mark.parametrize("values", ["normal", "int"])
def test_maxsim_rerank4k_sampled(values):
    """The benchmark's rerank batch (4096 documents, about 1.05 M rows) in the benchmark's
    launch configuration; the oracle checks 256 sampled documents."""
    w = make_maxsim("maxsim_rerank4k", values=values)
    got = run_maxsim(w)
    idx = np.random.default_rng(11).choice(w.num_docs, size=256, replace=False)
    if values == "int":
        ref, _ = oracle.maxsim(w.q, w.docs, w.offsets[idx], w.lengths[idx])
        np.testing.assert_array_equal(got[idx], ref)
    else:
        assert_close(w, got, idx)
