"""sel_mla_decode (sparse MLA decode attention over the selected slots) against the oracle's
double-precision definition, through the C ABI.

Tolerance, from the kernel's arithmetic. The logits are exact bf16 x bf16 products summed in
fp32 over 576 dims (relative error about 576 * 2^-24 of the sum of |terms|, negligible here).
The softmax weights p_j enter the second product rounded to bf16 (relative error <= 2^-9 each)
and are normalised by the sum of the rounded weights, so the kernel's output is
sum_j w'_j v_j with w'_j = w_j (1 + e_j) / (1 + e_avg), |e| <= 2^-9, and
|out - out*| = |sum_j (w'_j - w_j)(v_j - out*)| <= 2^-8 / (1 - 2^-9) * sum_j w_j |v_j - out*|.
The test allows B[r,h,d] = 1.01 * 2^-8 * sum_j w_j |v_jd - out*_d| + 1e-5 * (sum_j w_j |v_jd| + 1e-3),
with the exact weights w_j recomputed here in double. The log-sum-exp uses the unrounded fp32
weights and fp32 logits: |dlse| <= 2e-4 + 1e-5 |lse|.
"""

import numpy as np
import pytest
import torch

import oracle
from _gpu import DEV, lib
from workloads.mla import build_mla, make_mla

pytestmark = pytest.mark.gpu


def _f32(bits):
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def _tensors(w, alias_cache=True, dr=None):
    bf = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(DEV).view(torch.bfloat16)
    cache = bf(w.cache)
    dc = w.dc
    qn = bf(w.q_nope)
    if w.dr == 0:
        qp, kpe = None, None
        ckv = cache[:, :dc]
    elif alias_cache:
        qp, ckv, kpe = bf(w.q_pe), cache[:, :dc], cache[:, dc:]
    else:
        qp, ckv, kpe = bf(w.q_pe), bf(w.ckv), bf(w.kpe)
    slots = torch.from_numpy(w.slots).to(DEV)
    kv_len = torch.from_numpy(w.kv_len).to(DEV)
    return qn, qp, ckv, kpe, slots, kv_len


def _run(w, **kw):
    sel = lib()
    qn, qp, ckv, kpe, slots, kv_len = _tensors(w, **kw)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    out, lse = sel.sel_mla_decode(qn, qp, ckv, kpe, slots, kv_len, w.sm_scale, status=status)
    torch.cuda.synchronize()
    return out.cpu().numpy(), lse.cpu().numpy(), int(status.item())


def _bound(w):
    """Per-element output tolerance (module docstring) from a double recomputation."""
    rows, heads, dc = w.q_nope.shape
    qn = _f32(w.q_nope).astype(np.float64)
    qp = _f32(w.q_pe).astype(np.float64)
    B = np.zeros((rows, heads, dc))
    width = w.slots.shape[1]
    for r in range(rows):
        n = min(int(w.kv_len[r]), width)
        s = w.slots[r, :n].astype(np.int64)
        s = s[(s >= 0) & (s < w.cache.shape[0])]
        if s.size == 0:
            B[r] = 1e-8
            continue
        rowc = _f32(w.cache[s]).astype(np.float64)
        v = rowc[:, :dc]
        logit = w.sm_scale * (qn[r] @ v.T + (qp[r] @ rowc[:, dc:].T if w.dr else 0.0))  # [heads, n]
        p = np.exp(logit - logit.max(axis=1, keepdims=True))
        wgt = p / p.sum(axis=1, keepdims=True)
        o = wgt @ v                                                   # [heads, dc]
        dev = np.einsum("hn,hnd->hd", wgt, np.abs(v[None, :, :] - o[:, None, :]))
        mag = wgt @ np.abs(v)
        B[r] = 1.01 * 2.0 ** -8 * dev + 1e-5 * (mag + 1e-3)
    return B


def _check(w, out, lse, status):
    assert status == 0
    ref_o, ref_l = oracle.mla_decode(w.q_nope, w.q_pe, w.ckv, w.kpe, w.slots, w.kv_len, w.sm_scale)
    empty = np.isneginf(ref_l)
    assert np.array_equal(np.isneginf(lse), empty)
    assert np.all(out[empty] == 0.0)
    full = ~empty
    assert np.all(np.abs(lse[full] - ref_l[full]) <= 2e-4 + 1e-5 * np.abs(ref_l[full]))
    err = np.abs(out.astype(np.float64) - ref_o)
    B = _bound(w)
    bad = err > B
    assert not bad.any(), (f"{int(bad.sum())} outputs outside the bound; worst ratio "
                           f"{float((err / B).max()):.3g} at {np.unravel_index(np.argmax(err / B), err.shape)}")


def test_mla_small_mixed_lengths_and_holes():
    w = make_mla("mla_small")   # kv_len 1, 7, 2047, 2048, 2049, 2048; -1 and far slots inside kv_len
    out, lse, st = _run(w)
    _check(w, out, lse, st)


def test_mla_small_without_rotary_dims_and_separate_tensors():
    w = build_mla(name="mla_small_dr0", contexts=[5, 300, 2049, 4000], heads=16, dr=0, num_slots=1 << 15,
                  seed=3011, holes=True)
    out, lse, st = _run(w)
    _check(w, out, lse, st)
    w2 = make_mla("mla_small")
    out2, lse2, st2 = _run(w2, alias_cache=False)   # ckv and kpe as their own tensors
    _check(w2, out2, lse2, st2)


def test_mla_decode128k_every_row():
    w = make_mla("mla_decode128k")   # 40 rows x 2048..2051 entries over 2^20 slots
    out, lse, st = _run(w)
    _check(w, out, lse, st)


def test_mla_many_rows_whole_and_split():
    # 300 rows: most rows run whole inside one CTA (written directly), the rest are split and
    # merged; contexts include 0 (no entry: out 0, lse -inf) and values around tile edges
    rng = np.random.default_rng(77)
    ctx = rng.integers(0, 3000, size=300)
    ctx[:6] = [0, 1, 127, 128, 129, 2048]
    w = build_mla(name="mla_many", contexts=ctx, heads=16, num_slots=1 << 16, seed=3013, holes=True)
    out, lse, st = _run(w)
    _check(w, out, lse, st)


def test_mla_repeat_calls_identical():
    w = make_mla("mla_small")
    a = _run(w)
    b = _run(w)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_mla_launch_count_and_workspace():
    sel = lib()
    assert sel.sel_mla_launch_count(40) == 2 and sel.sel_mla_launch_count(0) == 0
    assert sel.sel_mla_workspace_bytes(40, 2052) > 0
