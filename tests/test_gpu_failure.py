"""Failure detection without a GPU fault: a bounded wait inside a kernel is made to run out
(the test hook leaves one tile of the launch unloaded and shortens every wait to 1 ms); the
launch must report SEL_ST_TIMEOUT and return, and the next normal call on the same buffers
must be exact again. Every wait in the kernels has such a limit, after which all roles of
the CTA leave without touching the missing data, any copy already issued lands first, and
the MaxSim workspace's work counters are still returned to zero."""

import numpy as np
import pytest
import torch

import oracle
import workloads
from _gpu import DEV, assert_select_bitexact, lib, oracle_select, run_select

pytestmark = pytest.mark.gpu

ST_TIMEOUT = 4


def test_scorer_wait_expires_then_next_call_is_exact():
    sel = lib()
    w = workloads.make_workload("decode32k")   # 4 segments x 64 tiles of 128 pools
    ref = oracle_select(w)
    sel.sel_debug_wait_limit(fault_tile=3, wait_ns=1_000_000)
    try:
        failed = run_select(w)
    finally:
        sel.sel_debug_wait_limit()
    assert failed["status"] & ST_TIMEOUT
    again = run_select(w)
    assert again["status"] == 0
    assert_select_bitexact(w, again, ref, np.arange(w.num_rows))


def test_maxsim_wait_expires_counters_back_at_zero_then_exact():
    from workloads.maxsim import make_maxsim
    sel = lib()
    wm = make_maxsim("maxsim_small", values="int")
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(DEV)
    q, docs, off, ln = t(wm.q), t(wm.docs), t(wm.offsets), t(wm.lengths)
    ws = sel.new_workspace(sel.sel_maxsim_workspace_bytes(), DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    sel.sel_debug_wait_limit(fault_tile=0, wait_ns=1_000_000)
    try:
        sel.sel_maxsim_rerank(q, docs, off, ln, status=status, ws=ws)
        torch.cuda.synchronize()
    finally:
        sel.sel_debug_wait_limit()
    assert int(status.item()) & ST_TIMEOUT
    assert int(ws.count_nonzero().item()) == 0          # the work counters are zero again
    status.zero_()
    scores = sel.sel_maxsim_rerank(q, docs, off, ln, status=status, ws=ws)
    torch.cuda.synchronize()
    ref, _ = oracle.maxsim(wm.q, wm.docs, wm.offsets, wm.lengths)
    assert int(status.item()) == 0
    np.testing.assert_array_equal(scores.cpu().numpy(), ref)
    assert int(ws.count_nonzero().item()) == 0
