"""Benchmark of the fused sparse-attention token selection (sel_select) on GB300.

One step = one pass of the whole selection (segment builder, tensor-core scorer, exact
top-k with expansion and remap, per chunk of rows) over one batch of the 128K-context
decode workload: 8 requests
x 5 rows at contexts 131,068..131,072, 4 heads x 128 dims fp16 queries and
compressed keys drawn from N(0,1)/sqrt(128), kpool 4, index_topk 2048, shuffled 64-token
blocks and key pages interleaved with other layers' pages. Inputs are synthetic and
seeded (workloads.make_workload("decode128k")).

Timing: the step is captured once in a CUDA graph and replayed; before every timed
replay a 2 x L2-sized buffer is written (outside the timed events) so the 64 MiB of
keys come from HBM. Each replay is bracketed by CUDA events on the replay stream.

Prints one JSON line (rank 0). --impl reference times the CPU oracle on the host
cores instead (the same workload, a bounded sample of rows per step).
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import workloads  # noqa: E402

METRIC = "selected rows/s and achieved HBM GB/s (% of GB300 peak) at 128K context"
UNIT = "rows/s"
WORKLOAD_DESC = ("decode 8 requests x 5 rows at 128K context (ctx 131,068..131,072), H=4, D=128 fp16 "
                 "N(0,1)/sqrt(128), kpool 4, index_topk 2048, 64-token blocks (stride 128 rows), "
                 "key pages interleaved (stride 2 pages)")


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", default="decode128k", choices=sorted(workloads.CONFIGS))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-remap", action="store_true", help="skip the stand-alone remap measurements")
    ap.add_argument("--no-maxsim", action="store_true", help="skip the MaxSim rerank measurement")
    ap.add_argument("--no-mla", action="store_true", help="skip the sparse MLA decode measurement")
    ap.add_argument("--no-flush", action="store_true", help="skip the L2 flush (profiling runs)")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the ragged and mixed workloads measured beside the headline")
    return ap.parse_args()


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    return rank, local, world


def max_over_ranks(x: float, world: int, device) -> float:
    """The largest of the ranks' values (every rank gets it); x itself with one rank."""
    if world <= 1:
        return float(x)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_rows_per_s(world: int, rows: int, steps: int, slowest_ms: float) -> float:
    """Whole-job throughput of N replicas: every rank processes `rows` rows per step, and the
    job takes as long as its slowest rank."""
    return world * rows * steps / (slowest_ms / 1e3)


# ---------------------------------------------------------------- byte accounting
def algorithmic_bytes(w):
    """Per-step algorithmic bytes of the selection (and of the scorer alone).

    Key-cache bytes each request's complete visible pools need, read once per request
    (only requests with a row whose context exceeds index_topk; 256 B per pool), the
    query rows that are scored (1 KiB each), the key-page-table and block-table rows
    (once per request), positions and query_start_loc, and the int32 slots [rows, W]
    plus valid counts written."""
    ctx = w.positions.astype(np.int64) + 1
    keys = q = kpt = bt = 0
    for i in range(w.num_reqs):
        lo, hi = int(w.qsl[i]), int(w.qsl[i + 1])
        c = ctx[lo:hi]
        big = c[c > w.index_topk]
        if big.size:
            pools = int(big.max()) // w.kpool
            keys += pools * 128 * 2
            q += big.size * 4 * 128 * 2
            kpt += -(-pools // 64) * 4
        if hi > lo:
            bt += -(-int(c.max()) // w.block_size) * 4
    meta = w.num_rows * 4 + (w.num_reqs + 1) * 4
    out = w.num_rows * w.out_width * 4 + w.num_rows * 4
    return dict(step=keys + q + kpt + bt + meta + out, scorer=keys + q + kpt, keys=keys, topk_out=out + bt)


def algorithmic_flops(w):
    """Tensor-core work of a step: 2 flops per multiply-add of every scored row (context above
    index_topk) against its own complete pools, 4 heads x 128 dims."""
    ctx = w.positions.astype(np.int64) + 1
    flops = 0
    for i in range(w.num_reqs):
        c = ctx[int(w.qsl[i]):int(w.qsl[i + 1])]
        flops += int((c[c > w.index_topk] // w.kpool).sum()) * 2 * 4 * 128
    return flops


def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            m = json.load(f)
        return float(m["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def measured_tensor_peak():
    """Dense bf16 tensor-core TFLOP/s sustained under the power cap (fp16 has the same nominal
    rate on this part), and where the number comes from."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            m = json.load(f)
        return float(m["bf16_tflops_sustained"]), "measured (bf16_tflops_sustained)"
    except Exception:
        return 1700.0, "fallback"


def recorded_traffic(kernel_file, workload):
    """DRAM bytes per launch recorded from an ncu capture in profiles/, valid only while
    the kernel source still has the hash recorded with it."""
    src = os.path.join(ROOT, "sparse_attention_kv_device_gb300", "csrc", kernel_file)
    prof = os.path.join(ROOT, "profiles", f"{kernel_file[:-3]}_{workload}.md")
    try:
        sha = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
        txt = open(prof).read()
        m_sha = re.search(r"source sha256\[:16\]:\s*([0-9a-f]{16})", txt)
        m_b = re.search(r"dram bytes per launch:\s*([0-9]+)", txt)
        if m_sha and m_b and m_sha.group(1) == sha:
            return int(m_b.group(1))
    except OSError:
        pass
    return None


# ---------------------------------------------------------------- clocks
class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.path = f"/tmp/sel_clocks_{os.getpid()}.csv"

    def start(self):
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.QUERY}",
                                          "--format=csv,noheader,nounits", "-lms", "20"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
            time.sleep(0.15)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.05)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.f.close()
        with open(self.path) as f:
            out = self.summarize(f)
        os.unlink(self.path)
        return out

    @staticmethod
    def summarize(lines):
        """Median SM clock, largest max clock and the throttle reasons seen active, from the
        CSV rows of QUERY (rows that do not parse are skipped); None without a sample."""
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": float(max(mx)), "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------- CPU oracle legs
def time_oracle(w, rows_per_step, steps, warmup, threads):
    import oracle
    n = w.num_rows
    times = []
    cursor = 0
    for s in range(warmup + steps):
        rows = (np.arange(rows_per_step) + cursor) % n
        cursor = (cursor + rows_per_step) % n
        t0 = time.perf_counter()
        oracle.select(w, rows=rows.astype(np.int32), nthreads=threads)
        dt = time.perf_counter() - t0
        if s >= warmup:
            times.append(dt)
    return float(np.sum(times)), times


def cpu_baseline(w, budget_s=12.0):
    import oracle
    threads = os.cpu_count() or 1
    rows = np.arange(w.num_rows, dtype=np.int32)
    done, t_total = 0, 0.0
    while t_total < budget_s and done < 50:
        t0 = time.perf_counter()
        oracle.select(w, rows=rows, nthreads=threads)
        t_total += time.perf_counter() - t0
        done += 1
    # one thread on a few rows as well (the oracle's per-core rate)
    one_rows = rows[:min(8, w.num_rows)]
    t0 = time.perf_counter()
    oracle.select(w, rows=one_rows, nthreads=1)
    t_one = time.perf_counter() - t0
    return {"value": done * w.num_rows / t_total, "unit": UNIT, "cores": threads, "kind": "oracle",
            "sample": f"{done} full steps ({w.num_rows} rows each) of the {w.name} workload, "
                      f"{threads} threads, {t_total:.1f} s",
            "single_thread": {"value": one_rows.size / t_one, "unit": UNIT,
                              "sample": f"{one_rows.size} rows, 1 thread, {t_one:.2f} s"}}


def run_reference(args):
    rank, _, world = dist_env()
    if rank != 0:
        return 0
    w = workloads.make_workload(args.config)
    threads = os.cpu_count() or 1
    rows_per_step = min(threads, w.num_rows)
    total, times = time_oracle(w, rows_per_step, args.steps, args.warmup, threads)
    value = rows_per_step * args.steps / total
    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": 1e3 * total / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "impl": "reference",
            "config": {"workload": WORKLOAD_DESC if args.config == "decode128k" else args.config,
                       "rows_per_step": rows_per_step, "l2": "n/a (CPU)"},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle",
                             "sample": f"{rows_per_step} rows of the {w.name} workload per step "
                                       f"(rotating over its {w.num_rows} rows), {threads} threads"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------- GPU arm
def remap_modes(sel, torch, dev, stream, flush, peak, iters):
    """The remap kernel's three modes (global slots, prefill workspace, one DCP rank with
    compaction) on the mixed step's output: 16 decode rows at 128K context (one request
    each) and 4,096 prefill rows of one request at contexts 60,001..64,096, 2,052 token
    columns shaped like the selection's output (ascending pools of 4 plus the trailing
    pool, -1 padding; 33.8 MB in, 33.8 MB out), a 2,048-block table row per request. Also
    the global mode on uniformly random token columns (the worst case for the block-table
    gather). CUDA events on the launching stream. `us`: per launch of a run of four
    back-to-back launches over four distinct token/slot buffer pairs (270 MB, above L2: each
    launch reads cold tokens), L2 flushed before each run; `us_single`: one launch between
    its own events, L2 flushed before it (this adds the launch latency to the kernel)."""
    rows, width, nreq, nb, nkv = 4112, 2052, 17, 2048, 40000
    rng = np.random.default_rng(77)
    bt = torch.from_numpy(rng.permutation(nkv)[:nreq * nb].reshape(nreq, nb).astype(np.int32)).to(dev)
    req_np = np.where(np.arange(rows) < 16, np.arange(rows), 16).astype(np.int32)
    ctx = np.where(np.arange(rows) < 16, 131072, 60001 + np.arange(rows) - 16)
    req = torch.from_numpy(req_np).to(dev)
    wsr = torch.from_numpy(np.where(np.arange(rows) < 16, -1, 0).astype(np.int32)).to(dev)
    starts = torch.tensor([1 << 20], dtype=torch.int32, device=dev)
    run = 4  # buffer pairs of one timed run
    tok = torch.from_numpy(workloads.selection_token_indices(ctx, width, seed=5)).to(dev)
    tok_rand = torch.from_numpy(workloads.random_token_indices(rows, width, nb * 64, seed=5)).to(dev)
    toks = [tok] + [tok.clone() for _ in range(run - 1)]
    toks_rand = [tok_rand] + [tok_rand.clone() for _ in range(run - 1)]
    slots = [torch.empty((rows, width), dtype=torch.int32, device=dev) for _ in range(run)]
    counts = [torch.empty(rows, dtype=torch.int32, device=dev) for _ in range(run)]
    calls = {
        "global": lambda i: sel.sel_remap_global(req, bt, toks[i], slots[i], num_kv_blocks=nkv,
                                                 valid_counts=counts[i], stream=stream),
        "workspace": lambda i: sel.sel_remap_workspace(req, bt, wsr, starts, toks[i], slots[i], num_kv_blocks=nkv,
                                                       valid_counts=counts[i], stream=stream),
        "dcp_compact": lambda i: sel.sel_remap_dcp(req, bt, toks[i], slots[i], num_kv_blocks=nkv, dcp_size=4,
                                                   dcp_rank=1, interleave=16, compact=True, valid_counts=counts[i],
                                                   stream=stream),
        "global_random_tokens": lambda i: sel.sel_remap_global(req, bt, toks_rand[i], slots[i], num_kv_blocks=nkv,
                                                               valid_counts=counts[i], stream=stream),
    }
    nbytes = 2 * rows * width * 4 + 3 * rows * 4 + nreq * nb * 4
    out = {"shape": f"{rows} rows x {width} tokens (selection-shaped; the last mode: random tokens)",
           "algorithmic_bytes": nbytes,
           "timing": f"us: per launch of {run} back-to-back launches over {run} distinct buffer pairs "
                     f"({run * 2 * rows * width * 4 / 1e6:.0f} MB, above L2), L2 flushed before each run; "
                     "us_single: one launch between its own events after an L2 flush"}
    with torch.cuda.stream(stream):
        for name, call in calls.items():
            for i in range(run):
                call(i)
            ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(iters)]
            for a, b in ev:
                flush()
                a.record(stream)
                for i in range(run):
                    call(i)
                b.record(stream)
            stream.synchronize()
            ms = float(np.mean([a.elapsed_time(b) for a, b in ev])) / run
            ev1 = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(iters)]
            for a, b in ev1:
                flush()
                a.record(stream)
                call(0)
                b.record(stream)
            stream.synchronize()
            ms1 = float(np.mean([a.elapsed_time(b) for a, b in ev1]))
            gbs = nbytes / (ms * 1e-3) / 1e9
            out[name] = {"us": ms * 1e3, "GB/s": gbs, "frac": gbs / peak, "us_single": ms1 * 1e3,
                         "frac_single": nbytes / (ms1 * 1e-3) / 1e9 / peak}
    return out


def maxsim_rerank(sel, torch, dev, stream, flush, peak, iters):
    """MaxSim rerank of a 32 x 128 query against 4,096 packed documents of 1..512 rows
    (about 1.05 M rows, 270 MB of fp16, above L2; L2 flushed before each call as well),
    CUDA events on the launching stream around each CUDA-graph replay of the call (one kernel).
    Algorithmic bytes: every document row once (d * 2 bytes), each document's offset,
    length and score (12 bytes), and the query once."""
    from workloads.maxsim import make_maxsim
    w = make_maxsim("maxsim_rerank4k")
    lq, d = w.q.shape
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)
    q, docs, off, ln = t(w.q), t(w.docs), t(w.offsets), t(w.lengths)
    scores = torch.empty(w.num_docs, dtype=torch.float32, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    ws = torch.zeros(sel.sel_maxsim_workspace_bytes(), dtype=torch.uint8, device=dev)
    call = lambda: sel.sel_maxsim_rerank(q, docs, off, ln, scores=scores, status=status, ws=ws, stream=stream)
    nbytes = w.doc_rows * d * 2 + w.num_docs * 12 + lq * d * 2
    with torch.cuda.stream(stream):
        for _ in range(3):
            call()
    stream.synchronize()
    graph = torch.cuda.CUDAGraph()  # timed as a graph replay, like the selection step
    with torch.cuda.graph(graph, stream=stream):
        call()
    with torch.cuda.stream(stream):
        graph.replay()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(iters)]
        for a, b in ev:
            flush()
            a.record(stream)
            graph.replay()
            b.record(stream)
    stream.synchronize()
    if int(status.item()) != 0:
        raise RuntimeError(f"device status {int(status.item())} in the MaxSim rerank")
    ms = float(np.mean([a.elapsed_time(b) for a, b in ev]))
    gbs = nbytes / (ms * 1e-3) / 1e9
    return {"workload": f"maxsim_rerank4k: lq {lq}, d {d}, {w.num_docs} docs, {w.doc_rows} rows",
            "algorithmic_bytes": nbytes, "us": ms * 1e3, "doc_rows_per_s": w.doc_rows / (ms * 1e-3),
            "docs_per_s": w.num_docs / (ms * 1e-3), "GB/s": gbs, "frac": gbs / peak,
            "traffic": recorded_traffic("k_maxsim.cu", "rerank4k"),
            "gpu_launches": sel.sel_maxsim_launch_count(lq, d)}


def mla_decode(sel, torch, dev, stream, flush, peak, tpeak, iters):
    """Sparse MLA decode attention over the selected slots of the 128K decode step: 40 rows x
    16 heads, 2,048..2,051 entries per row gathered from a 2^20-slot bf16 cache (1.2 GB) of
    512 latent + 64 rotary dims. CUDA-graph replay of the call (two kernels), L2 flushed before
    each replay, CUDA events on the launching stream. Algorithmic bytes: every valid entry's
    cache row once (1,152 B), the slot indices read (4 B per entry below kv_len), the queries,
    out (fp32) and lse written. FLOPs: both products, 2 * 16 * (576 + 512) per entry."""
    from workloads.mla import make_mla
    w = make_mla("mla_decode128k")
    bf = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev).view(torch.bfloat16)
    cache = bf(w.cache)
    qn, qp = bf(w.q_nope), bf(w.q_pe)
    ckv, kpe = cache[:, :w.dc], cache[:, w.dc:]
    slots = torch.from_numpy(w.slots).to(dev)
    kv_len = torch.from_numpy(w.kv_len).to(dev)
    rows, heads, dc = w.q_nope.shape
    out = torch.empty((rows, heads, dc), dtype=torch.float32, device=dev)
    lse = torch.empty((rows, heads), dtype=torch.float32, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    ws = sel.new_workspace(sel.sel_mla_workspace_bytes(rows, w.slots.shape[1]), dev)
    call = lambda: sel.sel_mla_decode(qn, qp, ckv, kpe, slots, kv_len, w.sm_scale, out=out, lse=lse,
                                      status=status, ws=ws, stream=stream)
    valid = 0
    for r in range(rows):
        s = w.slots[r, :int(w.kv_len[r])]
        valid += int(((s >= 0) & (s < w.cache.shape[0])).sum())
    entries = int(np.minimum(w.kv_len, w.slots.shape[1]).sum())
    nbytes = (valid * (w.dc + w.dr) * 2 + entries * 4 + rows * 4 + rows * heads * (w.dc + w.dr) * 2
              + rows * heads * (dc + 1) * 4)
    flops = 2 * heads * (w.dc + w.dr + w.dc) * valid
    with torch.cuda.stream(stream):
        for _ in range(3):
            call()
    stream.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        call()
    with torch.cuda.stream(stream):
        graph.replay()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(iters)]
        for a, b in ev:
            flush()
            a.record(stream)
            graph.replay()
            b.record(stream)
    stream.synchronize()
    if int(status.item()) != 0:
        raise RuntimeError(f"device status {int(status.item())} in the MLA decode")
    times = [a.elapsed_time(b) for a, b in ev]
    ms = float(np.mean(times))
    gbs = nbytes / (ms * 1e-3) / 1e9
    return {"workload": f"mla_decode128k: {rows} rows x {heads} heads, {entries} entries "
                        f"({valid} valid), dc {w.dc} + dr {w.dr} bf16, 2^20 cache slots",
            "algorithmic_bytes": nbytes, "us": ms * 1e3, "us_median": float(np.median(times)) * 1e3,
            "rows_per_s": rows / (ms * 1e-3), "GB/s": gbs, "frac": gbs / peak, "bound": "hbm",
            "algorithmic_flops": flops, "TFLOP/s": flops / (ms * 1e-3) / 1e12, "tensor_frac": flops / (ms * 1e-3) / 1e12 / tpeak,
            "traffic": recorded_traffic("k_mla.cu", "mla_decode128k"),
            "gpu_launches": sel.sel_mla_launch_count(rows)}


def eager_steps(sel, torch, prob, slots, counts, ws, stream, flush, rows, iters):
    """The same step launched eagerly (sel_select called from Python every step, no graph), L2
    flushed before each call, CUDA events on the stream around each call."""
    with torch.cuda.stream(stream):
        for _ in range(3):
            flush()
            sel.sel_select(prob, slots, counts, ws=ws, stream=stream)
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(iters)]
        for a, b in ev:
            flush()
            a.record(stream)
            sel.sel_select(prob, slots, counts, ws=ws, stream=stream)
            b.record(stream)
    stream.synchronize()
    ms = np.array([a.elapsed_time(b) for a, b in ev])
    med = float(np.median(ms))
    return {"median_ms": med, "p10_ms": float(np.percentile(ms, 10)), "p90_ms": float(np.percentile(ms, 90)),
            "rows_per_s": rows / (med * 1e-3), "launches_per_step": sel.sel_select_launch_count(prob)}


def graph_steps(sel, torch, prob, slots, counts, ws, stream, flush, iters, warmup=5, status=None):
    """CUDA-graph replays of one sel_select call, L2 flushed before each, CUDA events on the
    replay stream around each replay; returns the per-step times in ms."""
    with torch.cuda.stream(stream):
        sel.sel_select(prob, slots, counts, status=status, ws=ws)
    stream.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        sel.sel_select(prob, slots, counts, status=status, ws=ws)
    with torch.cuda.stream(stream):
        for _ in range(warmup):
            flush()
            graph.replay()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(iters)]
        for a, b in ev:
            flush()
            a.record(stream)
            graph.replay()
            b.record(stream)
    stream.synchronize()
    return np.array([a.elapsed_time(b) for a, b in ev])


def config_leg(sel, torch, dev, stream, flush, name, iters, peak, tpeak, chunk_rows=None):
    """One of the other workloads (ragged decode, the mixed step) timed like the headline:
    rows/s, time per step, algorithmic bytes and the fraction of the HBM copy peak; for a
    step with a large tensor-core share also the fraction of the tensor peak, and the
    larger of the two as the roofline fraction. chunk_rows overrides the workload's logits
    chunk (0: the library's own choice)."""
    w = workloads.make_workload(name)
    prob = sel.problem_from_workload(w, dev, **({} if chunk_rows is None else {"chunk_rows": chunk_rows}))
    slots = torch.empty((w.num_rows, w.out_width), dtype=torch.int32, device=dev)
    counts = torch.empty(w.num_rows, dtype=torch.int32, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    ws = sel.new_workspace(sel.sel_workspace_bytes(prob), dev)
    ms = graph_steps(sel, torch, prob, slots, counts, ws, stream, flush, iters, status=status)
    if int(status.item()) != 0:
        raise RuntimeError(f"device status {int(status.item())} on {name}")
    ab = algorithmic_bytes(w)
    fl = algorithmic_flops(w)
    mean = float(ms.mean())
    gbs = ab["step"] / (mean * 1e-3) / 1e9
    tfs = fl / (mean * 1e-3) / 1e12
    out = {"workload": name, "rows": w.num_rows, "requests": w.num_reqs,
           "us_per_step": {"mean": mean * 1e3, "median": float(np.median(ms)) * 1e3,
                           "p10": float(np.percentile(ms, 10)) * 1e3, "p90": float(np.percentile(ms, 90)) * 1e3},
           "rows_per_s": w.num_rows / (mean * 1e-3), "algorithmic_bytes": ab["step"], "GB/s": gbs,
           "hbm_frac": gbs / peak, "algorithmic_flops": fl, "TFLOP/s": tfs, "tensor_frac": tfs / tpeak,
           "launches_per_step": sel.sel_select_launch_count(prob)}
    out["bound"] = "tensor" if out["tensor_frac"] > out["hbm_frac"] else "hbm"
    out["frac"] = max(out["hbm_frac"], out["tensor_frac"])
    return out


def auxiliary(fn):
    """Runs one of the side measurements; a failure is reported in its place instead of
    suppressing the headline line."""
    try:
        return fn()
    except Exception as e:  # noqa: BLE001 -- any failure of a side measurement is reported as data
        return {"error": f"{type(e).__name__}: {e}"[:400]}


def run_ours(args):
    import torch
    import torch.distributed as dist

    import sparse_attention_kv_device_gb300 as sel

    rank, local, world = dist_env()
    if world > 1:
        dist.init_process_group("nccl", init_method="env://")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    w = workloads.make_workload(args.config)
    prob = sel.problem_from_workload(w, dev)
    rows = w.num_rows
    slots = torch.empty((rows, w.out_width), dtype=torch.int32, device=dev)
    counts = torch.empty(rows, dtype=torch.int32, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    ws = sel.new_workspace(sel.sel_workspace_bytes(prob), dev)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush_buf = torch.empty(max(2 * l2, 256 << 20) // 4, dtype=torch.float32, device=dev)

    stream = torch.cuda.Stream(device=dev)
    with torch.cuda.stream(stream):
        sel.sel_select(prob, slots, counts, status=status, ws=ws)
    stream.synchronize()
    if int(status.item()) != 0:
        raise RuntimeError(f"device status {int(status.item())} on the warm-up step")
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        sel.sel_select(prob, slots, counts, status=status, ws=ws)

    def flush():
        if not args.no_flush:
            flush_buf.zero_()

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            flush()
            graph.replay()
    stream.synchronize()

    # ---- timed region: K graph replays, each between its own events, L2 flushed before each
    ev_s = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ev_e = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    clocks = ClockSampler(local)
    clocks.start()
    t_wall = time.perf_counter()
    with torch.cuda.stream(stream):
        for i in range(args.steps):
            flush()
            ev_s[i].record(stream)
            graph.replay()
            ev_e[i].record(stream)
    torch.cuda.synchronize(dev)
    t_wall = time.perf_counter() - t_wall
    if world > 1:
        dist.barrier()
    clk = clocks.stop()
    step_ms = np.array([a.elapsed_time(b) for a, b in zip(ev_s, ev_e)])
    total_ms = max_over_ranks(float(step_ms.sum()), world, dev)
    value = job_rows_per_s(world, rows, args.steps, total_ms)
    ok_status = int(status.item())

    # ---- per-kernel times from trace events captured into a second graph
    trace = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
    sel.sel_set_trace_events(trace)
    try:
        tgraph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(tgraph, stream=stream):
            sel.sel_select(prob, slots, counts, status=status, ws=ws)
    finally:
        sel.sel_set_trace_events(None)
    n_tr = min(args.steps, 100)
    parts = np.zeros((n_tr, 3))
    with torch.cuda.stream(stream):
        for i in range(n_tr):
            flush()
            tgraph.replay()
            stream.synchronize()
            parts[i] = [trace[j].elapsed_time(trace[j + 1]) for j in range(3)]
    kern_ms = parts.mean(axis=0)   # builder, scorer, selection tail (the event nodes stop the PDL overlap)

    launches = sel.sel_select_launch_count(prob)
    ab = algorithmic_bytes(w)
    peak, peak_kind = measured_peaks()
    tpeak, tpeak_kind = measured_tensor_peak()
    names = ["k_build_segments", "k_score_segments", "k_select_rows"]
    dom = int(np.argmax(kern_ms))
    dom_bytes = [w.num_rows * 8 + (w.num_reqs + 1) * 4, ab["scorer"], ab["topk_out"]][dom]
    achieved = dom_bytes / (kern_ms[dom] * 1e-3) / 1e9
    traffic = recorded_traffic("k_score.cu", args.config) if dom == 1 else None
    step_gbs = ab["step"] / (total_ms / args.steps * 1e-3) / 1e9

    # ---- end to end through the host-buffer entry point (pinned host inputs and outputs)
    e2e = None
    if not args.no_e2e:
        hp = lambda a: torch.from_numpy(np.ascontiguousarray(a)).pin_memory()
        hprob = sel.Problem(query_start_loc=hp(w.qsl), positions=hp(w.positions), q=hp(w.q),
                            key_cache=prob.tensors[3], key_page_table=hp(w.key_page_table),
                            block_table=hp(w.block_table), index_topk=w.index_topk, kpool=w.kpool,
                            max_context=w.max_context, key_page_stride=w.key_page_stride,
                            num_key_pages=w.num_key_pages, num_kv_blocks=w.num_kv_blocks,
                            block_stride_rows=w.block_stride_rows, max_q_len=w.max_q_len,
                            max_key_pages_per_req=w.max_key_pages_per_req,
                            max_blocks_per_req=w.max_blocks_per_req, host_inputs=True)
        slots_h = torch.empty((rows, w.out_width), dtype=torch.int32).pin_memory()
        counts_h = torch.empty(rows, dtype=torch.int32).pin_memory()
        stage = torch.empty(sel.sel_host_stage_bytes(hprob, w.out_width), dtype=torch.uint8, device=dev)
        e_s = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
        e_e = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
        with torch.cuda.stream(stream):
            for _ in range(args.warmup):
                sel.sel_select_host(hprob, slots_h, counts_h, stage, ws, stream=stream)
            for i in range(args.steps):
                flush()
                e_s[i].record(stream)
                sel.sel_select_host(hprob, slots_h, counts_h, stage, ws, stream=stream)
                e_e[i].record(stream)
        torch.cuda.synchronize(dev)
        e2e_ms = max_over_ranks(float(sum(a.elapsed_time(b) for a, b in zip(e_s, e_e))), world, dev)
        h2d = (w.qsl.nbytes + w.positions.nbytes + w.q.nbytes + w.key_page_table.nbytes
               + w.block_table.nbytes)
        d2h = rows * w.out_width * 4 + rows * 4
        e2e = {"value": job_rows_per_s(world, rows, args.steps, e2e_ms), "unit": UNIT,
               "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h)}

    eager = auxiliary(lambda: eager_steps(sel, torch, prob, slots, counts, ws, stream, flush, rows, 50))
    configs = None
    if not args.no_configs:
        configs = {n: auxiliary(lambda n=n: config_leg(sel, torch, dev, stream, flush, n, 20, peak, tpeak))
                   for n in ("ragged", "mixed") if n != args.config}
        # the mixed step again with the library's default chunking (larger than the workload's
        # 256-row logits chunks; see chunk_rows in include/sel.h): for information, not the config
        configs["mixed_library_chunks"] = auxiliary(
            lambda: config_leg(sel, torch, dev, stream, flush, "mixed", 20, peak, tpeak, chunk_rows=0))
    remap = None
    if not args.no_remap:
        remap = auxiliary(lambda: remap_modes(sel, torch, dev, stream, flush, peak, 20))
    maxsim = None
    if not args.no_maxsim:
        maxsim = auxiliary(lambda: maxsim_rerank(sel, torch, dev, stream, flush, peak, 20))
    mla = None
    if not args.no_mla:
        mla = auxiliary(lambda: mla_decode(sel, torch, dev, stream, flush, peak, tpeak, 20))

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(w)

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": total_ms / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f16", "data": "synthetic",
            "config": {"workload": WORKLOAD_DESC if args.config == "decode128k" else args.config,
                       "rows": rows, "requests": w.num_reqs, "out_width": w.out_width,
                       "l2": "flushed before every step (2x L2 buffer written outside the timed events)"
                             if not args.no_flush else "not flushed",
                       "timing": "CUDA-graph replay of sel_select, CUDA events per step on the replay stream",
                       "parallelism": f"replicas x{world}"},
            "step_ms": {"median": float(np.median(step_ms)), "p10": float(np.percentile(step_ms, 10)),
                        "p90": float(np.percentile(step_ms, 90))},
            "hbm_gbs_step": step_gbs, "hbm_frac_step": step_gbs / peak,
            "algorithmic_bytes_per_step": ab["step"],
            "kernel_ms": {n: float(v) for n, v in zip(names, kern_ms)},
            "roofline": {"bound": "hbm", "kernel": names[dom], "achieved": achieved, "peak": peak,
                         "unit": "GB/s", "frac": achieved / peak, "traffic": traffic,
                         "algorithmic_bytes": dom_bytes, "launches_per_step": launches,
                         "peak_source": f"{peak_kind} (hbm_gbs, burst copy)",
                         "tensor": {"algorithmic_flops": algorithmic_flops(w),
                                    "TFLOP/s": algorithmic_flops(w) / (kern_ms[1] * 1e-3) / 1e12,
                                    "peak": tpeak, "peak_source": tpeak_kind}},
            "gpu_launches": launches * args.steps,
            "status": ok_status,
            "wall_s_timed_region": t_wall,
        }
        if clk:
            line["clocks"] = clk
        if e2e:
            line["e2e"] = e2e
        if cpu:
            line["cpu_baseline"] = cpu
        if eager:
            line["eager_step"] = eager
        if remap:
            line["remap_modes"] = remap
        if maxsim:
            line["maxsim_rerank"] = maxsim
        if mla:
            line["mla_decode"] = mla
        if configs:
            line["configs"] = configs
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


def main():
    args = parse()
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
