"""bench.py's host-side accounting, on CPU: the algorithmic bytes of each selection workload
(written out by hand for two of them), the gate that reports an ncu traffic figure only while
the kernel source still has the hash recorded with it, the peak lookup and the clock record."""

import hashlib
import json

import pytest

import bench
import workloads


def test_algorithmic_bytes_decode128k_by_hand():
    # 8 requests x 5 rows at ctx 131,068..131,072: every row is scored; per request the longest
    # row's 32,768 complete pools of 256 B are read once, its 512 key-page-table and 2,048
    # block-table entries once; each row's 4 x 128 fp16 query once; 40 positions and 9 query
    # start offsets; 40 rows of 2,052 int32 slots and 40 counts written.
    keys = 8 * 32768 * 256
    q = 40 * 4 * 128 * 2
    tables = 8 * 512 * 4 + 8 * 2048 * 4
    meta = 40 * 4 + 9 * 4
    out = 40 * 2052 * 4 + 40 * 4
    ab = bench.algorithmic_bytes(workloads.make_workload("decode128k"))
    assert ab["step"] == keys + q + tables + meta + out == 67_560_420
    assert ab["keys"] == keys
    assert ab["scorer"] == keys + q + 8 * 512 * 4


def test_algorithmic_bytes_tiny_by_hand():
    # requests of ctx 999, 1000 and 2999, 3000 (topk 256, kpool 4, W 260): 250 and 750 pools,
    # ceil(250/64) + ceil(750/64) key-page entries, ceil(1000/64) + ceil(3000/64) blocks
    keys = (250 + 750) * 256
    q = 4 * 1024
    tables = (4 + 12) * 4 + (16 + 47) * 4
    meta = 4 * 4 + 3 * 4
    out = 4 * 260 * 4 + 4 * 4
    assert bench.algorithmic_bytes(workloads.make_workload("tiny"))["step"] == keys + q + tables + meta + out


@pytest.mark.parametrize("name,step", [("decode32k", 8_546_724), ("ragged", 38_407_116), ("mixed", 176_483_676)])
def test_algorithmic_bytes_other_workloads(name, step):
    assert bench.algorithmic_bytes(workloads.make_workload(name))["step"] == step


def test_unscored_rows_read_no_query():
    # ragged_b's last request (7 rows, ctx 1,994..2,000 <= index_topk) is never scored: its
    # queries, keys and key-page-table row are not read (7 KiB less than counting its queries)
    assert bench.algorithmic_bytes(workloads.make_workload("ragged_b"))["step"] == 38_150_928 - 7 * 1024


def _fake_tree(tmp_path, src_text, prof_text):
    csrc = tmp_path / "sparse_attention_kv_device_gb300" / "csrc"
    csrc.mkdir(parents=True)
    (csrc / "k_x.cu").write_text(src_text)
    (tmp_path / "profiles").mkdir()
    if prof_text is not None:
        (tmp_path / "profiles" / "k_x_work.md").write_text(prof_text)


def test_recorded_traffic_only_for_the_captured_source(tmp_path, monkeypatch):
    src = "__global__ void k() {}\n"
    sha = hashlib.sha256(src.encode()).hexdigest()[:16]
    _fake_tree(tmp_path, src, f"source sha256[:16]: {sha}\ndram bytes per launch: 123456\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.recorded_traffic("k_x.cu", "work") == 123456
    (tmp_path / "sparse_attention_kv_device_gb300" / "csrc" / "k_x.cu").write_text(src + "// changed\n")
    assert bench.recorded_traffic("k_x.cu", "work") is None        # the kernel changed since the capture
    assert bench.recorded_traffic("k_x.cu", "other") is None       # no profile for that workload


def test_recorded_traffic_needs_both_lines(tmp_path, monkeypatch):
    src = "x"
    sha = hashlib.sha256(src.encode()).hexdigest()[:16]
    _fake_tree(tmp_path, src, f"source sha256[:16]: {sha}\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.recorded_traffic("k_x.cu", "work") is None


def test_measured_peaks_file_and_fallback(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.measured_peaks() == (6800.0, "fallback")
    (tmp_path / "MEASURED_PEAKS.json").write_text(json.dumps({"hbm_gbs": 7012.5, "bf16_tflops": 1800}))
    assert bench.measured_peaks() == (7012.5, "measured")


def test_clock_record_summary():
    rows = [
        "0, 2070, 2070, 900.1, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active",
        "0, 1995, 2070, 1350.0, 0x0000000000000004, Not Active, Not Active, Not Active, Active",
        "0, [N/A], 2070, 0.0, 0x0, Not Active, Not Active, Not Active, Not Active",   # skipped
        "garbage",
        "0, 2040, 2070, 1200.0, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active",
    ]
    out = bench.ClockSampler.summarize(rows)
    assert out == {"sm_mhz": 2040.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"], "samples": 3}
    assert bench.ClockSampler.summarize([]) is None
    hot = bench.ClockSampler.summarize(["0, 1500, 2070, 1400, 0x40, Active, Not Active, Active, Not Active"])
    assert hot["reasons"] == ["hw_slowdown", "sw_thermal_slowdown"]
