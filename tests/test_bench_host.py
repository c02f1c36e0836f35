"""Host-side logic of bench.py, without a GPU: the clock/throttle summary of the
timed window, and the rule that the committed DRAM traffic is reported only for the
kernel code it was measured on."""

import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _line(sm, mx, hw="Not Active", hwt="Not Active", swt="Not Active", pcap="Not Active"):
    # the fields of ClockSampler.FIELDS, as nvidia-smi prints them (csv, noheader, nounits)
    return ["0", str(sm), str(mx), "700.5", "0x0", hw, hwt, swt, pcap]


def test_clock_summary_uses_only_the_timed_window():
    s = bench.ClockSampler(0)
    s.samples = [_line(900, 2070, hw="Active")] + [_line(2070, 2070)] * 3 + [_line(1995, 2070)] + \
        [_line(600, 2070, swt="Active")]
    s.first, s.last = 1, 5  # the first and the last sample fall outside the timed region
    out = bench.ClockSampler.summary(s)
    assert out["sm_mhz"] == 2070.0 and out["sm_max_mhz"] == 2070.0
    assert out["reasons"] == [] and out["samples"] == 4


def test_clock_summary_reports_throttle_reasons():
    s = bench.ClockSampler(0)
    s.samples = [_line(1800, 2070, pcap="Active"), _line(1700, 2070, hwt="Active"), _line(1900, 2070)]
    s.first, s.last = 0, 3
    out = bench.ClockSampler.summary(s)
    assert out["reasons"] == ["hw_thermal_slowdown", "sw_power_cap"]
    assert out["sm_mhz"] == 1800.0


def test_clock_summary_without_samples_or_numbers():
    s = bench.ClockSampler(0)
    s.samples = []
    assert bench.ClockSampler.summary(s)["reasons"] == ["unsampled"]
    s.samples = [["0", "[N/A]", "[N/A]", "[N/A]", "0x0", "Not Active", "Not Active", "Not Active", "Not Active"]]
    s.first, s.last = 0, 1
    out = bench.ClockSampler.summary(s)
    assert out["sm_mhz"] is None and out["sm_max_mhz"] is None and out["reasons"] == []


def test_traffic_is_reported_only_for_the_measured_code(tmp_path, monkeypatch):
    # A profile keyed to the current code is reported; any code change drops it.
    import json

    real = bench.kernel_source_hash()
    (tmp_path / "profiles").mkdir()
    (tmp_path / "profiles" / "traffic.json").write_text(
        json.dumps({"gemm_8192": {"dram_bytes_per_launch": 123, "source_hash": real}}))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "kernel_source_hash", lambda: real)
    assert bench.profiled_traffic("gemm_8192") == 123
    monkeypatch.setattr(bench, "kernel_source_hash", lambda: "0" * 16)
    assert bench.profiled_traffic("gemm_8192") is None
    monkeypatch.setattr(bench, "kernel_source_hash", lambda: real)
    assert bench.profiled_traffic("no_such_kernel") is None


def test_kernel_hash_ignores_comments_but_not_code(tmp_path, monkeypatch):
    csrc = tmp_path / "nvfp4_block_scaled_gb300" / "csrc"
    csrc.mkdir(parents=True)
    for name in ("gemm_w4a4.cu", "pair_sched.h", "ptx.cuh"):
        (csrc / name).write_text("int f() { return 1; }  // a comment\n/* block\n comment */\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    h0 = bench.kernel_source_hash()
    (csrc / "ptx.cuh").write_text("int f() {\n  return 1;   // another comment\n}\n")
    assert bench.kernel_source_hash() == h0
    (csrc / "ptx.cuh").write_text("int f() { return 2; }\n")
    assert bench.kernel_source_hash() != h0
