"""Host logic of bench.py on the CPU: the clock-sample summary (nvidia-smi
lines as the sampler reads them) and the check that a recorded DRAM traffic
figure is only reported while the kernel's sources are unchanged."""
import json

import bench

LINE = "{sm}, 2070, 1180.5, 0x0000000000000000, {hw}, {hwt}, {swt}, {cap}"


def _line(sm, hw="Not Active", hwt="Not Active", swt="Not Active", cap="Not Active"):
    return LINE.format(sm=sm, hw=hw, hwt=hwt, swt=swt, cap=cap)


def test_clock_summary_inside_window():
    samples = [(0.0, _line(1000)), (1.0, _line(2070)), (1.1, _line(2070, cap="Active")), (1.2, _line(2055)),
               (5.0, _line(900, hwt="Active"))]
    c = bench.ClockSampler.summarize(samples, (0.95, 1.25))
    assert c == {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"], "samples": 3}


def test_clock_summary_reports_slowdowns_and_skips_bad_lines():
    samples = [(1.0, "garbled"), (1.0, _line("N/A")), (1.05, _line(1500, hw="Active", swt="Active"))]
    c = bench.ClockSampler.summarize(samples, (1.0, 1.1))
    assert c["reasons"] == ["hw_slowdown", "sw_thermal_slowdown"] and c["samples"] == 1


def test_clock_summary_nearest_sample_and_empty():
    samples = [(0.0, _line(1900)), (10.0, _line(2070))]
    assert bench.ClockSampler.summarize(samples, (4.0, 4.2))["sm_mhz"] == 1900.0
    assert bench.ClockSampler.summarize([], (0.0, 1.0)) is None


def test_traffic_only_while_sources_unchanged(tmp_path, monkeypatch):
    src = tmp_path / "k.cu"
    src.write_text("kernel v1")
    rec = tmp_path / "traffic.json"
    monkeypatch.setattr(bench, "KERNEL_SOURCES", [str(src)])
    monkeypatch.setattr(bench, "TRAFFIC_FILE", str(rec))
    assert bench.traffic_per_launch() is None  # no record
    rec.write_text(json.dumps({"sources_sha256": bench.sha_of([str(src)]), "bytes_per_launch": 123}))
    assert bench.traffic_per_launch() == 123
    src.write_text("kernel v2")  # the kernel changed since the capture
    assert bench.traffic_per_launch() is None
