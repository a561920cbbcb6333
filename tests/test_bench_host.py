"""Host logic of bench.py (no GPU): the nvidia-smi clock record, the DRAM-traffic lookup in the
committed ncu summary (null once the kernel source has changed), the measured-peak fallback, and
the workload's weight bytes."""
import json
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


class FinishedProcess:
    def terminate(self):
        pass

    def wait(self, timeout=None):
        return 0


def sampler_with(tmp_path, lines):
    s = bench.ClockSampler(0)
    s.path = str(tmp_path / "clocks.csv")
    with open(s.path, "w") as f:
        f.write("\n".join(lines) + "\n")
    s.fh = open(str(tmp_path / "unused"), "w")
    s.proc = FinishedProcess()
    return s


def test_clock_record_median_under_load_and_reasons(tmp_path):
    # index, sm, max, power, active mask, hw_slowdown, hw_thermal, sw_thermal, sw_power_cap
    lines = ["0, 345, 2070, 200.1, 0x0, Not Active, Not Active, Not Active, Not Active",  # idle, excluded
             "0, 2070, 2070, 900.0, 0x0, Not Active, Not Active, Not Active, Not Active",
             "0, 2055, 2070, 1300.0, 0x4, Not Active, Not Active, Not Active, Active",
             "0, 2070, 2070, 950.0, 0x0, Not Active, Not Active, Not Active, Not Active"]
    r = sampler_with(tmp_path, lines).stop()
    assert r["sm_mhz"] == 2070.0 and r["sm_max_mhz"] == 2070.0 and r["samples"] == 4
    assert r["reasons"] == ["sw_power_cap"]


def test_clock_record_reports_thermal_slowdown(tmp_path):
    lines = ["0, 1500, 2070, 1300.0, 0x40, Not Active, Active, Not Active, Not Active",
             "0, 1600, 2070, 1300.0, 0x40, Not Active, Active, Active, Not Active"]
    r = sampler_with(tmp_path, lines).stop()
    assert r["reasons"] == ["hw_thermal_slowdown", "sw_thermal_slowdown"]
    assert r["sm_mhz"] == 1550.0


def test_clock_record_without_samples(tmp_path):
    assert sampler_with(tmp_path, []).stop() is None
    s = bench.ClockSampler(0)  # nvidia-smi never started
    assert s.stop() is None


def test_traffic_lookup_follows_the_kernel_source(tmp_path, monkeypatch):
    prof = tmp_path / "profiles"
    prof.mkdir()
    (prof / "k.md").write_text("kernel_source_digest: `abc123`\ntraffic_bytes_per_launch: `34253151`\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "kernel_source_digest", lambda: "abc123")
    assert bench.profiled_traffic("k") == 34253151.0
    monkeypatch.setattr(bench, "kernel_source_digest", lambda: "def456")  # the kernel changed since
    assert bench.profiled_traffic("k") is None
    assert bench.profiled_traffic("missing") is None


def test_committed_profile_names_a_digest_and_traffic():
    text = open(os.path.join(ROOT, "profiles", "pn3t_gemv_m1_decode_step.md")).read()
    assert "kernel_source_digest:" in text and "traffic_bytes_per_launch:" in text
    assert len(bench.kernel_source_digest()) == 16


def test_measured_peak_and_fallback(tmp_path, monkeypatch):
    (tmp_path / "MEASURED_PEAKS.json").write_text(json.dumps({"hbm_gbs": 6688.5}))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.measured_peaks() == (6688.5, "measured")
    os.unlink(tmp_path / "MEASURED_PEAKS.json")
    assert bench.measured_peaks() == (6800.0, "fallback")


def test_workload_bytes():
    # gate/up/q pn3t, k/v/o/down pn4t: 172,130,304 bytes per layer, 64 layers per step
    assert bench.layer_bytes() == 172_130_304
    assert bench.row_bytes(bench.PN3T, 5120) == 2176 and bench.row_bytes(bench.PN4T, 17408) == 9248
    cfg = bench.workload_config(1, 64, 448, 1)
    assert cfg["weight_bytes_per_step"] == 11_016_339_456
    assert "448 pnq_gemv launches" in cfg["graph"]


def test_warmup_below_three_is_refused(monkeypatch):
    monkeypatch.setattr(sys, "argv", ["bench.py", "--warmup", "2"])
    with pytest.raises(SystemExit, match="warmup"):
        bench.main()
