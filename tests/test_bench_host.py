"""Host-side pieces of bench.py that need no GPU: the algorithmic byte counts
behind the roofline, the DRAM-traffic record lookup (valid only for the
kernel sources it was captured on), the measured-peak fallback and the
summary of nvidia-smi clock samples."""
import json

import bench
import bra_synth


def test_algorithmic_bytes_are_inputs_once_and_output_once():
    wl = bra_synth.WORKLOADS["stage1_bf16"]
    t = 64 * 56 * 56 * 64 * 2
    assert bench.algorithmic_bytes(wl) == {"route": 2 * t, "attend": 4 * t, "forward": 4 * t}
    assert bench.algorithmic_bytes(wl)["attend"] == 102_760_448
    tiny = bra_synth.WORKLOADS["tiny_f32"]
    assert bench.algorithmic_bytes(tiny)["route"] == 2 * 14 * 14 * 64 * 4


def test_recorded_traffic_only_for_matching_sources(tmp_path, monkeypatch):
    rec = {"attend": {"stage1_bf16": {"sources": bench.sources_digest(),
                                      "dram_bytes_per_launch": 123}},
           "route": {"stage1_bf16": {"sources": "0" * 16, "dram_bytes_per_launch": 456}}}
    path = tmp_path / "traffic.json"
    path.write_text(json.dumps(rec))
    monkeypatch.setattr(bench, "TRAFFIC_FILE", str(path))
    assert bench.recorded_traffic("attend", "stage1_bf16") == 123
    assert bench.recorded_traffic("route", "stage1_bf16") is None  # stale capture
    assert bench.recorded_traffic("attend", "seg512_bf16") is None  # none taken
    monkeypatch.setattr(bench, "TRAFFIC_FILE", str(tmp_path / "missing.json"))
    assert bench.recorded_traffic("attend", "stage1_bf16") is None


def test_sources_digest_covers_the_kernel_sources(tmp_path, monkeypatch):
    (tmp_path / "a.cu").write_text("x")
    (tmp_path / "notes.txt").write_text("y")
    monkeypatch.setattr(bench, "CSRC", str(tmp_path))
    d0 = bench.sources_digest()
    (tmp_path / "notes.txt").write_text("changed")
    assert bench.sources_digest() == d0
    (tmp_path / "b.cuh").write_text("z")
    assert bench.sources_digest() != d0


def test_measured_peak_falls_back_when_file_is_missing(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "PEAKS_FILE", str(tmp_path / "none.json"))
    assert bench.measured_peaks() == (6400.0, "fallback")
    p = tmp_path / "peaks.json"
    p.write_text(json.dumps({"hbm_gbs": 6514.2}))
    monkeypatch.setattr(bench, "PEAKS_FILE", str(p))
    assert bench.measured_peaks() == (6514.2, "measured")


def _row(mhz, hw="Not Active", power_cap="Not Active"):
    # index, clocks.sm, clocks.max.sm, power.draw, active, hw_slowdown,
    # hw_thermal_slowdown, sw_thermal_slowdown, sw_power_cap
    return ["0", str(mhz), "2032", "700.5", "0x0", hw, "Not Active", "Not Active", power_cap]


def test_clock_summary_uses_the_timed_window_and_flags_reasons():
    s = bench.ClockSampler("0")
    s.rows = [(0.5, _row(1000))] + [(1.0 + 0.1 * i, _row(2032)) for i in range(5)] + \
             [(1.3, _row(1980, power_cap="Active"))]
    out = s.summary(1.0, 2.0, "timed region")
    assert out["sm_mhz"] == 2032.0 and out["sm_max_mhz"] == 2032.0
    assert out["reasons"] == ["sw_power_cap"] and out["samples"] == 6
    assert out["window"] == "timed region"
    s.rows.append((1.2, _row(2032, hw="Active")))
    assert "hw_slowdown" in s.summary(1.0, 2.0, "timed region")["reasons"]


def test_clock_summary_short_window_and_no_samples():
    s = bench.ClockSampler("0")
    assert s.summary(0, 1, "timed region")["reasons"] == ["nvidia-smi unavailable"]
    s.rows = [(0.1, _row(2032)), (0.2, _row(2030)), (5.0, _row(2032))]
    out = s.summary(4.9, 5.1, "timed region")
    assert out["samples"] == 3 and "too short" in out["window"]
