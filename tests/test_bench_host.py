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
    src = bench.sources_digest(bench.kernel_sources("attend", "stage1_bf16"))
    rec = {"attend": {"stage1_bf16": {"sources": src, "dram_bytes_per_launch": 123}},
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
    # a kernel's own digest ignores the other kernels' files
    d1 = bench.sources_digest(["a.cu"])
    (tmp_path / "b.cuh").write_text("zz")
    assert bench.sources_digest(["a.cu"]) == d1
    (tmp_path / "a.cu").write_text("xx")
    assert bench.sources_digest(["a.cu"]) != d1


def test_kernel_sources_follow_the_kernel_each_workload_runs():
    assert bench.kernel_sources("route", "stage1_bf16") == ["route.cuh", "ptx.cuh"]
    assert bench.kernel_sources("route", "tiny_f32") == ["route.cuh", "ptx.cuh"]
    assert bench.kernel_sources("route", "stage3_bf16")[0] == "forward_image.cuh"
    assert bench.kernel_sources("attend", "tiny_f32")[0] == "attend_f32.cuh"
    assert bench.kernel_sources("attend", "stage3_bf16")[0] == "attend_image.cuh"
    for name in ("stage1_bf16", "stage2_bf16", "seg512_bf16"):
        assert bench.kernel_sources("attend", name)[0] == "attend_bf16.cuh"
    for kernel in ("route", "attend"):
        for name in bra_synth.WORKLOADS:
            for f in bench.kernel_sources(kernel, name):
                assert (bench.os.path.isfile(bench.os.path.join(bench.CSRC, f)))


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


# Per-forward algorithmic work of the five workloads, as tabled for the
# roofline: bytes, contraction GFLOP, other float32 GFLOP and exponentials.
SURVEY_TABLE = {
    "tiny_f32": (0.21e6, 0.0008, 0.0010, 6.3e3),
    "stage1_bf16": (102.8e6, 3.29, 0.68, 25.7e6),
    "stage2_bf16": (51.4e6, 1.64, 0.38, 12.8e6),
    "stage3_bf16": (25.7e6, 0.82, 0.25, 6.4e6),
    "seg512_bf16": (67.1e6, 8.59, 0.50, 67.1e6),
}


def test_algorithmic_work_matches_the_tabled_counts():
    for name, (nbytes, tc, alu, exps) in SURVEY_TABLE.items():
        wl = bra_synth.WORKLOADS[name]
        w = bench.algorithmic_work(wl)["forward"]
        assert abs(w["bytes"] - nbytes) / nbytes < 0.05, name  # tabled to 2-4 digits
        assert abs(w["exps"] - exps) / exps < 0.01, name
        if wl.dtype == "bf16":
            assert abs(w["tensor_flops"] / 1e9 - tc) / tc < 0.01, name
            assert abs(w["alu_flops"] / 1e9 - alu) / alu < 0.02, name
        else:  # the float32 path contracts on the FMA pipe
            assert w["tensor_flops"] == 0
            assert abs(w["alu_flops"] / 1e9 - (tc + alu)) / (tc + alu) < 0.05, name
    # the kernels' shares add up to the forward
    w = bench.algorithmic_work(bra_synth.WORKLOADS["stage3_bf16"])
    assert w["route"]["alu_flops"] + w["attend"]["alu_flops"] == w["forward"]["alu_flops"]
    assert w["attend"]["exps"] == w["forward"]["exps"]


def test_roofline_takes_the_slowest_pipe():
    pk = {"hbm_gbs": 6500.0, "tensor_tflops": 1750.0, "alu_tflops": 77.0,
          "ex2_per_s_f32": 4.8e12, "ex2_per_s_bf16": 9.6e12}
    hbm_bound = {"bytes": 65e6, "tensor_flops": 1e9, "alu_flops": 1e8, "exps": 1e6}
    r = bench.roofline(hbm_bound, pk, "bf16", 20e-6)
    assert r["bound"] == "hbm" and r["unit"] == "GB/s"
    assert abs(r["roof_us"] - 10.0) < 1e-9 and abs(r["frac"] - 0.5) < 1e-9
    assert abs(r["achieved"] - 3250.0) < 1e-6 and r["peak"] == 6500.0
    alu_bound = {"bytes": 6.5e6, "tensor_flops": 0, "alu_flops": 7.7e8, "exps": 0}
    r = bench.roofline(alu_bound, pk, "f32", 40e-6)
    assert r["bound"] == "alu" and abs(r["roof_us"] - 10.0) < 1e-9
    assert abs(r["frac"] - 0.25) < 1e-9
    mufu_bound = {"bytes": 0, "tensor_flops": 0, "alu_flops": 0, "exps": 9.6e7}
    assert bench.roofline(mufu_bound, pk, "bf16", 1e-5)["bound"] == "mufu"
    assert abs(bench.roofline(mufu_bound, pk, "f32", 1e-5)["roof_us"] - 20.0) < 1e-9


def test_peaks_derive_alu_and_mufu_from_unit_counts(tmp_path, monkeypatch):
    p = tmp_path / "peaks.json"
    p.write_text(json.dumps({"hbm_gbs": 6492.7, "bf16_tflops": 1744.1, "sm_max_mhz": 2032.0}))
    monkeypatch.setattr(bench, "PEAKS_FILE", str(p))
    pk = bench.peaks(148)
    assert pk["source"] == "measured" and pk["hbm_gbs"] == 6492.7
    assert abs(pk["alu_tflops"] - 148 * 128 * 2 * 2.032e9 / 1e12) < 1e-9
    assert abs(pk["ex2_per_s_bf16"] - 2 * pk["ex2_per_s_f32"]) < 1.0
    assert abs(pk["ex2_per_s_f32"] - 148 * 16 * 2.032e9) < 1.0


def test_workload_selection_and_config_numbers():
    assert bench.selected_workloads("all") == list(bra_synth.WORKLOADS)
    assert bench.selected_workloads("none") == []
    assert bench.selected_workloads("tiny_f32, stage3_bf16") == ["tiny_f32", "stage3_bf16"]
    assert bench.CONFIG_NUMBER["tiny_f32"] == 1 and bench.CONFIG_NUMBER["stage3_bf16"] == 4
    args = bench.parse_args([])
    assert args.workload == "stage1_bf16" and args.workloads == "all"


def test_block_work_counts_each_step_once():
    wl = bra_synth.WORKLOADS["stage1_bf16"]
    M, C = wl.B * wl.H * wl.W, wl.C
    w = bench.block_work(wl)
    fwd = bench.algorithmic_work(wl)["forward"]
    # LayerNorm 2 MC, projection 4 MC, forward 4 MC, residual add 3 MC (bf16)
    assert w["bytes"] == (2 + 4 + 4 + 3) * M * C * 2 + 3 * C * C * 2
    assert w["tensor_flops"] == fwd["tensor_flops"] + 2 * M * C * 3 * C
    assert w["exps"] == fwd["exps"]


def test_ffn_work_counts_each_step_once():
    wl = bra_synth.WORKLOADS["stage2_bf16"]
    M, C = wl.B * wl.H * wl.W, wl.C
    w = bench.ffn_work(wl)
    # LayerNorm 2, fc1 4, convolution + GELU 6, fc2 5 (M C elements, bf16)
    assert w["bytes"] == 17 * M * C * 2 + 2 * 3 * C * C * 2 + 10 * 3 * C * 4
    assert w["tensor_flops"] == 2 * (2 * M * C * 3 * C)


def test_backward_work_counts():
    wl = bra_synth.WORKLOADS["stage1_bf16"]
    T = wl.B * wl.H * wl.W * wl.C
    w = bench.backward_work(wl)
    # q, k, v, dout bf16 in; dq, dk, dv float32 out; LePE weights in and out
    assert w["bytes"] == 4 * T * 2 + 3 * T * 4 + 2 * wl.C * 25 * 4
    # six contractions of 2 * (k n) * d per query and head: 2 * 64 * C per token each
    assert w["tensor_flops"] == 6 * 2 * 64 * T
    assert w["alu_flops"] == 4 * 25 * T
    assert w["exps"] == wl.B * wl.H * wl.W * wl.heads * 64
    f = bench.backward_work(bra_synth.WORKLOADS["tiny_f32"])
    assert f["tensor_flops"] == 0 and f["alu_flops"] > 4 * 25 * 14 * 14 * 64
