"""The bench's host-side bookkeeping, on CPU: clock-sample summaries, the
committed DRAM-traffic record tied to the kernel's source, and the peaks."""
import json
import os

import pytest

import bench


def _sample(sm, mx, hw="Not Active", hw_th="Not Active", sw_th="Not Active", cap="Not Active"):
    # the nvidia-smi query columns, in the order ClockSampler asks for them
    return ["0", str(sm), str(mx), "900.0", "0x0", hw, hw_th, sw_th, cap]


def test_clock_summary_median_max_and_reasons():
    c = bench.ClockSampler(0)
    c.samples = [(10.0, _sample(2070, 2070)), (10.1, _sample(1965, 2070, cap="Active")),
                 (10.2, _sample(2070, 2070)), (50.0, _sample(900, 2070, hw_th="Active"))]
    s = c.summary(10.0, 10.2)
    # the late sample lies outside the window and is not counted
    assert s["samples"] == 3 and s["window"] == "timed window"
    assert s["sm_mhz"] == 2070.0 and s["sm_max_mhz"] == 2070.0
    assert s["reasons"] == ["sw_power_cap"]


def test_clock_summary_short_window_falls_back_to_the_whole_run():
    c = bench.ClockSampler(0)
    c.samples = [(1.0, _sample(2000, 2070)), (2.0, _sample(1000, 2070, hw="Active"))]
    s = c.summary(5.0, 5.01)
    assert s["samples"] == 2 and s["window"].startswith("whole run")
    assert s["sm_mhz"] == 1500.0
    assert s["reasons"] == ["hw_slowdown"]


def test_clock_summary_ignores_unreadable_fields_and_needs_samples():
    c = bench.ClockSampler(0)
    assert c.summary(0.0, 1.0) is None
    c.samples = [(0.5, _sample("[N/A]", "[N/A]")), (0.6, _sample(2070, 2070))]
    s = c.summary(0.0, 1.0)
    assert s["sm_mhz"] == 2070.0 and s["sm_max_mhz"] == 2070.0 and s["samples"] == 2


def _traffic_tree(tmp_path, source_text, recorded_hash=None):
    src = tmp_path / "kernel.cu"
    src.write_text(source_text)
    h = recorded_hash if recorded_hash is not None else bench.file_hash(str(src))
    prof = tmp_path / "profiles"
    prof.mkdir()
    (prof / "traffic.json").write_text(json.dumps(
        {"k_tc_gemm": {"outdoor": {"dram_bytes_per_launch": 1234, "source": "kernel.cu", "source_hash": h}}}))
    return src


def test_traffic_is_reported_only_for_the_kernel_it_was_taken_on(tmp_path, monkeypatch):
    src = _traffic_tree(tmp_path, "// kernel as captured\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.ncu_traffic("k_tc_gemm", "outdoor") == 1234
    assert bench.ncu_traffic("k_tc_gemm", "large") is None        # no capture for that workload
    assert bench.ncu_traffic("k_other", "outdoor") is None
    src.write_text("// kernel changed since the capture\n")
    assert bench.ncu_traffic("k_tc_gemm", "outdoor") is None


def test_traffic_without_a_record_or_source(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.ncu_traffic("k_tc_gemm", "outdoor") is None
    src = _traffic_tree(tmp_path, "x")
    os.remove(src)
    assert bench.ncu_traffic("k_tc_gemm", "outdoor") is None


def test_committed_traffic_records_name_existing_sources():
    with open(os.path.join(bench.ROOT, "profiles", "traffic.json")) as f:
        rec = json.load(f)
    for kernel, per_workload in rec.items():
        for workload, r in per_workload.items():
            assert os.path.exists(os.path.join(bench.ROOT, r["source"])), (kernel, workload)
            assert r["dram_bytes_per_launch"] > 0
            assert "--clock-control none" in r["command"]


def test_peaks_measured_and_fallback(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    p = bench.load_peaks()
    assert p["source"] == "fallback" and p["hbm"] == 6800.0 and p["bf16"] == 1900.0
    (tmp_path / "MEASURED_PEAKS.json").write_text(json.dumps({"hbm_gbs": 6670.9, "bf16_tflops": 1922.1}))
    p = bench.load_peaks()
    assert p["source"] == "measured" and p["hbm"] == pytest.approx(6670.9)
    assert p["bf16_sustained"] == pytest.approx(1922.1)   # no sustained figure: the burst one stands in
