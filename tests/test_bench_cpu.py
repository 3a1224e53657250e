"""Host-side logic of bench.py, without a GPU: the rule that the recorded
DRAM traffic is reported only for the kernel source it was measured on, the
roofline denominators, the parsing of the clock samples taken during the
timed region, and the whole-job throughput arithmetic."""

import json

import pytest

import bench


def test_traffic_reported_only_for_the_measured_source_and_workload(monkeypatch, tmp_path):
    summary = tmp_path / "profiles" / "traffic.md"
    summary.parent.mkdir()
    summary.write_text("# traffic\n\n- workload: `w16k`\n- kernel_source_sha: `abc123`\n"
                       "- traffic_bytes_per_launch: 251386112\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "TRAFFIC_SUMMARY", "profiles/traffic.md")
    monkeypatch.setattr(bench, "kernel_source_hash", lambda: "abc123")
    assert bench.recorded_traffic("w16k") == 251386112
    assert bench.recorded_traffic("w4k") is None                 # another workload
    monkeypatch.setattr(bench, "kernel_source_hash", lambda: "def456")
    assert bench.recorded_traffic("w16k") is None                # the kernel changed since the capture
    summary.unlink()
    assert bench.recorded_traffic("w16k") is None                # no capture at all


def test_committed_traffic_summary_names_a_workload_and_a_source_hash():
    fields = {}
    with open(f"{bench.ROOT}/{bench.TRAFFIC_SUMMARY}") as f:
        for line in f:
            if line.startswith("- ") and ":" in line:
                k, v = line[2:].split(":", 1)
                fields[k.strip()] = v.strip().strip("`")
    assert fields["workload"] in {w.name for w in bench.WORKLOADS}
    assert len(fields["kernel_source_sha"]) == 16
    assert int(fields["traffic_bytes_per_launch"]) > 0


def test_kernel_source_hash_is_stable_and_short():
    h = bench.kernel_source_hash()
    assert h == bench.kernel_source_hash() and len(h) == 16
    int(h, 16)


def test_peaks_from_the_measured_file_else_the_fallback(monkeypatch, tmp_path):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.measured_peaks() == {"bf16_tflops": 1900.0, "hbm_gbs": 6800.0, "source": "fallback"}
    (tmp_path / "MEASURED_PEAKS.json").write_text(json.dumps({"bf16_tflops": 1904.2, "hbm_gbs": 6790.3,
                                                              "bf16_tflops_sustained": 1700.0}))
    assert bench.measured_peaks() == {"bf16_tflops": 1904.2, "hbm_gbs": 6790.3, "source": "measured"}


def test_clock_summary_takes_the_median_and_every_active_reason():
    s = bench.ClockSampler(0)
    s.lines = [
        "0, 2070, 2070, 900.1, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active",
        "0, 1980, 2070, 1390.0, 0x0000000000000004, Not Active, Not Active, Not Active, Active",
        "0, 2055, 2070, 1200.0, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active",
        "garbled line",
        "0, [N/A], 2070, 0, 0, Not Active, Not Active, Not Active, Not Active",
    ]
    out = s.summary()
    assert out == {"sm_mhz": 2055.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"], "samples": 3}
    s.lines = ["0, 1500, 2070, 700, 0x8, Active, Active, Active, Not Active"]
    assert s.summary()["reasons"] == ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown"]


def test_clock_summary_without_samples():
    s = bench.ClockSampler(0)
    assert s.summary() == {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}


@pytest.mark.parametrize("world", [1, 2, 8])
def test_whole_job_throughput_counts_every_rank_at_the_slowest_time(world):
    # 2.2e12 FLOPs per step, 300 steps per rank, the slowest rank took 396 ms
    v = bench.whole_job_tflops(world, 2_199_157_473_280, 300, 396.0)
    assert v == pytest.approx(world * 2_199_157_473_280 * 300 / 0.396 / 1e12)
