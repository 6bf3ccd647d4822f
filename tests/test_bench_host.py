"""Host-side logic of bench.py that needs no GPU: the roofline `traffic`
figure comes from an ncu summary under profiles/ only while the kernel's
source still hashes to the value recorded beside the counters."""
import hashlib
import os

import bench


def _write(tmp_path, src_text, recorded_sha, workload="mid"):
    (tmp_path / "k.cu").write_text(src_text)
    (tmp_path / "profiles").mkdir()
    (tmp_path / "profiles" / "k_mid.md").write_text(
        "# summary\n\n```roofline-traffic\nkernel_source: k.cu\n"
        f"source_sha256: {recorded_sha}\nworkload: {workload}\ntraffic_bytes_per_launch: 123456\n```\n")


def test_traffic_reported_for_unchanged_source(tmp_path, monkeypatch):
    text = "__global__ void k() {}\n"
    _write(tmp_path, text, hashlib.sha256(text.encode()).hexdigest())
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.profiled_traffic("mid", "k.cu") == 123456
    assert bench.profiled_traffic("dsv3", "k.cu") is None  # another workload's counters do not apply


def test_traffic_null_once_source_changed(tmp_path, monkeypatch):
    _write(tmp_path, "__global__ void k() { /* edited */ }\n", hashlib.sha256(b"old").hexdigest())
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.profiled_traffic("mid", "k.cu") is None


def test_committed_summary_parses():
    """The committed fused-kernel summary holds a well-formed block (its value is
    reported only while the hash matches)."""
    path = os.path.join(bench.ROOT, "profiles", "grouped_mlp_bf16_fused_mid.md")
    text = open(path).read()
    assert "```roofline-traffic" in text and "traffic_bytes_per_launch:" in text


def test_clock_samples_summary():
    """Median clock and power under load, and every throttle reason seen Active."""
    lines = [
        "0, 2070, 2070, 512.30, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active",
        "0, 1995, 2070, 1390.10, 0x0000000000000004, Not Active, Not Active, Not Active, Active",
        "0, 2010, 2070, 1388.70, 0x0000000000000004, Not Active, Not Active, Not Active, Active",
        "garbage line",
        "0, [N/A], 2070, [N/A], 0x0, Not Active, Not Active, Not Active, Not Active",
    ]
    got = bench.ClockSampler.summarize(lines)
    assert got["sm_mhz"] == 2010.0 and got["sm_max_mhz"] == 2070.0
    assert got["reasons"] == ["sw_power_cap"] and got["samples"] == 3
    assert got["power_w"] == 1388.7


def test_clock_samples_summary_reports_slowdown_reasons():
    lines = ["0, 1500, 2070, 900.0, 0x8, Active, Not Active, Active, Not Active"]
    got = bench.ClockSampler.summarize(lines)
    assert got["reasons"] == ["hw_slowdown", "sw_thermal_slowdown"]


def test_pre_roll_keeps_the_gpu_busy_for_the_sampler():
    # half a second of 4 ms steps, never fewer than the warm-up count
    assert bench.pre_roll_count(4.0, 5) == 125
    assert bench.pre_roll_count(1000.0, 5) == 5
    assert bench.pre_roll_count(0.0, 3) == 25000  # a step timed at zero counts as 20 us
