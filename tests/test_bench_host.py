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
