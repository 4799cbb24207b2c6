"""CPU tests of the benchmark's evidence bookkeeping: DRAM traffic from the
committed ncu capture is reported only while the kernel's source is the one
that was captured, and the roofline peaks come from the measured file when
it exists."""
import hashlib
import json
import os

import bench


def _fake_root(tmp_path, src_text):
    src = tmp_path / "k.cu"
    src.write_text(src_text)
    (tmp_path / "profiles").mkdir()
    rec = {"kernels": {"k": {"kernel": "k_kernel", "source": "k.cu",
                             "sha256": hashlib.sha256(src_text.encode()).hexdigest(),
                             "dram_read_bytes": 1000, "dram_write_bytes": 24}}}
    (tmp_path / "profiles" / "traffic.json").write_text(json.dumps(rec))
    return src


def test_traffic_is_reported_only_for_the_captured_source(tmp_path, monkeypatch):
    src = _fake_root(tmp_path, "__global__ void k_kernel() {}\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.measured_traffic("k") == 1024
    assert bench.measured_traffic("other") is None
    src.write_text("__global__ void k_kernel() { /* changed */ }\n")
    assert bench.measured_traffic("k") is None
    os.remove(src)
    assert bench.measured_traffic("k") is None


def test_peaks_prefer_the_measured_file(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.peaks() == (6800.0, "fallback")
    (tmp_path / "MEASURED_PEAKS.json").write_text(json.dumps({"hbm_gbs": 6786.6}))
    assert bench.peaks() == (6786.6, "measured")
