"""bench.py's bookkeeping on the CPU: the committed ncu traffic is reported only for
the CUDA sources it was captured from, and the peak falls back when the measured
one is missing."""
import json
import os

import bench


def test_traffic_only_for_the_captured_sources(monkeypatch):
    path = os.path.join(bench.ROOT, "profiles", "ncu_traffic.json")
    records = json.load(open(path))
    assert records, "profiles/ncu_traffic.json holds no capture"
    key, rec = next(iter(records.items()))
    monkeypatch.setattr(bench, "kernel_source_hash", lambda: rec["source_sha"])
    assert bench.ncu_traffic(key) == rec["dram_bytes_per_launch"]
    assert bench.ncu_traffic("no such kernel") is None
    monkeypatch.setattr(bench, "kernel_source_hash", lambda: "0" * 16)  # sources changed
    assert bench.ncu_traffic(key) is None


def test_source_hash_covers_every_cuda_source(tmp_path, monkeypatch):
    before = bench.kernel_source_hash()
    assert len(before) == 16
    # a copy of the tree with one kernel byte changed hashes differently
    csrc = os.path.join(bench.ROOT, "walsh_hadamard_transform_gb300", "csrc")
    fake = tmp_path / "walsh_hadamard_transform_gb300" / "csrc"
    fake.mkdir(parents=True)
    for name in os.listdir(csrc):
        if name.endswith((".cu", ".cuh")):
            (fake / name).write_bytes(open(os.path.join(csrc, name), "rb").read())
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.kernel_source_hash() == before
    first = sorted(p for p in os.listdir(fake))[0]
    (fake / first).write_bytes((fake / first).read_bytes() + b"\n")
    assert bench.kernel_source_hash() != before


def test_peak_falls_back_without_the_measured_file(monkeypatch, tmp_path):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    peak, source = bench.measured_peaks()
    assert peak == bench.FALLBACK_HBM_GBS and source.startswith("fallback")
    (tmp_path / "MEASURED_PEAKS.json").write_text(json.dumps({"hbm_gbs": 1234.5}))
    peak, source = bench.measured_peaks()
    assert peak == 1234.5 and source.startswith("measured")
