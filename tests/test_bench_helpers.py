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


def test_headline_passes_have_fitted_records(monkeypatch):
    """The four n = 24 passes carry a batch-2/4 fit; bench.py reports its per-vector
    bytes and the fit at batch 16, only while the sources are those it was captured from."""
    path = os.path.join(bench.ROOT, "profiles", "ncu_traffic.json")
    records = json.load(open(path))
    keys = ["c64 row pass K=13 (n=24)", "c64 col pass K=11 (n=24)",
            "c32 row pass K=14 (n=24)", "c32 col pass K=10 (n=24)"]
    for key in keys:
        rec = records[key]
        fit = rec["batch_fit"]
        per = fit["read_per_vector"] + fit["write_per_vector"]
        assert rec["dram_bytes_per_vector"] == per
        at16 = fit["read_intercept"] + fit["write_intercept"] + 16 * per
        assert abs(rec["dram_bytes_per_launch"] - at16) <= 16
        # both captures lie on the fitted line
        for b, r, w in zip(fit["batches"], fit["read_bytes"], fit["write_bytes"]):
            assert abs(r - (fit["read_intercept"] + b * fit["read_per_vector"])) <= 4
            assert abs(w - (fit["write_intercept"] + b * fit["write_per_vector"])) <= 4
        monkeypatch.setattr(bench, "kernel_source_hash", lambda: rec["source_sha"])
        assert bench.ncu_bytes_per_vector(key) == per
        monkeypatch.setattr(bench, "kernel_source_hash", lambda: "f" * 16)
        assert bench.ncu_bytes_per_vector(key) is None


def test_cpu_leg_checks_gpu_results_against_the_oracle(monkeypatch):
    """The CPU leg's per-configuration check: exact results report ~0 error (float) or
    bit-exact (int32); a planted error of known size is reported at that size, and a
    changed int32 element is not bit-exact."""
    import dataclasses

    import numpy as np

    import oracle
    from walsh_hadamard_transform_gb300 import inputs

    monkeypatch.setattr(bench, "cpu_baseline", lambda parts, host, sample: {"value": 0.0})
    w32 = dataclasses.replace(inputs.WORKLOADS["n10_b64_c32"], batch=4)
    re, im = w32.generate()
    ore, oim = oracle.fwt_complex(re, im, normalize=True)
    bad_re = ore.copy()
    bad_re[2, 5] += 1e-4 * np.linalg.norm(np.concatenate([ore[2], oim[2]]))  # one element off
    wi = inputs.Workload("i8", 8, 3, "i32", 5, False, "uniform_int8")
    ire, iim = wi.generate()
    iore, ioim = oracle.fwt_complex(ire, iim, normalize=False)
    ibad = iore.copy()
    ibad[1, 7] += 1
    checks = [
        {"label": "good", "workload": w32, "rows": [0, 1, 2, 3], "host_in": (re, im),
         "got": (ore.astype(np.float32), oim.astype(np.float32))},
        {"label": "bad", "workload": w32, "rows": [0, 1, 2, 3], "host_in": (re, im), "got": (bad_re, oim)},
        {"label": "igood", "workload": wi, "rows": [0, 1, 2], "host_in": (ire, iim), "got": (iore, ioim)},
        {"label": "ibad", "workload": wi, "rows": [0, 1, 2], "host_in": (ire, iim), "got": (ibad, ioim)},
    ]
    _, errors = bench.cpu_leg([], [], 1, checks)
    assert errors["good"]["max_rel_l2_err"] < 1e-7
    assert 0.9e-4 < errors["bad"]["max_rel_l2_err"] < 1.1e-4
    assert errors["igood"]["bit_exact"] is True
    assert errors["ibad"]["bit_exact"] is False
    assert errors["good"]["oracle_check"] == "all 4 vectors"
