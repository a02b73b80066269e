"""The one JSON line bench.py prints, for both arms: every key the measurement contract
names, with values of the right kind.  The reference arm (the CPU oracle) runs here; our
arm needs a GPU."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

COMMON = {"metric": str, "value": float, "unit": str, "n_gpus": int, "steps": int, "warmup": int,
          "ms_per_step": float, "higher_is_better": bool, "scaling": str, "dtype": str,
          "data": str, "config": dict, "e2e": dict, "cpu_baseline": dict}


def _run(args, timeout):
    env = dict(os.environ)
    for k in ("RANK", "WORLD_SIZE", "LOCAL_RANK"):
        env.pop(k, None)
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], cwd=ROOT, env=env,
                       capture_output=True, text=True, timeout=timeout)
    assert r.returncode == 0, r.stderr[-4000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1, r.stdout
    return json.loads(lines[0])


def _check_common(d):
    for key, kind in COMMON.items():
        assert key in d, key
        assert isinstance(d[key], (int, float) if kind is float else kind), (key, d[key])
    assert d["value"] > 0 and d["ms_per_step"] > 0
    assert d["higher_is_better"] is True and d["scaling"] == "weak" and d["n_gpus"] == 1
    assert d["vs_baseline"] is None
    assert "workload" in d["config"]
    e2e = d["e2e"]
    for key in ("value", "unit", "h2d_bytes_per_step", "d2h_bytes_per_step"):
        assert key in e2e, key
    assert e2e["unit"] == d["unit"] == "vectors/s"
    cb = d["cpu_baseline"]
    for key in ("value", "unit", "cores", "kind", "sample"):
        assert key in cb, key
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] > 0


def test_reference_arm_line():
    d = _run(["--impl", "reference", "--workload", "n10_b64_c32", "--steps", "2", "--warmup", "1"],
             timeout=300)
    _check_common(d)
    assert d["impl"] == "reference"
    assert d["e2e"]["value"] == d["value"] == d["cpu_baseline"]["value"]
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0


@pytest.mark.gpu
def test_our_arm_line():
    d = _run(["--workload", "n12_b64_c32", "--steps", "5", "--warmup", "3", "--no-per-config",
              "--e2e-steps", "3"], timeout=600)
    _check_common(d)
    assert "impl" not in d or d["impl"] == "ours"
    assert d["steps"] == 5 and d["warmup"] == 3
    rf = d["roofline"]
    for key in ("bound", "achieved", "peak", "unit", "frac", "traffic"):
        assert key in rf, key
    assert rf["bound"] == "hbm" and rf["unit"] == "GB/s" and rf["peak"] > 0
    assert abs(rf["frac"] - rf["achieved"] / rf["peak"]) < 1e-3
    clocks = d["clocks"]
    for key in ("sm_mhz", "sm_max_mhz", "reasons"):
        assert key in clocks, key
    # one launch a step at n = 12 (a single tile), all of them the library's own
    assert d["gpu_launches"] == 5
    e2e = d["e2e"]
    assert e2e["h2d_bytes_per_step"] == e2e["d2h_bytes_per_step"] == 2 * 64 * 4096 * 4
    assert e2e["value"] > 0
