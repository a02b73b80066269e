"""Seeded input generators: deterministic, right shapes and value recipes (CPU only)."""
import numpy as np

from walsh_hadamard_transform_gb300 import inputs


def test_workload_table():
    w = inputs.WORKLOADS
    assert [(x.n, x.batch, x.dtype) for x in w.values()] == [
        (10, 64, "c32"), (12, 64, "c32"), (14, 64, "c32"), (18, 256, "i32"), (24, 16, "c64"), (24, 16, "c32")]
    assert w["n24_b16_c64"].bytes_in == 2 * 16 * (1 << 24) * 8


def test_deterministic_and_prefix():
    w = inputs.WORKLOADS["n12_b64_c32"]
    a = w.generate(batch=5)
    b = w.generate(batch=5)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])
    c = w.generate(batch=2)
    assert np.array_equal(a[0][:2], c[0])


def test_unit_norm_and_gaussian():
    re, im = inputs.draw("unit_gaussian", 10, 4, 2, "c64")
    norms = np.sqrt(np.sum(re * re + im * im, axis=1))
    assert np.allclose(norms, 1.0, rtol=0, atol=1e-14)
    re32, im32 = inputs.draw("unit_gaussian", 10, 4, 2, "c32")
    assert re32.dtype == np.float32 and np.array_equal(re32, re.astype(np.float32))
    g, _ = inputs.draw("gaussian", 14, 2, 0, "c64")
    assert abs(g.std() - 1.0) < 0.02


def test_int_recipe():
    re, im = inputs.WORKLOADS["n18_b256_i32"].generate(batch=2)
    assert re.dtype == np.int32 and re.min() == -8 and re.max() == 8
    assert not im.any()
