"""CUDA path vs the CPU oracle, element by element, through the C ABI (GPU only).

Tolerances: int32 bit-exact; fp32 and fp64 per-vector complex relative L2 error
<= 2e-6 and <= 1e-12 respectively (the transform's specification).
"""
import numpy as np
import pytest
import torch

import oracle
import walsh_hadamard_transform_gb300 as fwt
from helpers import NP_DTYPE, TOL, assert_matches, gpu_transform, host_threads, rel_err_per_vector
from walsh_hadamard_transform_gb300 import inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def need_cuda():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    fwt.library()


def _check(dtype, n, batch, normalize, seed, inplace=False, real_only=False):
    re, im = inputs.random_pair(n, batch, dtype, seed)
    if real_only:
        im = None
    gre, gim = gpu_transform(re, im, normalize, inplace=inplace)
    ore, oim = oracle.fwt_complex(re, im, normalize=normalize, nthreads=host_threads())
    assert_matches(dtype, gre, gim, ore, oim, f"{dtype} n={n} batch={batch} norm={normalize}")


@pytest.mark.parametrize("dtype", ["c32", "c64", "i32"])
@pytest.mark.parametrize("n", list(range(0, 21)))
def test_every_n_small_batch(dtype, n):
    # batch 3: several tiles and a ragged last tile wherever tiles pack short vectors
    for normalize in ((False,) if dtype == "i32" else (True, False)):
        _check(dtype, n, 3, normalize, seed=100 + n)


@pytest.mark.parametrize("dtype", ["c32", "c64", "i32"])
@pytest.mark.parametrize("n", [1, 7, 12, 15, 18, 22])
def test_in_place(dtype, n):
    _check(dtype, n, 2, dtype != "i32", seed=7 * n, inplace=True)


@pytest.mark.parametrize("n", [5, 14, 19])
def test_int32_real_only(n):
    _check("i32", n, 4, False, seed=n, real_only=True)


def _valid_plans(n, dtype):
    out = []
    for b in range(3, 16):
        for rest in ([n - b], *[[a2, n - b - a2] for a2 in range(3, 11)]):
            f = [b, *rest]
            if any(k <= 0 for k in f):
                continue
            try:
                fwt.set_plan(n, dtype, f)
            except fwt.FwtError:
                continue
            out.append(f)
    fwt.set_plan(n, dtype, None)
    return out


@pytest.mark.parametrize("tma", [2, 0], ids=["tma", "direct"])
@pytest.mark.parametrize("dtype", ["c32", "c64", "i32"])
@pytest.mark.parametrize("n", [16, 20, 21])
def test_every_kronecker_split(dtype, n, tma):
    """Each valid 2- and 3-factor split, for every column segment width, with
    TMA-staged and directly loaded column tiles (every compiled tile shape)."""
    re, im = inputs.random_pair(n, 2, dtype, seed=n)
    norm = dtype != "i32"
    ore, oim = oracle.fwt_complex(re, im, normalize=norm)
    width = fwt.column_bytes(dtype)
    fwt.set_tma(tma)
    try:
        for cb in ((16, 32, 64, 128) if tma == 2 else (32, 64, 128)):
            fwt.set_column_bytes(dtype, cb)
            plans = _valid_plans(n, dtype)
            assert plans, "no valid plan"
            for f in plans:
                fwt.set_plan(n, dtype, f)
                gre, gim = gpu_transform(re, im, norm)
                assert_matches(dtype, gre, gim, ore, oim, f"plan {f} cb={cb} tma={tma}")
    finally:
        fwt.set_plan(n, dtype, None)
        fwt.set_column_bytes(dtype, width)
        fwt.set_tma(fwt.TMA_AUTO)
    assert fwt.device_status() == fwt.FWT_OK


@pytest.mark.parametrize("name", ["n10_b64_c32", "n12_b64_c32", "n14_b64_c32", "n18_b256_i32"])
def test_workload_full_size(name):
    w = inputs.WORKLOADS[name]
    re, im = w.generate()
    gre, gim = gpu_transform(re, im, w.normalize)
    ore, oim = oracle.fwt_complex(re, im, normalize=w.normalize, nthreads=host_threads())
    assert_matches(w.dtype, gre, gim, ore, oim, name)
    if w.dtype == "i32":
        assert np.abs(gre).max() <= 8 << 18  # no overflow at this size


@pytest.mark.parametrize("name", ["n24_b16_c64", "n24_b16_c32"])
def test_workload_n24_full_batch(name):
    """Full batch on the GPU (the benchmarked call); the oracle checks two whole
    vectors and sampled entries of every vector from the definition."""
    w = inputs.WORKLOADS[name]
    re, im = w.generate()
    gre, gim = gpu_transform(re, im, w.normalize)
    full = [0, w.batch - 1]
    ore, oim = oracle.fwt_complex(re[full], im[full], normalize=True, nthreads=2)
    assert_matches(w.dtype, gre[full], gim[full], ore, oim, name + " whole vectors")
    rng = np.random.default_rng(0)
    ks = np.concatenate([[0, 1, w.N - 1], rng.integers(0, w.N, size=5)])
    for b in range(w.batch):
        sre = oracle.entries(re[b], ks, normalize=True)
        sim = oracle.entries(im[b], ks, normalize=True)
        err = rel_err_per_vector(gre[b, ks], gim[b, ks], sre, sim)
        assert err <= TOL[w.dtype], f"{name} vector {b}: sampled error {err:.3e}"
    # Parseval on every vector (unit-norm inputs stay unit-norm)
    norms = np.sqrt(np.sum(gre.astype(np.float64) ** 2 + gim.astype(np.float64) ** 2, axis=1))
    assert np.allclose(norms, 1.0, rtol=0, atol=4 * TOL[w.dtype])


def test_zero_batch_and_misaligned_on_device():
    x = torch.zeros(2, 64, device="cuda")
    y = torch.empty_like(x)
    assert fwt.fwt_batched_c32(x.data_ptr(), x.data_ptr(), y.data_ptr(), y.data_ptr(), 6, 0, 1,
                               None) == fwt.FWT_OK
    big = torch.zeros(4096, device="cuda")
    st = fwt.fwt_batched_c32(big.data_ptr() + 4, big[2048:].data_ptr(), y.data_ptr(),
                             y[1].data_ptr(), 5, 1, 1, None)
    assert st == fwt.FWT_ERR_MISALIGNED


def test_guard_bands_untouched():
    """Arrays embedded in larger buffers: nothing outside them is written."""
    for dtype, n, batch in (("c32", 13, 3), ("c32", 20, 2), ("c64", 22, 1), ("i32", 9, 5)):
        N = 1 << n
        pad = 4096
        re, im = inputs.random_pair(n, batch, dtype, seed=n)
        t = {"c32": torch.float32, "c64": torch.float64, "i32": torch.int32}[dtype]
        bufs = []
        for src in (re, im):
            b = torch.full((batch * N + 2 * pad,), 7, dtype=t, device="cuda")
            b[pad:pad + batch * N] = torch.from_numpy(src.reshape(-1)).cuda()
            bufs.append(b)
        outs = [torch.full_like(b, 9) for b in bufs]
        views = [b[pad:pad + batch * N].view(batch, N) for b in bufs + outs]
        fwt.transform(views[0], views[1], views[2], views[3], normalize=dtype != "i32")
        torch.cuda.synchronize()
        for b, fill in ((bufs[0], 7), (bufs[1], 7), (outs[0], 9), (outs[1], 9)):
            assert torch.all(b[:pad] == fill) and torch.all(b[-pad:] == fill), dtype
        ore, oim = oracle.fwt_complex(re, im, normalize=dtype != "i32")
        assert_matches(dtype, views[2].cpu().numpy(), views[3].cpu().numpy(), ore, oim, "guarded")


def test_deterministic():
    for dtype in ("c32", "c64"):
        re, im = inputs.random_pair(21, 2, dtype, seed=5)
        a = gpu_transform(re, im, True)
        b = gpu_transform(re, im, True)
        assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_nonfinite_values_propagate():
    for dtype in ("c32", "c64"):
        n = 16
        re = np.zeros((2, 1 << n), NP_DTYPE[dtype])
        im = np.zeros_like(re)
        re[0, 5] = np.inf
        re[1, 3] = np.inf
        re[1, 6] = -np.inf
        im[0, 9] = np.nan
        gre, gim = gpu_transform(re, im, False)
        ore, oim = oracle.fwt_complex(re, im, normalize=False)
        for g, o in ((gre, ore), (gim, oim)):
            assert np.array_equal(np.isnan(g), np.isnan(o)), dtype
            fin = ~np.isnan(o)
            assert np.array_equal(g[fin], o[fin].astype(g.dtype)), dtype


def test_fp64_wide_dynamic_range():
    """Entries from 1e-300 to 1e+300 (and subnormals) in one vector."""
    rng = np.random.default_rng(3)
    for n in (10, 14, 18, 24):
        N = 1 << n
        mags = 10.0 ** rng.uniform(-300, 300, size=(2, N))
        re = (mags[0] * rng.choice([-1.0, 1.0], size=N))[None, :]
        im = (mags[1] * rng.choice([-1.0, 1.0], size=N))[None, :]
        re[0, : min(N, 64)] = 5e-324 * np.arange(min(N, 64))  # subnormals
        for norm in (True, False):
            gre, gim = gpu_transform(re, im, norm)
            ore, oim = oracle.fwt_complex(re, im, normalize=norm, nthreads=2)
            assert_matches("c64", gre, gim, ore, oim, f"dynamic range n={n} norm={norm}")


def test_fp64_tiny_values_round_to_subnormals():
    n = 12
    re = np.full((1, 1 << n), 1e-310)
    re[0, 1::2] = -3e-311
    im = np.full_like(re, 2e-320)
    gre, gim = gpu_transform(re, im, True)
    ore, oim = oracle.fwt_complex(re, im, normalize=True)
    assert_matches("c64", gre, gim, ore, oim, "subnormal outputs")


@pytest.mark.parametrize("dtype", ["c32", "c64"])
def test_odd_n_normalisation(dtype):
    for n in (3, 11, 15, 17, 23, 25):
        _check(dtype, n, 1, True, seed=n)


def test_maximum_n_delta():
    """n = 30 (2^30 amplitudes, 8 GiB of fp32 re+im, three passes), in place: a delta
    at j gives s * (-1)^popc(k & j) everywhere; checked on sampled k."""
    n = 30
    N = 1 << n
    j = 0x2AAAAAAB & (N - 1)
    re = torch.zeros(1, N, device="cuda")
    im = torch.zeros(1, N, device="cuda")
    re[0, j] = 1.0
    im[0, 0] = -2.0
    fwt.transform(re, im, re, im, normalize=True)
    torch.cuda.synchronize()
    ks = torch.tensor(np.random.default_rng(1).integers(0, N, size=4096), device="cuda")
    s = 2.0 ** (-n / 2)
    par = torch.zeros_like(ks)
    v = ks & j
    while bool(v.any()):
        par ^= v & 1
        v = v >> 1
    expect = s * (1.0 - 2.0 * par.double())
    assert torch.allclose(re[0, ks].double(), expect, rtol=0, atol=1e-12)
    assert torch.allclose(im[0, ks].double(), torch.full_like(expect, -2.0 * s), rtol=0, atol=1e-12)
    total = float(re.double().pow(2).sum() + im.double().pow(2).sum())
    assert abs(total - 5.0) < 1e-4
    del re, im
    torch.cuda.empty_cache()


def test_involution_large():
    """Normalised transform applied twice is the identity (fp32, fp64; n = 26, 3 passes)."""
    for dtype, tol in (("c32", 4e-6), ("c64", 2e-12)):
        re, im = inputs.random_pair(26, 1, dtype, seed=9)
        t = torch.from_numpy(re).cuda(), torch.from_numpy(im).cuda()
        a = fwt.transform(*t, normalize=True)
        b = fwt.transform(*a, normalize=True)
        torch.cuda.synchronize()
        err = rel_err_per_vector(b[0].cpu().numpy(), b[1].cpu().numpy(), re, im)
        assert err.max() < tol, dtype
    x = torch.from_numpy(inputs.random_pair(26, 1, "i32", 1)[0]).cuda()
    y = fwt.transform(x, None, normalize=False)[0]
    z = fwt.transform(y, None, normalize=False)[0]
    assert torch.equal(z, x << 26)


@pytest.mark.parametrize("dtype", ["c32", "c64", "i32"])
def test_l2_chunked_schedules(dtype):
    """Every chunking of a multi-pass transform (one part at a time, pairs,
    ragged last group, off) gives the same result as the oracle, in and out of place."""
    n, batch = 17, 5
    vec = (8 if dtype == "c64" else 4) << n
    re, im = inputs.random_pair(n, batch, dtype, seed=31)
    norm = dtype != "i32"
    ore, oim = oracle.fwt_complex(re, im, normalize=norm)
    try:
        for budget in (vec, 2 * vec, 3 * vec, 4 * vec + 1, 0, -1):
            fwt.set_l2_chunk_bytes(budget)
            for inplace in (False, True):
                gre, gim = gpu_transform(re, im, norm, inplace=inplace)
                assert_matches(dtype, gre, gim, ore, oim, f"chunk budget {budget} inplace={inplace}")
        fwt.set_l2_chunk_bytes(vec)
        gre, _ = gpu_transform(re, None, False) if dtype == "i32" else (None, None)
        if dtype == "i32":
            assert np.array_equal(gre, ore)
    finally:
        fwt.set_l2_chunk_bytes(0)


def test_bounded_wait_gives_up_and_reports():
    """A wait on an mbarrier nobody arrives at gives up after ~1 s, records a
    timeout for fwt_device_status(), and leaves the context usable."""
    import time

    assert fwt.device_status() == fwt.FWT_OK
    t = time.time()
    assert fwt.selftest_bounded_wait() == fwt.FWT_OK
    torch.cuda.synchronize()
    assert 0.5 < time.time() - t < 30
    assert fwt.device_status() == fwt.FWT_ERR_TIMEOUT
    assert fwt.device_status() == fwt.FWT_OK  # cleared
    _check("c32", 12, 2, True, seed=1)  # the context still works


@pytest.mark.parametrize("dtype", ["c32", "i32"])
def test_cluster_one_pass(dtype):
    """n = 14..18 through the one-pass cluster kernels (forced from n = 14), in and
    out of place, and equal to the factor plans (bit-exact for int32)."""
    try:
        for n in (14, 15, 16, 17, 18):
            fwt.set_cluster(fwt.CLUSTER_FROM_14)
            assert fwt.plan_passes(n, dtype) == 1
            for inplace in (False, True):
                _check(dtype, n, 3, dtype != "i32", seed=90 + n, inplace=inplace)
            re, im = inputs.random_pair(n, 2, dtype, seed=n)
            a = gpu_transform(re, im, dtype != "i32")
            fwt.set_cluster(fwt.CLUSTER_NEVER)
            b = gpu_transform(re, im, dtype != "i32")
            if dtype == "i32":
                assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])
            else:
                assert rel_err_per_vector(a[0], a[1], b[0], b[1]).max() < 4e-6
    finally:
        fwt.set_cluster(fwt.CLUSTER_AUTO)


@pytest.mark.parametrize("dtype,n", [("c32", 12), ("c64", 24), ("i32", 16), ("c32", 20)])
def test_cuda_graph_capture_and_replay(dtype, n):
    """The entry points enqueue only stream work after their first call on a device,
    so a transform can be captured in a CUDA graph and replayed (launch-bound small
    batches); each replay must give the oracle's result for the current inputs."""
    batch = 2 if n >= 20 else 8
    norm = dtype != "i32"
    re, im = inputs.random_pair(n, batch, dtype, seed=11)
    a, b = torch.from_numpy(re).cuda(), torch.from_numpy(im).cuda()
    c, d = torch.empty_like(a), torch.empty_like(b)
    fwt.transform(a, b, c, d, normalize=norm)  # device set-up outside the capture
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        fwt.transform(a, b, c, d, normalize=norm)
    for seed in (12, 13):
        re2, im2 = inputs.random_pair(n, batch, dtype, seed=seed)
        a.copy_(torch.from_numpy(re2))
        b.copy_(torch.from_numpy(im2))
        g.replay()
        torch.cuda.synchronize()
        ore, oim = oracle.fwt_complex(re2, im2, normalize=norm, nthreads=host_threads())
        assert_matches(dtype, c.cpu().numpy(), d.cpu().numpy(), ore, oim, f"graph replay {dtype} n={n}")


def test_fp64_cluster_pairs():
    """fp64 vectors of 2^14 elements run one pass on CTA pairs (one fixed-point
    exponent over the pair); 2^14-element fp64 row passes of longer vectors use the
    same kernel.  Against the oracle, with the cluster kernel off for comparison,
    and through its rare paths: Inf/NaN (IEEE adds), a tiny-magnitude vector (exact
    integer rounding), and values across 1e-300 .. 1e300."""
    try:
        assert fwt.plan_passes(14, "c64") == 1
        for batch, seed in ((1, 1), (3, 2), (64, 3)):
            for inplace in (False, True):
                _check("c64", 14, batch, True, seed=seed, inplace=inplace)
            _check("c64", 14, batch, False, seed=seed + 10)
        # 2^25 elements: (14, 11), the 14-bit row pass on CTA pairs
        assert fwt.plan_factors(25, "c64") == [14, 11]
        _check("c64", 25, 1, True, seed=25)
        re, im = inputs.random_pair(14, 5, "c64", seed=7)
        a = gpu_transform(re, im, True)
        fwt.set_cluster(fwt.CLUSTER_NEVER)
        assert fwt.plan_passes(14, "c64") == 1
        b = gpu_transform(re, im, True)
        assert rel_err_per_vector(a[0], a[1], b[0], b[1]).max() < 2e-12
    finally:
        fwt.set_cluster(fwt.CLUSTER_AUTO)
    n = 14
    re = np.zeros((2, 1 << n)); im = np.zeros_like(re)
    re[0, 5] = np.inf; re[1, 8000] = -np.inf; re[1, 9000] = 3.0; im[0, 12000] = np.nan
    gre, gim = gpu_transform(re, im, False)
    ore, oim = oracle.fwt_complex(re, im, normalize=False)
    for g, o in ((gre, ore), (gim, oim)):
        assert np.array_equal(np.isnan(g), np.isnan(o))
        fin = ~np.isnan(o)
        assert np.array_equal(g[fin], o[fin])
    rng = np.random.default_rng(5)
    tiny = rng.standard_normal((2, 1 << n)) * 1e-310  # results subnormal: exact path
    gre, gim = gpu_transform(tiny, tiny[::-1].copy(), True)
    ore, oim = oracle.fwt_complex(tiny, tiny[::-1].copy(), normalize=True)
    assert np.array_equal(gre, ore) or rel_err_per_vector(gre, gim, ore, oim).max() <= TOL["c64"]
    mags = 10.0 ** rng.uniform(-300, 300, size=(2, 1 << n))
    wide = mags * rng.choice([-1.0, 1.0], size=mags.shape)
    gre, gim = gpu_transform(wide, wide[::-1].copy(), True)
    ore, oim = oracle.fwt_complex(wide, wide[::-1].copy(), normalize=True)
    assert_matches("c64", gre, gim, ore, oim, "cluster pair, wide dynamic range")


@pytest.mark.parametrize("dtype", ["c32", "c64", "i32"])
@pytest.mark.parametrize("n", [21, 22, 23, 25])
def test_default_plans_mid_and_large_n(dtype, n):
    """The measured default plans between the every-n range and the benchmark size
    (fp64: TMA-staged column tiles of 64/128-byte segments; 4-byte: 128-byte
    segments; n = 25: 32-byte 11-bit column factors), in and out of place."""
    for inplace in (False, True):
        _check(dtype, n, 1, dtype != "i32", seed=200 + n, inplace=inplace)


def test_concurrent_host_threads():
    """Two host threads issuing transforms on their own streams at the same time
    (settings and plans under locks, tracing per thread) give the single-threaded
    results exactly (same plan, same kernels: deterministic)."""
    import threading

    cases = [("c32", 18, 4), ("c64", 16, 4), ("i32", 20, 2), ("c64", 22, 1)]
    data, expect = [], []
    for i, (dtype, n, batch) in enumerate(cases):
        re, im = inputs.random_pair(n, batch, dtype, seed=300 + i)
        a, b = torch.from_numpy(re).cuda(), torch.from_numpy(im).cuda()
        data.append((dtype, a, b))
        expect.append(fwt.transform(a, b, normalize=dtype != "i32"))
    torch.cuda.synchronize()
    errors = []

    def worker(idx):
        try:
            s = torch.cuda.Stream()
            with torch.cuda.stream(s):
                for _ in range(10):
                    for k in range(idx, len(data), 2):
                        dtype, a, b = data[k]
                        out = fwt.transform(a, b, normalize=dtype != "i32")
                        s.synchronize()
                        if not (torch.equal(out[0], expect[k][0]) and torch.equal(out[1], expect[k][1])):
                            errors.append((idx, k))
        except Exception as e:  # pragma: no cover - reported below
            errors.append(repr(e))

    threads = [threading.Thread(target=worker, args=(i,)) for i in range(2)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors


def test_random_plans_widths_and_movers():
    """Seeded random cases over n = 14..23: a random valid 2- or 3-factor split, column
    width, TMA mode, batch, in or out of place, normalised or not."""
    rng = np.random.default_rng(2024)
    done = 0
    try:
        while done < 30:
            dtype = ["c32", "c64", "i32"][rng.integers(3)]
            n = int(rng.integers(14, 24))
            cb = int(rng.choice([16, 32, 64, 128]))
            tma = int(rng.integers(0, 3))
            if cb == 16:
                tma = 2
            fwt.set_tma(tma)
            fwt.set_column_bytes(dtype, cb)
            plans = _valid_plans(n, dtype)
            if not plans:
                continue
            plan = plans[int(rng.integers(len(plans)))]
            fwt.set_plan(n, dtype, plan)
            batch = int(rng.integers(1, 4))
            norm = dtype != "i32" and bool(rng.integers(2))
            re, im = inputs.random_pair(n, batch, dtype, seed=int(rng.integers(1 << 30)))
            ore, oim = oracle.fwt_complex(re, im, normalize=norm, nthreads=host_threads())
            gre, gim = gpu_transform(re, im, norm, inplace=bool(rng.integers(2)))
            assert_matches(dtype, gre, gim, ore, oim, f"{dtype} n={n} plan={plan} cb={cb} tma={tma}")
            fwt.set_plan(n, dtype, None)
            done += 1
    finally:
        for dt in ("c32", "c64", "i32"):
            fwt.set_column_bytes(dt, 0)
            for n in range(14, 24):
                fwt.set_plan(n, dt, None)
        fwt.set_tma(fwt.TMA_AUTO)
    assert fwt.device_status() == fwt.FWT_OK


def test_plan_log_environment_variable():
    """FWT_LOG=1 prints one plan line a call to stderr (a fresh process: the variable
    is read once); without it nothing is printed."""
    import os
    import subprocess
    import sys

    code = ("import torch, walsh_hadamard_transform_gb300 as fwt\n"
            "a = torch.randn(2, 1 << 24, dtype=torch.float64, device='cuda')\n"
            "fwt.transform(a, a.clone())\n"
            "x = torch.randn(3, 1 << 12, device='cuda')\n"
            "fwt.transform(x, x.clone(), bits=(3, 5))\n"
            "torch.cuda.synchronize()\n")
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    for value, expect in (("1", True), ("0", False)):
        env = dict(os.environ, FWT_LOG=value)
        r = subprocess.run([sys.executable, "-c", code], cwd=root, env=env, capture_output=True,
                           text=True, timeout=300)
        assert r.returncode == 0, r.stderr[-2000:]
        lines = [ln for ln in r.stderr.splitlines() if ln.startswith("fwt: ")]
        if not expect:
            assert lines == []
            continue
        assert len(lines) == 2, r.stderr[-2000:]
        assert lines[0].startswith("fwt: transform c64 n=24 batch=2 passes=2 | row K=13")
        assert "| col K=11 tile=2^13 stride=2^13 32B tma" in lines[0]
        assert lines[1].startswith("fwt: bits c32 n=12 batch=3 passes=1 | rowbits")
        assert "bits=[3,8)" in lines[1]


@pytest.mark.parametrize("dtype", ["c32", "c64", "i32"])
def test_overlapped_launches_keep_stream_order(dtype):
    """Pass kernels launched with programmatic stream serialisation (the default) may
    start while the previous kernel drains, and wait for it before touching memory.
    Chains of dependent in-place transforms on one stream must compose exactly as
    with plain launches: the transform twice is 2^n times the input (the identity
    when normalised), bit for bit equal to plain launches, for one-, two- and
    three-pass plans and cluster transforms."""
    norm = dtype != "i32"
    try:
        for n, batch in ((10, 64), (12, 33), (16, 5), (21, 2), (27, 1)):
            re, im = inputs.random_pair(n, batch, dtype, seed=400 + n)
            outs = {}
            for pdl in (0, 1):
                fwt.set_pdl(pdl)
                a, b = torch.from_numpy(re).cuda(), torch.from_numpy(im).cuda()
                for _ in range(4):  # four dependent transforms back to back, no sync
                    fwt.transform(a, b, a, b, normalize=norm)
                torch.cuda.synchronize()
                outs[pdl] = (a.cpu().numpy(), b.cpu().numpy())
            assert np.array_equal(outs[0][0], outs[1][0]) and np.array_equal(outs[0][1], outs[1][1]), \
                f"{dtype} n={n}: overlapped launches differ from plain ones"
            if dtype == "i32":  # H H x = 2^n x, four times: 2^(2n) x (mod 2^32)
                want = (re.astype(np.int64) << (2 * n)) % (1 << 32)
                want = np.where(want >= 1 << 31, want - (1 << 32), want).astype(np.int32)
                assert np.array_equal(outs[1][0], want)
            else:
                err = rel_err_per_vector(outs[1][0], outs[1][1], re, im)
                assert err.max() < 4 * TOL[dtype], f"{dtype} n={n}: {err.max():.3e}"
    finally:
        fwt.set_pdl(1)
    assert fwt.pdl() == 1
