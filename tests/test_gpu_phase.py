"""Fused diagonal phase + transform, y = s H (e^{i theta} . x), CUDA vs oracle (GPU only)."""
import numpy as np
import pytest
import torch

import oracle
import walsh_hadamard_transform_gb300 as fwt
from helpers import TOL, rel_err_per_vector
from walsh_hadamard_transform_gb300 import inputs

pytestmark = pytest.mark.gpu


def _run(re, im, th, norm, inplace=False):
    a, b = torch.from_numpy(re).cuda(), torch.from_numpy(im).cuda()
    t = torch.from_numpy(th).cuda()
    if inplace:
        fwt.phase_transform(a, b, t, a, b, normalize=norm)
        out = (a, b)
    else:
        out = fwt.phase_transform(a, b, t, normalize=norm)
    torch.cuda.synchronize()
    return out[0].cpu().numpy(), out[1].cpu().numpy()


@pytest.mark.parametrize("n", [0, 1, 2, 3, 5, 10, 12, 13, 14, 17, 20])
def test_phase_then_transform_matches_oracle(n):
    rng = np.random.default_rng(n)
    re, im = inputs.random_pair(n, 3, "c32", seed=60 + n)
    for shared in (False, True):
        th = rng.uniform(-np.pi, np.pi, size=(1 if shared else 3, 1 << n)).astype(np.float32)
        for norm in (True, False):
            ore, oim = oracle.phase_fwt(re, im, th, normalize=norm)
            gre, gim = _run(re, im, th, norm, inplace=norm)
            err = rel_err_per_vector(gre, gim, ore, oim)
            assert err.max() <= TOL["c32"], f"n={n} shared={shared} norm={norm}: {err.max():.3e}"


def test_phase_n24_full_batch():
    w = inputs.WORKLOADS["n24_b16_c32"]
    re, im = w.generate(batch=2)
    th = np.random.default_rng(5).uniform(0, 2 * np.pi, size=(2, w.N)).astype(np.float32)
    gre, gim = _run(re, im, th, True)
    ore, oim = oracle.phase_fwt(re, im, th, normalize=True)
    err = rel_err_per_vector(gre, gim, ore, oim)
    assert err.max() <= TOL["c32"], f"{err.max():.3e}"


def test_zero_phase_is_the_plain_transform():
    re, im = inputs.random_pair(16, 2, "c32", seed=3)
    th = np.zeros((1, 1 << 16), np.float32)
    gre, gim = _run(re, im, th, True)
    ore, oim = oracle.fwt_complex(re, im, normalize=True)
    assert rel_err_per_vector(gre, gim, ore, oim).max() <= TOL["c32"]


def test_phase_argument_errors():
    x = torch.zeros(2, 64, device="cuda")
    y = torch.empty_like(x)
    th = torch.zeros(128, device="cuda")
    p = (x.data_ptr(), x[1].data_ptr())
    o = (y.data_ptr(), y[1].data_ptr())
    assert fwt.fwt_phase_c32(*p, th.data_ptr(), 64, *o, 6, 1, 1, None) == fwt.FWT_OK
    assert fwt.fwt_phase_c32(*p, 0, 64, *o, 6, 1, 1, None) == fwt.FWT_ERR_INVALID_ARG  # no angles
    assert fwt.fwt_phase_c32(*p, th.data_ptr() + 4, 64, *o, 6, 1, 1, None) == fwt.FWT_ERR_MISALIGNED
    assert fwt.fwt_phase_c32(*p, th.data_ptr(), 6, *o, 6, 1, 1, None) == fwt.FWT_ERR_MISALIGNED
    assert fwt.fwt_phase_c32(*p, y.data_ptr(), 0, *o, 6, 1, 1, None) == fwt.FWT_ERR_INVALID_ARG  # overlap
    assert fwt.fwt_phase_c32(*p, th.data_ptr(), -1, *o, 6, 1, 1, None) == fwt.FWT_ERR_INVALID_ARG
    torch.cuda.synchronize()


@pytest.mark.parametrize("n", [0, 1, 2, 5, 12, 14, 16, 19])
def test_phase_fp64_matches_oracle(n):
    """fp64: phase element by element (double sincos), then the fp64 transform in
    place; shared and per-vector angles, in and out of place, angles up to 50 rad."""
    rng = np.random.default_rng(100 + n)
    re, im = inputs.random_pair(n, 3, "c64", seed=70 + n)
    for shared in (False, True):
        th = rng.uniform(-50.0, 50.0, size=(1 if shared else 3, 1 << n))
        for norm in (True, False):
            ore, oim = oracle.phase_fwt(re, im, th, normalize=norm)
            gre, gim = _run(re, im, th, norm, inplace=norm)
            err = rel_err_per_vector(gre, gim, ore, oim)
            assert err.max() <= TOL["c64"], f"n={n} shared={shared} norm={norm}: {err.max():.3e}"


def test_phase_fp64_n24_and_errors():
    w = inputs.WORKLOADS["n24_b16_c64"]
    re, im = w.generate(batch=1)
    th = np.random.default_rng(6).uniform(0, 2 * np.pi, size=(1, w.N))
    gre, gim = _run(re, im, th, True)
    ore, oim = oracle.phase_fwt(re, im, th, normalize=True)
    assert rel_err_per_vector(gre, gim, ore, oim).max() <= TOL["c64"]
    x = torch.zeros(2, 64, dtype=torch.float64, device="cuda")
    y = torch.empty_like(x)
    t = torch.zeros(128, dtype=torch.float64, device="cuda")
    p = (x.data_ptr(), x[1].data_ptr())
    o = (y.data_ptr(), y[1].data_ptr())
    assert fwt.fwt_phase_c64(*p, t.data_ptr(), 64, *o, 6, 1, 1, None) == fwt.FWT_OK
    assert fwt.fwt_phase_c64(*p, t.data_ptr() + 8, 64, *o, 6, 1, 1, None) == fwt.FWT_ERR_MISALIGNED
    assert fwt.fwt_phase_c64(*p, t.data_ptr(), 3, *o, 6, 1, 1, None) == fwt.FWT_ERR_MISALIGNED
    assert fwt.fwt_phase_c64(*p, y.data_ptr(), 0, *o, 6, 1, 1, None) == fwt.FWT_ERR_INVALID_ARG
    torch.cuda.synchronize()


def test_phase_fp64_angles_to_1e3_match_oracle():
    """fp64 phase with angles of up to 1e3 rad (fixed-point sine and cosine), then the
    transform: within the fp64 specification of the oracle (libm sin/cos, double)."""
    rng = np.random.default_rng(7)
    for n, batch in ((12, 3), (16, 2), (24, 1)):
        re, im = inputs.random_pair(n, batch, "c64", seed=80 + n)
        th = rng.uniform(-1e3, 1e3, size=(batch, 1 << n))
        ore, oim = oracle.phase_fwt(re, im, th, normalize=True)
        gre, gim = _run(re, im, th, True)
        err = rel_err_per_vector(gre, gim, ore, oim)
        assert err.max() <= TOL["c64"], f"n={n}: {err.max():.3e}"


def _angles(rng, size):
    parts = [rng.uniform(-1e3, 1e3, size), rng.uniform(-np.pi, np.pi, size),
             np.round(rng.uniform(-600, 600, size)) * (np.pi / 2) + rng.uniform(-1e-9, 1e-9, size),
             rng.uniform(-1e-6, 1e-6, size), rng.uniform(-1e12, 1e12, size),
             np.array([0.0, -0.0, 5e-324, -1e-300, 1e-150, np.pi, -np.pi / 2, 2 * np.pi, 1e11,
                       -1.0995e12])]
    return np.concatenate(parts)


def test_phase_fp64_rotation_matches_cuda_sincos():
    """n = 0 and x = 1: the phase alone, (cos t, sin t), against CUDA's double-precision
    cos and sin (torch on the device), for angles across [-1e12, 1e12] including
    multiples of pi/2, tiny angles and signed zeros; non-finite angles and angles
    beyond 2^40 rad (the fp64 sincos fallback) give what CUDA's sincos gives."""
    rng = np.random.default_rng(11)
    th = _angles(rng, 4000)
    th = np.concatenate([th, [np.inf, -np.inf, np.nan, 3e12, -1e15, 1e300]])
    one = np.ones((th.size, 1)); zero = np.zeros_like(one)
    gre, gim = _run(one, zero, th[:, None], False)
    t = torch.from_numpy(th).cuda()
    cre, cim = torch.cos(t).cpu().numpy(), torch.sin(t).cpu().numpy()
    fin = np.isfinite(cre)
    assert np.array_equal(np.isnan(gre[:, 0]), np.isnan(cre)) and np.array_equal(np.isnan(gim[:, 0]), np.isnan(cim))
    assert np.max(np.abs(gre[fin, 0] - cre[fin])) <= 5e-16
    assert np.max(np.abs(gim[fin, 0] - cim[fin])) <= 5e-16


def test_phase_fp64_element_magnitudes():
    """Elements from subnormal to 1e250 (one exponent per element pair in the fixed
    point rotation; results near the subnormal range take the exact integer rounding),
    and Inf/NaN elements (the fp64 fallback), against the oracle."""
    rng = np.random.default_rng(12)
    n = 10
    re, im = inputs.random_pair(n, 4, "c64", seed=90)
    re[0] *= 1e250; im[0] *= 1e-250
    re[1] *= 1e-300; im[1] *= 1e-305
    re[2] = 4e-320 * np.sign(re[2]); im[2] = -7e-321
    th = rng.uniform(-1e3, 1e3, size=(4, 1 << n))
    ore, oim = oracle.phase_fwt(re, im, th, normalize=True)
    gre, gim = _run(re, im, th, True)
    err = rel_err_per_vector(gre, gim, ore, oim)
    assert err[:2].max() <= TOL["c64"] and err[3] <= TOL["c64"], err
    # subnormal elements: the oracle's own double products round on the subnormal grid
    # (5e-324 apart), so compare absolutely (2^10 terms, each off by a few grid steps)
    assert max(np.abs(gre[2] - ore[2]).max(), np.abs(gim[2] - oim[2]).max()) <= 1e-319
    re2, im2 = re.copy(), im.copy()
    re2[3, 5] = np.inf; im2[3, 7] = np.nan
    gre, gim = _run(re2, im2, th, False)
    assert np.isnan(gre[3]).any() and np.isnan(gim[3]).any()
    ore, oim = oracle.phase_fwt(re2[:2], im2[:2], th[:2], normalize=False)
    assert rel_err_per_vector(gre[:2], gim[:2], ore, oim).max() <= TOL["c64"]
