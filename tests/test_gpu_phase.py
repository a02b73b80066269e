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
