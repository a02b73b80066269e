"""Shared test helpers: GPU calls through the C ABI and oracle comparisons."""
from __future__ import annotations

import os

import numpy as np

TOL = {"c32": 2e-6, "c64": 1e-12}
NP_DTYPE = {"c32": np.float32, "c64": np.float64, "i32": np.int32}


def host_threads() -> int:
    return max(1, min(16, os.cpu_count() or 1))


def gpu_transform(re, im, normalize, inplace=False):
    """Run the CUDA transform on host arrays; returns host (re, im) results."""
    import torch

    import walsh_hadamard_transform_gb300 as fwt

    dre = torch.from_numpy(np.ascontiguousarray(re)).cuda()
    dim_ = None if im is None else torch.from_numpy(np.ascontiguousarray(im)).cuda()
    if inplace:
        ore, oim = fwt.transform(dre, dim_, dre, dim_, normalize=normalize)
    else:
        ore, oim = fwt.transform(dre, dim_, normalize=normalize)
    torch.cuda.synchronize()
    return ore.cpu().numpy(), None if oim is None else oim.cpu().numpy()


def rel_err_per_vector(gre, gim, ore, oim) -> np.ndarray:
    """Complex relative L2 error of each vector (re and im together).

    Both sides are divided by the vector's largest reference magnitude before
    squaring, so entries near 1e300 neither overflow nor lose the ratio."""
    gre = np.atleast_2d(gre).astype(np.float64); ore = np.atleast_2d(ore).astype(np.float64)
    parts = [(gre, ore)]
    if gim is not None:
        parts.append((np.atleast_2d(gim).astype(np.float64), np.atleast_2d(oim).astype(np.float64)))
    scale = np.max([np.max(np.abs(o), axis=-1) for _, o in parts], axis=0)
    scale = np.where(scale > 0, scale, 1.0)[:, None]
    num = sum(np.sum(((g - o) / scale) ** 2, axis=-1) for g, o in parts)
    den = sum(np.sum((o / scale) ** 2, axis=-1) for _, o in parts)
    return np.sqrt(num) / np.where(den > 0, np.sqrt(den), 1.0)


def assert_matches(dtype, gre, gim, ore, oim, what=""):
    if dtype == "i32":
        assert np.array_equal(gre, ore), f"int32 real part differs {what}"
        if oim is not None:
            assert np.array_equal(gim, oim), f"int32 imaginary part differs {what}"
        return
    err = rel_err_per_vector(gre, gim, ore, oim)
    assert err.max() <= TOL[dtype], f"{what}: max relative L2 error {err.max():.3e} > {TOL[dtype]}"
