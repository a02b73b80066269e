"""Host-buffer entry points (fwt_host_*) vs the CPU oracle (GPU only): the chunked
copy-in / transform / copy-out pipeline must give the same results as the device
entry points for every chunking the workspace allows."""
import numpy as np
import pytest
import torch

import oracle
import walsh_hadamard_transform_gb300 as fwt
from helpers import assert_matches, host_threads
from walsh_hadamard_transform_gb300 import inputs

pytestmark = pytest.mark.gpu


def _host_pair(re, im, pinned):
    a = torch.from_numpy(np.ascontiguousarray(re))
    b = None if im is None else torch.from_numpy(np.ascontiguousarray(im))
    if pinned:
        a = a.pin_memory()
        b = None if b is None else b.pin_memory()
    return a, b


def _run(dtype, n, batch, ws_fraction=1.0, pinned=True, inplace=False, real_only=False, seed=0):
    re, im = inputs.random_pair(n, batch, dtype, seed)
    if real_only:
        im = None
    norm = dtype != "i32"
    ore, oim = oracle.fwt_complex(re, im, normalize=norm, nthreads=host_threads())
    a, b = _host_pair(re.copy(), None if im is None else im.copy(), pinned)
    full = fwt.fwt_host_workspace_bytes(fwt.DTYPES[dtype], n, batch, im is not None)
    one_vector = (1 if im is None else 2) * (((re.itemsize << n) + 255) // 256 * 256)
    nbytes = max(int(full * ws_fraction) // 16 * 16, one_vector)
    ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    if inplace:
        out = fwt.transform_host(a, b, a, b, normalize=norm, workspace=ws)
    else:
        out = fwt.transform_host(a, b, normalize=norm, workspace=ws)
    gim = None if out[1] is None else out[1].numpy()
    assert_matches(dtype, out[0].numpy(), gim, ore, oim,
                   f"host {dtype} n={n} batch={batch} ws={ws_fraction}")


@pytest.mark.parametrize("dtype", ["c32", "c64", "i32"])
@pytest.mark.parametrize("n,batch", [(0, 5), (3, 7), (10, 33), (14, 9), (17, 5), (20, 3)])
def test_host_matches_oracle(dtype, n, batch):
    _run(dtype, n, batch, seed=n + batch)


@pytest.mark.parametrize("dtype", ["c32", "c64", "i32"])
@pytest.mark.parametrize("fraction", [0.34, 0.2, 0.05])
def test_host_small_workspace_rotates_slots(dtype, fraction):
    # smaller workspaces: fewer vectors a chunk and / or fewer than three slots
    _run(dtype, 12, 50, ws_fraction=fraction, seed=3)
    _run(dtype, 19, 6, ws_fraction=fraction, seed=4)


def test_host_workspace_below_one_vector_is_rejected():
    re, im = inputs.random_pair(15, 2, "c64", 1)
    a, b = _host_pair(re, im, True)
    ws = torch.empty(2 * 8 << 15, dtype=torch.uint8, device="cuda")[: (2 * 8 << 15) - 16]
    with pytest.raises(fwt.FwtError):
        fwt.transform_host(a, b, workspace=ws)


@pytest.mark.parametrize("dtype", ["c32", "i32"])
def test_host_in_place_pageable_and_real_only(dtype):
    _run(dtype, 13, 11, inplace=True, seed=5)
    _run(dtype, 13, 11, pinned=False, seed=6)
    if dtype == "i32":
        _run(dtype, 13, 11, real_only=True, seed=7)
        _run(dtype, 13, 11, real_only=True, pinned=False, inplace=True, seed=8)


def test_host_waits_for_earlier_work_on_the_stream():
    """Work the caller queued on the stream before the call finishes before the
    first copy: a kernel that fills the workspace must not clobber chunk data."""
    re, im = inputs.random_pair(16, 8, "c32", 9)
    a, b = _host_pair(re, im, True)
    ws = torch.empty(fwt.fwt_host_workspace_bytes(fwt.FWT_C32, 16, 8),
                     dtype=torch.uint8, device="cuda")
    s = torch.cuda.Stream()
    big = torch.empty(1 << 28, dtype=torch.uint8, device="cuda")
    with torch.cuda.stream(s):
        for _ in range(4):  # a few ms of work on `s` that writes the workspace last
            big.fill_(1)
        ws.fill_(0x7f)
        out = fwt.transform_host(a, b, normalize=True, workspace=ws, stream=s)
    ore, oim = oracle.fwt_complex(re, im, normalize=True, nthreads=host_threads())
    assert_matches("c32", out[0].numpy(), out[1].numpy(), ore, oim, "stream order")


def test_host_rejects_device_tensors_and_bad_shapes():
    with pytest.raises(ValueError):
        fwt.transform_host(torch.zeros(2, 8, device="cuda"), torch.zeros(2, 8, device="cuda"))
    with pytest.raises(ValueError):
        fwt.transform_host(torch.zeros(2, 6), torch.zeros(2, 6))


@pytest.mark.parametrize("name", ["n24_b16_c64", "n24_b16_c32"])
def test_host_benchmark_workload(name):
    """The end-to-end call the benchmark times (n = 24, batch 16, pinned host arrays, the
    full-depth workspace): the first and last vectors against the oracle, and every
    vector's norm against Parseval (the normalised transform is orthogonal)."""
    w = inputs.WORKLOADS[name]
    re, im = w.generate()
    a, b = _host_pair(re, im, pinned=True)
    ws = torch.empty(fwt.fwt_host_workspace_bytes(fwt.DTYPES[w.dtype], w.n, w.batch, True),
                     dtype=torch.uint8, device="cuda")
    gre, gim = fwt.transform_host(a, b, normalize=True, workspace=ws)
    gre, gim = gre.numpy(), gim.numpy()
    rows = [0, w.batch - 1]
    ore, oim = oracle.fwt_complex(re[rows], im[rows], normalize=True, nthreads=host_threads())
    assert_matches(w.dtype, gre[rows], gim[rows], ore, oim, f"host {name} vectors {rows}")
    tol = 1e-5 if w.dtype == "c32" else 1e-11
    for v in range(w.batch):
        n_in = np.sum(re[v].astype(np.float64) ** 2 + im[v].astype(np.float64) ** 2)
        n_out = np.sum(gre[v].astype(np.float64) ** 2 + gim[v].astype(np.float64) ** 2)
        assert abs(n_out - n_in) <= tol * n_in, (name, v, n_in, n_out)
