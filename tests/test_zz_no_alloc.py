"""Host-buffer entry points over the library's static device workspace
(fwt_host_static_*): same results as the oracle, several chunks and slots, calls
on two streams serialised on the shared buffer, nothing allocated per call, and
vectors larger than the workspace rejected.  Collected last."""
import numpy as np
import pytest

import oracle
import walsh_hadamard_transform_gb300 as fwt
from helpers import assert_matches, host_threads
from walsh_hadamard_transform_gb300 import inputs


def test_static_entry_points_are_declared_and_check_arguments():
    lib = fwt.library()
    for name in ("fwt_host_static_c32", "fwt_host_static_c64", "fwt_host_static_i32",
                 "fwt_host_static_workspace_bytes"):
        assert hasattr(lib, name)
    assert fwt.fwt_host_static_workspace_bytes() >= 64 << 20
    a, b, c, d = 0x10000, 0x20000, 0x30000, 0x40000
    assert fwt.fwt_host_static_c32(a, b, c, d, -1, 1, 1, None) == fwt.FWT_ERR_INVALID_ARG
    assert fwt.fwt_host_static_c64(a, b, c, d, 31, 1, 1, None) == fwt.FWT_ERR_INVALID_ARG
    assert fwt.fwt_host_static_c32(None, None, None, None, 4, 0, 1, None) == fwt.FWT_OK
    assert fwt.fwt_host_static_c64(a, None, c, None, 4, 1, 1, None) == fwt.FWT_ERR_INVALID_ARG
    assert fwt.fwt_host_static_i32(a, None, c, None, 4, 1, 1, None) == fwt.FWT_ERR_UNSUPPORTED


def _pinned(x):
    import torch

    return None if x is None else torch.from_numpy(np.ascontiguousarray(x)).pin_memory()


def _run(dtype, n, batch, seed, real_only=False, stream=None):
    import torch

    re, im = inputs.random_pair(n, batch, dtype, seed)
    if real_only:
        im = None
    norm = dtype != "i32"
    ore, oim = oracle.fwt_complex(re, im, normalize=norm, nthreads=host_threads())
    a, b = _pinned(re), _pinned(im)
    oa = torch.empty_like(a).pin_memory()
    ob = None if b is None else torch.empty_like(b).pin_memory()
    f = {"c32": fwt.fwt_host_static_c32, "c64": fwt.fwt_host_static_c64,
         "i32": fwt.fwt_host_static_i32}[dtype]
    handle = None if stream is None else stream.cuda_stream
    st = f(a.data_ptr(), None if b is None else b.data_ptr(), oa.data_ptr(),
           None if ob is None else ob.data_ptr(), n, batch, norm, handle)
    assert st == fwt.FWT_OK, fwt.status_string(st)
    return (oa, ob), (ore, oim), stream


@pytest.mark.gpu
def test_static_workspace_matches_oracle():
    import torch

    for dtype, n, batch in (("c32", 10, 300), ("c64", 16, 40), ("i32", 18, 7), ("c64", 22, 3),
                            ("c32", 0, 5)):
        (oa, ob), (ore, oim), _ = _run(dtype, n, batch, seed=n)
        torch.cuda.synchronize()
        assert_matches(dtype, oa.numpy(), ob.numpy(), ore, oim, f"static {dtype} n={n}")
    (oa, _), (ore, _), _ = _run("i32", 12, 9, seed=3, real_only=True)
    torch.cuda.synchronize()
    assert np.array_equal(oa.numpy(), ore)


@pytest.mark.gpu
def test_static_workspace_calls_on_two_streams_do_not_overlap():
    """Two calls on different streams share the static buffer; the second waits for
    the first to have copied its last chunk out, so both results are right."""
    import torch

    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    r1 = _run("c64", 20, 24, seed=1, stream=s1)
    r2 = _run("c64", 20, 24, seed=2, stream=s2)
    torch.cuda.synchronize()
    for (oa, ob), (ore, oim), _ in (r1, r2):
        assert_matches("c64", oa.numpy(), ob.numpy(), ore, oim, "two streams")


@pytest.mark.gpu
def test_static_workspace_allocates_nothing_per_call():
    import torch

    _run("c32", 16, 64, seed=4)
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    for seed in range(3):
        _run("c32", 16, 64, seed=5 + seed)
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free0 - free1 < (8 << 20)  # no per-call device allocation (pinned outputs are host)


@pytest.mark.gpu
def test_static_workspace_rejects_vectors_larger_than_it():
    """A vector (both parts) that does not fit the static workspace is an argument
    error, returned before anything is enqueued (the fake host addresses below are
    never dereferenced)."""
    ws = fwt.fwt_host_static_workspace_bytes()
    n = 1
    while (2 * 8 << n) <= ws:
        n += 1
    A, G = 1 << 40, 1 << 34
    st = fwt.fwt_host_static_c64(A, A + G, A + 2 * G, A + 3 * G, n, 1, 1, None)
    assert st == fwt.FWT_ERR_INVALID_ARG
