"""Host-buffer entry points over the library's static device workspace
(fwt_host_static_*), the form for callers that cannot allocate device memory:
same results as the oracle, several chunks and slots, calls on two streams
serialised on the shared buffer, nothing allocated per call, and vectors larger
than the workspace rejected before any CUDA call.  Collected last, so that a run
stopping at the first failure has run every other test first."""
import numpy as np
import pytest

import oracle
import walsh_hadamard_transform_gb300 as fwt
from helpers import assert_matches, host_threads
from walsh_hadamard_transform_gb300 import inputs

_STATIC = {"c32": "fwt_host_static_c32", "c64": "fwt_host_static_c64",
           "i32": "fwt_host_static_i32"}


def test_static_entry_points_are_declared_and_check_arguments():
    lib = fwt.library()
    for name in (*_STATIC.values(), "fwt_host_static_workspace_bytes"):
        assert hasattr(lib, name)
    assert fwt.fwt_host_static_workspace_bytes() >= 64 << 20
    a, b, c, d = 0x10000, 0x20000, 0x30000, 0x40000
    assert fwt.fwt_host_static_c32(a, b, c, d, -1, 1, 1, None) == fwt.FWT_ERR_INVALID_ARG
    assert fwt.fwt_host_static_c64(a, b, c, d, 31, 1, 1, None) == fwt.FWT_ERR_INVALID_ARG
    assert fwt.fwt_host_static_c32(None, None, None, None, 4, 0, 1, None) == fwt.FWT_OK
    assert fwt.fwt_host_static_c64(a, None, c, None, 4, 1, 1, None) == fwt.FWT_ERR_INVALID_ARG
    assert fwt.fwt_host_static_i32(a, None, c, None, 4, 1, 1, None) == fwt.FWT_ERR_UNSUPPORTED
    # overlapping host arrays: an argument error, found before any CUDA call
    assert fwt.fwt_host_static_c32(a, b, a + 4, d, 4, 1, 1, None) == fwt.FWT_ERR_INVALID_ARG


def test_static_workspace_rejects_vectors_larger_than_it():
    """A vector (both parts) that does not fit the static workspace is an argument
    error, returned before any CUDA call (so this runs without a GPU; the fake host
    addresses are never dereferenced)."""
    ws = fwt.fwt_host_static_workspace_bytes()
    n = 1
    while (2 * 8 << n) <= ws:
        n += 1
    A, G = 1 << 40, 1 << 34
    st = fwt.fwt_host_static_c64(A, A + G, A + 2 * G, A + 3 * G, n, 1, 1, None)
    assert st == fwt.FWT_ERR_INVALID_ARG
    # one vector that fits exactly is accepted by the checks (n - 1: 2 x 8 B x 2^(n-1))
    assert (2 * 8 << (n - 1)) <= ws


def _pinned(x):
    import torch

    return None if x is None else torch.from_numpy(np.ascontiguousarray(x)).pin_memory()


class _Call:
    """Inputs, pinned host buffers and the oracle's result of one static call.  The
    pinned inputs stay referenced here until the caller has synchronised."""

    def __init__(self, dtype, n, batch, seed, real_only=False):
        import torch

        re, im = inputs.random_pair(n, batch, dtype, seed)
        if real_only:
            im = None
        self.dtype, self.n, self.batch = dtype, n, batch
        self.norm = dtype != "i32"
        self.expect = oracle.fwt_complex(re, im, normalize=self.norm, nthreads=host_threads())
        self.a, self.b = _pinned(re), _pinned(im)
        self.oa = torch.empty_like(self.a).pin_memory()
        self.ob = None if self.b is None else torch.empty_like(self.b).pin_memory()

    def issue(self, stream=None):
        f = getattr(fwt, _STATIC[self.dtype])
        handle = None if stream is None else stream.cuda_stream
        st = f(self.a.data_ptr(), None if self.b is None else self.b.data_ptr(),
               self.oa.data_ptr(), None if self.ob is None else self.ob.data_ptr(),
               self.n, self.batch, self.norm, handle)
        assert st == fwt.FWT_OK, fwt.status_string(st)

    def check(self, what):
        ore, oim = self.expect
        assert_matches(self.dtype, self.oa.numpy(), None if self.ob is None else self.ob.numpy(),
                       ore, oim, what)


@pytest.mark.gpu
def test_static_workspace_matches_oracle():
    import torch

    for dtype, n, batch in (("c32", 10, 300), ("c64", 16, 40), ("i32", 18, 7), ("c64", 22, 3),
                            ("c32", 0, 5)):
        call = _Call(dtype, n, batch, seed=n)
        call.issue()
        torch.cuda.synchronize()
        call.check(f"static {dtype} n={n}")
    call = _Call("i32", 12, 9, seed=3, real_only=True)
    call.issue()
    torch.cuda.synchronize()
    call.check("static int32 real only")


@pytest.mark.gpu
def test_static_workspace_calls_on_two_streams_do_not_overlap():
    """Two calls on different streams share the static buffer; the second must wait
    for the first to have copied its last chunk out.  The first call moves 1.5 GiB
    each way (many chunks through the three slots), and the second is enqueued right
    behind it: the test checks that the first is still in flight at that moment, so
    without the wait the second call's copies would overwrite slots the first still
    uses."""
    import torch

    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    first = _Call("c64", 20, 96, seed=1)
    second = _Call("c64", 20, 24, seed=2)
    torch.cuda.synchronize()
    first.issue(s1)
    mark = torch.cuda.Event()
    mark.record(s1)
    second.issue(s2)
    in_flight = not mark.query()
    torch.cuda.synchronize()
    assert in_flight, "the first call finished before the second was enqueued"
    first.check("two streams, first call")
    second.check("two streams, second call")


@pytest.mark.gpu
def test_static_workspace_allocates_nothing_per_call():
    import torch

    warm = _Call("c32", 16, 64, seed=4)
    warm.issue()
    torch.cuda.synchronize()
    calls = [_Call("c32", 16, 64, seed=5 + seed) for seed in range(3)]
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    for call in calls:
        call.issue()
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free0 - free1 < (8 << 20)  # no per-call device allocation (pinned buffers are host)
    for i, call in enumerate(calls):
        call.check(f"call {i}")


@pytest.mark.gpu
def test_static_entry_matches_workspace_entry_twice():
    """The static-buffer entry point against the caller-workspace entry point on the
    same inputs, two calls in a row (the second reuses the buffer the first left)."""
    import torch

    for dtype, n, batch in (("c64", 18, 20), ("c32", 21, 6)):
        ref = _Call(dtype, n, batch, seed=40 + n)
        ws = torch.empty(fwt.fwt_host_workspace_bytes(fwt.DTYPES[dtype], n, batch),
                         dtype=torch.uint8, device="cuda")
        f = getattr(fwt, "fwt_host_" + dtype)
        wa = torch.empty_like(ref.oa).pin_memory()
        wb = torch.empty_like(ref.ob).pin_memory()
        st = f(ref.a.data_ptr(), ref.b.data_ptr(), wa.data_ptr(), wb.data_ptr(), n, batch,
               ref.norm, ws.data_ptr(), ws.numel(), None)
        assert st == fwt.FWT_OK
        torch.cuda.synchronize()
        for rep in range(2):
            ref.oa.zero_()
            ref.ob.zero_()
            ref.issue()
            torch.cuda.synchronize()
            assert_matches(dtype, ref.oa.numpy(), ref.ob.numpy(), wa.numpy(), wb.numpy(),
                           f"static vs workspace, call {rep}")
            ref.check(f"static call {rep}")
