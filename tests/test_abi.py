"""The C-ABI library: builds, exports every declared symbol, validates arguments
on the host before any CUDA call, and its tile shapes pass the host self-check.
CPU only: no call here reaches the GPU."""
import ctypes
import os
import re

import pytest

import walsh_hadamard_transform_gb300 as fwt
from walsh_hadamard_transform_gb300 import build as fbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fwt.h")


@pytest.fixture(scope="module")
def lib():
    fbuild.build()
    return fwt.library()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(fwt_\w+)\s*\(", text)))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for must in ("fwt_batched_c32", "fwt_batched_c64", "fwt_batched_i32", "fwt_status_string",
                 "fwt_plan_passes"):
        assert must in names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), f"{name} declared in include/fwt.h but not exported"


def test_status_strings(lib):
    for st in range(6):
        assert fwt.status_string(st)
    assert fwt.status_string(99) == "unknown status"


def test_selfcheck_of_all_tile_shapes(lib):
    assert fwt.selfcheck() == 0


A = 0x10000  # fake, 16-byte aligned host addresses; validation never dereferences them
GiB = 1 << 30


@pytest.mark.parametrize("fn", ["fwt_batched_c32", "fwt_batched_c64", "fwt_batched_i32"])
def test_argument_errors_return_before_launch(lib, fn):
    f = getattr(fwt, fn)
    norm = 0 if fn.endswith("i32") else 1
    a, b, c, d = A, A + GiB, A + 2 * GiB, A + 3 * GiB
    assert f(a, b, c, d, -1, 1, norm, None) == fwt.FWT_ERR_INVALID_ARG
    assert f(a, b, c, d, 31, 1, norm, None) == fwt.FWT_ERR_INVALID_ARG
    assert f(a, b, c, d, 4, -1, norm, None) == fwt.FWT_ERR_INVALID_ARG
    assert f(None, None, None, None, 4, 0, norm, None) == fwt.FWT_OK  # empty batch
    assert f(None, b, c, d, 4, 1, norm, None) == fwt.FWT_ERR_INVALID_ARG
    assert f(a, b, None, d, 4, 1, norm, None) == fwt.FWT_ERR_INVALID_ARG
    assert f(a, b, c, None, 4, 1, norm, None) == fwt.FWT_ERR_INVALID_ARG  # im half missing
    assert f(a + 4, b, c, d, 4, 1, norm, None) == fwt.FWT_ERR_MISALIGNED
    assert f(a, b, c, d + 8, 4, 1, norm, None) == fwt.FWT_ERR_MISALIGNED
    # outputs overlapping anything other than their own input exactly
    assert f(a, b, a + 16, d, 4, 1, norm, None) == fwt.FWT_ERR_INVALID_ARG
    assert f(a, b, c, c, 4, 1, norm, None) == fwt.FWT_ERR_INVALID_ARG
    assert f(a, b, b, d, 4, 1, norm, None) == fwt.FWT_ERR_INVALID_ARG
    assert f(a, b, c, a, 4, 1, norm, None) == fwt.FWT_ERR_INVALID_ARG
    # size overflow
    assert f(a, b, c, d, 30, 1 << 40, norm, None) == fwt.FWT_ERR_INVALID_ARG


def test_int32_rules(lib):
    a, c = A, A + 2 * GiB
    assert fwt.fwt_batched_i32(a, None, c, None, 4, 1, 1, None) == fwt.FWT_ERR_UNSUPPORTED
    assert fwt.fwt_batched_c32(a, None, c, None, 4, 1, 1, None) == fwt.FWT_ERR_INVALID_ARG
    assert fwt.fwt_batched_c64(a, None, c, None, 4, 1, 0, None) == fwt.FWT_ERR_INVALID_ARG


def test_plans(lib):
    for dt, rmax in (("c32", 15), ("c64", 14), ("i32", 15)):
        for n in range(0, 31):
            f = fwt.plan_factors(n, dt)
            assert sum(f) == n and 1 <= len(f) <= 3
            assert fwt.plan_passes(n, dt) == len(f)
            # one-pass cluster plans on a GPU
            cluster_ok = (dt != "c64" and 15 <= n <= 17) or (dt == "c64" and n == 14)
            assert (len(f) == 1) == (n <= rmax) or (cluster_ok and len(f) == 1)
    assert fwt.plan_factors(24, "c32") == [14, 10]
    assert fwt.plan_factors(24, "c64") == [13, 11]
    if fwt.column_bytes("c32") == 0 and fwt.column_bytes("c64") == 0:
        # measured two-pass splits with narrower column segments for large n
        assert fwt.plan_factors(26, "c32") == [15, 11]
        assert fwt.plan_factors(27, "c32") == [12, 7, 8]
        assert fwt.plan_factors(28, "i32") == [13, 8, 7]
        assert fwt.plan_factors(25, "c64") == [14, 11]
        assert fwt.plan_factors(26, "c64") == [12, 6, 8]
        assert fwt.plan_factors(27, "c64") == [12, 8, 7]
        assert fwt.plan_factors(30, "c64") == [12, 9, 9]
    assert lib.fwt_plan_passes(31, 0) == -1 and lib.fwt_plan_passes(10, 7) == -1


def test_plan_override_roundtrip(lib):
    default = fwt.plan_factors(20, "c32")
    width = fwt.column_bytes("c32")
    fwt.set_column_bytes("c32", 128)  # 5-bit column factors exist for 128-byte tiles
    try:
        fwt.set_plan(20, "c32", [10, 5, 5])
        assert fwt.plan_factors(20, "c32") == [10, 5, 5]
        assert fwt.plan_passes(20, "c32") == 3
    finally:
        fwt.set_plan(20, "c32", None)
        fwt.set_column_bytes("c32", width)
    assert fwt.plan_factors(20, "c32") == default
    fwt.set_column_bytes("c32", 64)
    try:
        for bad in ([10, 9], [16, 4], [2, 18], [3, 7, 10], [10, 11], [10, 5, 5]):
            with pytest.raises(fwt.FwtError):
                fwt.set_plan(20, "c32", bad)
    finally:
        fwt.set_column_bytes("c32", width)
    assert fwt.plan_factors(20, "c32") == default
    # with the width chosen per plan, a plan takes the first width that has tiles
    # for all its factors: 5-bit column factors need 128-byte segments, a 3-bit row
    # factor segments of at most 2^3 elements
    if width == 0:
        try:
            for ok in ([10, 5, 5], [3, 7, 10]):
                fwt.set_plan(20, "c32", ok)
                assert fwt.plan_factors(20, "c32") == ok
        finally:
            fwt.set_plan(20, "c32", None)
        for bad in ([10, 9], [16, 4], [2, 18], [10, 11], [3, 3, 14]):
            with pytest.raises(fwt.FwtError):
                fwt.set_plan(20, "c32", bad)


def test_column_bytes_setting(lib):
    for dt in ("c32", "c64", "i32"):
        assert fwt.column_bytes(dt) in (0, 16, 32, 64, 128)
    with pytest.raises(fwt.FwtError):
        fwt.set_column_bytes("c32", 96)
    with pytest.raises(fwt.FwtError):
        fwt.set_column_bytes("c32", 256)
    assert lib.fwt_get_column_bytes(5) == -1


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    monkeypatch.setattr(fwt, "_lib", None)
    monkeypatch.setattr(fwt, "LIBRARY", str(tmp_path / "absent.so"))
    with pytest.raises(RuntimeError, match="missing"):
        fwt.library()


def test_l2_chunk_setting(lib):
    assert fwt.l2_chunk_bytes() == 0
    fwt.set_l2_chunk_bytes(-1)
    assert fwt.l2_chunk_bytes() == -1
    fwt.set_l2_chunk_bytes(0)
    with pytest.raises(fwt.FwtError):
        fwt.set_l2_chunk_bytes(-2)


def test_tma_setting(lib):
    assert fwt.tma() == fwt.TMA_AUTO
    fwt.set_tma(fwt.TMA_NEVER)
    assert fwt.tma() == fwt.TMA_NEVER
    with pytest.raises(fwt.FwtError):
        fwt.set_tma(3)
    fwt.set_tma(fwt.TMA_AUTO)


@pytest.mark.parametrize("fn", ["fwt_bits_c32", "fwt_bits_c64", "fwt_bits_i32"])
def test_bit_range_argument_errors_before_launch(lib, fn):
    f = getattr(fwt, fn)
    a, b, c, d = A, A + GiB, A + 2 * GiB, A + 3 * GiB
    assert f(a, b, c, d, 8, 1, 0, 9, 0, None) == fwt.FWT_ERR_INVALID_ARG   # past n
    assert f(a, b, c, d, 8, 1, -1, 2, 0, None) == fwt.FWT_ERR_INVALID_ARG  # lo < 0
    assert f(a, b, c, d, 8, 1, 2, -1, 0, None) == fwt.FWT_ERR_INVALID_ARG  # nbits < 0
    assert f(a, b, c, d, 31, 1, 0, 1, 0, None) == fwt.FWT_ERR_INVALID_ARG  # n > 30
    assert f(a + 4, b, c, d, 8, 1, 0, 3, 0, None) == fwt.FWT_ERR_MISALIGNED
    assert f(a, b, b, d, 8, 1, 0, 3, 0, None) == fwt.FWT_ERR_INVALID_ARG   # re_out over im_in
    assert f(None, None, None, None, 8, 0, 0, 3, 0, None) == fwt.FWT_OK     # empty batch


def test_pdl_setting(lib):
    assert fwt.pdl() == 1
    fwt.set_pdl(0)
    assert fwt.pdl() == 0
    with pytest.raises(fwt.FwtError):
        fwt.set_pdl(2)
    with pytest.raises(fwt.FwtError):
        fwt.set_pdl(-1)
    fwt.set_pdl(1)
    assert fwt.pdl() == 1


def test_cluster_setting(lib):
    assert fwt.cluster() == fwt.CLUSTER_AUTO
    fwt.set_cluster(fwt.CLUSTER_NEVER)
    assert fwt.cluster() == fwt.CLUSTER_NEVER
    with pytest.raises(fwt.FwtError):
        fwt.set_cluster(5)
    fwt.set_cluster(fwt.CLUSTER_AUTO)


@pytest.mark.parametrize("fn", ["fwt_host_c32", "fwt_host_c64", "fwt_host_i32"])
def test_host_entry_argument_errors_before_any_cuda_call(lib, fn):
    f = getattr(fwt, fn)
    norm = 0 if fn.endswith("i32") else 1
    a, b, c, d, w = A, A + GiB, A + 2 * GiB, A + 3 * GiB, A + 4 * GiB
    ws = 1 << 30
    assert f(a, b, c, d, -1, 1, norm, w, ws, None) == fwt.FWT_ERR_INVALID_ARG
    assert f(a, b, c, d, 31, 1, norm, w, ws, None) == fwt.FWT_ERR_INVALID_ARG
    assert f(a, b, c, d, 4, -1, norm, w, ws, None) == fwt.FWT_ERR_INVALID_ARG
    assert f(None, None, None, None, 4, 0, norm, None, 0, None) == fwt.FWT_OK  # empty batch
    assert f(a, b, c, d, 4, 1, norm, None, ws, None) == fwt.FWT_ERR_INVALID_ARG  # no workspace
    assert f(a, b, c, d, 4, 1, norm, w + 8, ws, None) == fwt.FWT_ERR_MISALIGNED
    assert f(a, b, c, None, 4, 1, norm, w, ws, None) == fwt.FWT_ERR_INVALID_ARG
    # outputs overlapping anything but their own input exactly
    assert f(a, b, a + 16, d, 4, 1, norm, w, ws, None) == fwt.FWT_ERR_INVALID_ARG
    assert f(a, b, c, c, 4, 1, norm, w, ws, None) == fwt.FWT_ERR_INVALID_ARG
    assert f(a, b, b, d, 4, 1, norm, w, ws, None) == fwt.FWT_ERR_INVALID_ARG
    # a workspace too small for one vector (both parts)
    esz = 8 if fn.endswith("c64") else 4
    assert f(a, b, c, d, 10, 2, norm, w, 2 * esz * 1024 - 16, None) == fwt.FWT_ERR_INVALID_ARG
    assert f(a, b, c, d, 30, 1 << 40, norm, w, ws, None) == fwt.FWT_ERR_INVALID_ARG
    if fn.endswith("i32"):
        assert f(a, None, c, None, 4, 1, 1, w, ws, None) == fwt.FWT_ERR_UNSUPPORTED
    else:
        assert f(a, None, c, None, 4, 1, norm, w, ws, None) == fwt.FWT_ERR_INVALID_ARG


def test_host_workspace_size(lib):
    ws = fwt.fwt_host_workspace_bytes
    # n = 24 batch 16 fp64: chunks of one vector (2 parts x 128 MiB), three slots
    assert ws(fwt.FWT_C64, 24, 16) == 3 * 2 * (8 << 24)
    # small vectors: chunks of at least 32 MiB, never more than the batch
    assert ws(fwt.FWT_C32, 10, 64) == 2 * 64 * 4096  # the whole batch is one chunk
    # many vectors: chunks of batch / 16 vectors (here above the 32 MiB floor)
    assert ws(fwt.FWT_I32, 12, 1 << 16, with_im=False) == 3 * 4096 * (4 << 12)
    assert ws(fwt.FWT_I32, 12, 1 << 14, with_im=False) == 3 * 2048 * (4 << 12)
    assert ws(fwt.FWT_C32, 4, 0) == 0 and ws(fwt.FWT_C32, 31, 1) == 0 and ws(7, 4, 1) == 0


@pytest.mark.parametrize("fn", ["fwt_mask_c32", "fwt_mask_c64", "fwt_mask_i32"])
def test_mask_argument_errors_before_launch(lib, fn):
    f = getattr(fwt, fn)
    norm = 0 if fn.endswith("i32") else 1
    a, b, c, d = A, A + GiB, A + 2 * GiB, A + 3 * GiB
    assert f(a, b, c, d, 4, 1, 1 << 4, norm, None) == fwt.FWT_ERR_INVALID_ARG  # bit 4 of n = 4
    assert f(a, b, c, d, -1, 1, 0, norm, None) == fwt.FWT_ERR_INVALID_ARG
    assert f(a, b, c, d, 31, 1, 1, norm, None) == fwt.FWT_ERR_INVALID_ARG
    assert f(None, None, None, None, 4, 0, 0b101, norm, None) == fwt.FWT_OK  # empty batch
    assert f(a + 4, b, c, d, 4, 1, 0b101, norm, None) == fwt.FWT_ERR_MISALIGNED
    assert f(a, b, a + 16, d, 4, 1, 0b101, norm, None) == fwt.FWT_ERR_INVALID_ARG


@pytest.mark.parametrize("fn", ["fwt_phase_c32", "fwt_phase_c64"])
def test_phase_argument_errors_before_launch(lib, fn):
    f = getattr(fwt, fn)
    a, b, c, d, th = A, A + GiB, A + 2 * GiB, A + 3 * GiB, A + 4 * GiB
    E = fwt.FWT_ERR_INVALID_ARG
    assert f(a, b, th, -4, c, d, 4, 2, 1, None) == E             # negative stride
    assert f(a, b, th, 16, c, d, 31, 1, 1, None) == E            # n > 30
    assert f(a, b, None, 16, c, d, 4, 2, 1, None) == E           # no angles
    assert f(a, None, th, 16, c, None, 4, 2, 1, None) == E       # both parts required
    assert f(a, b, th + 4, 16, c, d, 4, 2, 1, None) == fwt.FWT_ERR_MISALIGNED
    assert f(a, b, th, 1, c, d, 4, 2, 1, None) == fwt.FWT_ERR_MISALIGNED  # odd stride
    assert f(a, b, th, 1 << 61, c, d, 4, 3, 1, None) == E        # angle extent overflows
    assert f(a, b, c, 16, c, d, 4, 2, 1, None) == E              # angles overlap re_out
    assert f(None, None, None, 0, None, None, 4, 0, 1, None) == fwt.FWT_OK  # empty batch


def test_default_plans_valid_for_every_width_setting(lib):
    """Whatever column width is set, the default plan of every n and dtype is one the
    library accepts (re-submitting it through fwt_set_plan validates it on the host)."""
    try:
        for dt in ("c32", "c64", "i32"):
            for cb in (0, 16, 32, 64, 128):
                fwt.set_column_bytes(dt, cb)
                for n in range(0, 31):
                    f = fwt.plan_factors(n, dt)
                    assert sum(f) == n, (dt, cb, n, f)
                    if len(f) > 1:
                        fwt.set_plan(n, dt, f)  # raises FwtError if the plan is invalid
                        assert fwt.plan_factors(n, dt) == f
                        fwt.set_plan(n, dt, None)
    finally:
        for dt in ("c32", "c64", "i32"):
            fwt.set_column_bytes(dt, 0)
            for n in range(0, 31):
                fwt.set_plan(n, dt, None)
