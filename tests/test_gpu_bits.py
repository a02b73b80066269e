"""Transform on a range of index bits (I x H_k x I), CUDA vs the oracle (GPU only).

Ranges inside the contiguous row tile, straddling it, and wholly in the strided
column region; empty ranges; out of place and in place; every dtype."""
import numpy as np
import pytest
import torch

import oracle
import walsh_hadamard_transform_gb300 as fwt
from helpers import assert_matches
from walsh_hadamard_transform_gb300 import inputs

pytestmark = pytest.mark.gpu

T = {"c32": torch.float32, "c64": torch.float64, "i32": torch.int32}


def _gpu_bits(re, im, lo, k, norm, inplace=False):
    dre, dim_ = torch.from_numpy(re).cuda(), torch.from_numpy(im).cuda()
    if inplace:
        fwt.transform(dre, dim_, dre, dim_, normalize=norm, bits=(lo, k))
        out = (dre, dim_)
    else:
        out = fwt.transform(dre, dim_, normalize=norm, bits=(lo, k))
    torch.cuda.synchronize()
    return out[0].cpu().numpy(), out[1].cpu().numpy()


def _ranges(n, rmax):
    r = {(0, n), (0, 0), (n, 0), (0, 1), (n - 1, 1), (1, min(3, n - 1)), (0, min(n, 3))}
    if n >= 8:
        r |= {(2, 5), (3, n - 3), (n - 6, 6), (n // 2, n - n // 2)}
    if n > rmax:
        r |= {(rmax, n - rmax), (rmax - 2, 4), (rmax + 1, min(4, n - rmax - 1)), (5, n - 5)}
    return sorted((lo, k) for lo, k in r if lo >= 0 and k >= 0 and lo + k <= n)


@pytest.mark.parametrize("dtype", ["c32", "c64", "i32"])
@pytest.mark.parametrize("n", [4, 9, 12, 16, 19, 22])
def test_bit_ranges_match_oracle(dtype, n):
    rmax = 14 if dtype == "c64" else 15
    re, im = inputs.random_pair(n, 3, dtype, seed=40 + n)
    for lo, k in _ranges(n, rmax):
        for norm in ((False,) if dtype == "i32" else (True, False)):
            ore = oracle.fwt_bits(re, lo, k, normalize=norm)
            oim = oracle.fwt_bits(im, lo, k, normalize=norm)
            gre, gim = _gpu_bits(re, im, lo, k, norm, inplace=(lo + k) % 2 == 1)
            assert_matches(dtype, gre, gim, ore, oim, f"bits [{lo}, {lo + k}) n={n} norm={norm}")
    assert fwt.device_status() == fwt.FWT_OK


@pytest.mark.parametrize("dtype", ["c32", "c64", "i32"])
def test_ranges_compose_to_whole_transform(dtype):
    n = 23
    re, im = inputs.random_pair(n, 2, dtype, seed=7)
    norm = dtype != "i32"
    dre, dim_ = torch.from_numpy(re).cuda(), torch.from_numpy(im).cuda()
    for lo, k in ((0, 4), (4, 9), (13, 3), (16, 7)):
        fwt.transform(dre, dim_, dre, dim_, normalize=norm, bits=(lo, k))
    whole = fwt.transform(torch.from_numpy(re).cuda(), torch.from_numpy(im).cuda(), normalize=norm)
    torch.cuda.synchronize()
    ore, oim = oracle.fwt_complex(re, im, normalize=norm)
    assert_matches(dtype, dre.cpu().numpy(), dim_.cpu().numpy(), ore, oim, "composed ranges")
    assert_matches(dtype, whole[0].cpu().numpy(), whole[1].cpu().numpy(), ore, oim, "whole")


def test_bit_range_argument_errors():
    x = torch.zeros(2, 64, device="cuda")
    y = torch.empty_like(x)
    p = (x.data_ptr(), x[1].data_ptr(), y.data_ptr(), y[1].data_ptr())
    assert fwt.fwt_bits_c32(*p, 5, 1, 0, 6, 1, None) == fwt.FWT_ERR_INVALID_ARG
    assert fwt.fwt_bits_c32(*p, 5, 1, -1, 2, 1, None) == fwt.FWT_ERR_INVALID_ARG
    assert fwt.fwt_bits_c32(*p, 5, 1, 2, -1, 1, None) == fwt.FWT_ERR_INVALID_ARG
    assert fwt.fwt_bits_c32(*p, 5, 1, 1, 4, 1, None) == fwt.FWT_OK
    torch.cuda.synchronize()


def _gpu_mask(re, im, mask, norm, inplace=False):
    dre, dim_ = torch.from_numpy(re).cuda(), torch.from_numpy(im).cuda()
    if inplace:
        fwt.transform(dre, dim_, dre, dim_, normalize=norm, mask=mask)
        out = (dre, dim_)
    else:
        out = fwt.transform(dre, dim_, normalize=norm, mask=mask)
    torch.cuda.synchronize()
    return out[0].cpu().numpy(), out[1].cpu().numpy()


def _masks(n, rmax):
    full = (1 << n) - 1
    m = {0, full, 1, 1 << (n - 1), full & 0x5555_5555, full & 0xAAAA_AAAA}
    if n >= 6:
        m |= {0b101101, (1 << (n - 1)) | 1, full & ~(1 << (n // 2))}
    if n > rmax:  # runs above the row tiles, and one crossing their limit
        m |= {(1 << rmax) | 0b110, (0b11 << (rmax - 1)) | (1 << (n - 1)),
              full & ~((1 << rmax) - 1) & ~(1 << (rmax + 2)) | 0b1001}
    return sorted(x & full for x in m)


@pytest.mark.parametrize("dtype", ["c32", "c64", "i32"])
@pytest.mark.parametrize("n", [3, 9, 13, 17, 21])
def test_bit_masks_match_oracle(dtype, n):
    """Any set of index bits: the set bits within the row tiles in one run-time-mask
    pass, runs above them in column passes; against the oracle's composition of
    bit ranges, in and out of place."""
    rmax = 14 if dtype == "c64" else 15
    batch = 3 if n < 20 else 1
    norm_opts = (False,) if dtype == "i32" else (True, False)
    re, im = inputs.random_pair(n, batch, dtype, seed=40 + n)
    for i, mask in enumerate(_masks(n, rmax)):
        for norm in norm_opts:
            gre, gim = _gpu_mask(re, im, mask, norm, inplace=(i % 2 == 1))
            ore = oracle.fwt_mask(re, mask, normalize=norm, nthreads=4)
            oim = oracle.fwt_mask(im, mask, normalize=norm, nthreads=4)
            assert_matches(dtype, gre, gim, ore, oim, f"{dtype} n={n} mask={mask:#x} norm={norm}")


def test_bit_mask_argument_errors():
    a = torch.zeros(2, 1 << 5, device="cuda")
    with pytest.raises(fwt.FwtError):
        fwt.transform(a, a.clone(), mask=1 << 5)
    with pytest.raises(ValueError):
        fwt.transform(a, a.clone(), mask=1, bits=(0, 1))


@pytest.mark.parametrize("dtype", ["c32", "c64", "i32"])
def test_out_of_place_ranges_on_16_byte_column_tiles(dtype):
    """Ranges from bit 2 (4-byte types) or bit 1 (fp64) long enough for column passes:
    at that row stride the only column tile is a 16-byte TMA tile, which runs in
    place, so an out-of-place call copies the input to the output first.  Both forms
    against the oracle."""
    lo = 1 if dtype == "c64" else 2
    n = 17
    re, im = inputs.random_pair(n, 3, dtype, seed=77)
    for k in (8, 9, 10, 12, n - lo):
        for norm in ((False,) if dtype == "i32" else (True,)):
            ore = oracle.fwt_bits(re, lo, k, normalize=norm)
            oim = oracle.fwt_bits(im, lo, k, normalize=norm)
            for inplace in (False, True):
                gre, gim = _gpu_bits(re, im, lo, k, norm, inplace=inplace)
                assert_matches(dtype, gre, gim, ore, oim,
                               f"bits [{lo}, {lo + k}) n={n} in_place={inplace}")
    assert fwt.device_status() == fwt.FWT_OK
