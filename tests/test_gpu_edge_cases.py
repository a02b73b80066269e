"""Edge cases of the two exact arithmetics, CUDA vs the CPU oracle (GPU only).

fp64 runs its butterflies in int64 fixed point: each tile's elements are
converted to integers with one common binary exponent and their magnitudes
truncated, so the conversion error of a pass is largest when every element
carries a full mantissa, and relative to the vector's norm largest when one entry
per tile dominates the others.  These tests drive every fp64 pass shape (the
n = 24 two-pass plan at every column-segment width and with both column movers,
the 2^14-element tile on a CTA pair, a single 2^13 tile, a three-pass plan) with
such inputs and require the specification's 1e-12 relative L2 error; the measured
errors are printed beside the a-priori bound sqrt(T) 2^-F per pass.

int32 runs in wrap-around arithmetic modulo 2^32: full-range inputs make nearly
every intermediate sum wrap, through the row, column (both movers), cluster,
bit-range and bit-mask kernels at n = 1..22; results must equal the oracle's bit
for bit.
"""
import numpy as np
import pytest
import torch

import oracle
import walsh_hadamard_transform_gb300 as fwt
from helpers import TOL, assert_matches, gpu_transform, host_threads, rel_err_per_vector
from walsh_hadamard_transform_gb300 import inputs

pytestmark = pytest.mark.gpu

FP64_KINDS = ("fp64_one_signed", "fp64_below_pow2", "fp64_spike")
MEASURED = []  # (case, max relative error) for the summary printed at the end


@pytest.fixture(scope="module", autouse=True)
def need_cuda():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    fwt.library()
    yield
    for case, err in MEASURED:
        print(f"fp64 worst-case input {case}: max relative L2 error {err:.3e} (limit 1e-12)")


def _fp64_case(kind, n, batch, seed, tile_bits=13):
    re, im = inputs.edge_pair(kind, n, batch, seed, tile_bits=tile_bits)
    ore, oim = oracle.fwt_complex(re, im, normalize=True, nthreads=host_threads())
    return re, im, ore, oim


def _fp64_check(re, im, ore, oim, what):
    gre, gim = gpu_transform(re, im, True)
    err = float(rel_err_per_vector(gre, gim, ore, oim).max())
    MEASURED.append((what, err))
    assert err <= TOL["c64"], f"{what}: max relative L2 error {err:.3e} > 1e-12"


@pytest.mark.parametrize("kind", FP64_KINDS)
def test_fp64_worst_case_n24_every_width_and_mover(kind):
    """n = 24: the default (13, 11) plan, then each column-segment width (32, 64,
    128 bytes) with TMA-staged and directly loaded column tiles; 128-byte segments
    give (14, 10), whose 14-bit row pass runs on CTA pairs."""
    n = 24
    re, im, ore, oim = _fp64_case(kind, n, 1, seed=24)
    assert fwt.plan_factors(n, "c64") == [13, 11]
    _fp64_check(re, im, ore, oim, f"{kind} n=24 default plan")
    try:
        for cb in (32, 64, 128):
            for tma in (fwt.TMA_ALWAYS, fwt.TMA_NEVER):
                fwt.set_column_bytes("c64", cb)
                fwt.set_tma(tma)
                plan = fwt.plan_factors(n, "c64")
                _fp64_check(re, im, ore, oim, f"{kind} n=24 plan {plan} {cb}B tma={tma}")
    finally:
        fwt.set_column_bytes("c64", 0)
        fwt.set_tma(fwt.TMA_AUTO)
    assert fwt.device_status() == fwt.FWT_OK


@pytest.mark.parametrize("kind", FP64_KINDS)
def test_fp64_worst_case_single_tiles(kind):
    """One-pass shapes: a single 2^13-element tile (truncating conversion, 13 bits)
    and the 2^14-element vector on a CTA pair (one exponent over the pair)."""
    for n, batch, tb in ((13, 8, 13), (14, 8, 14), (14, 4, 13)):
        re, im, ore, oim = _fp64_case(kind, n, batch, seed=n + tb, tile_bits=tb)
        _fp64_check(re, im, ore, oim, f"{kind} n={n} spikes per 2^{tb}")


def _kron3(u, v, w):
    t = [torch.from_numpy(np.ascontiguousarray(x)).cuda() for x in (u, v, w)]
    return torch.kron(t[0], torch.kron(t[1], t[2]))


@pytest.mark.parametrize("kind", ["fp64_one_signed", "fp64_spike"])
def test_fp64_worst_case_three_passes(kind):
    """n = 26: the default three-pass fp64 plan on x = u (x) v (x) w, whose exact
    transform is (H u) (x) (H v) (x) (H w) (the oracle transforms the short factors).
    One-signed full-mantissa factors, or factors with one spike each."""
    n, sizes = 26, (9, 9, 8)
    assert fwt.plan_passes(n, "c64") == 3
    parts, expect = [], []
    for c in range(2):
        facs, hfacs = [], []
        for i, k in enumerate(sizes):
            a, _ = inputs.edge_pair(kind, k, 1, seed=500 + 10 * c + i, tile_bits=k)
            facs.append(a[0])
            hfacs.append(oracle.fwt(a[0], normalize=True))
        parts.append(_kron3(*facs).unsqueeze(0))
        expect.append(hfacs)
    out = fwt.transform(parts[0], parts[1], normalize=True)
    torch.cuda.synchronize()
    num = den = 0.0
    for got, h in zip(out, expect):
        want = _kron3(*h)
        num += float((got[0] - want).pow(2).sum())
        den += float(want.pow(2).sum())
    err = (num / den) ** 0.5
    MEASURED.append((f"{kind} n=26 plan {fwt.plan_factors(n, 'c64')}", err))
    assert err <= TOL["c64"], f"{kind} n=26: relative L2 error {err:.3e}"


# ---- int32: full-range inputs (every intermediate wraps) ------------------------------

def _i32(n, batch, seed, real_only=False):
    re, im = inputs.edge_pair("int32_full", n, batch, seed)
    return re, None if real_only else im


def _i32_check(re, im, what, inplace=False):
    gre, gim = gpu_transform(re, im, False, inplace=inplace)
    ore, oim = oracle.fwt_complex(re, im, normalize=False, nthreads=host_threads())
    assert_matches("i32", gre, gim, ore, oim, what)


def test_int32_full_range_default_plans():
    """Every n = 1..22 with its default plan (single tiles to n = 14, clusters at
    n = 15..17, two passes above), in and out of place; real-only at a few sizes."""
    for n in range(1, 23):
        re, im = _i32(n, 3 if n <= 20 else 1, seed=700 + n)
        _i32_check(re, im, f"int32 full range n={n}", inplace=n % 2 == 1)
    for n in (9, 16, 21):
        re, _ = _i32(n, 2, seed=800 + n, real_only=True)
        _i32_check(re, None, f"int32 full range real only n={n}")


def test_int32_full_range_clusters():
    try:
        fwt.set_cluster(fwt.CLUSTER_FROM_14)
        for n in range(14, 19):
            assert fwt.plan_passes(n, "i32") == 1
            re, im = _i32(n, 3, seed=900 + n)
            _i32_check(re, im, f"int32 full range cluster n={n}", inplace=n % 2 == 0)
    finally:
        fwt.set_cluster(fwt.CLUSTER_AUTO)


def _sample_plans(n):
    plans = []
    for b in range(3, 16):
        for rest in ([n - b], *[[a2, n - b - a2] for a2 in range(3, 11)]):
            f = [b, *rest]
            if any(k <= 0 for k in f):
                continue
            try:
                fwt.set_plan(n, "i32", f)
            except fwt.FwtError:
                continue
            plans.append(f)
    fwt.set_plan(n, "i32", None)
    return plans


@pytest.mark.parametrize("tma", [fwt.TMA_ALWAYS, fwt.TMA_NEVER], ids=["tma", "direct"])
def test_int32_full_range_column_passes(tma):
    """Two- and three-factor plans at n = 16, 20, 21 for each column width and mover
    (a sample of the valid plans: the first, middle and last of each width)."""
    try:
        fwt.set_tma(tma)
        for n in (16, 20, 21):
            re, im = _i32(n, 2, seed=1000 + n)
            ore, oim = oracle.fwt_complex(re, im, normalize=False, nthreads=host_threads())
            for cb in ((16, 32, 64, 128) if tma == fwt.TMA_ALWAYS else (32, 64, 128)):
                fwt.set_column_bytes("i32", cb)
                plans = _sample_plans(n)
                assert plans
                for f in {tuple(plans[0]), tuple(plans[len(plans) // 2]), tuple(plans[-1])}:
                    fwt.set_plan(n, "i32", list(f))
                    gre, gim = gpu_transform(re, im, False)
                    assert_matches("i32", gre, gim, ore, oim, f"int32 n={n} plan {f} cb={cb}")
                fwt.set_plan(n, "i32", None)
    finally:
        fwt.set_column_bytes("i32", 0)
        fwt.set_tma(fwt.TMA_AUTO)
        for n in (16, 20, 21):
            fwt.set_plan(n, "i32", None)
    assert fwt.device_status() == fwt.FWT_OK


def test_int32_full_range_bit_ranges_and_masks():
    """Bit ranges inside, across and above the row tile, and bit masks (runs inside
    and above it), bit for bit against the oracle's restricted butterflies."""
    n = 20
    re, im = _i32(n, 2, seed=1100)
    dre, dim_ = torch.from_numpy(re).cuda(), torch.from_numpy(im).cuda()
    for lo, k in ((0, 20), (0, 9), (3, 9), (13, 5), (15, 5), (2, 16), (17, 3), (7, 0)):
        gre, gim = fwt.transform(dre, dim_, normalize=False, bits=(lo, k))
        torch.cuda.synchronize()
        ore = oracle.fwt_bits(re, lo, k, normalize=False)
        oim = oracle.fwt_bits(im, lo, k, normalize=False)
        assert_matches("i32", gre.cpu().numpy(), gim.cpu().numpy(), ore, oim, f"bits [{lo}, {lo + k})")
    n = 21
    re, im = _i32(n, 2, seed=1200)
    dre, dim_ = torch.from_numpy(re).cuda(), torch.from_numpy(im).cuda()
    for mask in (0x15555, (1 << 3) | (1 << 20), 0x1F0F0F, 0x100001, 0xFFF00):
        gre, gim = fwt.transform(dre, dim_, normalize=False, mask=mask)
        torch.cuda.synchronize()
        ore = oracle.fwt_mask(re, mask, normalize=False)
        oim = oracle.fwt_mask(im, mask, normalize=False)
        assert_matches("i32", gre.cpu().numpy(), gim.cpu().numpy(), ore, oim, f"mask {mask:#x}")
    assert fwt.device_status() == fwt.FWT_OK
