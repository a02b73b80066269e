"""Default plans at n = 26..30 vs the oracle, through the C ABI (GPU only).

At these sizes the oracle cannot transform whole vectors in test time, so the
inputs are Kronecker products x = u (x) v (x) w of short seeded vectors.  Because
H_n = H_a (x) H_b (x) H_c for any split a + b + c = n (the factorisation every pass
plan is built on), the exact transform is (H_a u) (x) (H_b v) (x) (H_c w), scaled by
2^{-n/2} = 2^{-a/2} 2^{-b/2} 2^{-c/2}: the oracle transforms the three short
vectors and PyTorch multiplies them out on the device.  Every output element is
compared: int32 bit for bit (wrapped mod 2^32), floats by the per-vector relative
L2 error of the specification.  These sizes run the three-pass default plans
(fp64 from n = 26, 4-byte types from n = 27) and the largest two-pass ones.
"""
import numpy as np
import pytest
import torch

import oracle
import walsh_hadamard_transform_gb300 as fwt
from helpers import TOL
from walsh_hadamard_transform_gb300 import inputs

pytestmark = pytest.mark.gpu

LOW_BITS, MID_BITS = 8, 9  # w: 2^8 elements, v: 2^9, u: the rest (2^9 .. 2^13)
TORCH = {"c32": torch.float32, "c64": torch.float64, "i32": torch.int32}


@pytest.fixture(scope="module", autouse=True)
def need_cuda():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    fwt.library()


def _factors(dtype, n, seed):
    """Three short seeded vectors (float64 or int64) and their oracle transforms."""
    sizes = (n - LOW_BITS - MID_BITS, MID_BITS, LOW_BITS)  # u, v, w
    norm = dtype != "i32"
    vecs, hvecs = [], []
    for i, k in enumerate(sizes):
        re, _ = inputs.random_pair(k, 1, dtype, seed * 7 + i)
        x = re[0]
        hx = oracle.fwt(x, normalize=norm)
        if dtype == "i32":
            vecs.append(x.astype(np.int64))
            hvecs.append(hx.astype(np.int64))  # exact: |H x| <= 8 * 2^13
        else:
            vecs.append(x.astype(np.float64))
            hvecs.append(hx)
    return vecs, hvecs


def _kron3(a, b, c, dtype):
    t = [torch.from_numpy(v).cuda() for v in (a, b, c)]
    return torch.kron(t[0], torch.kron(t[1], t[2]))  # index = iu * 2^17 + iv * 2^8 + iw


def _to_elem(full, dtype):
    if dtype == "i32":  # int64 products, wrapped to int32 two's complement
        return (torch.remainder(full + 2**31, 2**32) - 2**31).to(torch.int32)
    return full.to(TORCH[dtype])


def _batch(dtype, n, batch, seed):
    """(re, im) device inputs of shape (batch, 2^n) and their factor transforms."""
    re = torch.empty(batch, 1 << n, dtype=TORCH[dtype], device="cuda")
    im = torch.empty_like(re)
    expect = []
    for b in range(batch):
        pair = []
        for part, dst in ((0, re), (1, im)):
            vecs, hvecs = _factors(dtype, n, seed + 2 * b + part)
            dst[b] = _to_elem(_kron3(*vecs, dtype), dtype)
            pair.append(hvecs)
        expect.append(pair)
    return re, im, expect


def _check_vector(dtype, got_re, got_im, hre, him, what):
    if dtype == "i32":
        for got, h in ((got_re, hre), (got_im, him)):
            want = _to_elem(_kron3(*h, dtype), dtype)
            assert torch.equal(got, want), f"{what}: int32 result differs"
            del want
        return
    num = 0.0
    den = 0.0
    for got, h in ((got_re, hre), (got_im, him)):
        want = _kron3(*h, dtype)  # float64 products of the oracle's transforms
        num += float((got.double() - want).pow(2).sum())
        den += float(want.pow(2).sum())
        del want
    err = (num ** 0.5) / (den ** 0.5)
    assert err <= TOL[dtype], f"{what}: relative L2 error {err:.3e} > {TOL[dtype]}"


@pytest.mark.parametrize("dtype", ["c32", "c64", "i32"])
@pytest.mark.parametrize("n,batch,inplace", [(26, 2, False), (27, 2, True), (28, 1, False),
                                             (29, 1, True), (30, 1, False)])
def test_default_plans_large_n_kronecker_inputs(dtype, n, batch, inplace):
    norm = dtype != "i32"
    re, im, expect = _batch(dtype, n, batch, seed=1000 + n)
    if inplace:
        out = fwt.transform(re, im, re, im, normalize=norm)
    else:
        out = fwt.transform(re, im, normalize=norm)
        del re, im
    torch.cuda.synchronize()
    plan = fwt.plan_factors(n, dtype)
    for b in range(batch):
        _check_vector(dtype, out[0][b], out[1][b], expect[b][0], expect[b][1],
                      f"{dtype} n={n} vector {b} plan {plan} in_place={inplace}")
    del out
    torch.cuda.empty_cache()
