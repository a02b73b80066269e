"""Seeded random cases across every entry point and setting, CUDA vs the oracle
(GPU only).

Each case draws a dtype, n (0..24), batch, normalisation, in or out of place, real-
only int32, a column segment width, a TMA mode, and one of: a random valid pass
plan, the default plan, a random bit range, a random bit mask, a cluster mode, the
diagonal phase (shared or per-vector angles), the host-buffer pipeline (pinned or
pageable, random workspace size) or an L2-chunk budget.  Every result is compared
with the oracle: int32 bit for bit, floats within the specified relative L2 error.
"""
import numpy as np
import pytest
import torch

import oracle
import walsh_hadamard_transform_gb300 as fwt
from helpers import assert_matches, host_threads
from test_gpu_parity import _valid_plans
from walsh_hadamard_transform_gb300 import inputs

pytestmark = pytest.mark.gpu

KINDS = ["plan", "default", "bits", "mask", "cluster", "phase", "host", "chunk"]


def _case(rng):
    dtype = ["c32", "c64", "i32"][rng.integers(3)]
    n = int(rng.integers(0, 25))
    batch = int(rng.integers(1, max(2, min(9, (1 << 24) >> n) + 1)))
    kind = KINDS[rng.integers(len(KINDS))]
    if kind == "phase" and dtype == "i32":
        dtype = "c32"
    norm = dtype != "i32" and bool(rng.integers(2))
    cb = int(rng.choice([0, 16, 32, 64, 128]))
    tma = 2 if cb == 16 else int(rng.integers(0, 3))
    re, im = inputs.random_pair(n, batch, dtype, seed=int(rng.integers(1 << 30)))
    if dtype == "i32" and kind != "phase" and rng.integers(2):
        im = None  # real-only int32
    return dict(dtype=dtype, n=n, batch=batch, kind=kind, norm=norm, cb=cb, tma=tma, re=re, im=im,
                inplace=bool(rng.integers(2)))


def _run(c, rng):
    dtype, n, batch, norm, re, im, inplace = (c[k] for k in
                                              ("dtype", "n", "batch", "norm", "re", "im", "inplace"))
    what = f"{dtype} n={n} batch={batch} {c['kind']} cb={c['cb']} tma={c['tma']} in_place={inplace}"
    fwt.set_tma(c["tma"])
    fwt.set_column_bytes(dtype, c["cb"])
    kw = {"normalize": norm}
    if c["kind"] == "plan" and n >= 3:
        plans = _valid_plans(n, dtype)
        if plans:
            plan = plans[int(rng.integers(len(plans)))]
            fwt.set_plan(n, dtype, plan)
            what += f" plan={plan}"
    if c["kind"] == "cluster":
        fwt.set_cluster(int(rng.integers(0, 3)))
    if c["kind"] == "chunk":
        fwt.set_l2_chunk_bytes(int(rng.choice([-1, 1 << 20, 8 << 20, 64 << 20])))
    if c["kind"] == "phase":
        # fp64 angles at several scales: the fixed-point reduction (up to 2^40 rad) and the
        # fp64 sincos beyond it
        span = np.pi if re.dtype == np.float32 else float(rng.choice([np.pi, 1e3, 1e9, 1e13]))
        theta = rng.uniform(-span, span, size=(int(rng.choice([1, batch])), 1 << n)).astype(re.dtype)
        ore, oim = oracle.phase_fwt(re, im, theta, normalize=norm)
        a, b, t = (torch.from_numpy(v).cuda() for v in (re, im, theta))
        out = (fwt.phase_transform(a, b, t, a, b, normalize=norm) if inplace
               else fwt.phase_transform(a, b, t, normalize=norm))
        torch.cuda.synchronize()
        return what, (out[0].cpu().numpy(), out[1].cpu().numpy()), (ore, oim)
    if c["kind"] == "bits" and n >= 1:
        lo = int(rng.integers(0, n))
        k = int(rng.integers(0, n - lo + 1))
        kw["bits"] = (lo, k)
        what += f" bits=[{lo}, {lo + k})"
        ore = oracle.fwt_bits(re, lo, k, normalize=norm, nthreads=host_threads())
        oim = None if im is None else oracle.fwt_bits(im, lo, k, normalize=norm,
                                                      nthreads=host_threads())
    elif c["kind"] == "mask" and n >= 1:
        mask = int(rng.integers(0, 1 << n))
        kw["mask"] = mask
        what += f" mask={mask:#x}"
        ore = oracle.fwt_mask(re, mask, normalize=norm, nthreads=host_threads())
        oim = None if im is None else oracle.fwt_mask(im, mask, normalize=norm,
                                                      nthreads=host_threads())
    else:
        ore, oim = oracle.fwt_complex(re, im, normalize=norm, nthreads=host_threads())
    if c["kind"] == "host":
        ha = torch.from_numpy(re.copy())
        hb = None if im is None else torch.from_numpy(im.copy())
        if rng.integers(2):
            ha = ha.pin_memory()
            hb = None if hb is None else hb.pin_memory()
        full = fwt.fwt_host_workspace_bytes(fwt.DTYPES[dtype], n, batch, im is not None)
        one = (1 if im is None else 2) * (((re.itemsize << n) + 255) // 256 * 256)
        nbytes = max(int(full * float(rng.uniform(0.05, 1.0))) // 16 * 16, one)
        ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
        what += f" host workspace={nbytes}"
        out = (fwt.transform_host(ha, hb, ha, hb, workspace=ws, **kw) if inplace
               else fwt.transform_host(ha, hb, workspace=ws, **kw))
        return what, (out[0].numpy(), None if out[1] is None else out[1].numpy()), (ore, oim)
    a = torch.from_numpy(re).cuda()
    b = None if im is None else torch.from_numpy(im).cuda()
    out = fwt.transform(a, b, a, b, **kw) if inplace else fwt.transform(a, b, **kw)
    torch.cuda.synchronize()
    return what, (out[0].cpu().numpy(), None if out[1] is None else out[1].cpu().numpy()), (ore, oim)


@pytest.mark.parametrize("seed", [31, 32])
def test_random_cases_every_entry_point(seed):
    rng = np.random.default_rng(seed)
    for _ in range(40):
        c = _case(rng)
        try:
            what, (gre, gim), (ore, oim) = _run(c, rng)
            assert_matches(c["dtype"], gre, gim, ore, oim, what)
        finally:
            fwt.set_plan(c["n"], c["dtype"], None)
            fwt.set_column_bytes(c["dtype"], 0)
            fwt.set_tma(fwt.TMA_AUTO)
            fwt.set_cluster(fwt.CLUSTER_AUTO)
            fwt.set_l2_chunk_bytes(0)
    assert fwt.device_status() == fwt.FWT_OK
