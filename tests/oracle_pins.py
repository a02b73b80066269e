"""Pins that tie the CPU oracle to facts outside itself.

Each ``pin_*`` takes an ``oracle.Oracle`` and raises AssertionError on a mismatch.
They check the oracle against:

* the dense popc-rule matrix (``oracle.dense``), itself checked against
  ``scipy.linalg.hadamard`` (Sylvester's construction) -- the plain definition;
* hand-worked examples in ``tests/golden/hand_examples.json``;
* closed forms (delta -> Walsh row, constant -> scaled delta, y_0 = s * sum x);
* invariants (involution H H = 2^n I, Parseval, linearity, the Sylvester block
  recursion H_{n} = [[H, H], [H, -H]], the Kronecker split H_n = H_a (x) H_b);
* int32 wrap-around modulo 2^32.

``test_oracle_pins.py`` runs them on the real oracle; ``test_oracle_mutants.py``
plants mistakes in a copy of the oracle source and checks that some pin fails.
"""
from __future__ import annotations

import json
import os

import numpy as np

from oracle import dense

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "hand_examples.json")


def _popc_parity(a):
    a = np.asarray(a, dtype=np.int64)
    return dense.popcount(a) & 1


def _rel(a, b):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    den = np.linalg.norm(b)
    return np.linalg.norm(a - b) / (den if den > 0 else 1.0)


def pin_dense_is_sylvester():
    """The popc matrix equals scipy's Sylvester Hadamard matrix for n <= 10."""
    import scipy.linalg

    for n in range(0, 11):
        H = dense.hadamard_popc(n)
        S = scipy.linalg.hadamard(1 << n, dtype=np.int64)
        assert np.array_equal(H, S), f"popc matrix differs from Sylvester at n={n}"


def pin_butterfly_vs_dense_float(orc):
    rng = np.random.default_rng(1234)
    for n in range(0, 11):
        x = rng.standard_normal((3, 1 << n))
        for norm in (False, True):
            y = orc.fwt(x, normalize=norm)
            ref = dense.dense_fwt(x, normalize=norm)
            for b in range(3):
                assert _rel(y[b], ref[b]) < 1e-13, f"float mismatch n={n} normalize={norm}"


def pin_butterfly_vs_dense_int(orc):
    rng = np.random.default_rng(99)
    for n in range(0, 11):
        # full-range int32: intermediate sums wrap; the dense product is exact in
        # int64 (|sum| < 2^41), reduced modulo 2^32 afterwards.
        x = rng.integers(-(2 ** 31), 2 ** 31, size=(2, 1 << n), dtype=np.int64).astype(np.int32)
        y = orc.fwt(x, normalize=False)
        ref = (dense.dense_fwt(x.astype(np.int64)) % (1 << 32)).astype(np.uint32).view(np.int32)
        assert np.array_equal(y, ref), f"int32 mismatch n={n}"


def pin_golden(orc):
    with open(GOLDEN) as f:
        data = json.load(f)
    for case in data["cases"]:
        x = np.array(case["x"], dtype=np.float64)
        y = orc.fwt(x[None, :], normalize=case["normalize"])[0]
        assert np.array_equal(y, np.array(case["y"], dtype=np.float64)), case["what"]
        y32 = orc.fwt(x.astype(np.float32)[None, :], normalize=case["normalize"])[0]
        assert np.array_equal(y32, np.array(case["y"], dtype=np.float64)), case["what"]
    for case in data["int32_wrap_cases"]:
        x = np.array(case["x"], dtype=np.int64).astype(np.int32)
        y = orc.fwt(x[None, :], normalize=False)[0]
        assert np.array_equal(y, np.array(case["y"], dtype=np.int64).astype(np.int32)), case["what"]


def pin_closed_forms(orc):
    for n in (0, 1, 2, 3, 5, 8, 11, 14, 16):
        N = 1 << n
        s = 2.0 ** (-n / 2.0)
        k = np.arange(N)
        for j in sorted({j for j in (0, 1, N - 1, N // 3, N // 2) if j < N}):
            x = np.zeros((1, N))
            x[0, j] = 1.0
            y = orc.fwt(x, normalize=True)[0]
            walsh = s * (1.0 - 2.0 * _popc_parity(k & j))
            assert _rel(y, walsh) < 1e-15, f"delta at {j}, n={n}"
            yi = orc.fwt(x.astype(np.int32), normalize=False)[0]
            assert np.array_equal(yi, (1 - 2 * _popc_parity(k & j)).astype(np.int32))
        y = orc.fwt(np.ones((1, N)), normalize=True)[0]
        expect = np.zeros(N)
        expect[0] = N * s
        assert _rel(y, expect) < 1e-15, f"constant input, n={n}"
        x = np.random.default_rng(n).standard_normal((1, N))
        y0 = orc.fwt(x, normalize=True)[0][0]
        assert abs(y0 - s * np.sum(x)) <= 1e-12 * max(1.0, np.sum(np.abs(x))), f"y_0, n={n}"


def pin_involution(orc):
    rng = np.random.default_rng(7)
    for n in (1, 2, 5, 9, 12, 15):
        x = rng.standard_normal((2, 1 << n))
        yy = orc.fwt(orc.fwt(x, normalize=True), normalize=True)
        assert _rel(yy, x) < 1e-14, f"normalised transform is not an involution, n={n}"
        xi = rng.integers(-(2 ** 31), 2 ** 31, size=(2, 1 << n), dtype=np.int64).astype(np.int32)
        zz = orc.fwt(orc.fwt(xi, normalize=False), normalize=False)
        expect = ((xi.astype(np.int64) << n) % (1 << 32)).astype(np.uint32).view(np.int32)
        assert np.array_equal(zz, expect), f"H H != 2^n I modulo 2^32 at n={n}"


def pin_parseval_and_linearity(orc):
    rng = np.random.default_rng(11)
    for n in (0, 3, 7, 13, 16):
        x = rng.standard_normal((2, 1 << n))
        z = rng.standard_normal((2, 1 << n))
        y = orc.fwt(x, normalize=True)
        for b in range(2):
            assert abs(np.linalg.norm(y[b]) / np.linalg.norm(x[b]) - 1.0) < 1e-14, f"Parseval n={n}"
        lhs = orc.fwt(2.5 * x - 0.75 * z, normalize=False)
        rhs = 2.5 * orc.fwt(x, normalize=False) - 0.75 * orc.fwt(z, normalize=False)
        assert _rel(lhs, rhs) < 1e-13, f"linearity n={n}"


def pin_sylvester_recursion(orc):
    """H_n [lo; hi] = [H_{n-1} lo + H_{n-1} hi; H_{n-1} lo - H_{n-1} hi]."""
    rng = np.random.default_rng(5)
    for n in range(1, 18):
        h = 1 << (n - 1)
        x = rng.standard_normal((1, 2 * h))
        y = orc.fwt(x, normalize=False)[0]
        lo = orc.fwt(x[:, :h], normalize=False)[0]
        hi = orc.fwt(x[:, h:], normalize=False)[0]
        assert _rel(y[:h], lo + hi) < 1e-13 and _rel(y[h:], lo - hi) < 1e-13, f"n={n}"
        xi = rng.integers(-(2 ** 31), 2 ** 31, size=(1, 2 * h), dtype=np.int64).astype(np.int32)
        yi = orc.fwt(xi, normalize=False)[0].view(np.uint32)
        loi = orc.fwt(xi[:, :h], normalize=False)[0].view(np.uint32)
        hii = orc.fwt(xi[:, h:], normalize=False)[0].view(np.uint32)
        assert np.array_equal(yi[:h], loi + hii) and np.array_equal(yi[h:], loi - hii), f"int n={n}"


def pin_kronecker(orc):
    """H_{a+b} x = (H_a (x) H_b) x, i.e. Y = H_a X H_b^T for X = x viewed as 2^a x 2^b."""
    rng = np.random.default_rng(3)
    for a, b in ((1, 1), (3, 5), (7, 7), (6, 9), (8, 8)):
        n = a + b
        x = rng.standard_normal((1, 1 << n))
        Ha = dense.hadamard_popc(a).astype(np.float64)
        Hb = dense.hadamard_popc(b).astype(np.float64)
        X = x.reshape(1 << a, 1 << b)
        ref = (Ha @ X @ Hb.T).reshape(-1) * 2.0 ** (-n / 2.0)
        y = orc.fwt(x, normalize=True)[0]
        assert _rel(y, ref) < 1e-13, f"Kronecker split a={a} b={b}"


def pin_entries(orc):
    rng = np.random.default_rng(17)
    for n in (0, 1, 4, 10):
        x = rng.standard_normal(1 << n)
        ref = dense.dense_fwt(x[None, :], normalize=True)[0]
        ks = np.arange(1 << n)
        got = orc.entries(x, ks, normalize=True)
        assert _rel(got, ref) < 1e-14, f"entry vs dense n={n}"
        xi = rng.integers(-(2 ** 31), 2 ** 31, size=1 << n, dtype=np.int64).astype(np.int32)
        refi = (dense.dense_fwt(xi[None, :].astype(np.int64))[0] % (1 << 32)).astype(np.uint32).view(np.int32)
        assert np.array_equal(orc.entries(xi, ks), refi), f"int entry vs dense n={n}"
    n = 16
    x = rng.standard_normal(1 << n)
    y = orc.fwt(x[None, :], normalize=True)[0]
    ks = rng.integers(0, 1 << n, size=24)
    assert _rel(orc.entries(x, ks, normalize=True), y[ks]) < 1e-14, "entry vs butterfly n=16"


def pin_scale(orc):
    for n in range(0, 31):
        s = orc.scale(n, True)
        assert abs(s * s * 2.0 ** n - 1.0) < 4e-16, f"scale^2 * 2^n != 1 at n={n}"
        if n % 2 == 0:
            assert s == 2.0 ** (-n // 2), f"even-n scale not exact at n={n}"
        assert orc.scale(n, False) == 1.0


def pin_fp32_promotion(orc):
    rng = np.random.default_rng(21)
    x = rng.standard_normal((2, 1 << 9)).astype(np.float32)
    assert np.array_equal(orc.fwt(x, normalize=True), orc.fwt(x.astype(np.float64), normalize=True))


def pin_bit_range(orc):
    """The transform over index bits [lo, lo+k): I (x) H_k (x) I_{2^lo} (dense Kronecker
    product of popc matrices), the whole transform for [0, n), and a partition of
    [0, n) into ranges composes to the whole transform."""
    rng = np.random.default_rng(23)
    for n in (1, 3, 6, 9):
        x = rng.standard_normal((2, 1 << n))
        xi = rng.integers(-(2 ** 31), 2 ** 31, size=(2, 1 << n), dtype=np.int64).astype(np.int32)
        for lo in range(0, n):
            for k in range(1, n - lo + 1):
                M = np.kron(np.kron(np.eye(1 << (n - lo - k)), dense.hadamard_popc(k)), np.eye(1 << lo))
                ref = x @ M.T * 2.0 ** (-k / 2.0)
                assert _rel(orc.fwt_bits(x, lo, k, normalize=True), ref) < 1e-14, f"n={n} lo={lo} k={k}"
                refi = ((xi.astype(np.int64) @ M.T.astype(np.int64)) % (1 << 32)).astype(np.uint32).view(np.int32)
                assert np.array_equal(orc.fwt_bits(xi, lo, k, normalize=False), refi), f"int n={n} lo={lo} k={k}"
    for n in (5, 12, 16):
        x = rng.standard_normal((1, 1 << n))
        assert _rel(orc.fwt_bits(x, 0, n, normalize=True), orc.fwt(x, normalize=True)) < 1e-15
        cuts = sorted(set([0, n // 3, (2 * n) // 3, n]))
        y = x
        for a, b in zip(cuts[:-1], cuts[1:]):
            y = orc.fwt_bits(y, a, b - a, normalize=True)
        assert _rel(y, orc.fwt(x, normalize=True)) < 1e-14, f"composition n={n}"
        xi = rng.integers(-(2 ** 31), 2 ** 31, size=(1, 1 << n), dtype=np.int64).astype(np.int32)
        twice = orc.fwt_bits(orc.fwt_bits(xi, 2, 3, normalize=False), 2, 3, normalize=False)
        assert np.array_equal(twice, ((xi.astype(np.int64) << 3) % (1 << 32)).astype(np.uint32).view(np.int32))


def pin_phase_then_transform(orc):
    """y = s H (e^{i theta} . x): dense complex product for n <= 8; theta = 0 is the
    plain transform; a constant phase commutes with H; theta = pi/2 multiplies by i;
    |e^{i theta}| = 1 keeps the norm (Parseval)."""
    rng = np.random.default_rng(29)
    for n in (0, 1, 3, 8):
        re, im = rng.standard_normal((2, 2, 1 << n))
        th = rng.uniform(-np.pi, np.pi, size=(2, 1 << n))
        H = dense.hadamard_popc(n).astype(np.float64) * 2.0 ** (-n / 2.0)
        z = (re + 1j * im) * np.exp(1j * th)
        ref = z @ H.T
        yr, yi = orc.phase_fwt(re, im, th, normalize=True)
        assert np.linalg.norm((yr + 1j * yi) - ref) <= 1e-13 * np.linalg.norm(ref), f"dense n={n}"
        shared = th[:1]
        yr1, yi1 = orc.phase_fwt(re, im, shared, normalize=True)
        ref1 = ((re + 1j * im) * np.exp(1j * shared)) @ H.T
        assert np.linalg.norm((yr1 + 1j * yi1) - ref1) <= 1e-13 * np.linalg.norm(ref1), "shared theta"
    n = 12
    re, im = rng.standard_normal((2, 3, 1 << n))
    yr, yi = orc.phase_fwt(re, im, np.zeros((1, 1 << n)), normalize=True)
    assert _rel(yr, orc.fwt(re)) < 1e-15 and _rel(yi, orc.fwt(im)) < 1e-15, "theta = 0"
    phi = 0.7
    yr, yi = orc.phase_fwt(re, im, np.full((1, 1 << n), phi), normalize=True)
    plain = orc.fwt(re) + 1j * orc.fwt(im)
    assert np.linalg.norm((yr + 1j * yi) - np.exp(1j * phi) * plain) <= 1e-13 * np.linalg.norm(plain)
    yr, yi = orc.phase_fwt(re, im, np.full((1, 1 << n), np.pi / 2), normalize=True)
    assert _rel(yr, -orc.fwt(im)) < 1e-14 and _rel(yi, orc.fwt(re)) < 1e-14, "theta = pi/2"
    th = rng.uniform(0, 2 * np.pi, size=(3, 1 << n))
    yr, yi = orc.phase_fwt(re, im, th, normalize=True)
    for b in range(3):
        a = np.sqrt(np.sum(yr[b] ** 2 + yi[b] ** 2))
        e = np.sqrt(np.sum(re[b] ** 2 + im[b] ** 2))
        assert abs(a / e - 1) < 1e-14, "Parseval with phase"


def pin_bit_mask(orc):
    """The transform over an arbitrary set of index bits equals the dense Kronecker
    product, index bit n-1 leftmost, of H_1 (the popc matrix of one bit) where the
    bit is set and I_2 where it is not, scaled by 2^{-popcount/2}; for int32 the
    same product modulo 2^32.  The empty set copies; the full set is the transform."""
    rng = np.random.default_rng(31)
    h1 = dense.hadamard_popc(1).astype(np.float64)
    for n in (1, 4, 7, 9):
        x = rng.standard_normal((2, 1 << n))
        xi = rng.integers(-(2 ** 31), 2 ** 31, size=(2, 1 << n), dtype=np.int64).astype(np.int32)
        masks = {0, (1 << n) - 1, 1, 1 << (n - 1)} | {int(m) for m in rng.integers(0, 1 << n, size=8)}
        for mask in sorted(masks):
            M = np.ones((1, 1))
            for bit in reversed(range(n)):
                M = np.kron(M, h1 if (mask >> bit) & 1 else np.eye(2))
            k = bin(mask).count("1")
            ref = x @ M.T * 2.0 ** (-k / 2.0)
            assert _rel(orc.fwt_mask(x, mask, normalize=True), ref) < 1e-14, f"n={n} mask={mask:#x}"
            refi = ((xi.astype(np.int64) @ M.T.astype(np.int64)) % (1 << 32)).astype(np.uint32).view(np.int32)
            assert np.array_equal(orc.fwt_mask(xi, mask, normalize=False), refi), f"int n={n} mask={mask:#x}"
    x = rng.standard_normal((1, 1 << 12))
    assert _rel(orc.fwt_mask(x, (1 << 12) - 1), orc.fwt(x)) < 1e-15
    assert np.array_equal(orc.fwt_mask(x, 0, normalize=True), x)


def pin_complex_parts(orc):
    """A split complex vector transforms part by part (H is real): the real output is
    the dense popc product of the real input, the imaginary output that of the
    imaginary input, for float and wrapping int32; an int32 vector without an
    imaginary part gives none."""
    rng = np.random.default_rng(57)
    for n in (0, 1, 5, 9):
        re, im = rng.standard_normal((2, 3, 1 << n))
        gr, gi = orc.fwt_complex(re, im, normalize=True)
        assert _rel(gr, dense.dense_fwt(re, normalize=True)) < 1e-14, f"real part n={n}"
        assert _rel(gi, dense.dense_fwt(im, normalize=True)) < 1e-14, f"imaginary part n={n}"
        ri, ii = rng.integers(-(2 ** 31), 2 ** 31, size=(2, 2, 1 << n), dtype=np.int64).astype(np.int32)
        gr, gi = orc.fwt_complex(ri, ii, normalize=False)
        for got, x in ((gr, ri), (gi, ii)):
            ref = (dense.dense_fwt(x.astype(np.int64)) % (1 << 32)).astype(np.uint32).view(np.int32)
            assert np.array_equal(got, ref), f"int32 part n={n}"
        gr, gi = orc.fwt_complex(ri, None, normalize=False)
        assert gi is None and np.array_equal(
            gr, (dense.dense_fwt(ri.astype(np.int64)) % (1 << 32)).astype(np.uint32).view(np.int32))


ORACLE_PINS = [
    pin_butterfly_vs_dense_float,
    pin_butterfly_vs_dense_int,
    pin_golden,
    pin_closed_forms,
    pin_involution,
    pin_parseval_and_linearity,
    pin_sylvester_recursion,
    pin_kronecker,
    pin_entries,
    pin_scale,
    pin_fp32_promotion,
    pin_bit_range,
    pin_bit_mask,
    pin_phase_then_transform,
    pin_complex_parts,
]
