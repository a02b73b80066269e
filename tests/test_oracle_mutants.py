"""Plant plausible mistakes in a copy of the oracle and check that a pin catches each.

The mistakes are planted in the oracle's C source on the CPU (a temporary copy,
compiled with gcc); the real oracle is never touched.
"""
import os

import numpy as np
import pytest

import oracle
import oracle_pins

# (name, original text, replacement, which occurrence (0-based)) -- occurrence 0 of the
# butterfly lines is the double routine, occurrence 1 the uint32 routine.
MUTANTS = [
    ("f64 swapped outputs", "x[j] = u + v;\n        x[j + h] = u - v;",
     "x[j] = u - v;\n        x[j + h] = u + v;", 0),
    ("f64 wrong sign", "x[j + h] = u - v;", "x[j + h] = v - u;", 0),
    ("f64 dropped stage 0", "for (int64_t h = 1; h < N; h *= 2)", "for (int64_t h = 2; h < N; h *= 2)", 0),
    ("f64 last stage missing", "for (int64_t h = 1; h < N; h *= 2)", "for (int64_t h = 1; 2 * h < N; h *= 2)", 0),
    ("f64 wrong partner", "double v = x[j + h];", "double v = x[i + h + (j - i + 1) % h];", 0),
    ("u32 wrong sign", "x[j + h] = u - v;", "x[j + h] = v - u;", 1),
    ("u32 dropped stage", "for (int64_t h = 1; h < N; h *= 2)", "for (int64_t h = 2; h < N; h *= 2)", 1),
    ("even scale wrong", "return ldexp(1.0, -n / 2);", "return ldexp(1.0, -n);", 0),
    ("odd scale inverted", "/ sqrt(2.0);", "* sqrt(2.0);", 0),
    ("entry uses OR", "double t = popc_parity((uint64_t)(k & i))", "double t = popc_parity((uint64_t)(k | i))", 0),
    ("int entry transposed sign", "if (popc_parity((uint64_t)(k & i))) acc -= x[i];",
     "if (!popc_parity((uint64_t)(k & i))) acc -= x[i];", 0),
    ("scale skipped", "if (jb->scale != 1.0)", "if (jb->scale == 12345.0)", 0),
    ("phase rotation sign", "const double r = xr[i] * c - xi[i] * sn;", "const double r = xr[i] * c + xi[i] * sn;", 0),
    ("phase uses cos for sin", "const double c = cos(th[i]), sn = sin(th[i]);", "const double c = cos(th[i]), sn = cos(th[i]);", 0),
    ("bit range starts one stage late", "for (int64_t h = (int64_t)1 << lo;",
     "for (int64_t h = (int64_t)2 << lo;", 0),
    ("bit range scale uses n", "oracle_scale(nbits, normalize), 0, nthreads, lo, nbits)",
     "oracle_scale(n, normalize), 0, nthreads, lo, nbits)", 0),
    ("u32 bit range drops the last stage", "for (int64_t h = (int64_t)1 << lo; h < ((int64_t)1 << (lo + nbits)); h *= 2) {\n    for (int64_t i = 0; i < N; i += 2 * h) {\n      for (int64_t j = i; j < i + h; ++j) {\n        uint32_t",
     "for (int64_t h = (int64_t)1 << lo; 2 * h < ((int64_t)1 << (lo + nbits)); h *= 2) {\n    for (int64_t i = 0; i < N; i += 2 * h) {\n      for (int64_t j = i; j < i + h; ++j) {\n        uint32_t", 0),
]


def _replace_nth(text, old, new, nth):
    start = -1
    for _ in range(nth + 1):
        start = text.find(old, start + 1)
        assert start >= 0, f"mutation anchor not found: {old!r}"
    return text[:start] + new + text[start + len(old):]


@pytest.mark.parametrize("name,old,new,nth", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_planted_mistake(tmp_path, name, old, new, nth):
    src = open(oracle.SOURCE).read()
    mutated = _replace_nth(src, old, new, nth)
    assert mutated != src
    path = tmp_path / "mutant.c"
    path.write_text(mutated)
    so = oracle.compile_library(str(path), str(tmp_path / "libmutant.so"))
    orc = oracle.Oracle(so)
    caught = []
    for pin in oracle_pins.ORACLE_PINS:
        try:
            pin(orc)
        except AssertionError as e:  # the planted mistake was seen
            caught.append((pin.__name__, str(e)))
    assert caught, f"no pin caught the planted mistake {name!r}"


def test_unmutated_copy_passes(tmp_path):
    so = oracle.compile_library(oracle.SOURCE, str(tmp_path / "libcopy.so"))
    orc = oracle.Oracle(so)
    for pin in oracle_pins.ORACLE_PINS:
        pin(orc)
    assert os.path.exists(so)


# Mistakes in the oracle's Python layer (the bit-mask composition and the split
# complex form), planted on one Oracle instance by replacing a method.
def _mask_as_one_range(orc):
    def fwt_mask(x, mask, normalize=True, nthreads=1):
        if mask == 0:
            return orc.fwt_bits(x, 0, 0, normalize, nthreads)
        lo, hi = (mask & -mask).bit_length() - 1, mask.bit_length()
        return orc.fwt_bits(x, lo, hi - lo, normalize, nthreads)
    orc.fwt_mask = fwt_mask


def _mask_drops_top_run(orc):
    right = orc.fwt_mask

    def fwt_mask(x, mask, normalize=True, nthreads=1):
        b = mask.bit_length() - 1
        while b >= 0 and (mask >> b) & 1:
            mask &= ~(1 << b)
            b -= 1
        return right(x, mask, normalize, nthreads)
    orc.fwt_mask = fwt_mask


def _mask_scales_by_n(orc):
    right = orc.fwt_mask

    def fwt_mask(x, mask, normalize=True, nthreads=1):
        y = right(x, mask, False, nthreads)
        if normalize:
            n = int(np.asarray(x).shape[-1]).bit_length() - 1
            y = y * 2.0 ** (-n / 2)
        return y
    orc.fwt_mask = fwt_mask


def _complex_swaps_parts(orc):
    def fwt_complex(re, im, normalize=True, nthreads=1):
        if im is None:
            return orc.fwt(re, normalize, nthreads), None
        return orc.fwt(im, normalize, nthreads), orc.fwt(re, normalize, nthreads)
    orc.fwt_complex = fwt_complex


def _complex_imag_from_real(orc):
    def fwt_complex(re, im, normalize=True, nthreads=1):
        out = orc.fwt(re, normalize, nthreads)
        return out, None if im is None else out.copy()
    orc.fwt_complex = fwt_complex


PY_MUTANTS = [_mask_as_one_range, _mask_drops_top_run, _mask_scales_by_n, _complex_swaps_parts,
              _complex_imag_from_real]


@pytest.mark.parametrize("plant", PY_MUTANTS, ids=[m.__name__.strip("_") for m in PY_MUTANTS])
def test_pins_catch_planted_python_mistake(plant):
    orc = oracle.Oracle(oracle.build())
    plant(orc)
    caught = []
    for pin in oracle_pins.ORACLE_PINS:
        try:
            pin(orc)
        except AssertionError as e:
            caught.append((pin.__name__, str(e)))
    assert caught, f"no pin caught the planted mistake {plant.__name__!r}"
