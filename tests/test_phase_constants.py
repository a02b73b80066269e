"""The fixed-point constants of the fp64 phase kernel: the CUDA source holds exactly
the values phase_constants.py derives, and its pi (Machin's formula) agrees with an
independent series (Bailey-Borwein-Plouffe) to far beyond the bits the constants use."""
import os
import re
from fractions import Fraction

from walsh_hadamard_transform_gb300 import phase_constants

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bbp_pi(terms: int = 80) -> Fraction:
    total = Fraction(0)
    for k in range(terms):
        total += Fraction(1, 16 ** k) * (Fraction(4, 8 * k + 1) - Fraction(2, 8 * k + 4)
                                         - Fraction(1, 8 * k + 5) - Fraction(1, 8 * k + 6))
    return total


def test_pi_by_two_independent_series():
    assert abs(phase_constants.pi_fraction() - _bbp_pi()) < Fraction(1, 1 << 300)


def test_constants_scale_as_documented():
    c = phase_constants.constants()
    pi = _bbp_pi()
    inv = Fraction((c["kInv2PiHi"] << 64) | c["kInv2PiLo"], 1 << 128)
    assert abs(inv - 1 / (2 * pi)) <= Fraction(1, 1 << 128)
    assert abs(Fraction(c["kTwoPiQ61"], 1 << 61) - 2 * pi) <= Fraction(1, 1 << 61)
    for name, d in (("kInv6Q32", 6), ("kInv24Q32", 24), ("kInv120Q32", 120)):
        assert abs(Fraction(c[name], 1 << 32) - Fraction(1, d)) <= Fraction(1, 1 << 32)


def test_cuda_source_holds_the_derived_values():
    src = open(os.path.join(ROOT, "walsh_hadamard_transform_gb300", "csrc", "rows_c64.cu")).read()
    found = dict(re.findall(r"constexpr unsigned long long (k\w+) = (0x[0-9a-f]+)ull;", src))
    for name, value in phase_constants.constants().items():
        assert int(found[name], 16) == value, name
