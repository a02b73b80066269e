"""Fixed-point constants of the fp64 diagonal phase (the sine and cosine of the
angles, evaluated in 64-bit integer arithmetic by ``fwt_phase_c64``).

The kernels reduce an angle to a fraction of a turn and evaluate the sine and
cosine from a table and two short series, all in integers.  Their constants are
derived here from pi, itself computed with Machin's formula
pi = 16 atan(1/5) - 4 atan(1/239) (each arctangent by its Taylor series) in exact
rational arithmetic, so that every digit can be checked without any floating-point
library.  ``python phase_constants.py`` prints the C definitions; a CPU test checks
that the CUDA source holds exactly these values.
"""
from __future__ import annotations

from fractions import Fraction


def _atan_inv(k: int, terms: int) -> Fraction:
    """atan(1/k) from its Taylor series, summed to `terms` terms."""
    total = Fraction(0)
    for i in range(terms):
        total += Fraction((-1) ** i, (2 * i + 1) * k ** (2 * i + 1))
    return total


def pi_fraction(bits: int = 256) -> Fraction:
    """pi to well beyond 2^-bits (Machin's formula)."""
    terms = bits // 4 + 8  # atan(1/5): each term gains log2(25) > 4 bits
    return 16 * _atan_inv(5, terms) - 4 * _atan_inv(239, terms)


def _round(x: Fraction) -> int:
    return int(x + Fraction(1, 2)) if x >= 0 else -int(-x + Fraction(1, 2))


def constants() -> dict:
    pi = pi_fraction()
    inv2pi_q128 = _round(Fraction(1 << 128) / (2 * pi))  # 1/(2 pi) in units of 2^-128
    return {
        # 1/(2 pi) * 2^128 as two 64-bit words (high, low): turns = angle * this / 2^128
        "kInv2PiHi": inv2pi_q128 >> 64,
        "kInv2PiLo": inv2pi_q128 & ((1 << 64) - 1),
        # 2 pi * 2^61: radians = turns (Q64) * this / 2^125
        "kTwoPiQ61": _round(2 * pi * (1 << 61)),
        # 1/6, 1/24, 1/120 in units of 2^-32 (series coefficients)
        "kInv6Q32": _round(Fraction(1 << 32, 6)),
        "kInv24Q32": _round(Fraction(1 << 32, 24)),
        "kInv120Q32": _round(Fraction(1 << 32, 120)),
    }


def c_definitions() -> str:
    return "\n".join(f"constexpr unsigned long long {k} = 0x{v:0{16 if 'Q32' not in k else 8}x}ull;"
                     for k, v in constants().items())


if __name__ == "__main__":
    print(c_definitions())
