"""Seeded synthetic inputs for the batched Walsh-Hadamard transform.

This module holds no transform arithmetic: it only draws the input states that
both the CUDA path and the CPU oracle consume, so the two can be compared on the
same bytes.  It imports neither.

Recipe (the source pages give the shapes, not the generator):

* NumPy ``Generator(PCG64(seed))``.
* Gaussian states: ``standard_normal((batch, 2, N))`` in float64; ``[:, 0]`` is the
  real part, ``[:, 1]`` the imaginary part.  "Unit L2" states divide each vector
  by its joint complex norm sqrt(sum re^2 + im^2), in float64, before any cast.
* fp32 workloads are the float64 draw rounded once to float32.
* int32 workloads: ``integers(-8, 9, (batch, N))`` (uniform on -8..8 inclusive),
  imaginary part all zero.

Edge-case recipes (``edge_pair``), for tests only: full-range int32 (every
intermediate wraps), and fp64 inputs that drive a fixed-point conversion to its
worst case (one-signed values with full mantissas; every element just below a
power of two; one large entry per tile with full-mantissa entries far below it).
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np


@dataclass(frozen=True)
class Workload:
    """One named batch shape: 2^n amplitudes x batch, split re/im arrays."""

    name: str
    n: int
    batch: int
    dtype: str  # "c32" (float32 pairs), "c64" (float64 pairs) or "i32" (int32 pairs)
    seed: int
    normalize: bool
    values: str  # "gaussian", "unit_gaussian" or "uniform_int8"

    @property
    def N(self) -> int:
        return 1 << self.n

    @property
    def elem_bytes(self) -> int:
        return {"c32": 4, "c64": 8, "i32": 4}[self.dtype]

    @property
    def bytes_in(self) -> int:
        """Bytes of input (re + im) for the whole batch."""
        return 2 * self.batch * self.N * self.elem_bytes

    def generate(self, batch: int | None = None):
        """Return (re, im) host arrays of shape (batch, 2^n).

        A smaller ``batch`` gives exactly the first rows of the full draw: the
        generator fills the (batch, 2, N) block in row order."""
        b = self.batch if batch is None else int(batch)
        return draw(self.values, self.n, b, self.seed, self.dtype)


def draw(values: str, n: int, batch: int, seed: int, dtype: str):
    """Seeded (re, im) pair of (batch, 2^n) arrays; see the module docstring."""
    rng = np.random.Generator(np.random.PCG64(seed))
    N = 1 << n
    if values == "uniform_int8":
        re = rng.integers(-8, 9, size=(batch, N), dtype=np.int32)
        im = np.zeros((batch, N), dtype=np.int32)
        return re, im
    z = rng.standard_normal((batch, 2, N))  # float64
    if values == "unit_gaussian":
        norms = np.sqrt(np.sum(z * z, axis=(1, 2)))
        norms[norms == 0] = 1.0
        z /= norms[:, None, None]
    elif values != "gaussian":
        raise ValueError(f"unknown value recipe {values!r}")
    ftype = {"c32": np.float32, "c64": np.float64}[dtype]
    return np.ascontiguousarray(z[:, 0], dtype=ftype), np.ascontiguousarray(z[:, 1], dtype=ftype)


# The five shapes the transform is specified on.  The last one appears twice: the
# same fp64 states, and those states rounded to fp32.
WORKLOADS = {
    w.name: w
    for w in [
        Workload("n10_b64_c32", 10, 64, "c32", 0, True, "gaussian"),
        Workload("n12_b64_c32", 12, 64, "c32", 1, True, "unit_gaussian"),
        Workload("n14_b64_c32", 14, 64, "c32", 2, True, "unit_gaussian"),
        Workload("n18_b256_i32", 18, 256, "i32", 3, False, "uniform_int8"),
        Workload("n24_b16_c64", 24, 16, "c64", 4, True, "unit_gaussian"),
        Workload("n24_b16_c32", 24, 16, "c32", 4, True, "unit_gaussian"),
    ]
}


def random_pair(n: int, batch: int, dtype: str, seed: int):
    """Small seeded case for sweeps: Gaussian floats or uniform -8..8 ints."""
    if dtype == "i32":
        return draw("uniform_int8", n, batch, seed, dtype)
    return draw("gaussian", n, batch, seed, dtype)


def edge_pair(kind: str, n: int, batch: int, seed: int, tile_bits: int = 13):
    """Seeded (re, im) pair of (batch, 2^n) edge-case arrays:

    * ``"int32_full"``: int32 uniform over the whole range [-2^31, 2^31), both parts.
    * ``"fp64_one_signed"``: fp64 uniform in [1, 2) (full 52-bit mantissas), both parts.
    * ``"fp64_below_pow2"``: every element nextafter(2^e, 0) for a per-vector e in
      [-20, 20) (all 53 significand bits set); the imaginary part negated.
    * ``"fp64_spike"``: per block of 2^tile_bits contiguous elements one entry of
      magnitude 2^e (e per vector in [-20, 20)), the others full-mantissa values in
      [1, 2) * 2^(e - 30); signs random.
    """
    rng = np.random.Generator(np.random.PCG64(seed))
    N = 1 << n
    if kind == "int32_full":
        z = rng.integers(-(1 << 31), 1 << 31, size=(batch, 2, N), dtype=np.int64).astype(np.int32)
        return np.ascontiguousarray(z[:, 0]), np.ascontiguousarray(z[:, 1])
    e = rng.integers(-20, 20, size=batch)
    if kind == "fp64_one_signed":
        z = 1.0 + rng.random((batch, 2, N))
    elif kind == "fp64_below_pow2":
        v = np.nextafter(np.ldexp(1.0, e), 0.0)
        z = np.empty((batch, 2, N))
        z[:, 0] = v[:, None]
        z[:, 1] = -v[:, None]
    elif kind == "fp64_spike":
        z = np.ldexp(1.0 + rng.random((batch, 2, N)), (e - 30)[:, None, None])
        tb = min(tile_bits, n)
        blocks = N >> tb
        pos = rng.integers(0, 1 << tb, size=(batch, 2, blocks)) + (np.arange(blocks) << tb)
        for b in range(batch):
            for c in range(2):
                z[b, c, pos[b, c]] = np.ldexp(1.0, int(e[b]))
        z *= rng.choice([-1.0, 1.0], size=z.shape)
    else:
        raise ValueError(f"unknown edge-case recipe {kind!r}")
    return np.ascontiguousarray(z[:, 0]), np.ascontiguousarray(z[:, 1])
