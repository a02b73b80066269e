"""Dense Walsh-Hadamard matrix straight from the popc sign rule.

TEST INFRASTRUCTURE ONLY (see the package docstring).

``H[k, i] = (-1)^popc(k & i)`` ("[QDP] [feature] Pr4 kronecker fwt", section
"How": the on-the-fly Hadamard value of the naive GEMM placeholder).  Multiplying
by this matrix is the plain O(N^2) definition of the transform; it pins the
butterfly oracle for small n.  Integer products are exact in int64.
"""
from __future__ import annotations

import numpy as np


def popcount(a: np.ndarray) -> np.ndarray:
    """Number of set bits of each non-negative integer entry (bit by bit)."""
    a = np.asarray(a, dtype=np.int64).copy()
    count = np.zeros_like(a)
    while np.any(a):
        count += a & 1
        a >>= 1
    return count


def hadamard_popc(n: int) -> np.ndarray:
    """The 2^n x 2^n matrix with entries (-1)^popc(k & i), as int64."""
    if n < 0 or n > 12:
        raise ValueError("dense matrix only for 0 <= n <= 12")
    idx = np.arange(1 << n, dtype=np.int64)
    signs = popcount(idx[:, None] & idx[None, :]) & 1
    return (1 - 2 * signs).astype(np.int64)


def dense_fwt(x, normalize: bool = False) -> np.ndarray:
    """y = s * H x along the last axis by a dense matrix product.

    Integer input: exact int64 result (no scaling allowed).  Float input: float64.
    """
    x = np.asarray(x)
    n = x.shape[-1].bit_length() - 1
    H = hadamard_popc(n)
    if np.issubdtype(x.dtype, np.integer):
        if normalize:
            raise ValueError("integer transform has no normalised form")
        return x.astype(np.int64) @ H.T
    y = x.astype(np.float64) @ H.T.astype(np.float64)
    if normalize:
        y = y * 2.0 ** (-n / 2.0)
    return y
