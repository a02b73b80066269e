"""CPU oracle for the batched Walsh-Hadamard transform.

TEST INFRASTRUCTURE ONLY.  The product library never imports, links or runs
anything in this package; only the test suite, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` do.  It shares no code with the CUDA path.

Two independent statements of what the transform computes:

* ``fwt_oracle.c`` (wrapped here): the textbook in-place butterfly network in
  double (uint32 for int32 data), plus single output entries evaluated straight
  from the definition ``y[k] = s * sum_i (-1)^popc(k & i) x[i]``
  ("[QDP] [feature] Pr4 kronecker fwt", section "How"; iThome "Day 18" FWT post,
  section "Tensor Core wants matrix multiplication" for the stage structure).
* ``dense.py``: the Hadamard matrix built entry by entry from the same popc rule
  and multiplied densely (n <= 12), used to pin the butterfly.

fp32 inputs are promoted to double before the transform, so the oracle result is
the exact transform to within about n * 2^-53 relative error.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(_HERE, "fwt_oracle.c")
LIBRARY = os.path.join(_HERE, "liboracle_fwt.so")

_lock = threading.Lock()


def compile_library(source: str = SOURCE, output: str = LIBRARY) -> str:
    """Compile an oracle C source into a shared library with gcc; returns its path."""
    cmd = ["gcc", "-O2", "-std=c99", "-Wall", "-shared", "-fPIC", "-o", output, source,
           "-lpthread", "-lm"]
    subprocess.run(cmd, check=True, capture_output=True, text=True)
    return output


def build(force: bool = False) -> str:
    """Build ``liboracle_fwt.so`` next to its source if missing or stale."""
    with _lock:
        stale = (not os.path.exists(LIBRARY)
                 or os.path.getmtime(LIBRARY) < os.path.getmtime(SOURCE))
        if force or stale:
            compile_library()
    return LIBRARY


class Oracle:
    """ctypes view of one compiled oracle library (the default one, or a test copy)."""

    def __init__(self, path: str):
        lib = ctypes.CDLL(path)
        i64, dp, up = ctypes.c_int64, ctypes.POINTER(ctypes.c_double), ctypes.POINTER(ctypes.c_uint32)
        lib.oracle_scale.argtypes = [ctypes.c_int, ctypes.c_int]
        lib.oracle_scale.restype = ctypes.c_double
        lib.oracle_fwt_f64.argtypes = [dp, dp, ctypes.c_int, i64, ctypes.c_int, ctypes.c_int]
        lib.oracle_fwt_f64.restype = ctypes.c_int
        lib.oracle_fwt_u32.argtypes = [up, up, ctypes.c_int, i64, ctypes.c_int]
        lib.oracle_fwt_u32.restype = ctypes.c_int
        lib.oracle_fwt_bits_f64.argtypes = [dp, dp, ctypes.c_int, i64, ctypes.c_int, ctypes.c_int,
                                            ctypes.c_int, ctypes.c_int]
        lib.oracle_fwt_bits_f64.restype = ctypes.c_int
        lib.oracle_fwt_bits_u32.argtypes = [up, up, ctypes.c_int, i64, ctypes.c_int, ctypes.c_int,
                                            ctypes.c_int]
        lib.oracle_fwt_bits_u32.restype = ctypes.c_int
        lib.oracle_phase_fwt_f64.argtypes = [dp, dp, dp, i64, dp, dp, ctypes.c_int, i64, ctypes.c_int]
        lib.oracle_phase_fwt_f64.restype = ctypes.c_int
        lib.oracle_fwt_entry_f64.argtypes = [dp, ctypes.c_int, i64, ctypes.c_int]
        lib.oracle_fwt_entry_f64.restype = ctypes.c_double
        lib.oracle_fwt_entry_u32.argtypes = [up, ctypes.c_int, i64]
        lib.oracle_fwt_entry_u32.restype = ctypes.c_uint32
        self.lib = lib
        self.path = path

    # -- helpers -----------------------------------------------------------------
    @staticmethod
    def _n_of(length: int) -> int:
        n = int(length).bit_length() - 1
        if length < 1 or (1 << n) != length:
            raise ValueError(f"vector length {length} is not a power of two")
        return n

    def scale(self, n: int, normalize: bool = True) -> float:
        return float(self.lib.oracle_scale(int(n), int(bool(normalize))))

    # -- whole transforms --------------------------------------------------------
    def fwt(self, x, normalize: bool = True, nthreads: int = 1) -> np.ndarray:
        """Transform every length-2^n row of ``x`` (last axis).

        float16/32/64 input -> float64 result; int32/uint32 input -> int32 result
        (wrap-around modulo 2^32; ``normalize`` must be False).
        """
        x = np.asarray(x)
        n = self._n_of(x.shape[-1])
        count = x.size // x.shape[-1] if x.size else 0
        if x.dtype in (np.int32, np.uint32):
            if normalize:
                raise ValueError("int32 transform has no normalised form")
            src = np.ascontiguousarray(x).view(np.uint32)
            out = np.empty_like(src)
            rc = self.lib.oracle_fwt_u32(
                src.ctypes.data_as(ctypes.POINTER(ctypes.c_uint32)),
                out.ctypes.data_as(ctypes.POINTER(ctypes.c_uint32)), n, count, int(nthreads))
            if rc:
                raise RuntimeError(f"oracle_fwt_u32 failed ({rc})")
            return out.view(np.int32)
        src = np.ascontiguousarray(x, dtype=np.float64)
        out = np.empty_like(src)
        rc = self.lib.oracle_fwt_f64(
            src.ctypes.data_as(ctypes.POINTER(ctypes.c_double)),
            out.ctypes.data_as(ctypes.POINTER(ctypes.c_double)), n, count,
            int(bool(normalize)), int(nthreads))
        if rc:
            raise RuntimeError(f"oracle_fwt_f64 failed ({rc})")
        return out

    def fwt_bits(self, x, lo: int, nbits: int, normalize: bool = True, nthreads: int = 1):
        """Transform over index bits [lo, lo+nbits) of every row of ``x`` (last axis):
        I (x) H_nbits (x) I_{2^lo}, scaled by 2^{-nbits/2} when normalising."""
        x = np.asarray(x)
        n = self._n_of(x.shape[-1])
        count = x.size // x.shape[-1] if x.size else 0
        if x.dtype in (np.int32, np.uint32):
            if normalize:
                raise ValueError("int32 transform has no normalised form")
            src = np.ascontiguousarray(x).view(np.uint32)
            out = np.empty_like(src)
            rc = self.lib.oracle_fwt_bits_u32(
                src.ctypes.data_as(ctypes.POINTER(ctypes.c_uint32)),
                out.ctypes.data_as(ctypes.POINTER(ctypes.c_uint32)), n, count, int(lo), int(nbits),
                int(nthreads))
            if rc:
                raise RuntimeError(f"oracle_fwt_bits_u32 failed ({rc})")
            return out.view(np.int32)
        src = np.ascontiguousarray(x, dtype=np.float64)
        out = np.empty_like(src)
        rc = self.lib.oracle_fwt_bits_f64(
            src.ctypes.data_as(ctypes.POINTER(ctypes.c_double)),
            out.ctypes.data_as(ctypes.POINTER(ctypes.c_double)), n, count, int(lo), int(nbits),
            int(bool(normalize)), int(nthreads))
        if rc:
            raise RuntimeError(f"oracle_fwt_bits_f64 failed ({rc})")
        return out

    def fwt_mask(self, x, mask: int, normalize: bool = True, nthreads: int = 1):
        """Transform over the index bits set in ``mask``: the stages of those bits
        commute, so this is the bit-range transform of each maximal run of set bits
        in turn (the same butterfly loop, restricted to a run at a time), scaled by
        2^{-popcount(mask)/2} in all when normalising."""
        x = np.asarray(x)
        n = self._n_of(x.shape[-1])
        mask = int(mask)
        if mask < 0 or mask >> n:
            raise ValueError(f"mask {mask:#x} has bits at or above n = {n}")
        runs, b = [], 0
        while b < n:
            if (mask >> b) & 1:
                a = b
                while b < n and (mask >> b) & 1:
                    b += 1
                runs.append((a, b - a))
            else:
                b += 1
        y = x
        for lo, k in runs:
            y = self.fwt_bits(y, lo, k, normalize, nthreads)
        if not runs:  # nothing transformed: a copy in the result type
            y = self.fwt_bits(x, 0, 0, normalize, nthreads)
        return y

    def fwt_complex(self, re, im, normalize: bool = True, nthreads: int = 1):
        """H is real, so a split complex vector transforms component by component."""
        out_im = None if im is None else self.fwt(im, normalize, nthreads)
        return self.fwt(re, normalize, nthreads), out_im

    def phase_fwt(self, re, im, theta, normalize: bool = True):
        """y = s * H (e^{i theta} . x) for split complex rows; ``theta`` has one row
        per vector, or a single row shared by all vectors.  Returns float64 (re, im)."""
        re = np.ascontiguousarray(re, dtype=np.float64)
        im = np.ascontiguousarray(im, dtype=np.float64)
        th = np.ascontiguousarray(np.atleast_2d(theta), dtype=np.float64)
        n = self._n_of(re.shape[-1])
        count = re.size // re.shape[-1] if re.size else 0
        stride = 0 if th.shape[0] == 1 else re.shape[-1]
        if th.shape[-1] != re.shape[-1] or (stride and th.shape[0] != count):
            raise ValueError("theta must have one row per vector or a single shared row")
        out_r, out_i = np.empty_like(re), np.empty_like(im)
        dp = ctypes.POINTER(ctypes.c_double)
        rc = self.lib.oracle_phase_fwt_f64(re.ctypes.data_as(dp), im.ctypes.data_as(dp),
                                           th.ctypes.data_as(dp), stride, out_r.ctypes.data_as(dp),
                                           out_i.ctypes.data_as(dp), n, count, int(bool(normalize)))
        if rc:
            raise RuntimeError(f"oracle_phase_fwt_f64 failed ({rc})")
        return out_r, out_i

    # -- single entries from the definition ----------------------------------------
    def entry(self, vec, k: int, normalize: bool = True):
        """y[k] of one vector from the popc definition (compensated sum for floats)."""
        vec = np.asarray(vec)
        n = self._n_of(vec.shape[-1])
        if vec.dtype in (np.int32, np.uint32):
            v = np.ascontiguousarray(vec).view(np.uint32)
            r = self.lib.oracle_fwt_entry_u32(v.ctypes.data_as(ctypes.POINTER(ctypes.c_uint32)),
                                              n, int(k))
            return np.uint32(r).view(np.int32)
        v = np.ascontiguousarray(vec, dtype=np.float64)
        return float(self.lib.oracle_fwt_entry_f64(
            v.ctypes.data_as(ctypes.POINTER(ctypes.c_double)), n, int(k), int(bool(normalize))))

    def entries(self, vec, ks, normalize: bool = True) -> np.ndarray:
        vals = [self.entry(vec, int(k), normalize) for k in ks]
        vec = np.asarray(vec)
        dtype = np.int32 if vec.dtype in (np.int32, np.uint32) else np.float64
        return np.array(vals, dtype=dtype)


_default: Oracle | None = None


def default() -> Oracle:
    """The oracle built from ``fwt_oracle.c`` (compiled on first use)."""
    global _default
    if _default is None:
        _default = Oracle(build())
    return _default


def fwt(x, normalize: bool = True, nthreads: int = 1) -> np.ndarray:
    return default().fwt(x, normalize, nthreads)


def fwt_complex(re, im, normalize: bool = True, nthreads: int = 1):
    return default().fwt_complex(re, im, normalize, nthreads)


def fwt_bits(x, lo: int, nbits: int, normalize: bool = True, nthreads: int = 1) -> np.ndarray:
    return default().fwt_bits(x, lo, nbits, normalize, nthreads)


def fwt_mask(x, mask: int, normalize: bool = True, nthreads: int = 1) -> np.ndarray:
    return default().fwt_mask(x, mask, normalize, nthreads)


def phase_fwt(re, im, theta, normalize: bool = True):
    return default().phase_fwt(re, im, theta, normalize)


def entry(vec, k: int, normalize: bool = True):
    return default().entry(vec, k, normalize)


def entries(vec, ks, normalize: bool = True) -> np.ndarray:
    return default().entries(vec, ks, normalize)


def scale(n: int, normalize: bool = True) -> float:
    return default().scale(n, normalize)
