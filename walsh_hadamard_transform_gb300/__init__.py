"""Batched Walsh-Hadamard transform on GB300 (sm_103a): Python binding.

``y[k] = s * sum_i (-1)^popc(k & i) x[i]`` on batches of 2^n-amplitude complex
vectors held as split real / imaginary arrays ("[QDP] [feature] Pr4 kronecker
fwt", section "How"), with s = 2^{-n/2} when normalised.

The functions named like the C ABI (``fwt_batched_c32`` ...) take raw device
pointers and marshal arguments only; every step of the transform runs in the
CUDA kernels of ``libfwt_gb300.so``.  ``transform`` is the tensor-level wrapper:
it checks dtypes, devices and contiguity, then calls the C ABI on the current
PyTorch stream.  There is no CPU fallback: without the compiled library (see
``build.py``) every call raises.
"""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIBRARY = os.path.join(_HERE, "libfwt_gb300.so")

FWT_OK, FWT_ERR_INVALID_ARG, FWT_ERR_MISALIGNED = 0, 1, 2
FWT_ERR_UNSUPPORTED, FWT_ERR_CUDA, FWT_ERR_TIMEOUT = 3, 4, 5
FWT_C32, FWT_C64, FWT_I32 = 0, 1, 2
DTYPES = {"c32": FWT_C32, "c64": FWT_C64, "i32": FWT_I32}


class FwtError(RuntimeError):
    """A non-zero status from the C ABI."""

    def __init__(self, status: int, what: str):
        self.status = status
        msg = f"{what}: {status_string(status)} ({status})"
        if status == FWT_ERR_CUDA:
            msg += f", cudaError {last_cuda_error()}"
        super().__init__(msg)


_lib = None


def library() -> ctypes.CDLL:
    """The loaded C library; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIBRARY):
            raise RuntimeError(
                f"{LIBRARY} is missing: build it with "
                "`python -c 'import __graft_entry__ as g; g.build()'` "
                "(or python walsh_hadamard_transform_gb300/build.py)")
        lib = ctypes.CDLL(LIBRARY)
        vp, i64, ci = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
        for name in ("fwt_batched_c32", "fwt_batched_c64", "fwt_batched_i32"):
            f = getattr(lib, name)
            f.argtypes = [vp, vp, vp, vp, ci, i64, ci, vp]
            f.restype = ci
        for name in ("fwt_bits_c32", "fwt_bits_c64", "fwt_bits_i32"):
            f = getattr(lib, name)
            f.argtypes = [vp, vp, vp, vp, ci, i64, ci, ci, ci, vp]
            f.restype = ci
        for name in ("fwt_mask_c32", "fwt_mask_c64", "fwt_mask_i32"):
            f = getattr(lib, name)
            f.argtypes = [vp, vp, vp, vp, ci, i64, ctypes.c_uint32, ci, vp]
            f.restype = ci
        for name in ("fwt_phase_c32", "fwt_phase_c64"):
            f = getattr(lib, name)
            f.argtypes = [vp, vp, vp, i64, vp, vp, ci, i64, ci, vp]
            f.restype = ci
        for name in ("fwt_host_c32", "fwt_host_c64", "fwt_host_i32"):
            f = getattr(lib, name)
            f.argtypes = [vp, vp, vp, vp, ci, i64, ci, vp, ctypes.c_size_t, vp]
            f.restype = ci
        lib.fwt_host_workspace_bytes.argtypes = [ci, ci, i64, ci]
        lib.fwt_host_workspace_bytes.restype = ctypes.c_size_t
        for name in ("fwt_host_static_c32", "fwt_host_static_c64", "fwt_host_static_i32"):
            f = getattr(lib, name)
            f.argtypes = [vp, vp, vp, vp, ci, i64, ci, vp]
            f.restype = ci
        lib.fwt_host_static_workspace_bytes.argtypes = []
        lib.fwt_host_static_workspace_bytes.restype = ctypes.c_size_t
        lib.fwt_status_string.argtypes = [ci]
        lib.fwt_status_string.restype = ctypes.c_char_p
        lib.fwt_last_cuda_error.argtypes = []
        lib.fwt_last_cuda_error.restype = ci
        lib.fwt_plan_passes.argtypes = [ci, ci]
        lib.fwt_plan_passes.restype = ci
        lib.fwt_plan_factors.argtypes = [ci, ci, ctypes.POINTER(ci), ci]
        lib.fwt_plan_factors.restype = ci
        lib.fwt_set_plan.argtypes = [ci, ci, ci, ctypes.POINTER(ci)]
        lib.fwt_set_plan.restype = ci
        lib.fwt_selfcheck.argtypes = []
        lib.fwt_selfcheck.restype = ci
        lib.fwt_set_column_bytes.argtypes = [ci, ci]
        lib.fwt_set_column_bytes.restype = ci
        lib.fwt_get_column_bytes.argtypes = [ci]
        lib.fwt_get_column_bytes.restype = ci
        lib.fwt_set_tma.argtypes = [ci]
        lib.fwt_set_tma.restype = ci
        lib.fwt_get_tma.argtypes = []
        lib.fwt_get_tma.restype = ci
        lib.fwt_set_pdl.argtypes = [ci]
        lib.fwt_set_pdl.restype = ci
        lib.fwt_get_pdl.argtypes = []
        lib.fwt_get_pdl.restype = ci
        lib.fwt_set_cluster.argtypes = [ci]
        lib.fwt_set_cluster.restype = ci
        lib.fwt_get_cluster.argtypes = []
        lib.fwt_get_cluster.restype = ci
        lib.fwt_set_tma_l2_promotion.argtypes = [ci]
        lib.fwt_set_tma_l2_promotion.restype = ci
        lib.fwt_selftest_bounded_wait.argtypes = [vp]
        lib.fwt_selftest_bounded_wait.restype = ci
        lib.fwt_device_status.argtypes = []
        lib.fwt_device_status.restype = ci
        lib.fwt_set_l2_chunk_bytes.argtypes = [ctypes.c_longlong]
        lib.fwt_set_l2_chunk_bytes.restype = ci
        lib.fwt_get_l2_chunk_bytes.argtypes = []
        lib.fwt_get_l2_chunk_bytes.restype = ctypes.c_longlong
        lib.fwt_trace_events.argtypes = [ctypes.POINTER(ctypes.c_void_p), ci]
        lib.fwt_trace_events.restype = ci
        lib.fwt_trace_count.argtypes = []
        lib.fwt_trace_count.restype = ci
        _lib = lib
    return _lib


# ---- C ABI, one Python function per entry point (argument marshalling only) -------

def fwt_batched_c32(re_in, im_in, re_out, im_out, n, batch, normalize, stream) -> int:
    return library().fwt_batched_c32(re_in, im_in, re_out, im_out, n, batch, int(normalize), stream)


def fwt_batched_c64(re_in, im_in, re_out, im_out, n, batch, normalize, stream) -> int:
    return library().fwt_batched_c64(re_in, im_in, re_out, im_out, n, batch, int(normalize), stream)


def fwt_batched_i32(re_in, im_in, re_out, im_out, n, batch, normalize, stream) -> int:
    return library().fwt_batched_i32(re_in, im_in, re_out, im_out, n, batch, int(normalize), stream)


def fwt_bits_c32(re_in, im_in, re_out, im_out, n, batch, lo, nbits, normalize, stream) -> int:
    return library().fwt_bits_c32(re_in, im_in, re_out, im_out, n, batch, lo, nbits,
                                  int(normalize), stream)


def fwt_bits_c64(re_in, im_in, re_out, im_out, n, batch, lo, nbits, normalize, stream) -> int:
    return library().fwt_bits_c64(re_in, im_in, re_out, im_out, n, batch, lo, nbits,
                                  int(normalize), stream)


def fwt_bits_i32(re_in, im_in, re_out, im_out, n, batch, lo, nbits, normalize, stream) -> int:
    return library().fwt_bits_i32(re_in, im_in, re_out, im_out, n, batch, lo, nbits,
                                  int(normalize), stream)


def fwt_mask_c32(re_in, im_in, re_out, im_out, n, batch, mask, normalize, stream) -> int:
    return library().fwt_mask_c32(re_in, im_in, re_out, im_out, n, batch, mask, int(normalize),
                                  stream)


def fwt_mask_c64(re_in, im_in, re_out, im_out, n, batch, mask, normalize, stream) -> int:
    return library().fwt_mask_c64(re_in, im_in, re_out, im_out, n, batch, mask, int(normalize),
                                  stream)


def fwt_mask_i32(re_in, im_in, re_out, im_out, n, batch, mask, normalize, stream) -> int:
    return library().fwt_mask_i32(re_in, im_in, re_out, im_out, n, batch, mask, int(normalize),
                                  stream)


def fwt_phase_c64(re_in, im_in, theta, theta_stride, re_out, im_out, n, batch, normalize,
                  stream) -> int:
    return library().fwt_phase_c64(re_in, im_in, theta, theta_stride, re_out, im_out, n, batch,
                                   int(normalize), stream)


def fwt_phase_c32(re_in, im_in, theta, theta_stride, re_out, im_out, n, batch, normalize,
                  stream) -> int:
    return library().fwt_phase_c32(re_in, im_in, theta, theta_stride, re_out, im_out, n, batch,
                                   int(normalize), stream)


def fwt_host_c32(re_in, im_in, re_out, im_out, n, batch, normalize, workspace, workspace_bytes,
                 stream) -> int:
    return library().fwt_host_c32(re_in, im_in, re_out, im_out, n, batch, int(normalize),
                                  workspace, workspace_bytes, stream)


def fwt_host_c64(re_in, im_in, re_out, im_out, n, batch, normalize, workspace, workspace_bytes,
                 stream) -> int:
    return library().fwt_host_c64(re_in, im_in, re_out, im_out, n, batch, int(normalize),
                                  workspace, workspace_bytes, stream)


def fwt_host_i32(re_in, im_in, re_out, im_out, n, batch, normalize, workspace, workspace_bytes,
                 stream) -> int:
    return library().fwt_host_i32(re_in, im_in, re_out, im_out, n, batch, int(normalize),
                                  workspace, workspace_bytes, stream)


def fwt_host_static_c32(re_in, im_in, re_out, im_out, n, batch, normalize, stream) -> int:
    return library().fwt_host_static_c32(re_in, im_in, re_out, im_out, n, batch, int(normalize),
                                         stream)


def fwt_host_static_c64(re_in, im_in, re_out, im_out, n, batch, normalize, stream) -> int:
    return library().fwt_host_static_c64(re_in, im_in, re_out, im_out, n, batch, int(normalize),
                                         stream)


def fwt_host_static_i32(re_in, im_in, re_out, im_out, n, batch, normalize, stream) -> int:
    return library().fwt_host_static_i32(re_in, im_in, re_out, im_out, n, batch, int(normalize),
                                         stream)


def fwt_host_static_workspace_bytes() -> int:
    return int(library().fwt_host_static_workspace_bytes())


def fwt_host_workspace_bytes(dtype, n, batch, with_im=True) -> int:
    return int(library().fwt_host_workspace_bytes(int(dtype), int(n), int(batch), int(bool(with_im))))


def phase_transform(re, im, theta, out_re=None, out_im=None, normalize: bool = True, stream=None):
    """y = s * H (e^{i theta} . x) for float32 or float64 CUDA tensors of shape
    (batch, 2^n) (fwt_phase_c32 / fwt_phase_c64).

    ``theta`` holds angles of the same dtype: shape (batch, 2^n) (one row per
    vector) or (2^n,) / (1, 2^n) (shared by the batch).  Returns (out_re, out_im)."""
    import torch

    if im is None or re.dtype not in (torch.float32, torch.float64) or im.dtype != re.dtype:
        raise TypeError("phase_transform takes float32 or float64 re and im of one dtype")
    if theta.dtype != re.dtype or not theta.is_cuda or not theta.is_contiguous():
        raise ValueError("theta must be a contiguous CUDA tensor of the data's dtype")
    batch, N = re.shape
    n = int(N).bit_length() - 1
    if N < 1 or (1 << n) != N:
        raise ValueError(f"row length {N} is not a power of two")
    th2 = theta.reshape(-1, N)
    if th2.shape[0] not in (1, batch):
        raise ValueError("theta must have one row per vector or one shared row")
    stride = 0 if th2.shape[0] == 1 else N
    if out_re is None:
        out_re = torch.empty_like(re)
    if out_im is None:
        out_im = torch.empty_like(im)
    for t in (re, im, out_re, out_im):
        if t.shape != re.shape or t.device != re.device or not t.is_contiguous():
            raise ValueError("re, im and outputs must be contiguous CUDA tensors of one shape")
    if stream is None:
        stream = torch.cuda.current_stream(re.device)
    handle = stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)
    entry, name = ((fwt_phase_c64, "fwt_phase_c64") if re.dtype == torch.float64
                   else (fwt_phase_c32, "fwt_phase_c32"))
    with torch.cuda.device(re.device):
        st = entry(re.data_ptr(), im.data_ptr(), theta.data_ptr(), stride, out_re.data_ptr(),
                   out_im.data_ptr(), n, batch, normalize, handle)
    if st != FWT_OK:
        raise FwtError(st, f"{name}(n={n}, batch={batch})")
    return out_re, out_im


def status_string(status: int) -> str:
    return library().fwt_status_string(int(status)).decode()


def last_cuda_error() -> int:
    return library().fwt_last_cuda_error()


def plan_factors(n: int, dtype: str) -> list[int]:
    buf = (ctypes.c_int * 3)()
    k = library().fwt_plan_factors(int(n), DTYPES[dtype], buf, 3)
    if k < 0:
        raise ValueError(f"no plan for n={n} dtype={dtype}")
    return list(buf)[:k]


def plan_passes(n: int, dtype: str) -> int:
    return library().fwt_plan_passes(int(n), DTYPES[dtype])


def set_plan(n: int, dtype: str, factors) -> None:
    """Override the Kronecker factors for (n, dtype); ``None`` or [] restores the default."""
    factors = list(factors or [])
    buf = (ctypes.c_int * max(1, len(factors)))(*factors)
    st = library().fwt_set_plan(int(n), DTYPES[dtype], len(factors), buf)
    if st != FWT_OK:
        raise FwtError(st, f"fwt_set_plan(n={n}, {dtype}, {factors})")


def set_column_bytes(dtype: str, nbytes: int) -> None:
    """Column-pass segment width (16, 32, 64 or 128 bytes; 0 = chosen per plan, the
    default) for later plans of ``dtype``."""
    st = library().fwt_set_column_bytes(DTYPES[dtype], int(nbytes))
    if st != FWT_OK:
        raise FwtError(st, f"fwt_set_column_bytes({dtype}, {nbytes})")


def column_bytes(dtype: str) -> int:
    return library().fwt_get_column_bytes(DTYPES[dtype])


TMA_NEVER, TMA_AUTO, TMA_ALWAYS = 0, 1, 2


def set_tma(mode: int) -> None:
    """Column-pass staging: TMA_ALWAYS, TMA_NEVER (vector loads) or TMA_AUTO (default)."""
    st = library().fwt_set_tma(int(mode))
    if st != FWT_OK:
        raise FwtError(st, f"fwt_set_tma({mode})")


def tma() -> int:
    return library().fwt_get_tma()


def set_pdl(mode: int) -> None:
    """Launch pass kernels with programmatic stream serialisation (1, the default:
    a kernel may be scheduled while the previous one on the stream finishes, and
    waits for it before touching memory) or plainly (0); results are identical."""
    st = library().fwt_set_pdl(int(mode))
    if st != FWT_OK:
        raise FwtError(st, f"fwt_set_pdl({mode})")


def pdl() -> int:
    return library().fwt_get_pdl()


CLUSTER_NEVER, CLUSTER_AUTO, CLUSTER_FROM_14 = 0, 1, 2


def set_cluster(mode: int) -> None:
    """One-pass cluster transforms of 2^14..2^18-element fp32/int32 vectors:
    CLUSTER_AUTO (default: 4-byte n = 15..17, fp64 n = 14 on CTA pairs), CLUSTER_FROM_14
    (4-byte n = 14..18) or CLUSTER_NEVER."""
    st = library().fwt_set_cluster(int(mode))
    if st != FWT_OK:
        raise FwtError(st, f"fwt_set_cluster({mode})")


def cluster() -> int:
    return library().fwt_get_cluster()


def set_tma_l2_promotion(nbytes: int) -> None:
    """L2 sector promotion of TMA column-tile copies: 0, 64, 128 (default) or 256 bytes."""
    st = library().fwt_set_tma_l2_promotion(int(nbytes))
    if st != FWT_OK:
        raise FwtError(st, f"fwt_set_tma_l2_promotion({nbytes})")


def device_status() -> int:
    """FWT_ERR_TIMEOUT if a kernel gave up a bounded TMA wait since the last call."""
    return library().fwt_device_status()


def selftest_bounded_wait(stream=None) -> int:
    """Enqueue the bounded-wait self-test (one CTA, ~1 s); see fwt_selftest_bounded_wait."""
    return library().fwt_selftest_bounded_wait(stream)


def set_l2_chunk_bytes(nbytes: int) -> None:
    """L2 chunk budget for multi-pass transforms: -1 = half the L2, 0 = off (default)."""
    st = library().fwt_set_l2_chunk_bytes(int(nbytes))
    if st != FWT_OK:
        raise FwtError(st, f"fwt_set_l2_chunk_bytes({nbytes})")


def l2_chunk_bytes() -> int:
    return library().fwt_get_l2_chunk_bytes()


def selfcheck() -> int:
    return library().fwt_selfcheck()


class PassTrace:
    """Record a CUDA event pair around every pass this thread launches.

    ``events`` are ``torch.cuda.Event(enable_timing=True)`` objects (two per
    traced pass).  Use as a context manager; ``durations_ms()`` afterwards gives
    one device time per traced pass, in launch order."""

    def __init__(self, events):
        self.events = list(events)
        for e in self.events:
            e.record()  # makes torch create the underlying cudaEvent_t
        self._handles = (ctypes.c_void_p * len(self.events))(*[e.cuda_event for e in self.events])
        self.count = 0

    def __enter__(self):
        st = library().fwt_trace_events(self._handles, len(self.events))
        if st != FWT_OK:
            raise FwtError(st, "fwt_trace_events")
        return self

    def __exit__(self, *exc):
        self.count = library().fwt_trace_count()
        library().fwt_trace_events(None, 0)
        return False

    def durations_ms(self):
        return [self.events[2 * i].elapsed_time(self.events[2 * i + 1])
                for i in range(self.count // 2)]


# ---- tensor-level wrapper ---------------------------------------------------------

_ENTRY = {"c32": fwt_batched_c32, "c64": fwt_batched_c64, "i32": fwt_batched_i32}
_BITS_ENTRY = {"c32": fwt_bits_c32, "c64": fwt_bits_c64, "i32": fwt_bits_i32}
_HOST_ENTRY = {"c32": fwt_host_c32, "c64": fwt_host_c64, "i32": fwt_host_i32}
_MASK_ENTRY = {"c32": fwt_mask_c32, "c64": fwt_mask_c64, "i32": fwt_mask_i32}


_torch = None
_DTYPE_KEYS = None


def _torch_mod():
    global _torch, _DTYPE_KEYS
    if _torch is None:
        import torch

        _DTYPE_KEYS = {torch.float32: "c32", torch.float64: "c64", torch.int32: "i32"}
        _torch = torch
    return _torch


def _dtype_key(t) -> str:
    _torch_mod()
    key = _DTYPE_KEYS.get(t.dtype)
    if key is None:
        raise TypeError(f"unsupported dtype {t.dtype}: use float32, float64 or int32")
    return key


_raw_stream = None
_get_device = None


def _stream_handle(stream, device):
    """The raw cudaStream_t of ``stream`` (default: the current PyTorch stream of
    ``device``)."""
    global _raw_stream
    if stream is not None:
        return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)
    if _raw_stream is None:
        torch = _torch_mod()
        _raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None) or (
            lambda index: torch.cuda.current_stream(index).cuda_stream)
    return _raw_stream(device.index)


def _on_device(device, call):
    """Runs ``call`` with ``device`` current (switching only when it is not)."""
    global _get_device
    if _get_device is None:
        torch = _torch_mod()
        _get_device = getattr(torch._C, "_cuda_getDevice", None) or torch.cuda.current_device
    if device.index == _get_device():
        return call()
    with _torch_mod().cuda.device(device):
        return call()


def transform(re, im=None, out_re=None, out_im=None, normalize: bool = True, stream=None,
              bits=None, mask=None):
    """Transform the rows of ``re`` / ``im`` (CUDA tensors of shape (batch, 2^n)).

    Outputs are new tensors unless ``out_re`` / ``out_im`` are given (they may be
    the inputs themselves, for an in-place transform).  ``im`` may be None only
    for int32 (real-only input).  Runs on ``stream`` (default: the current
    PyTorch stream); the call does not synchronise.  ``bits=(lo, nbits)``
    transforms index bits [lo, lo + nbits) only (I (x) H_nbits (x) I); ``mask``
    (an int below 2^n) transforms the index bits set in it.  Returns
    (out_re, out_im).
    """
    torch = _torch or _torch_mod()
    key = _dtype_key(re)
    dtype, shape, device = re.dtype, re.shape, re.device
    if device.type != "cuda":
        raise ValueError("transform() needs CUDA tensors; use transform_host() for host arrays")
    if len(shape) != 2:
        raise ValueError("expected a (batch, 2^n) tensor")
    batch, N = shape
    n = int(N).bit_length() - 1
    if N < 1 or (1 << n) != N:
        raise ValueError(f"row length {N} is not a power of two")
    if bits is not None and mask is not None:
        raise ValueError("give bits or mask, not both")
    if not re.is_contiguous():
        raise ValueError("tensors must be contiguous")
    # outputs made here match re; tensors given by the caller are checked
    given = [t for t in (im, out_re, out_im) if t is not None]
    if out_re is None:
        out_re = torch.empty_like(re)
    if im is not None and out_im is None:
        out_im = torch.empty_like(im)
    for t in given:
        if t.dtype != dtype or t.shape != shape or t.device != device:
            raise ValueError("re, im and outputs must share dtype, shape and device")
        if not t.is_contiguous():
            raise ValueError("tensors must be contiguous")
    handle = _stream_handle(stream, device)
    ptrs = (re.data_ptr(), im.data_ptr() if im is not None else None, out_re.data_ptr(),
            out_im.data_ptr() if out_im is not None else None)
    if mask is not None:
        call = lambda: _MASK_ENTRY[key](*ptrs, n, batch, int(mask), normalize, handle)  # noqa: E731
    elif bits is None:
        call = lambda: _ENTRY[key](*ptrs, n, batch, normalize, handle)  # noqa: E731
    else:
        call = lambda: _BITS_ENTRY[key](*ptrs, n, batch, int(bits[0]), int(bits[1]),  # noqa: E731
                                        normalize, handle)
    st = _on_device(device, call)
    if st != FWT_OK:
        what = (f"fwt_mask_{key}(mask={mask:#x})" if mask is not None else
                f"fwt_batched_{key}" if bits is None else f"fwt_bits_{key}(bits={tuple(bits)})")
        raise FwtError(st, f"{what}(n={n}, batch={batch})")
    return out_re, out_im


def transform_host(re, im=None, out_re=None, out_im=None, normalize: bool = True, device="cuda",
                   stream=None, workspace=None, synchronize: bool = True):
    """End-to-end transform of HOST tensors through ``fwt_host_*``: the batch is
    copied to ``device`` in chunks, transformed and copied back, the three stages of
    successive chunks overlapping.

    ``re`` / ``im`` are contiguous CPU tensors of shape (batch, 2^n); page-locked
    (pinned) memory lets the copies overlap.  Outputs are new host tensors (pinned
    when the input is) unless ``out_re`` / ``out_im`` are given (they may be the
    inputs).  ``workspace`` is a CUDA tensor of at least
    ``fwt_host_workspace_bytes(...)`` bytes for full overlap (allocated here when
    None).  With ``synchronize`` the call returns once the outputs are complete;
    otherwise they are complete when ``stream`` reaches the call.  Returns
    (out_re, out_im).
    """
    import torch

    key = _dtype_key(re)
    if re.is_cuda or (im is not None and im.is_cuda):
        raise ValueError("transform_host() takes host tensors; use transform() for CUDA tensors")
    if re.dim() != 2:
        raise ValueError("expected a (batch, 2^n) tensor")
    batch, N = re.shape
    n = int(N).bit_length() - 1
    if N < 1 or (1 << n) != N:
        raise ValueError(f"row length {N} is not a power of two")
    if out_re is None:
        out_re = torch.empty(re.shape, dtype=re.dtype, pin_memory=re.is_pinned())
    if im is not None and out_im is None:
        out_im = torch.empty(im.shape, dtype=im.dtype, pin_memory=im.is_pinned())
    for t in (re, im, out_re, out_im):
        if t is None:
            continue
        if t.dtype != re.dtype or t.shape != re.shape or t.is_cuda:
            raise ValueError("re, im and outputs must be host tensors of one dtype and shape")
        if not t.is_contiguous():
            raise ValueError("tensors must be contiguous")
    device = torch.device(device)
    dt = DTYPES[key]
    if workspace is None:
        nbytes = fwt_host_workspace_bytes(dt, n, max(batch, 1), im is not None)
        workspace = torch.empty(max(nbytes, 16), dtype=torch.uint8, device=device)
    if not workspace.is_cuda or not workspace.is_contiguous():
        raise ValueError("workspace must be a contiguous CUDA tensor")
    if stream is None:
        stream = torch.cuda.current_stream(workspace.device)
    handle = stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)
    ws_bytes = workspace.numel() * workspace.element_size()
    with torch.cuda.device(workspace.device):
        st = _HOST_ENTRY[key](re.data_ptr(), im.data_ptr() if im is not None else None,
                              out_re.data_ptr(), out_im.data_ptr() if out_im is not None else None,
                              n, batch, normalize, workspace.data_ptr(), ws_bytes, handle)
    if st != FWT_OK:
        raise FwtError(st, f"fwt_host_{key}(n={n}, batch={batch}, workspace={ws_bytes} B)")
    if synchronize:
        if hasattr(stream, "synchronize"):
            stream.synchronize()
        else:
            torch.cuda.synchronize(workspace.device)
    return out_re, out_im
