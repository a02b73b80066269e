"""The Python binding's own checks, which run before any CUDA call (CPU only):
dtypes, devices, shapes and the host-buffer wrapper's argument rules."""
import os

import pytest
import torch

import walsh_hadamard_transform_gb300 as fwt


def test_transform_rejects_unsupported_dtype_and_host_tensors():
    with pytest.raises(TypeError):
        fwt.transform(torch.zeros(2, 8, dtype=torch.float16))
    with pytest.raises(ValueError, match="CUDA tensors"):
        fwt.transform(torch.zeros(2, 8), torch.zeros(2, 8))


def test_phase_transform_rejects_bad_types_and_host_angles():
    with pytest.raises(TypeError):
        fwt.phase_transform(torch.zeros(2, 8, dtype=torch.int32), torch.zeros(2, 8, dtype=torch.int32),
                            torch.zeros(8, dtype=torch.int32))
    with pytest.raises(TypeError):  # the imaginary part is required
        fwt.phase_transform(torch.zeros(2, 8), None, torch.zeros(8))
    with pytest.raises(ValueError, match="theta"):
        fwt.phase_transform(torch.zeros(2, 8), torch.zeros(2, 8), torch.zeros(8))


def test_transform_host_argument_rules():
    with pytest.raises(ValueError, match="power of two"):
        fwt.transform_host(torch.zeros(2, 6), torch.zeros(2, 6))
    with pytest.raises(ValueError, match="batch, 2\\^n"):
        fwt.transform_host(torch.zeros(8), torch.zeros(8))
    with pytest.raises(ValueError, match="one dtype and shape"):
        fwt.transform_host(torch.zeros(2, 8), torch.zeros(2, 8, dtype=torch.float64))
    with pytest.raises(ValueError, match="one dtype and shape"):
        fwt.transform_host(torch.zeros(2, 8), torch.zeros(3, 8))
    with pytest.raises(ValueError, match="contiguous"):
        fwt.transform_host(torch.zeros(8, 2).t(), torch.zeros(2, 8))
    with pytest.raises(TypeError):
        fwt.transform_host(torch.zeros(2, 8, dtype=torch.int16))


def test_dtype_codes_match_the_header():
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    text = open(os.path.join(root, "include", "fwt.h")).read()
    for name, value in (("FWT_C32", fwt.FWT_C32), ("FWT_C64", fwt.FWT_C64), ("FWT_I32", fwt.FWT_I32),
                        ("FWT_OK", fwt.FWT_OK), ("FWT_ERR_INVALID_ARG", fwt.FWT_ERR_INVALID_ARG),
                        ("FWT_ERR_MISALIGNED", fwt.FWT_ERR_MISALIGNED),
                        ("FWT_ERR_UNSUPPORTED", fwt.FWT_ERR_UNSUPPORTED),
                        ("FWT_ERR_CUDA", fwt.FWT_ERR_CUDA), ("FWT_ERR_TIMEOUT", fwt.FWT_ERR_TIMEOUT)):
        assert f"{name} = {value}" in text, name
