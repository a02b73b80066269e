"""The C ABI from a plain C99 program (tests/c_consumer.c), without Python in between.

The header must compile as C99 under -Wall -Wextra -pedantic -Werror, the program must
link against the library and the CUDA runtime, and its checks must pass: argument
errors, plans and the tile self-check on the CPU; on a GPU, transforms of device
arrays (from cudaMalloc, on a stream the program creates) and of host arrays, checked
against closed forms of the sign rule and against sums taken from the definition.
"""
import os
import shutil
import subprocess

import pytest

from walsh_hadamard_transform_gb300 import build as fbuild

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)


def _cuda_home() -> str:
    return os.path.dirname(os.path.dirname(os.path.realpath(fbuild.nvcc())))


@pytest.fixture(scope="module")
def consumer(tmp_path_factory):
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    lib = fbuild.build()
    libdir = os.path.dirname(lib)
    cuda = _cuda_home()
    cuda_lib = os.path.join(cuda, "lib64")
    exe = str(tmp_path_factory.mktemp("c_consumer") / "c_consumer")
    cmd = [cc, "-std=c99", "-O1", "-Wall", "-Wextra", "-pedantic", "-Werror", "-DFWT_CONSUMER_CUDA",
           "-I", os.path.join(ROOT, "include"), "-isystem", os.path.join(cuda, "include"),
           os.path.join(HERE, "c_consumer.c"), "-o", exe,
           "-L", libdir, "-l:" + os.path.basename(lib), "-L", cuda_lib, "-lcudart", "-lm",
           "-Wl,-rpath," + libdir, "-Wl,-rpath," + cuda_lib]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, f"C build failed:\n{' '.join(cmd)}\n{r.stdout}\n{r.stderr}"
    return exe


def test_header_needs_no_cuda_headers():
    """include/fwt.h stands alone: the program's CPU part compiles as C99 with no CUDA
    include path and no CUDA define."""
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    cmd = [cc, "-std=c99", "-fsyntax-only", "-Wall", "-Wextra", "-pedantic", "-Werror",
           "-I", os.path.join(ROOT, "include"), os.path.join(HERE, "c_consumer.c")]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr


def _run(exe, mode, timeout):
    r = subprocess.run([exe, mode], capture_output=True, text=True, timeout=timeout)
    assert r.returncode == 0, f"c_consumer {mode} exited {r.returncode}:\n{r.stdout}\n{r.stderr}"
    assert f"{mode} checks: 0 failure(s)" in r.stdout


def test_c_program_host_checks(consumer):
    _run(consumer, "cpu", timeout=120)


@pytest.mark.gpu
def test_c_program_transforms_on_gpu(consumer):
    _run(consumer, "gpu", timeout=600)
