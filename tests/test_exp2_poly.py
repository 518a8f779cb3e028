"""The kernels' polynomial exp2 (range reduction to [-1/2, 1/2] plus a fitted
degree-3 minimax polynomial) against CUDA's exp2f on the GPU.

Bound: relative error <= 1e-4 over the inputs the kernels feed it
(x in [-100, 8]); the fit itself guarantees 7.5e-5 (fit_exp2_poly.py). Far
below bf16's 2^-9 rounding of the probabilities that consume it."""

import ctypes
import os
import subprocess

import numpy as np
import pytest

from conftest import ROOT

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def checker(tmp_path_factory):
    d = tmp_path_factory.mktemp("exp2")
    so = str(d / "exp2_poly_check.so")
    src = os.path.join(ROOT, "tests", "cuda", "exp2_poly_check.cu")
    inc = os.path.join(ROOT, "exact_io_aware_33_gb300", "csrc")
    subprocess.run(["nvcc", "-shared", "-Xcompiler", "-fPIC", "-O3", "-gencode",
                    "arch=compute_103a,code=sm_103a", "-I" + inc, src, "-o", so], check=True)
    lib = ctypes.CDLL(so)
    lib.exp2_poly_check.argtypes = [ctypes.c_void_p] * 3 + [ctypes.c_int]
    return lib


def test_polynomial_exp2_against_exp2f(checker):
    x = torch.cat([torch.linspace(-100.0, 8.0, 2_000_000),
                   torch.arange(-100, 9, dtype=torch.float32) + 0.5,      # rounding ties
                   torch.arange(-100, 9, dtype=torch.float32)]).cuda()     # integers
    if x.numel() % 2:
        x = torch.cat([x, x[:1]])
    poly = torch.empty_like(x)
    ref = torch.empty_like(x)
    assert checker.exp2_poly_check(x.data_ptr(), poly.data_ptr(), ref.data_ptr(), x.numel()) == 0
    rel = ((poly.double() - ref.double()).abs() / ref.double()).max().item()
    assert rel <= 1e-4, rel
    # far below the clamp the result is tiny and non-negative
    y = torch.tensor([-200.0, -1e30, float("-inf"), -126.0], device="cuda")
    p2, r2 = torch.empty_like(y), torch.empty_like(y)
    assert checker.exp2_poly_check(y.data_ptr(), p2.data_ptr(), r2.data_ptr(), 4) == 0
    assert (p2 >= 0).all() and (p2 < 1e-37).all()
