"""The hardware approximations behind the INT8 epilogue's fast path stay
within the bounds its exactness argument assumes (see test_requant_fast.py):
ex2.approx.ftz.f32 within 4.8e-7 relative over every float in [-116, 116],
rcp.approx.ftz.f32 within 2.4e-7 over every float in [1, 2^116].  Measured
exhaustively on the GPU by a probe this test builds (tests/probes)."""
import ctypes
import os
import shutil
import subprocess
import tempfile

import pytest

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))


def test_hardware_approximations_within_assumed_bounds():
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    with tempfile.TemporaryDirectory() as d:
        so = os.path.join(d, "approx_error.so")
        subprocess.run([nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-shared", "-Xcompiler", "-fPIC",
                        "-o", so, os.path.join(HERE, "probes", "approx_error.cu")], check=True)
        lib = ctypes.CDLL(so)
        ex2, rcp = ctypes.c_double(-1), ctypes.c_double(-1)
        assert lib.approx_worst(ctypes.byref(ex2), ctypes.byref(rcp)) == 0
    print(f"ex2.approx worst relative error {ex2.value:.3e}, rcp.approx {rcp.value:.3e}")
    assert 0 <= ex2.value <= 4.8e-7
    assert 0 <= rcp.value <= 2.4e-7
