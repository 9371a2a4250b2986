"""A bounded wait that runs out (failure detection without a GPU fault).

Compiles tests/cuda/wait_timeout_probe.cu, which runs the library's own
mbarrier wait helper on a barrier nothing ever completes.  The wait must give
up after the library's limit (2 s), report the timeout bit in the error word,
and return; the context must stay usable, which a GEMM call afterwards
checks against the oracle.
"""
import ctypes
import os
import subprocess

import pytest
import torch

from dense_gemm_12_gb300 import _build
from dense_gemm_12_gb300.workloads import make_inputs
from gpu_helpers import oracle_sgemm, ratio, run_sgemm, tol_fp32

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))
TIMEOUT_BIT = 1  # kErrWaitTimeout


@pytest.fixture(scope="module")
def probe(tmp_path_factory, cuda_device):
    out = tmp_path_factory.mktemp("probe") / "libwaitprobe.so"
    subprocess.run([_build.nvcc_path(), *_build.ARCH, "-O2", "-std=c++17", "-Xcompiler", "-fPIC",
                    "-shared", os.path.join(HERE, "cuda", "wait_timeout_probe.cu"), "-o", str(out)],
                   check=True)
    lib = ctypes.CDLL(str(out))
    lib.probe_wait_timeout.restype = ctypes.c_int
    lib.probe_wait_timeout.argtypes = [ctypes.POINTER(ctypes.c_int), ctypes.POINTER(ctypes.c_int),
                                       ctypes.POINTER(ctypes.c_uint),
                                       ctypes.POINTER(ctypes.c_double)]
    return lib


def test_wait_runs_out_and_reports(probe, gemm_lib):
    completed, aborted = ctypes.c_int(-1), ctypes.c_int(-1)
    err, secs = ctypes.c_uint(0), ctypes.c_double(0)
    rc = probe.probe_wait_timeout(ctypes.byref(completed), ctypes.byref(aborted),
                                  ctypes.byref(err), ctypes.byref(secs))
    assert rc == 0
    assert completed.value == 0          # the wait gave up
    assert aborted.value == 1            # and raised the CTA abort flag
    assert err.value & TIMEOUT_BIT       # and recorded the timeout
    assert 1.5 <= secs.value <= 20.0     # after the 2 s limit, not never
    # the context is still usable
    M, N, K = 200, 300, 400
    A, B, C = make_inputs(M, N, K, seed=3)
    out, st, _, _, _ = run_sgemm(A, B, C, 1.0, 0.5)
    assert st == 0
    _, ref64, den = oracle_sgemm(A, B, C, 1.0, 0.5)
    assert ratio(out, ref64, den) <= tol_fp32(K)
    assert torch.cuda.is_available()
