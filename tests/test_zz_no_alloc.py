"""gemm_bf16gemm_decode_static: the decode GEMM for callers that cannot
allocate device memory (its scratch lives in a fixed array the library owns).

Each case calls the new entry point through the C ABI twice in a row, each
time on a fresh copy of the same C, and checks both results against the
result of gemm_bf16gemm on the same inputs, within the bf16 bound used by the
other tests: 8e-3 of |alpha| (|A||B|)_ij + |beta||C_ij|.  The cases cover the
whole-column-group layout (no partial sums) and the split-K layout, which
uses the fixed array for partial sums and arrival counters.  This file is
named so that pytest collects it after every other test file.
"""
import pytest
import torch

import dense_gemm_12_gb300 as g
from dense_gemm_12_gb300.workloads import WORKLOADS, make_inputs, workload_inputs
from gpu_helpers import TOL_BF16, check_device_error, oracle_bf16, ratio

pytestmark = pytest.mark.gpu

UNSUPPORTED = 3


@pytest.fixture(scope="module", autouse=True)
def _lib(gemm_lib, cuda_device):
    yield


def _call(fn, A, B, C0, alpha, beta):
    M, K = A.shape
    N = B.shape[1]
    dA, dB = A.cuda(), B.cuda()
    dC = C0.clone().cuda()
    st = fn(M, N, K, alpha, dA.data_ptr(), K, dB.data_ptr(), N, beta, dC.data_ptr(), N, 0)
    torch.cuda.synchronize()
    return st, dC.cpu()


CASES = [
    # the decode workload: one CTA per 128-column group, no partial sums
    ("decode_16x12288x4096", None),
    # few column groups: k split over the SMs, partial sums and counters
    ("split_16x1024x4096", (16, 1024, 4096)),
    ("split_5x384x8192", (5, 384, 8192)),
]


@pytest.mark.parametrize("name,shape", CASES, ids=[c[0] for c in CASES])
def test_static_scratch_matches_allocating_entry_point(name, shape):
    if shape is None:
        w = WORKLOADS["decode_16"]
        A, B, C0 = workload_inputs(w)
        alpha, beta = w.alpha, w.beta
    else:
        M, N, K = shape
        A, B, C0 = make_inputs(M, N, K, ("normal", 1.0), ("normal", 0.02), ("uniform", None),
                               seed=M + N + K, dtype="bf16")
        alpha, beta = 0.75, 1.0
    st, ref = _call(g.gemm_bf16gemm, A, B, C0, alpha, beta)
    assert st == 0
    _, _, den = oracle_bf16(A, B, C0, alpha, beta)
    for _ in range(2):  # two calls in a row share the same fixed array
        st, out = _call(g.gemm_bf16gemm_decode_static, A, B, C0, alpha, beta)
        assert st == 0, g.gemm_status_string(st)
        assert ratio(out, ref.numpy().astype("float64"), den) <= TOL_BF16
    check_device_error()


def test_static_scratch_rejects_what_does_not_fit():
    # 512 column groups with K = 64 need more partial-sum space than the
    # fixed array holds: refused before anything is launched.
    M, N, K = 16, 65536, 64
    A, B, C0 = make_inputs(M, N, K, seed=1, dtype="bf16")
    st, out = _call(g.gemm_bf16gemm_decode_static, A, B, C0, 1.0, 1.0)
    assert st == UNSUPPORTED
    assert torch.equal(out, C0)
    # not decode-shaped: refused too
    A, B, C0 = make_inputs(17, 256, 128, seed=2, dtype="bf16")
    st, out = _call(g.gemm_bf16gemm_decode_static, A, B, C0, 1.0, 1.0)
    assert st == UNSUPPORTED
    assert torch.equal(out, C0)
