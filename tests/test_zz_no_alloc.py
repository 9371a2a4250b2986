"""gemm_bf16gemm_decode_static: the decode GEMM for callers that cannot
allocate device memory (a server that reserves all of its device memory at
start-up, code running inside an allocator's callbacks).  Its scratch lives
in one fixed array the library owns on each device.

The kernel uses that array only when the 128-column groups outnumber the
SMs: each CTA then streams a run of groups, and the groups cut at run
boundaries meet through partial sums and arrival counters in the array.
With fewer groups (one CTA per group, or clusters adding their partial sums
in shared memory) no scratch is touched.  The cases cover both layouts; the
run-split ones are sized from the device's SM count so that they really
take that layout, and stay within the array (N <= 256 x SMs).

Each case calls the entry point through the C ABI twice in a row, each time
on a fresh copy of the same C, right after a call of another run-split shape
has left other partial sums in the array, and checks both results against
the oracle within the bf16 bound of the other tests
(8e-3 of |alpha| (|A||B|)_ij + |beta||C_ij|) and against gemm_bf16gemm on
the same inputs within the same bound.  This file is named so that pytest
collects it after every other test file.
"""
import pytest
import torch

import dense_gemm_12_gb300 as g
from dense_gemm_12_gb300.workloads import WORKLOADS, make_inputs, workload_inputs
from gpu_helpers import TOL_BF16, check_device_error, oracle_bf16, ratio

pytestmark = pytest.mark.gpu

UNSUPPORTED = 3
GROUP = 128   # columns of C per column group of the decode kernel


@pytest.fixture(scope="module", autouse=True)
def _lib(gemm_lib, cuda_device):
    yield


def _sms():
    return torch.cuda.get_device_properties(0).multi_processor_count


def _call(fn, A, B, C0, alpha, beta):
    M, K = A.shape
    N = B.shape[1]
    dA, dB = A.cuda(), B.cuda()
    dC = C0.clone().cuda()
    st = fn(M, N, K, alpha, dA.data_ptr(), K, dB.data_ptr(), N, beta, dC.data_ptr(), N, 0)
    torch.cuda.synchronize()
    return st, dC.cpu()


def _inputs(M, N, K, seed):
    return make_inputs(M, N, K, ("normal", 1.0), ("normal", 0.02), ("uniform", None),
                       seed=seed, dtype="bf16")


def _shape(name):
    """(M, N, K, run_split) of a case; run-split shapes have more column
    groups than the device has SMs."""
    sms = _sms()
    if name == "decode_16x12288x4096":
        return 16, 12288, 4096, False
    if name == "clusters_16x1024x4096":
        return 16, 1024, 4096, False
    if name == "runs_16_groups1.5xSMs_2048":
        return 16, GROUP * (sms + sms // 2), 2048, True
    if name == "runs_1_groups+5_1024":
        return 1, GROUP * (sms + 5) - 40, 1024, True
    if name == "runs_7_groups2xSMs_512":
        return 7, GROUP * 2 * sms, 512, True
    raise KeyError(name)


CASES = ["decode_16x12288x4096", "clusters_16x1024x4096", "runs_16_groups1.5xSMs_2048",
         "runs_1_groups+5_1024", "runs_7_groups2xSMs_512"]


def _dirty_the_array():
    # another run-split shape: leaves its own partial sums in the array
    sms = _sms()
    M, N, K = 9, GROUP * (sms + 20), 768
    A, B, C0 = _inputs(M, N, K, seed=99)
    st, _ = _call(g.gemm_bf16gemm_decode_static, A, B, C0, -1.25, 0.5)
    assert st == 0, g.gemm_status_string(st)


@pytest.mark.parametrize("name", CASES)
def test_static_scratch_matches_oracle_two_calls_in_a_row(name):
    M, N, K, run_split = _shape(name)
    groups = (N + GROUP - 1) // GROUP
    assert (groups > _sms()) == run_split
    if name == "decode_16x12288x4096":
        w = WORKLOADS["decode_16"]
        A, B, C0 = workload_inputs(w)
        alpha, beta = w.alpha, w.beta
    else:
        A, B, C0 = _inputs(M, N, K, seed=M + N + K)
        alpha, beta = 0.75, 1.0
    _, ref64, den = oracle_bf16(A, B, C0, alpha, beta)
    st, ref_gpu = _call(g.gemm_bf16gemm, A, B, C0, alpha, beta)
    assert st == 0
    _dirty_the_array()
    for _ in range(2):  # two calls in a row share the same fixed array
        st, out = _call(g.gemm_bf16gemm_decode_static, A, B, C0, alpha, beta)
        assert st == 0, g.gemm_status_string(st)
        assert ratio(out, ref64, den) <= TOL_BF16
        assert ratio(out, ref_gpu.numpy().astype("float64"), den) <= TOL_BF16
    check_device_error()


def test_static_scratch_integers_exact_after_other_shape():
    # small integers: every partial sum is exact in fp32, so the run-split
    # result must equal the oracle's bit for bit, whatever the array held
    sms = _sms()
    M, N, K = 16, GROUP * (sms + sms // 2) - 8, 1536
    A, B, C0 = make_inputs(M, N, K, ("int", None), ("int", None), ("int", None), seed=5,
                           dtype="bf16")
    ref32, _, _ = oracle_bf16(A, B, C0, 1.5, -0.5, want64=False)
    for _ in range(2):
        _dirty_the_array()
        st, out = _call(g.gemm_bf16gemm_decode_static, A, B, C0, 1.5, -0.5)
        assert st == 0, g.gemm_status_string(st)
        assert torch.equal(out, torch.from_numpy(ref32))
    check_device_error()


def test_static_scratch_rejects_what_does_not_fit():
    # more than twice as many column groups as SMs: the partial sums would
    # not fit in the fixed array, refused before anything is launched
    sms = _sms()
    M, N, K = 16, GROUP * (2 * sms + 1), 64
    A, B, C0 = make_inputs(M, N, K, seed=1, dtype="bf16")
    st, out = _call(g.gemm_bf16gemm_decode_static, A, B, C0, 1.0, 1.0)
    assert st == UNSUPPORTED
    assert torch.equal(out, C0)
    # not decode-shaped: refused too
    A, B, C0 = make_inputs(17, 256, 128, seed=2, dtype="bf16")
    st, out = _call(g.gemm_bf16gemm_decode_static, A, B, C0, 1.0, 1.0)
    assert st == UNSUPPORTED
    assert torch.equal(out, C0)
