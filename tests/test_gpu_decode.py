"""Decode-shaped bf16 GEMM (M <= 16) on the GPU: the swapped-operand tcgen05
kernel with split-K and the fixed-order fix-up, against the CPU oracle.

Bound: 8e-3 of |alpha| (|A||B|)_ij + |beta||C_ij| (same bf16-rounded inputs);
bit-exact on small integers; bitwise identical across repeated launches (the
partial sums are added in k order whatever order the CTAs finish in).
"""
import numpy as np
import pytest
import torch

import dense_gemm_12_gb300 as g
from dense_gemm_12_gb300.workloads import WORKLOADS, make_inputs, workload_inputs
from gpu_helpers import TOL_BF16, check_device_error, oracle_bf16, ratio, run_bf16gemm

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib(gemm_lib, cuda_device):
    yield


def test_decode_full_workload():
    w = WORKLOADS["decode_16"]
    A, B, C = workload_inputs(w)
    assert g.gemm_select_path(1, w.M, w.N, w.K, w.alpha, 1 << 20, w.K, 1 << 20, w.N) == "tc_decode"
    out, st, _, _, dC = run_bf16gemm(A, B, C, w.alpha, w.beta)
    assert st == 0
    check_device_error()
    _, ref64, den = oracle_bf16(A, B, C, w.alpha, w.beta)
    r = ratio(out, ref64, den)
    assert r <= TOL_BF16, r
    assert dC.untouched_outside()


def test_decode_integers_exact():
    M, N, K = 16, 1536, 2048
    A, B, C = make_inputs(M, N, K, ("int", None), ("int", None), ("int", None), seed=3,
                          dtype="bf16")
    out, st, _, _, _ = run_bf16gemm(A, B, C, 1.0, 1.0)
    assert st == 0
    ref32, _, _ = oracle_bf16(A, B, C, 1.0, 1.0)
    assert np.array_equal(out.numpy(), ref32)


@pytest.mark.parametrize("M", [1, 2, 5, 8, 15, 16])
@pytest.mark.parametrize("N,K", [(128, 64), (1000, 1000), (12288, 4096), (200, 8192), (4096, 72)])
def test_decode_shapes(M, N, K):
    if N * K > 12288 * 4096 // 2 and M not in (1, 16):
        pytest.skip("large shape checked at M = 1 and 16 only")
    A, B, C = make_inputs(M, N, K, ("normal", 1.0), ("normal", 0.02), ("uniform", None),
                          seed=M * 1000 + N + K, dtype="bf16")
    out, st, _, _, dC = run_bf16gemm(A, B, C, 0.5, 1.0)
    assert st == 0
    _, ref64, den = oracle_bf16(A, B, C, 0.5, 1.0)
    assert ratio(out, ref64, den) <= TOL_BF16
    assert dC.untouched_outside()
    check_device_error()


@pytest.mark.parametrize("N,K", [(128, 8192), (384, 4096), (256, 16384), (1000, 2048)])
def test_decode_many_contributors(N, K):
    # few column groups, long k: up to ~128 CTAs add into one group, which
    # exercises the arrival-counter hand-off and both fix-up paths
    M = 16
    A, B, C = make_inputs(M, N, K, ("normal", 1.0), ("normal", 0.02), ("uniform", None),
                          seed=N + K, dtype="bf16")
    outs = []
    for _ in range(3):
        out, st, _, _, dC = run_bf16gemm(A, B, C, 1.25, -0.75)
        assert st == 0
        outs.append(out)
    _, ref64, den = oracle_bf16(A, B, C, 1.25, -0.75)
    assert ratio(outs[0], ref64, den) <= TOL_BF16
    for o in outs[1:]:
        assert torch.equal(o.view(torch.int32), outs[0].view(torch.int32))
    check_device_error()


def test_decode_beta_zero_nan():
    M, N, K = 16, 2048, 1024
    A, B, _ = make_inputs(M, N, K, seed=7, dtype="bf16")
    C = torch.full((M, N), float("nan"))
    out, st, _, _, _ = run_bf16gemm(A, B, C, 1.0, 0.0)
    assert st == 0 and torch.isfinite(out).all()


def test_decode_deterministic_and_counters_reset():
    w = WORKLOADS["decode_16"]
    A, B, C = workload_inputs(w)
    outs = [run_bf16gemm(A, B, C, w.alpha, w.beta)[0] for _ in range(5)]
    for o in outs[1:]:
        assert torch.equal(o.view(torch.int32), outs[0].view(torch.int32))
    check_device_error()
