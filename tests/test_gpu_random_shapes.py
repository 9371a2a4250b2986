"""Seeded random shapes, scalars, leading dimensions and base offsets against
the oracle: every kernel path automatic dispatch can take for small and
medium problems (CUDA-core fp32 with TMA, generic or staged loads; bf16
decode, single-CTA and CTA-pair tensor-core kernels, staged bf16 operands),
with sentinel-filled padding that must stay untouched.

Integer inputs must match the oracle bit for bit; random inputs within
2e-6 sqrt(K) (fp32) or 8e-3 (bf16) of |alpha| (|A||B|)_ij + |beta| |C_ij|.
"""
import math

import numpy as np
import pytest
import torch

from dense_gemm_12_gb300.workloads import make_inputs
from gpu_helpers import (TOL_BF16, check_device_error, oracle_bf16, oracle_sgemm, ratio,
                         run_bf16gemm, run_sgemm, tol_fp32)

pytestmark = pytest.mark.gpu

INT = ("int", None)


@pytest.fixture(scope="module", autouse=True)
def _lib(gemm_lib, cuda_device):
    yield


def _cases(seed, count, m_max, bf16):
    rng = np.random.default_rng(seed)
    out = []
    for i in range(count):
        M = int(math.exp(rng.uniform(0, math.log(m_max))))
        N = int(math.exp(rng.uniform(0, math.log(1500))))
        K = int(math.exp(rng.uniform(0, math.log(1500))))
        alpha = float(rng.choice([1.0, -0.75, 1.5, 0.0], p=[0.4, 0.25, 0.25, 0.1]))
        beta = float(rng.choice([0.0, 1.0, -0.5, 0.25]))
        pads = [int(rng.integers(0, 9)) if rng.random() < 0.5 else 0 for _ in range(3)]
        offs = [int(rng.integers(0, 4)) if rng.random() < 0.3 else 0 for _ in range(3)]
        integer = bool(rng.random() < 0.4)
        out.append((i, M, N, K, alpha, beta, pads, offs, integer))
    return out


def _check(bf16, case):
    i, M, N, K, alpha, beta, pads, offs, integer = case
    dist = (INT, INT, INT) if integer else (("normal", 1.0), ("normal", 1.0), ("uniform", None))
    A, B, C = make_inputs(M, N, K, *dist, seed=1000 + i, dtype="bf16" if bf16 else "f32")
    run = run_bf16gemm if bf16 else run_sgemm
    out, st, dA, dB, dC = run(A, B, C, alpha, beta, lda=K + pads[0], ldb=N + pads[1],
                              ldc=N + pads[2], offsets=tuple(offs))
    assert st == 0, case
    ref32, ref64, den = (oracle_bf16 if bf16 else oracle_sgemm)(A, B, C, alpha, beta)
    if integer:
        # small integers and dyadic scalars: every partial sum and the result
        # are exact in fp32
        assert np.array_equal(out.numpy(), ref32), case
    else:
        tol = TOL_BF16 if bf16 else tol_fp32(K)
        assert ratio(out, ref64, den) <= tol, case
    assert dA.untouched_outside() and dB.untouched_outside() and dC.untouched_outside(), case


@pytest.mark.parametrize("case", _cases(11, 40, 1500, bf16=False), ids=lambda c: "f32_%d" % c[0])
def test_fp32_random_shapes(case):
    _check(False, case)


@pytest.mark.parametrize("case", _cases(12, 40, 400, bf16=True), ids=lambda c: "bf16_%d" % c[0])
def test_bf16_random_shapes(case):
    _check(True, case)


def test_random_shapes_left_no_device_error():
    check_device_error()
