"""bf16-input / fp32-output GEMM on the GPU (tcgen05 tensor-core kernel, and the
CUDA-core fallback for operands TMA cannot describe) against the CPU oracle
run on the same bf16-rounded inputs.

Bound per element: |C - C_ref| <= 8e-3 * (|alpha| (|A||B|)_ij + |beta||C_ij|).
Small-integer inputs are exact in bf16 and every partial sum is an integer
below 2^24, so those cases must match bit for bit.
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


def _inputs(M, N, K, seed, dist=("normal", 1.0), dist_c=("uniform", None)):
    return make_inputs(M, N, K, dist, dist, dist_c, seed=seed, dtype="bf16")


def test_single_tile_integers_exact():
    # one 128 x 256 tile, one k-block, on the single-CTA tile kernel (pinned:
    # automatic dispatch sends this shape to the decode kernel): exercises the
    # descriptors directly
    M, N, K = 128, 256, 64
    A, B, C = make_inputs(M, N, K, ("int", None), ("int", None), ("int", None), seed=1,
                          dtype="bf16")
    dA, dB, dC = A.cuda(), B.cuda(), torch.full((M, N), float("nan"), device="cuda")
    st = g.gemm_bf16gemm_config(M, N, K, 1.0, dA.data_ptr(), K, dB.data_ptr(), N, 0.0,
                                dC.data_ptr(), N, {"kernel": "single_cta"}, 0)
    torch.cuda.synchronize()
    assert st == 0
    ref32, _, _ = oracle_bf16(A, B, C, 1.0, 0.0)
    assert np.array_equal(dC.cpu().numpy(), ref32)
    check_device_error()


def test_multi_tile_integers_exact():
    M, N, K = 384, 768, 512
    A, B, C = make_inputs(M, N, K, ("int", None), ("int", None), ("int", None), seed=2,
                          dtype="bf16")
    out, st, _, _, _ = run_bf16gemm(A, B, C, 1.5, -0.5)
    assert st == 0
    ref32, _, _ = oracle_bf16(A, B, C, 1.5, -0.5)
    assert np.array_equal(out.numpy(), ref32)


@pytest.mark.parametrize("M,N,K", [
    (17, 8, 8), (128, 256, 64), (129, 264, 72), (300, 520, 200), (1000, 1000, 1000),
    (255, 257 + 7, 1999 + 1), (513, 1032, 4096), (33, 2048, 136),
])
def test_ragged_tensor_core(M, N, K):
    A, B, C = _inputs(M, N, K, seed=M + N + K)
    out, st, _, _, dC = run_bf16gemm(A, B, C, 0.7, 0.3)
    assert st == 0
    # small M runs the decode kernel (bound by streaming B): M <= 32; M <= 128
    # (two row blocks above 64) up to N = 16384; M <= 512 (row blocks of 64)
    # while column groups x row blocks stay within 128 (160 for K >= 4096).
    # The tile kernels at small M are covered with pinned configurations in
    # test_gpu_config.py
    units = -(-N // 128) * -(-M // 64)
    decode = M <= 32 or (M <= 128 and N <= 16384) or \
        (M <= 512 and units <= (160 if K >= 4096 else 128))
    single = g.gemm_get_config(1, M, N, K)[0]["kernel"] == "single_cta"
    expect = "tc_decode" if decode else "tc_bf16" if single else "tc_bf16_pair"
    assert g.gemm_select_path(1, M, N, K, 0.7, 1 << 20, K, 1 << 20, N) == expect
    _, ref64, den = oracle_bf16(A, B, C, 0.7, 0.3)
    r = ratio(out, ref64, den)
    assert r <= TOL_BF16, r
    assert dC.untouched_outside()
    check_device_error()


@pytest.mark.parametrize("M,N,K", [(50, 70, 30), (129, 131, 257), (17, 9, 1999)])
def test_unaligned_fallback(M, N, K):
    A, B, C = _inputs(M, N, K, seed=M * N)
    # odd pitches: TMA cannot describe them, the CUDA-core kernel widens bf16
    out, st, _, _, dC = run_bf16gemm(A, B, C, 1.0, 1.0, lda=K + 1, ldb=N + 3, ldc=N + 1)
    assert st == 0
    assert g.gemm_select_path(1, M, N, K, 1.0, 1 << 20, K + 1, 1 << 20, N + 3) == "simt_bf16"
    _, ref64, den = oracle_bf16(A, B, C, 1.0, 1.0)
    assert ratio(out, ref64, den) <= TOL_BF16
    assert dC.untouched_outside()


def test_padded_pitches_tensor_core():
    M, N, K = 200, 304, 264
    A, B, C = _inputs(M, N, K, seed=21)
    out, st, dA, dB, dC = run_bf16gemm(A, B, C, 2.0, -1.0, lda=K + 8, ldb=N + 16, ldc=N + 5)
    assert st == 0
    _, ref64, den = oracle_bf16(A, B, C, 2.0, -1.0)
    assert ratio(out, ref64, den) <= TOL_BF16
    assert dA.untouched_outside() and dB.untouched_outside() and dC.untouched_outside()


def test_beta_zero_ignores_nan_c():
    M, N, K = 256, 512, 128
    A, B, _ = _inputs(M, N, K, seed=22)
    C = torch.full((M, N), float("nan"))
    out, st, _, _, _ = run_bf16gemm(A, B, C, 1.0, 0.0)
    assert st == 0 and torch.isfinite(out).all()


def test_deterministic_repeats():
    M, N, K = 640, 768, 1024
    A, B, C = _inputs(M, N, K, seed=23)
    outs = [run_bf16gemm(A, B, C, 1.0, 0.5)[0] for _ in range(5)]
    for o in outs[1:]:
        assert torch.equal(o.view(torch.int32), outs[0].view(torch.int32))


def test_full_8192_sampled_rows():
    w = WORKLOADS["bf16_8192"]
    A, B, C = workload_inputs(w)
    out, st, _, _, dC = run_bf16gemm(A, B, C, w.alpha, w.beta)
    assert st == 0
    check_device_error()
    gen = torch.Generator().manual_seed(0)
    idx = torch.randperm(w.M, generator=gen)[:24].sort().values
    # tile (128) and CTA-pair tile (256) boundaries
    idx = torch.cat([idx, torch.tensor([0, 127, 128, 255, 256, 383, 384, w.M - 1])]).unique()
    _, ref64, den = oracle_bf16(A[idx].contiguous(), B, C[idx].contiguous(), w.alpha, w.beta)
    r = ratio(out[idx], ref64, den)
    assert r <= TOL_BF16, r
    assert dC.untouched_outside()


# ---- the last round's work items cut along k (split-K tail) ---------------
# The plan depends on how many CTAs (pairs) are resident and on the sweep's
# table; each case asserts that it really splits (the shapes lie in classes
# the table leaves to the cost model).

@pytest.mark.parametrize("M,N,K", [
    (512, 10240, 4096),   # pair kernel: 80 pair tiles on at most 76 clusters
    (128, 16640, 4096),   # single-CTA kernel: 65 tiles on 152 SMs
])
def test_split_integers_exact(M, N, K):
    # |partial sums| <= 16 K < 2^24: exact in fp32 in any order and any split
    assert g.gemm_split_parts(1, M, N, K) > 1
    A, B, C = make_inputs(M, N, K, ("int", None), ("int", None), ("int", None), seed=31,
                          dtype="bf16")
    out, st, _, _, dC = run_bf16gemm(A, B, C, 1.5, -0.5)
    assert st == 0
    ref32, _, _ = oracle_bf16(A, B, C, 1.5, -0.5)
    assert np.array_equal(out.numpy(), ref32)
    assert dC.untouched_outside()
    check_device_error()


@pytest.mark.parametrize("M,N,K", [
    (512, 10240, 4096),   # pair kernel
    (500, 10232, 4000),   # pair kernel, ragged M, N and K (last part ends on a partial k-block)
    (100, 16640, 4096),   # single-CTA kernel
])
def test_split_matches_oracle_and_repeats(M, N, K):
    assert g.gemm_split_parts(1, M, N, K) > 1
    A, B, C = _inputs(M, N, K, seed=M + K)
    outs = [run_bf16gemm(A, B, C, 0.7, 0.3)[0] for _ in range(3)]
    for o in outs[1:]:
        assert torch.equal(o.view(torch.int32), outs[0].view(torch.int32))
    gen = torch.Generator().manual_seed(2)
    idx = torch.randperm(M, generator=gen)[:48].sort().values
    idx = torch.cat([idx, torch.tensor([0, M - 1])]).unique()
    _, ref64, den = oracle_bf16(A[idx].contiguous(), B, C[idx].contiguous(), 0.7, 0.3)
    r = ratio(outs[0][idx], ref64, den)
    assert r <= TOL_BF16, r
    check_device_error()


def test_split_parts_of_the_benchmark_shapes():
    # 8192^3: 1024 pair tiles on up to 76 clusters leave a partial round
    assert g.gemm_split_parts(1, 8192, 8192, 8192) >= 1
    # decode shapes plan their own split
    assert g.gemm_split_parts(1, 16, 12288, 4096) == 1
    # fp32 4092^3: 1024 tiles on 152 SMs, tail of 112 tiles split
    assert g.gemm_split_parts(0, 4092, 4092, 4092) > 1
