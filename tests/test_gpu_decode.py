"""Decode-shaped bf16 GEMM (small M, up to 512 rows in row blocks of 64) on the
GPU: the swapped-operand tcgen05 kernel with split-K and the fixed-order
fix-up, against the CPU oracle.

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


@pytest.mark.parametrize("M", [1, 2, 5, 8, 15, 16, 17, 31, 32, 40, 64])
@pytest.mark.parametrize("N,K", [(128, 64), (1000, 1000), (12288, 4096), (200, 8192), (4096, 72)])
def test_decode_shapes(M, N, K):
    # M <= 16, <= 32 and <= 64 run the kernel's 16-, 32- and 64-row instances
    if N * K > 12288 * 4096 // 2 and M not in (1, 16, 32, 64):
        pytest.skip("large shape checked at M = 1, 16, 32 and 64 only")
    A, B, C = make_inputs(M, N, K, ("normal", 1.0), ("normal", 0.02), ("uniform", None),
                          seed=M * 1000 + N + K, dtype="bf16")
    out, st, _, _, dC = run_bf16gemm(A, B, C, 0.5, 1.0)
    assert st == 0
    _, ref64, den = oracle_bf16(A, B, C, 0.5, 1.0)
    assert ratio(out, ref64, den) <= TOL_BF16
    assert dC.untouched_outside()
    check_device_error()


@pytest.mark.parametrize("M,N,K", [
    (16, 1024, 4096),   # 8 column groups: clusters of 8 CTAs
    (8, 2048, 1000),    # 16 groups: clusters of 4 (16 clusters of 8 do not fit at once)
    (16, 4096, 4096),   # 32 groups x 4
    (5, 8192, 2048),    # 64 groups x 2
    (16, 1000, 300),    # ragged N; 3 k-blocks: clusters of 2
    (3, 200, 8192),     # 2 groups x 8, the last one mostly past N
    (1, 9000, 777),     # 71 groups x 2, K not a multiple of 128
])
def test_decode_cluster_split_integers_exact(M, N, K):
    _cluster_exact(M, N, K)


@pytest.mark.parametrize("M,N,K", [
    (32, 1024, 4096),   # 32-row instance, clusters of 8
    (64, 2048, 1000),   # 64-row instance, clusters of 4
    (48, 8192, 2048),   # 64-row instance, clusters of 2
    (20, 12288, 512),   # 32-row instance, whole groups
    (64, 200, 8192),    # ragged N, clusters of 8
])
def test_decode_wide_rows_integers_exact(M, N, K):
    _cluster_exact(M, N, K)


# 64 < M <= 128: two row blocks of 64 rows (the launch's y dimension), each
# streaming B for its own rows; the second sees rows 64.. of A, C and D.
@pytest.mark.parametrize("M,N,K", [
    (65, 4096, 1024),    # one row in the second block; clusters of 2
    (96, 1024, 4096),    # 8 column groups x 2 row blocks: clusters of 4
    (128, 8192, 2048),   # 64 groups x 2 row blocks = 128 CTAs: whole groups
    (100, 1000, 296),    # ragged N and K
    (128, 200, 8192),    # 2 groups, the last one mostly past N
])
def test_decode_two_row_blocks_integers_exact(M, N, K):
    assert g.gemm_select_path(1, M, N, K, 1.0, 1 << 20, K, 1 << 20, N) == "tc_decode"
    _cluster_exact(M, N, K)


@pytest.mark.parametrize("M,N,K", [(72, 4096, 4096), (128, 8192, 1024),
                                   (96, 16384, 1024)])   # more groups than SMs per block
def test_decode_two_row_blocks_random_within_bound(M, N, K):
    A, B, C = make_inputs(M, N, K, ("normal", 1.0), ("normal", 0.02), ("uniform", None),
                          seed=M + N, dtype="bf16")
    out, st, _, _, dC = run_bf16gemm(A, B, C, 0.5, 1.0, ldc=N + 5)
    assert st == 0
    _, ref64, den = oracle_bf16(A, B, C, 0.5, 1.0)
    assert ratio(out, ref64, den) <= TOL_BF16
    assert dC.untouched_outside()
    check_device_error()


# 128 < M <= 512: three to eight row blocks, each reading all of B (from L2
# after the first); the last block may be mostly past M.
@pytest.mark.parametrize("M,N,K", [
    (160, 1000, 1024),   # 3 blocks, the last with 32 rows; ragged N
    (256, 4096, 4096),   # 4 blocks x 32 groups = 128 CTAs: whole groups
    (320, 2048, 2048),   # 5 blocks x 16 groups
    (512, 1024, 8192),   # 8 blocks x 8 groups: clusters of 2 per group
    (500, 296, 1000),    # 8 blocks, the last with 52 rows; ragged N and K
    (384, 3328, 4096),   # 26 groups > 25 SMs per block: runs of groups
])
def test_decode_many_row_blocks_integers_exact(M, N, K):
    assert g.gemm_select_path(1, M, N, K, 1.0, 1 << 20, K, 1 << 20, N) == "tc_decode"
    _cluster_exact(M, N, K)


@pytest.mark.parametrize("M,N,K", [(200, 4000, 4096), (448, 1500, 2048)])
def test_decode_many_row_blocks_random_within_bound(M, N, K):
    A, B, C = make_inputs(M, N, K, ("normal", 1.0), ("normal", 0.02), ("uniform", None),
                          seed=M + N, dtype="bf16")
    out, st, _, _, dC = run_bf16gemm(A, B, C, 0.5, 1.0, ldc=N + 5)
    assert st == 0
    _, ref64, den = oracle_bf16(A, B, C, 0.5, 1.0)
    assert ratio(out, ref64, den) <= TOL_BF16
    assert dC.untouched_outside()
    check_device_error()


def test_decode_range_boundaries():
    path = lambda M, N, K: g.gemm_select_path(1, M, N, K, 1.0, 1 << 20, K, 1 << 20, N)
    assert path(129, 4096, 4096) == "tc_decode"      # 32 groups x 3 blocks
    assert path(512, 2048, 1024) == "tc_decode"      # 16 x 8 = 128
    assert path(320, 4096, 4096) == "tc_decode"      # 32 x 5 = 160, K >= 4096
    tile = ("tc_bf16", "tc_bf16_pair")                # whichever the table picks
    assert path(320, 4096, 1024) in tile             # 160 > 128 at small K
    assert path(256, 8192, 4096) in tile             # 64 x 4 = 256
    assert path(513, 1024, 1024) in tile             # beyond eight row blocks
    assert path(100, 16392, 4096) == "tc_bf16"       # M <= 128 beyond N = 16384


def _cluster_exact(M, N, K):
    # few column groups: clusters of CTAs split each group's k range and add
    # their partial sums, in k order, through distributed shared memory
    A, B, C = make_inputs(M, N, K, ("int", None), ("int", None), ("int", None),
                          seed=M + N + K, dtype="bf16")
    ref32, _, _ = oracle_bf16(A, B, C, 1.5, -0.5)
    for _ in range(3):  # every repeat bit-exact: the partial sums add in k order
        out, st, _, _, dC = run_bf16gemm(A, B, C, 1.5, -0.5, ldc=N + 3)
        assert st == 0
        assert np.array_equal(out.numpy().view(np.uint32), ref32.view(np.uint32))
        assert dC.untouched_outside()
    check_device_error()


@pytest.mark.parametrize("M,N,K", [(16, 28672, 2048), (1, 20000, 1024), (7, 19500, 3000),
                                   (32, 20000, 1024), (24, 19500, 2000)])
def test_decode_runs_of_groups(M, N, K):
    # more column groups than SMs: each CTA takes a run of whole groups and
    # the groups at run boundaries are combined through the workspace
    A, B, C = make_inputs(M, N, K, ("normal", 1.0), ("normal", 0.02), ("uniform", None),
                          seed=N + K, dtype="bf16")
    outs = []
    for _ in range(3):
        out, st, _, _, dC = run_bf16gemm(A, B, C, 0.75, 0.5)
        assert st == 0
        assert dC.untouched_outside()
        outs.append(out)
    _, ref64, den = oracle_bf16(A, B, C, 0.75, 0.5)
    assert ratio(outs[0], ref64, den) <= TOL_BF16
    for o in outs[1:]:
        assert torch.equal(o.view(torch.int32), outs[0].view(torch.int32))
    check_device_error()


@pytest.mark.parametrize("N,K", [(128, 8192), (384, 4096), (256, 16384), (1000, 2048)])
def test_decode_many_contributors(N, K):
    # few column groups, long k: clusters of 8 CTAs per group
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
