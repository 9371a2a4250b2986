"""fp32 SGEMM on the GPU (CUDA-core kernel) against the CPU oracle.

Bound per element: |C - C_ref| <= 2e-6 * sqrt(K) * (|alpha| (|A||B|)_ij + |beta||C_ij|),
bit-exact on small-integer inputs.  Covers the TMA-fed and the generic-load
variants, ragged edges, padded leading dimensions (padding must stay
untouched), guard bands around C, the alpha/beta special cases, determinism,
and the full-size workloads on sampled rows.
"""
import numpy as np
import pytest
import torch

import dense_gemm_12_gb300 as g
from dense_gemm_12_gb300.workloads import WORKLOADS, make_inputs, workload_inputs
from gpu_helpers import (check_device_error, oracle_sgemm, ratio, run_sgemm, tol_fp32)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib(gemm_lib, cuda_device):
    yield


def _inputs(M, N, K, seed, dist=("uniform", None)):
    return make_inputs(M, N, K, dist, dist, dist, seed=seed)


def test_256_uniform():
    w = WORKLOADS["sgemm_256"]
    A, B, C = workload_inputs(w)
    out, st, _, _, dC = run_sgemm(A, B, C, w.alpha, w.beta)
    assert st == 0
    assert g.gemm_select_path(0, w.M, w.N, w.K, w.alpha, 1 << 20, w.K, 1 << 20, w.N) == "simt_tma"
    ref32, ref64, den = oracle_sgemm(A, B, C, w.alpha, w.beta)
    assert ratio(out, ref64, den) <= tol_fp32(w.K)
    assert dC.untouched_outside()
    check_device_error()


def test_256_integers_bit_exact():
    w = WORKLOADS["sgemm_256_int"]
    A, B, C = workload_inputs(w)
    out, st, _, _, _ = run_sgemm(A, B, C, w.alpha, w.beta)
    assert st == 0
    ref32, _, _ = oracle_sgemm(A, B, C, w.alpha, w.beta)
    assert np.array_equal(out.numpy().view(np.uint32), ref32.view(np.uint32))


def test_256_integers_bit_exact_generic_loader():
    w = WORKLOADS["sgemm_256_int"]
    A, B, C = workload_inputs(w)
    # pitch 257 floats is not a multiple of 16 bytes: both operands take cp.async loads
    out, st, _, _, _ = run_sgemm(A, B, C, w.alpha, w.beta, lda=257, ldb=257, ldc=259)
    assert st == 0
    ref32, _, _ = oracle_sgemm(A, B, C, w.alpha, w.beta)
    assert np.array_equal(out.numpy().view(np.uint32), ref32.view(np.uint32))


EDGE = [1, 2, 3, 5, 7, 8, 9, 127, 128, 129, 255, 257]
RAGGED = [(M, N, K) for M in EDGE for N in (1, 9, 129, 257) for K in (1, 8, 33, 257)
          if (M * N * K) % 7 in (0, 3)] + [(300, 300, 300), (129, 257, 1999), (1, 1, 1)]


@pytest.mark.parametrize("M,N,K", RAGGED)
def test_ragged_tma(M, N, K):
    A, B, C = _inputs(M, N, K, seed=M * 10007 + N * 101 + K)
    # pad the pitches to multiples of 4 floats so TMA is legal
    lda, ldb, ldc = (K + 3) // 4 * 4, (N + 3) // 4 * 4, (N + 3) // 4 * 4
    out, st, dA, dB, dC = run_sgemm(A, B, C, 0.7, 0.3, lda=lda, ldb=ldb, ldc=ldc)
    assert st == 0
    _, ref64, den = oracle_sgemm(A, B, C, 0.7, 0.3)
    assert ratio(out, ref64, den) <= tol_fp32(K)
    assert dC.untouched_outside()


@pytest.mark.parametrize("M,N,K", RAGGED[::3])
def test_ragged_generic(M, N, K):
    A, B, C = _inputs(M, N, K, seed=M * 7 + N * 13 + K)
    # dense odd pitches and a misaligned base: generic loads for A and B
    out, st, dA, dB, dC = run_sgemm(A, B, C, -1.25, 0.5, offsets=(1, 3, 1))
    assert st == 0
    _, ref64, den = oracle_sgemm(A, B, C, -1.25, 0.5)
    assert ratio(out, ref64, den) <= tol_fp32(K)
    assert dC.untouched_outside()


@pytest.mark.parametrize("mix", ["a_generic", "b_generic"])
def test_mixed_loaders(mix):
    M, N, K = 200, 264, 300
    A, B, C = _inputs(M, N, K, seed=5)
    if mix == "a_generic":
        kw = dict(lda=301, ldb=264)      # A pitch 1204 B (not /16), B pitch 1056 B
    else:
        kw = dict(lda=300, ldb=265)
    out, st, _, _, dC = run_sgemm(A, B, C, 1.0, -1.0, **kw)
    assert st == 0
    _, ref64, den = oracle_sgemm(A, B, C, 1.0, -1.0)
    assert ratio(out, ref64, den) <= tol_fp32(K)
    assert dC.untouched_outside()


def test_padded_leading_dimensions_sentinels():
    M, N, K = 333, 517, 129
    A, B, C = _inputs(M, N, K, seed=11)
    out, st, dA, dB, dC = run_sgemm(A, B, C, 0.5, 2.0, lda=K + 7, ldb=N + 11, ldc=N + 3)
    assert st == 0
    _, ref64, den = oracle_sgemm(A, B, C, 0.5, 2.0)
    assert ratio(out, ref64, den) <= tol_fp32(K)
    assert dA.untouched_outside() and dB.untouched_outside() and dC.untouched_outside()


def test_beta_zero_ignores_nan_c():
    M, N, K = 130, 140, 150
    A, B, _ = _inputs(M, N, K, seed=12)
    C = torch.full((M, N), float("nan"))
    out, st, _, _, _ = run_sgemm(A, B, C, 1.0, 0.0)
    assert st == 0 and torch.isfinite(out).all()
    _, ref64, den = oracle_sgemm(A, B, torch.zeros(M, N), 1.0, 0.0)
    assert ratio(out, ref64, den) <= tol_fp32(K)


def test_alpha_zero_and_k_zero():
    M, N, K = 70, 90, 40
    A, B, C = _inputs(M, N, K, seed=13)
    out, st, _, _, _ = run_sgemm(A, B, C, 0.0, -0.5)
    assert st == 0 and torch.equal(out, -0.5 * C)
    out, st, _, _, _ = run_sgemm(torch.zeros(M, 0), torch.zeros(0, N), C, 2.0, 3.0)
    assert st == 0 and torch.equal(out, 3.0 * C)
    out, st, _, _, _ = run_sgemm(torch.zeros(M, 0), torch.zeros(0, N), C, 2.0, 0.0)
    assert st == 0 and torch.equal(out, torch.zeros(M, N))
    # alpha = 0, beta = 1: C unchanged bit for bit
    out, st, _, _, _ = run_sgemm(A, B, C, 0.0, 1.0)
    assert st == 0 and torch.equal(out.view(torch.int32), C.view(torch.int32))


def test_deterministic_repeats():
    M, N, K = 515, 643, 777
    A, B, C = _inputs(M, N, K, seed=14)
    outs = [run_sgemm(A, B, C, 0.7, 0.3)[0] for _ in range(5)]
    for o in outs[1:]:
        assert torch.equal(o.view(torch.int32), outs[0].view(torch.int32))


def _sampled_rows_check(w, rows=48, seed=0):
    A, B, C = workload_inputs(w)
    out, st, _, _, dC = run_sgemm(A, B, C, w.alpha, w.beta)
    assert st == 0
    check_device_error()
    gen = torch.Generator().manual_seed(seed)
    idx = torch.randperm(w.M, generator=gen)[:rows].sort().values
    idx = torch.cat([idx, torch.tensor([0, w.M - 1])]).unique()
    _, ref64, den = oracle_sgemm(A[idx].contiguous(), B, C[idx].contiguous(), w.alpha, w.beta)
    r = ratio(out[idx], ref64, den)
    assert r <= tol_fp32(w.K), r
    assert dC.untouched_outside()
    return r


def test_full_4092():
    _sampled_rows_check(WORKLOADS["sgemm_4092"])


def test_full_4096():
    _sampled_rows_check(WORKLOADS["sgemm_4096"])


def test_full_ragged_3000x5000x1999():
    w = WORKLOADS["sgemm_ragged"]
    # A's 7996-byte rows are not TMA-describable: A is staged (copied to a
    # 16-byte pitch) and the TMA-fed kernel runs
    assert g.gemm_select_path(0, w.M, w.N, w.K, 1.0, 1 << 20, w.K, 1 << 20, w.N) == "simt_staged"
    _sampled_rows_check(w)


def test_stream_argument():
    M, N, K = 256, 384, 512
    A, B, C = _inputs(M, N, K, seed=15)
    s = torch.cuda.Stream()
    out, st, _, _, _ = run_sgemm(A, B, C, 1.0, 1.0, stream=s.cuda_stream)
    assert st == 0
    _, ref64, den = oracle_sgemm(A, B, C, 1.0, 1.0)
    assert ratio(out, ref64, den) <= tol_fp32(K)


def test_tensor_helper():
    M, N, K = 100, 200, 300
    A, B, C = _inputs(M, N, K, seed=16)
    dC = C.cuda()
    g.sgemm(A.cuda(), B.cuda(), dC, alpha=0.5, beta=0.25)
    torch.cuda.synchronize()
    _, ref64, den = oracle_sgemm(A, B, C, 0.5, 0.25)
    assert ratio(dC.cpu(), ref64, den) <= tol_fp32(K)


@pytest.mark.parametrize("M,N,K", [
    (128 * 13, 128 * 13, 2048),   # 169 tiles: 152 whole, the last 17 split along k
    (128 * 16, 128 * 10, 1024),   # 160 tiles: 8-tile tail
    (512, 512, 2048),             # 16 tiles, fewer than the SMs: every tile split
    (100, 3000, 4096),            # one tile row, ragged
])
def test_split_k_tiles_match_oracle_and_repeat(M, N, K):
    A, B, C = _inputs(M, N, K, seed=M + N + K)
    outs = [run_sgemm(A, B, C, 0.7, 0.3)[0] for _ in range(3)]
    for o in outs[1:]:
        assert torch.equal(o.view(torch.int32), outs[0].view(torch.int32))
    gen = torch.Generator().manual_seed(1)
    idx = torch.randperm(M, generator=gen)[:64].sort().values
    idx = torch.cat([idx, torch.tensor([0, M - 1])]).unique()
    _, ref64, den = oracle_sgemm(A[idx].contiguous(), B, C[idx].contiguous(), 0.7, 0.3)
    assert ratio(outs[0][idx], ref64, den) <= tol_fp32(K)
    check_device_error()


def test_split_k_integers_exact():
    # small integers: every partial sum and their total are exact in fp32
    M, N, K = 512, 640, 1024
    A, B, C = make_inputs(M, N, K, ("int", None), ("int", None), ("int", None), seed=9)
    out, st, _, _, _ = run_sgemm(A, B, C, 1.5, -0.5)
    assert st == 0
    ref32, _, _ = oracle_sgemm(A, B, C, 1.5, -0.5)
    assert np.array_equal(out.numpy().view(np.uint32), ref32.view(np.uint32))
