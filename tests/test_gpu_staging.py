"""Operands the TMA engine cannot describe (base not 16-byte aligned, row pitch
not a multiple of 16 bytes), staged: the library copies them into an aligned
per-stream buffer and runs the TMA-fed kernels (fp32: CUDA-core kernel with
128x256 tiles and the stream-K tail; bf16: the tcgen05 tile kernels and, for
the fused output stage, the decode kernel).

Every case compares against the oracle on the same inputs: small-integer
inputs, whose products and sums are exact in fp32 in any order, must match
bit for bit; the operands and the padding around every matrix must be left
unchanged (the copy only reads them).
"""
import numpy as np
import pytest
import torch

import dense_gemm_12_gb300 as g
import oracle
from dense_gemm_12_gb300.workloads import make_inputs
from gpu_helpers import (DeviceMatrix, TOL_BF16, bits, check_device_error, oracle_bf16,
                         oracle_sgemm, ratio, run_bf16gemm, run_sgemm, tol_fp32)

pytestmark = pytest.mark.gpu

INT = ("int", None)


@pytest.fixture(scope="module", autouse=True)
def _lib(gemm_lib, cuda_device):
    yield


def _u32(t):
    return t.numpy().view(np.uint32)


@pytest.mark.parametrize("M,N,K,lda,ldb,offsets", [
    (1024, 1280, 2047, 2047, 1280, (0, 0, 0)),       # A pitch 8188 B
    (1280, 1280, 1311, 1311, 1281, (0, 0, 0)),       # both pitches odd
    (1280, 1536, 1024, 1024, 1536, (1, 0, 0)),       # A base 4 bytes past a 16-B boundary
    (512, 2304, 2048, 2048, 2305, (0, 3, 0)),        # B pitch and base
])
def test_fp32_staged_exact_on_integers(M, N, K, lda, ldb, offsets):
    A, B, C = make_inputs(M, N, K, INT, INT, INT, seed=M + K)
    aptr = 0x10000 + offsets[0] * 4
    bptr = 0x10000 + offsets[1] * 4
    assert g.gemm_select_path(0, M, N, K, 1.5, aptr, lda, bptr, ldb) == "simt_staged"
    out, st, dA, dB, dC = run_sgemm(A, B, C, 1.5, -0.5, lda=lda, ldb=ldb, ldc=N + 3,
                                    offsets=offsets)
    assert st == 0
    ref32, _, _ = oracle_sgemm(A, B, C, 1.5, -0.5, want64=False)
    assert np.array_equal(_u32(out), ref32.view(np.uint32))
    assert dA.untouched_outside() and dB.untouched_outside() and dC.untouched_outside()
    assert torch.equal(dA.logical(), A) and torch.equal(dB.logical(), B)
    check_device_error()


def test_fp32_staged_matches_generic_loader_result_bound():
    # The same ragged problem below the staging threshold (generic loads) and
    # above it (staged): both within the fp32 bound of the oracle.
    for M, N, K, expect in ((900, 1000, 999, "simt_generic"), (1100, 1000, 999, "simt_staged")):
        A, B, C = make_inputs(M, N, K, ("normal", 1.0), ("normal", 1.0), ("uniform", None),
                              seed=M)
        assert g.gemm_select_path(0, M, N, K, 0.7, 0x10000, K, 0x10000, N) == expect
        out, st, _, _, dC = run_sgemm(A, B, C, 0.7, 0.3)
        assert st == 0
        _, ref64, den = oracle_sgemm(A, B, C, 0.7, 0.3)
        assert ratio(out, ref64, den) <= tol_fp32(K), expect
        assert dC.untouched_outside()


@pytest.mark.parametrize("M,N,K,lda,ldb,offsets,kernel", [
    (512, 640, 257, 258, 640, (0, 0, 0), "decode"),   # A pitch 516 B; 8 row blocks
    (100, 512, 333, 333, 517, (0, 0, 0), "decode"),   # both pitches odd
    (384, 768, 512, 512, 768, (1, 0, 0), "decode"),   # A base 2 bytes off
    (640, 768, 512, 512, 768, (1, 0, 0), "pair"),     # A base 2 bytes off
    (256, 256, 1000, 1001, 257, (0, 5, 0), "decode"),  # B pitch and base
    (1024, 256, 1000, 1001, 257, (0, 5, 0), "pair"),  # B pitch and base
])
def test_bf16_staged_tensor_cores_exact_on_integers(M, N, K, lda, ldb, offsets, kernel):
    A, B, C = make_inputs(M, N, K, INT, INT, INT, seed=M * 7 + K, dtype="bf16")
    aptr = 0x10000 + offsets[0] * 2
    bptr = 0x10000 + offsets[1] * 2
    assert g.gemm_select_path(1, M, N, K, 1.5, aptr, lda, bptr, ldb) == "tc_staged"
    out, st, dA, dB, dC = run_bf16gemm(A, B, C, 1.5, -0.5, lda=lda, ldb=ldb, ldc=N + 1,
                                       offsets=offsets)
    assert st == 0
    ref32, _, _ = oracle_bf16(A, B, C, 1.5, -0.5, want64=False)
    assert np.array_equal(_u32(out), ref32.view(np.uint32))
    assert dA.untouched_outside() and dB.untouched_outside() and dC.untouched_outside()
    assert torch.equal(dA.logical(), A) and torch.equal(dB.logical(), B)
    check_device_error()


def test_bf16_staged_random_within_bound():
    M, N, K = 640, 896, 1999
    A, B, C = make_inputs(M, N, K, ("normal", 1.0), ("normal", 1.0), ("uniform", None),
                          seed=77, dtype="bf16")
    out, st, _, _, _ = run_bf16gemm(A, B, C, 0.7, 0.3, lda=K, ldb=N)
    assert st == 0
    _, ref64, den = oracle_bf16(A, B, C, 0.7, 0.3)
    assert ratio(out, ref64, den) <= TOL_BF16


def _fused_relu(M, N, K, lda, ldb, seed):
    """gemm_bf16gemm_epilogue (bias + ReLU, fp32 D) with odd pitches."""
    A, B, C = make_inputs(M, N, K, INT, INT, INT, seed=seed, dtype="bf16")
    bias = torch.randint(-8, 9, (N,), generator=torch.Generator().manual_seed(seed)).float()
    dA = DeviceMatrix(A, lda)
    dB = DeviceMatrix(B, ldb)
    dC = DeviceMatrix(C, N + 2)
    dbias = bias.cuda()
    dD = DeviceMatrix(torch.zeros(M, N), N + 5)
    st = g.gemm_bf16gemm_epilogue(M, N, K, 0.5, dA.ptr, dA.ld, dB.ptr, dB.ld, 2.0, dC.ptr, dC.ld,
                                  dbias.data_ptr(), 1, dD.ptr, dD.ld, 0, 0)
    torch.cuda.synchronize()
    assert st == 0, g.gemm_status_string(st)
    _, ref64, _ = oracle_bf16(A, B, C, 0.5, 2.0)
    v = oracle.epilogue(ref64, bias=bias.numpy(), act="relu")
    assert np.array_equal(dD.logical().numpy(), v.astype(np.float32))
    assert dA.untouched_outside() and dB.untouched_outside() and dD.untouched_outside()


@pytest.mark.parametrize("M,N,K,lda,ldb", [
    (16, 63, 64, 64, 63),        # decode kernel on the staged B
    (8, 1000, 777, 777, 1000),   # decode, A pitch 1554 B
    (40, 300, 130, 131, 300),    # decode kernel, 64-row instance, small
    (100, 300, 130, 131, 300),   # decode kernel, two row blocks
    (300, 520, 270, 270, 521),   # decode kernel, five row blocks
    (640, 520, 270, 270, 521),   # CTA pairs
])
def test_fused_output_stage_on_staged_operands(M, N, K, lda, ldb):
    _fused_relu(M, N, K, lda, ldb, seed=M + N)
    check_device_error()


def test_staging_buffer_grows_and_is_reused_on_one_stream():
    s = torch.cuda.Stream()
    for (M, N, K) in ((512, 512, 131), (1024, 768, 515), (256, 512, 131)):
        A, B, C = make_inputs(M, N, K, INT, INT, INT, seed=K + M, dtype="bf16")
        out, st, _, _, _ = run_bf16gemm(A, B, C, 1.0, 1.0, lda=K, ldb=N + 1,
                                        stream=s.cuda_stream)
        assert st == 0
        ref32, _, _ = oracle_bf16(A, B, C, 1.0, 1.0, want64=False)
        assert np.array_equal(_u32(out), ref32.view(np.uint32))
    check_device_error()


def test_staged_calls_on_two_streams_back_to_back():
    # Each stream copies into its own staging buffer; the calls are queued
    # before either is waited for.
    M, N, K = 1024, 1280, 1999
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    ins = [make_inputs(M, N, K, INT, INT, INT, seed=s) for s in (1, 2)]
    mats = []
    for (A, B, C), s in zip(ins, (s1, s2)):
        dA, dB, dC = DeviceMatrix(A), DeviceMatrix(B), DeviceMatrix(C)
        torch.cuda.synchronize()
        st = g.gemm_sgemm(M, N, K, 1.0, dA.ptr, dA.ld, dB.ptr, dB.ld, 1.0, dC.ptr, dC.ld,
                          s.cuda_stream)
        assert st == 0
        mats.append(dC)
    torch.cuda.synchronize()
    for (A, B, C), dC in zip(ins, mats):
        ref32, _, _ = oracle_sgemm(A, B, C, 1.0, 1.0, want64=False)
        assert np.array_equal(_u32(dC.logical()), ref32.view(np.uint32))
    check_device_error()
