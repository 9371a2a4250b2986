"""bf16 GEMM with the fused output stage, D = act(alpha*A*B + beta*C + bias),
on the GPU against the oracle's definition (oracle.epilogue on the fp64 GEMM
result).

Bound per element: L * 8e-3 * (den + |bias_j|) (+ 2^-8 |D_ref| when D is
bf16), where den = |alpha| (|A||B|)_ij + |beta||C_ij| is the bf16 GEMM's
error scale and L the activation's largest slope (1 for none and ReLU, 1.13
for GELU).
"""
import numpy as np
import pytest
import torch

import dense_gemm_12_gb300 as g
import oracle
from dense_gemm_12_gb300.workloads import make_inputs
from gpu_helpers import TOL_BF16, check_device_error, oracle_bf16

pytestmark = pytest.mark.gpu

SLOPE = {"none": 1.0, "relu": 1.0, "gelu": 1.13}


@pytest.fixture(scope="module", autouse=True)
def _lib(gemm_lib, cuda_device):
    yield


def _run(A, B, C, alpha, beta, bias, act, out, d_ld=None):
    M, K = A.shape
    N = B.shape[1]
    dt = torch.bfloat16 if out == "bf16" else torch.float32
    ldd = d_ld or N
    Dbuf = torch.full((M, ldd), 7.0, dtype=dt, device="cuda")
    D = Dbuf[:, :N]
    g.bf16gemm_epilogue(A.cuda(), B.cuda(), D, C=C.cuda() if beta != 0 else None, alpha=alpha,
                        beta=beta, bias=bias.cuda() if bias is not None else None, act=act)
    torch.cuda.synchronize()
    if ldd > N:  # padding untouched
        assert torch.all(Dbuf[:, N:] == 7.0)
    return D.float().cpu()


def _check(A, B, C, alpha, beta, bias, act, out, D):
    _, ref64, den = oracle_bf16(A, B, C, alpha, beta)
    bias_np = bias.numpy() if bias is not None else None
    ref = oracle.epilogue(ref64, bias_np, act)
    scale = den + (np.abs(bias_np)[None, :] if bias_np is not None else 0.0)
    bound = SLOPE[act] * TOL_BF16 * scale + 1e-30
    if out == "bf16":
        bound = bound + 2.0 ** -8 * np.abs(ref)
    err = np.abs(D.numpy().astype(np.float64) - ref)
    assert np.all(err <= bound), float(np.max(err / bound))


@pytest.mark.parametrize("act", ["none", "relu", "gelu"])
@pytest.mark.parametrize("out", ["f32", "bf16"])
@pytest.mark.parametrize("with_bias", [False, True])
@pytest.mark.parametrize("beta", [0.0, 0.5])
def test_tile_kernel_epilogues(act, out, with_bias, beta):
    M, N, K = 300, 520, 200
    A, B, C = make_inputs(M, N, K, ("normal", 1.0), ("normal", 0.1), ("uniform", None),
                          seed=11, dtype="bf16")
    bias = torch.randn(N, generator=torch.Generator().manual_seed(5)) if with_bias else None
    D = _run(A, B, C, 0.8, beta, bias, act, out)
    _check(A, B, C, 0.8, beta, bias, act, out, D)


@pytest.mark.parametrize("act,out", [("gelu", "bf16"), ("relu", "f32"), ("none", "bf16")])
def test_decode_kernel_epilogues(act, out):
    M, N, K = 7, 1000, 1024
    A, B, C = make_inputs(M, N, K, ("normal", 1.0), ("normal", 0.05), ("uniform", None),
                          seed=12, dtype="bf16")
    bias = torch.randn(N, generator=torch.Generator().manual_seed(6))
    D = _run(A, B, C, 1.0, 1.0, bias, act, out)
    _check(A, B, C, 1.0, 1.0, bias, act, out, D)
    check_device_error()


@pytest.mark.parametrize("M,N,K,act,out", [
    (100, 16640, 4096, "gelu", "bf16"),  # single-CTA kernel, tiles split along k
    (512, 10240, 4096, "relu", "f32"),   # pair kernel, last round split along k
])
def test_split_tiles_epilogue(M, N, K, act, out):
    # the output stage runs once, on the summed parts
    assert g.gemm_split_parts(1, M, N, K) > 1
    A, B, C = make_inputs(M, N, K, ("normal", 1.0), ("normal", 0.05), ("uniform", None),
                          seed=15, dtype="bf16")
    bias = torch.randn(N, generator=torch.Generator().manual_seed(8))
    D = _run(A, B, C, 0.9, 0.5, bias, act, out)
    _check(A, B, C, 0.9, 0.5, bias, act, out, D)
    check_device_error()


def test_padded_output_and_ragged():
    M, N, K = 129, 264, 72
    A, B, C = make_inputs(M, N, K, seed=13, dtype="bf16")
    bias = torch.linspace(-1, 1, N)
    D = _run(A, B, C, 1.5, -0.25, bias, "gelu", "bf16", d_ld=N + 8)
    _check(A, B, C, 1.5, -0.25, bias, "gelu", "bf16", D)


def test_relu_integers_exact():
    # integer inputs: the pre-activation is an exact small integer, so ReLU's
    # fp32 output must equal the definition exactly
    M, N, K = 256, 512, 128
    A, B, C = make_inputs(M, N, K, ("int", None), ("int", None), ("int", None), seed=14,
                          dtype="bf16")
    bias = torch.randint(-8, 9, (N,), generator=torch.Generator().manual_seed(7)).float()
    D = _run(A, B, C, 1.0, 1.0, bias, "relu", "f32")
    _, ref64, _ = oracle_bf16(A, B, C, 1.0, 1.0)
    assert np.array_equal(D.numpy().astype(np.float64), oracle.epilogue(ref64, bias.numpy(), "relu"))


def test_empty_product():
    M, N = 40, 96
    A, B, C = make_inputs(M, N, 0, seed=15, dtype="bf16")
    bias = torch.randn(N, generator=torch.Generator().manual_seed(8))
    D = _run(A, B, C, 1.0, 0.5, bias, "gelu", "f32")
    ref = oracle.epilogue(0.5 * C.numpy().astype(np.float64), bias.numpy(), "gelu")
    assert np.all(np.abs(D.numpy() - ref) <= 1e-6 * (1 + np.abs(ref)))


def test_in_place_fp32_matches_plain_gemm():
    M, N, K = 200, 304, 256
    A, B, C = make_inputs(M, N, K, seed=16, dtype="bf16")
    plain = C.cuda()
    g.bf16gemm(A.cuda(), B.cuda(), plain, alpha=0.5, beta=2.0)
    inplace = C.cuda()
    g.bf16gemm_epilogue(A.cuda(), B.cuda(), inplace, C=inplace, alpha=0.5, beta=2.0)
    torch.cuda.synchronize()
    assert torch.equal(plain, inplace)


def test_invalid_arguments():
    A, B, C = make_inputs(16, 64, 64, seed=17, dtype="bf16")
    dA, dB = A.cuda(), B.cuda()
    D = torch.empty(16, 64, device="cuda")
    st = g.gemm_bf16gemm_epilogue(16, 64, 64, 1.0, dA.data_ptr(), 64, dB.data_ptr(), 64, 0.0, 0, 64,
                                  0, 7, D.data_ptr(), 64, 0, 0)
    assert st == 1  # unknown activation
    st = g.gemm_bf16gemm_epilogue(16, 64, 64, 1.0, dA.data_ptr(), 64, dB.data_ptr(), 64, 0.0, 0, 64,
                                  0, 0, D.data_ptr(), 64, 9, 0)
    assert st == 1  # unknown output type
    # odd pitch: TMA cannot describe B, so it is staged (results checked in
    # test_gpu_staging.py)
    st = g.gemm_bf16gemm_epilogue(16, 63, 64, 1.0, dA.data_ptr(), 64, dB.data_ptr(), 63, 0.0, 0, 63,
                                  0, 0, D.data_ptr(), 63, 0, 0)
    assert st == 0
