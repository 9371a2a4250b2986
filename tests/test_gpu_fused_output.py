"""bf16 GEMM with the general fused output stage (gemm_bf16gemm_fused):

    v = act(alpha*A*B + beta*C + bias) + R,   D = convert(d_scale * v),
    amax = max |v|

on the GPU against the oracle: oracle.epilogue gives v in fp64, and
oracle.quantize rounds the exact product d_scale * v once to the output
format (the plain reading of "scaling, then fp8/int8 quantisation" in "Tiled
matrix multiplication", "Implementation notes").

Integer inputs with power-of-two scales make v and d_scale * v exact on both
sides, so the fp8 E4M3 / int8 codes must be identical.  Otherwise the
kernel's value carries the bf16 GEMM's bound slope * 8e-3 * (den + |bias|),
plus two fp32 roundings the definition does not have -- the residual add and
the product d_scale * v, which the kernel forms in fp32 before converting --
of at most 2^-24 |v| each.  With b their sum, each code must lie between the
codes of d_scale * (v - b) and d_scale * (v + b): the conversion is monotone,
so that is exactly the set of codes a value within the bound can produce.
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
TORCH_TYPE = {"f32": torch.float32, "bf16": torch.bfloat16, "s8": torch.int8,
              "f8e4m3": getattr(torch, "float8_e4m3fn", None)}
FILL = 0x5A  # byte pattern of D's padding, checked untouched


@pytest.fixture(scope="module", autouse=True)
def _lib(gemm_lib, cuda_device):
    yield


def _run(A, B, C, alpha, beta, bias, act, residual, d_scale, out, with_amax=True, amax0=0.0,
         pad=8):
    M, K = A.shape
    N = B.shape[1]
    dt = TORCH_TYPE[out]
    if dt is None:
        pytest.skip("torch without float8_e4m3fn")
    esize = torch.tensor([], dtype=dt).element_size()
    ldd = N + pad
    raw = torch.full((M, ldd * esize), FILL, dtype=torch.uint8, device="cuda")
    D = raw.view(dt)[:, :N]
    amax = torch.full((1,), amax0, dtype=torch.float32, device="cuda") if with_amax else None
    g.bf16gemm_fused(A.cuda(), B.cuda(), D, C=C.cuda() if beta != 0 else None, alpha=alpha,
                     beta=beta, bias=bias.cuda() if bias is not None else None, act=act,
                     residual=residual.cuda() if residual is not None else None,
                     d_scale=d_scale, amax=amax)
    torch.cuda.synchronize()
    check_device_error()
    host = raw.cpu()
    assert torch.all(host[:, N * esize:] == FILL), "padding of D written"
    Dh = host.view(dt)[:, :N]
    return Dh, (float(amax.item()) if amax is not None else None)


def _codes(Dh, out):
    if out == "f8e4m3":
        return Dh.view(torch.uint8).numpy()
    if out == "s8":
        return Dh.numpy()
    return Dh.float().numpy()


def _decode(codes, out):
    if out == "f8e4m3":
        return oracle.e4m3_decode(codes)
    return np.asarray(codes, dtype=np.float64)


def _reference(A, B, C, alpha, beta, bias, act, residual):
    _, ref64, den = oracle_bf16(A, B, C, alpha, beta)
    v = oracle.epilogue(ref64, bias.numpy() if bias is not None else None, act,
                        residual.numpy() if residual is not None else None)
    scale = den + (np.abs(bias.numpy())[None, :] if bias is not None else 0.0)
    # the GEMM's bound through the activation, plus the kernel's fp32
    # roundings of the residual add and of d_scale * v (2^-24 |v| each)
    b = SLOPE[act] * TOL_BF16 * scale + 2 * 2.0 ** -24 * np.abs(v) + 1e-30
    return v, b


def _check_within(codes, v, b, out, d_scale):
    got = _decode(codes, out)
    lo = _decode(oracle.quantize(v - b, out, d_scale), out)
    hi = _decode(oracle.quantize(v + b, out, d_scale), out)
    ok = (got >= lo) & (got <= hi)
    assert ok.all(), "%d codes outside the bound, first at %s" % (
        int((~ok).sum()), np.argwhere(~ok)[0].tolist())


def _int_case(M, N, K, seed):
    A, B, C = make_inputs(M, N, K, ("int", None), ("int", None), ("int", None), seed=seed,
                          dtype="bf16")
    gen = torch.Generator().manual_seed(seed + 1)
    bias = torch.randint(-8, 9, (N,), generator=gen).float()
    res = torch.randint(-32, 33, (M, N), generator=gen).float()
    return A, B, C, bias, res


# Integer inputs: every partial sum is an integer below 2^24 and the scales
# are powers of two, so v and d_scale * v are exact on both sides.
INT_SHAPES = [
    (8, 1000, 512),       # decode kernel (M <= 16), clusters of 4
    (40, 1000, 512),      # decode kernel, 64-row instance
    (24, 16384, 256),     # decode kernel, 32-row instance, whole column groups
    (100, 520, 256),      # decode kernel, two row blocks of 64
    (100, 16392, 256),    # single-CTA kernel, ragged N
    (384, 512, 256),      # decode kernel, six row blocks of 64
    (640, 512, 256),      # CTA-pair kernel, odd number of tile rows
    (100, 16640, 4096),   # single-CTA kernel, tiles split along k
]


@pytest.mark.parametrize("M,N,K", INT_SHAPES)
@pytest.mark.parametrize("out,d_scale", [("f8e4m3", 2.0 ** -3), ("s8", 2.0 ** -4),
                                         ("f32", 0.5)])
def test_integers_exact(M, N, K, out, d_scale):
    A, B, C, bias, res = _int_case(M, N, K, seed=M + N)
    Dh, amax = _run(A, B, C, 1.0, -0.5, bias, "relu", res, d_scale, out)
    v, _ = _reference(A, B, C, 1.0, -0.5, bias, "relu", res)
    want = oracle.quantize(v, out, d_scale)
    got = _codes(Dh, out)
    if out == "f8e4m3":
        # compare values (+0 and -0 are both zero codes)
        assert np.array_equal(oracle.e4m3_decode(got), oracle.e4m3_decode(want))
    else:
        assert np.array_equal(got, want)
    assert amax == float(np.max(np.abs(v)))


@pytest.mark.parametrize("M,N,K", [(8, 1000, 512), (100, 520, 256), (384, 512, 256),
                                   (640, 512, 256)])
def test_empty_product_integers_exact(M, N, K):
    # alpha = 0: the output stage alone (v = act(beta*C + bias) + R)
    A, B, C, bias, res = _int_case(M, N, K, seed=7)
    Dh, amax = _run(A, B, C, 0.0, 0.75, bias, "relu", res, 2.0 ** -2, "s8")
    v = oracle.epilogue(0.75 * C.numpy().astype(np.float64), bias.numpy(), "relu", res.numpy())
    assert np.array_equal(_codes(Dh, "s8"), oracle.quantize(v, "s8", 2.0 ** -2))
    assert amax == float(np.max(np.abs(v)))


@pytest.mark.parametrize("M,N,K", [
    (16, 12288, 1024),    # decode kernel
    (64, 4096, 2048),     # decode kernel, 64-row instance, clusters of 4
    (128, 16640, 512),    # single-CTA kernel
    (120, 2048, 512),     # decode kernel, two row blocks
    (640, 1280, 1000),    # CTA-pair kernel, ragged K
    (512, 10240, 4096),   # CTA-pair kernel, last round split along k
])
@pytest.mark.parametrize("out,act", [("f8e4m3", "gelu"), ("s8", "none"), ("bf16", "relu")])
def test_random_within_bound(M, N, K, out, act):
    A, B, C = make_inputs(M, N, K, ("normal", 1.0), ("normal", 0.05), ("uniform", None),
                          seed=M + K, dtype="bf16")
    gen = torch.Generator().manual_seed(3)
    bias = torch.randn(N, generator=gen)
    res = torch.randn(M, N, generator=gen)
    d_scale = 24.0 if out == "s8" else 40.0
    Dh, amax = _run(A, B, C, 0.9, 0.5, bias, act, res, d_scale, out)
    v, b = _reference(A, B, C, 0.9, 0.5, bias, act, res)
    if out == "bf16":
        got = Dh.float().numpy().astype(np.float64)
        bound = d_scale * b + 2.0 ** -8 * np.abs(d_scale * v)
        assert np.all(np.abs(got - d_scale * v) <= bound)
    else:
        _check_within(_codes(Dh, out), v, b, out, d_scale)
    worst = np.max(np.abs(v))
    assert abs(amax - worst) <= np.max(b)


def test_amax_is_raised_not_reset():
    A, B, C, bias, res = _int_case(100, 520, 256, seed=3)
    _, amax = _run(A, B, C, 1.0, -0.5, bias, "relu", res, 1.0, "f32", amax0=1e9)
    assert amax == 1e9
    _, amax = _run(A, B, C, 1.0, -0.5, bias, "relu", res, 1.0, "f32", amax0=0.0)
    v, _ = _reference(A, B, C, 1.0, -0.5, bias, "relu", res)
    assert amax == float(np.max(np.abs(v)))


@pytest.mark.parametrize("M", [8, 100, 384])
def test_residual_in_place(M):
    # D is the residual itself (fp32, ldd == ldr): x <- x + relu(A B + bias)
    N, K = 512, 256
    A, B, C, bias, res = _int_case(M, N, K, seed=11)
    X = res.cuda().contiguous()
    g.bf16gemm_fused(A.cuda(), B.cuda(), X, bias=bias.cuda(), act="relu", residual=X)
    torch.cuda.synchronize()
    _, ref64, _ = oracle_bf16(A, B, C, 1.0, 0.0)
    want = oracle.epilogue(ref64, bias.numpy(), "relu", res.numpy())
    assert np.array_equal(X.cpu().numpy().astype(np.float64), want)


@pytest.mark.parametrize("M", [8, 100])
def test_fp32_output_to_separate_padded_d(M):
    # plain output stage (no bias, no activation) into a D that is not C,
    # with ldd != ldc: every kernel must use D's own leading dimension
    N, K = 512, 256
    A, B, C = make_inputs(M, N, K, ("int", None), ("int", None), ("int", None), seed=12,
                          dtype="bf16")
    Dbuf = torch.full((M, N + 24), 7.0, device="cuda")
    D = Dbuf[:, :N]
    g.bf16gemm_epilogue(A.cuda(), B.cuda(), D, C=C.cuda(), alpha=1.0, beta=1.0)
    torch.cuda.synchronize()
    ref32, _, _ = oracle_bf16(A, B, C, 1.0, 1.0)
    assert np.array_equal(D.cpu().numpy(), ref32)
    assert torch.all(Dbuf[:, N:] == 7.0)


def test_invalid_arguments():
    M, N, K = 64, 64, 64
    A = torch.zeros(M, K, dtype=torch.bfloat16, device="cuda")
    B = torch.zeros(K, N, dtype=torch.bfloat16, device="cuda")
    D = torch.zeros(M, N, device="cuda")
    amax = torch.zeros(4, device="cuda")

    def call(**kw):
        o = g.GemmOutput()
        o.beta, o.C, o.ldc, o.bias, o.act = 0.0, 0, N, 0, 0
        o.residual, o.ldr, o.d_scale, o.amax = 0, N, 1.0, 0
        o.D, o.ldd, o.d_type = D.data_ptr(), N, 0
        for k, v in kw.items():
            setattr(o, k, v)
        return g.gemm_bf16gemm_fused(M, N, K, 1.0, A.data_ptr(), K, B.data_ptr(), N, o, 0)

    assert call() == 0
    assert call(d_type=7) == 1
    assert call(act=5) == 1
    assert call(amax=amax.data_ptr() + 2) == 1
    assert call(residual=D.data_ptr(), ldr=N - 1) == 1
    assert call(residual=D.data_ptr() + 2, ldr=N) == 1
    assert call(D=0) == 1
    assert call(beta=1.0, C=0) == 1
    torch.cuda.synchronize()
