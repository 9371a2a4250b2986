"""Pins of the CPU oracle against facts fixed outside it.

Every function takes an oracle object (``oracle.default()`` or a mutated copy)
and raises AssertionError when the oracle disagrees with:
  * closed forms: identity A, rank-1 A and B, K = 1 outer products;
  * the alpha/beta semantics: alpha = 0, beta = 0 with NaN in C, beta = 1;
  * exact rational arithmetic (fractions.Fraction) on tiny shapes;
  * numpy's float64 matmul, an independent library routine;
  * invariants: (AB)^T = B^T A^T, row permutation, scaling in alpha,
    leading dimensions larger than the row length;
  * the error scale den = |alpha| |A||B| + |beta| |C| on sign-mixed inputs;
  * the definition of bf16 (the upper half of an IEEE binary32);
  * the fused output stage's activations: ReLU on signed values, GELU(0) = 0,
    GELU(x) - GELU(-x) = x, and tabulated values of the normal CDF.

The GEMM being pinned is C <- alpha (A x B) + beta C ("GEMM Worklog I: Naive
to Tiled", opening equation; "A GEMM Kernel, Step by Step", "The ladder we
are climbing").  None of these checks evaluates the oracle's own loop again.
"""
from __future__ import annotations

import itertools
from fractions import Fraction

import numpy as np
import pytest

F32 = np.float32


def _rng(seed):
    return np.random.default_rng(seed)


def _ints(rng, shape, lo=-4, hi=4):
    return rng.integers(lo, hi + 1, size=shape).astype(F32)


def pin_identity(orc):
    """A = I (M = K): C = alpha * B + beta * C exactly on small integers."""
    rng = _rng(1)
    M, N = 7, 5
    A = np.eye(M, dtype=F32)
    B = _ints(rng, (M, N))
    C = _ints(rng, (M, N))
    out, out64, _ = orc.sgemm(1.5, A, B, -0.5, C, want64=True)
    expect = 1.5 * B.astype(np.float64) - 0.5 * C.astype(np.float64)
    assert np.array_equal(out64, expect), "identity: alpha*B + beta*C"
    assert np.array_equal(out, expect.astype(F32))


def pin_identity_right(orc):
    """B = I (K = N): C = alpha * A exactly (beta = 0)."""
    rng = _rng(2)
    A = _ints(rng, (6, 9))
    B = np.eye(9, dtype=F32)
    _, out64, _ = orc.sgemm(-2.0, A, B, 0.0, None, want64=True)
    assert np.array_equal(out64, -2.0 * A.astype(np.float64)), "right identity"


def pin_rank1(orc):
    """A = u v^T, B = w z^T  =>  A B = (v . w) u z^T."""
    rng = _rng(3)
    M, K, N = 5, 8, 6
    u, v = _ints(rng, M), _ints(rng, K)
    w, z = _ints(rng, K), _ints(rng, N)
    A = np.outer(u, v).astype(F32)
    B = np.outer(w, z).astype(F32)
    C = _ints(rng, (M, N))
    vw = float(np.dot(v.astype(np.float64), w.astype(np.float64)))
    _, out64, _ = orc.sgemm(0.5, A, B, 2.0, C, want64=True)
    expect = 0.5 * vw * np.outer(u, z).astype(np.float64) + 2.0 * C.astype(np.float64)
    assert np.array_equal(out64, expect), "rank-1 closed form"


def pin_k1_outer(orc):
    """K = 1: C = alpha * a b^T + beta * C."""
    rng = _rng(4)
    a = _ints(rng, (7, 1))
    b = _ints(rng, (1, 3))
    C = _ints(rng, (7, 3))
    _, out64, _ = orc.sgemm(3.0, a, b, -1.0, C, want64=True)
    expect = 3.0 * (a.astype(np.float64) @ b.astype(np.float64)) - C.astype(np.float64)
    # a (7x1) @ b (1x3) has a single term per entry: exact in any routine
    assert np.array_equal(out64, expect), "K = 1 outer product"


def pin_alpha_zero(orc):
    """alpha = 0: C <- beta * C and A, B are not read (NaN there is harmless)."""
    rng = _rng(5)
    A = np.full((4, 6), np.nan, dtype=F32)
    B = np.full((6, 5), np.inf, dtype=F32)
    C = _ints(rng, (4, 5))
    out, _, den = orc.sgemm(0.0, A, B, 0.25, C)
    assert np.array_equal(out, (0.25 * C).astype(F32)), "alpha = 0 gives beta*C"
    assert np.array_equal(den, 0.25 * np.abs(C.astype(np.float64)))


def pin_beta_zero_nan(orc):
    """beta = 0: C is not read; NaN in C does not reach the result."""
    rng = _rng(6)
    A = _ints(rng, (3, 4))
    B = _ints(rng, (4, 2))
    C = np.full((3, 2), np.nan, dtype=F32)
    out, _, _ = orc.sgemm(1.0, A, B, 0.0, C)
    assert np.all(np.isfinite(out)), "beta = 0 must not read C"
    assert np.array_equal(out, (A.astype(np.float64) @ B.astype(np.float64)).astype(F32))


def pin_beta_one_alpha_zero(orc):
    """alpha = 0, beta = 1 leaves C bit-for-bit unchanged."""
    rng = _rng(7)
    C = rng.standard_normal((5, 7)).astype(F32)
    A = rng.standard_normal((5, 3)).astype(F32)
    B = rng.standard_normal((3, 7)).astype(F32)
    out, _, _ = orc.sgemm(0.0, A, B, 1.0, C)
    assert np.array_equal(out.view(np.uint32), C.view(np.uint32)), "C unchanged"


def pin_k_zero(orc):
    """K = 0: the product is empty, C <- beta * C."""
    C = np.arange(12, dtype=F32).reshape(3, 4)
    A = np.zeros((3, 0), dtype=F32)
    B = np.zeros((0, 4), dtype=F32)
    out, _, _ = orc.sgemm(5.0, A, B, -1.0, C)
    assert np.array_equal(out, -C), "K = 0"


def _exact_gemm(alpha, A, B, beta, C):
    """Exact rational C_ij = alpha sum_k A_ik B_kj + beta C_ij (tiny shapes)."""
    M, K = A.shape
    N = B.shape[1]
    fa, fb = Fraction(float(alpha)), Fraction(float(beta))
    res = [[None] * N for _ in range(M)]
    for i in range(M):
        for j in range(N):
            s = Fraction(0)
            for k in range(K):
                s += Fraction(float(A[i, k])) * Fraction(float(B[k, j]))
            res[i][j] = fa * s + (fb * Fraction(float(C[i, j])) if beta != 0 else 0)
    return res


def pin_bruteforce_dyadic(orc):
    """Tiny shapes, dyadic inputs: the fp64 result equals exact arithmetic."""
    rng = _rng(8)
    for M, N, K in itertools.product((1, 2, 3, 5), (1, 2, 4), (1, 2, 3, 6)):
        A = (rng.integers(-16, 17, size=(M, K)) / 8.0).astype(F32)
        B = (rng.integers(-16, 17, size=(K, N)) / 4.0).astype(F32)
        C = (rng.integers(-16, 17, size=(M, N)) / 2.0).astype(F32)
        _, out64, _ = orc.sgemm(0.75, A, B, -1.25, C, want64=True)
        ex = _exact_gemm(0.75, A, B, -1.25, C)
        for i in range(M):
            for j in range(N):
                assert Fraction(float(out64[i, j])) == ex[i][j], (M, N, K, i, j)


def pin_bruteforce_float(orc):
    """Tiny shapes, general floats: within fp64 rounding of exact arithmetic,
    and the fp32 output is the exact value rounded once (1 ulp)."""
    rng = _rng(9)
    for M, N, K in ((1, 1, 1), (2, 3, 4), (4, 1, 6), (3, 5, 2), (6, 6, 6)):
        A = rng.standard_normal((M, K)).astype(F32)
        B = rng.standard_normal((K, N)).astype(F32)
        C = rng.standard_normal((M, N)).astype(F32)
        out, out64, den = orc.sgemm(0.7, A, B, 0.3, C, want64=True)
        ex = _exact_gemm(0.7, A, B, 0.3, C)
        for i in range(M):
            for j in range(N):
                e = float(ex[i][j])
                # k-sum of K terms in fp64 plus the alpha/beta step
                bound = (K + 3) * 2.0 ** -52 * den[i, j] + 1e-300
                assert abs(out64[i, j] - e) <= bound, (M, N, K, i, j)
                assert abs(float(out[i, j]) - e) <= 2.0 ** -23 * abs(e) + bound


def pin_numpy_matmul(orc):
    """Against numpy's float64 matmul (independent BLAS routine)."""
    rng = _rng(10)
    M, K, N = 37, 61, 53
    A = rng.uniform(-1, 1, (M, K)).astype(F32)
    B = rng.uniform(-1, 1, (K, N)).astype(F32)
    C = rng.uniform(-1, 1, (M, N)).astype(F32)
    _, out64, den = orc.sgemm(1.5, A, B, -0.5, C, want64=True)
    ref = 1.5 * (A.astype(np.float64) @ B.astype(np.float64)) - 0.5 * C.astype(np.float64)
    assert np.all(np.abs(out64 - ref) <= 4 * K * 2.0 ** -52 * den), "numpy float64 matmul"


def pin_transpose(orc):
    """(A B)^T = B^T A^T, element for element (same k order per entry)."""
    rng = _rng(11)
    A = rng.standard_normal((9, 13)).astype(F32)
    B = rng.standard_normal((13, 6)).astype(F32)
    _, ab, _ = orc.sgemm(1.0, A, B, 0.0, None, want64=True)
    _, bt_at, _ = orc.sgemm(1.0, np.ascontiguousarray(B.T), np.ascontiguousarray(A.T), 0.0,
                            None, want64=True)
    assert np.array_equal(ab.T, bt_at), "(AB)^T = B^T A^T"
    assert ab.shape == (9, 6)


def pin_row_permutation(orc):
    """Permuting the rows of A and C permutes the rows of the result."""
    rng = _rng(12)
    A = rng.standard_normal((8, 5)).astype(F32)
    B = rng.standard_normal((5, 7)).astype(F32)
    C = rng.standard_normal((8, 7)).astype(F32)
    perm = rng.permutation(8)
    _, r1, _ = orc.sgemm(0.9, A, B, 1.1, C, want64=True)
    _, r2, _ = orc.sgemm(0.9, A[perm], B, 1.1, C[perm], want64=True)
    assert np.array_equal(r1[perm], r2), "row permutation"


def pin_column_permutation(orc):
    """Permuting the columns of B and C permutes the columns of the result."""
    rng = _rng(13)
    A = rng.standard_normal((4, 6)).astype(F32)
    B = rng.standard_normal((6, 9)).astype(F32)
    C = rng.standard_normal((4, 9)).astype(F32)
    perm = rng.permutation(9)
    _, r1, _ = orc.sgemm(1.3, A, B, -0.7, C, want64=True)
    _, r2, _ = orc.sgemm(1.3, A, B[:, perm], -0.7, C[:, perm], want64=True)
    assert np.array_equal(r1[:, perm], r2), "column permutation"


def pin_alpha_scaling(orc):
    """Scaling alpha by 2 scales the (beta = 0) result by 2 exactly."""
    rng = _rng(14)
    A = rng.standard_normal((6, 10)).astype(F32)
    B = rng.standard_normal((10, 4)).astype(F32)
    _, r1, _ = orc.sgemm(0.625, A, B, 0.0, None, want64=True)
    _, r2, _ = orc.sgemm(1.25, A, B, 0.0, None, want64=True)
    assert np.array_equal(2.0 * r1, r2), "linearity in alpha"


def pin_leading_dimensions(orc):
    """Row strides larger than the row length give the dense result; the
    padding (NaN) is never read."""
    rng = _rng(15)
    M, K, N = 5, 7, 6
    A = rng.standard_normal((M, K)).astype(F32)
    B = rng.standard_normal((K, N)).astype(F32)
    C = rng.standard_normal((M, N)).astype(F32)
    Ap = np.full((M, K + 3), np.nan, dtype=F32)
    Ap[:, :K] = A
    Bp = np.full((K, N + 5), np.nan, dtype=F32)
    Bp[:, :N] = B
    Cp = np.full((M, N + 2), np.nan, dtype=F32)
    Cp[:, :N] = C
    _, dense, _ = orc.sgemm(0.5, A, B, 2.0, C, want64=True)
    _, strided, _ = orc.sgemm(0.5, Ap[:, :K], Bp[:, :N], 2.0, Cp[:, :N], want64=True)
    assert np.array_equal(dense, strided), "leading dimensions"


def pin_denominator(orc):
    """den = |alpha| sum_k |A_ik| |B_kj| + |beta| |C_ij| on sign-mixed inputs
    whose signed sum cancels to zero."""
    A = np.array([[1, -1, 2, -2]], dtype=F32)
    B = np.array([[3], [3], [1], [1]], dtype=F32)
    C = np.array([[-4]], dtype=F32)
    out, _, den = orc.sgemm(-2.0, A, B, 0.5, C)
    # signed sum: 3 - 3 + 2 - 2 = 0  -> result 0.5 * -4 = -2
    assert out[0, 0] == -2.0, "signed sum"
    # magnitudes: 3 + 3 + 2 + 2 = 10 -> |alpha| 10 + |beta| 4 = 22
    assert den[0, 0] == 22.0, "error scale"


def pin_dims_nonsquare(orc):
    """Result has shape (M, N) and entry (i, j) pairs row i of A with column j
    of B (catches a transposed operand on a non-square shape)."""
    A = np.array([[1, 0, 0], [0, 1, 0]], dtype=F32)        # 2 x 3 selector
    B = np.arange(12, dtype=F32).reshape(3, 4)             # 3 x 4
    out, _, _ = orc.sgemm(1.0, A, B, 0.0, None)
    assert out.shape == (2, 4)
    assert np.array_equal(out, B[:2]), "row selector picks rows of B"


def pin_bf16_definition(orc):
    """bf16 bit patterns widen to the binary32 with that upper half."""
    cases = {0x3F80: 1.0, 0xBF80: -1.0, 0x4000: 2.0, 0x3F81: 1.0 + 2.0 ** -7,
             0x4049: 3.140625, 0x0001: 2.0 ** -133, 0x3C00: 2.0 ** -7, 0x0000: 0.0}
    one = np.array([[0x3F80]], dtype=np.uint16)
    for bits, value in cases.items():
        a = np.array([[bits]], dtype=np.uint16)
        _, out64, _ = orc.bf16gemm(1.0, a, one, 0.0, None, want64=True)
        assert out64[0, 0] == value, hex(bits)


def pin_bf16_matches_widened_fp32(orc):
    """The bf16 oracle equals the fp32 oracle on the widened values."""
    rng = _rng(16)
    A32 = rng.standard_normal((11, 17)).astype(F32)
    B32 = rng.standard_normal((17, 9)).astype(F32)
    # truncate to bf16 precision so the fp32 copy holds exactly the bf16 value
    Ab = (A32.view(np.uint32) >> 16).astype(np.uint16)
    Bb = (B32.view(np.uint32) >> 16).astype(np.uint16)
    Aw = (Ab.astype(np.uint32) << 16).view(F32)
    Bw = (Bb.astype(np.uint32) << 16).view(F32)
    C = rng.standard_normal((11, 9)).astype(F32)
    _, r16, d16 = orc.bf16gemm(0.8, Ab, Bb, 0.2, C, want64=True)
    _, r32, d32 = orc.sgemm(0.8, Aw, Bw, 0.2, C, want64=True)
    assert np.array_equal(r16, r32) and np.array_equal(d16, d32)


def pin_thread_count_invariance(orc):
    """The split of rows over threads does not change any bit."""
    rng = _rng(17)
    A = rng.standard_normal((33, 40)).astype(F32)
    B = rng.standard_normal((40, 21)).astype(F32)
    C = rng.standard_normal((33, 21)).astype(F32)
    _, r1, _ = orc.sgemm(1.1, A, B, 0.9, C, nthreads=1, want64=True)
    _, r4, _ = orc.sgemm(1.1, A, B, 0.9, C, nthreads=4, want64=True)
    assert np.array_equal(r1, r4)


def pin_epilogue_relu(orc):
    """ReLU keeps non-negative values and zeroes negative ones."""
    import oracle
    x = np.array([[-2.5, -0.0, 0.0, 1e-30, 3.25]])
    assert np.array_equal(oracle.activation(x, "relu"), np.array([[0.0, 0.0, 0.0, 1e-30, 3.25]]))
    assert np.array_equal(oracle.activation(x, "none"), x)


def pin_epilogue_gelu(orc):
    """GELU(x) = x Phi(x): GELU(0) = 0, GELU(x) - GELU(-x) = x, and the
    standard normal CDF at 1 and 3 (0.8413447460685429, 0.9986501019683699)."""
    import oracle
    g = lambda v: float(oracle.activation(np.array([[v]]), "gelu")[0, 0])
    assert g(0.0) == 0.0
    for v in (0.3, 1.0, 2.7, 5.0):
        assert abs((g(v) - g(-v)) - v) <= 4e-16 * max(1.0, v)
    assert abs(g(1.0) - 0.8413447460685429) <= 2e-16
    assert abs(g(-1.0) + (1.0 - 0.8413447460685429)) <= 2e-16
    assert abs(g(3.0) - 3.0 * 0.9986501019683699) <= 1e-15


def pin_epilogue_bias_broadcast(orc):
    """The bias is added per column, to every row."""
    import oracle
    ref = np.arange(6, dtype=np.float64).reshape(2, 3)
    bias = np.array([10.0, -20.0, 0.5])
    out = oracle.epilogue(ref, bias, "none")
    assert np.array_equal(out, np.array([[10.0, -19.0, 2.5], [13.0, -16.0, 5.5]]))
    assert np.array_equal(oracle.epilogue(ref, bias, "relu"), np.maximum(out, 0.0))


def pin_epilogue_residual(orc):
    """The residual is added after the activation, element by element."""
    import oracle
    ref = np.array([[-3.0, 2.0], [0.5, -0.25]])
    res = np.array([[1.0, -1.0], [10.0, 0.75]])
    out = oracle.epilogue(ref, None, "relu", res)
    assert np.array_equal(out, np.array([[1.0, 1.0], [10.5, 0.75]]))
    bias = np.array([4.0, 0.0])
    assert np.array_equal(oracle.epilogue(ref, bias, "none", res),
                          np.array([[2.0, 1.0], [14.5, 0.5]]))


def pin_e4m3_format_values(orc):
    """Values of the OCP 8-bit floating point (E4M3) definition: largest
    finite 448 = 0x7E, smallest normal 2^-6 = 0x08, largest subnormal
    7 * 2^-9 = 0x07, smallest subnormal 2^-9 = 0x01, 1 = 0x38, -2 = 0xC0,
    NaN = S.1111.111; saturation of anything larger to 448."""
    import oracle
    enc = lambda v: int(oracle.e4m3_encode(np.array([v], dtype=np.float32))[0])
    assert enc(448.0) == 0x7E and enc(-448.0) == 0xFE
    assert enc(2.0 ** -6) == 0x08 and enc(7 * 2.0 ** -9) == 0x07 and enc(2.0 ** -9) == 0x01
    assert enc(1.0) == 0x38 and enc(-2.0) == 0xC0 and enc(0.0) == 0x00
    assert enc(1e6) == 0x7E and enc(-np.inf) == 0xFE and enc(np.inf) == 0x7E
    assert enc(np.nan) & 0x7F == 0x7F
    assert np.isnan(oracle.e4m3_decode(np.array([0x7F, 0xFF], dtype=np.uint8))).all()
    assert oracle.e4m3_decode(np.array([0x7E], dtype=np.uint8))[0] == 448.0


def pin_e4m3_ties_to_even(orc):
    """Halfway cases go to the even mantissa: 2^-10 -> 0, 3 * 2^-10 -> 2^-8,
    1 + 1/16 -> 1, 1 + 3/16 -> 1.25, 17 -> 16, 19 -> 20, 464 (halfway to the
    NaN pattern's slot) -> 448."""
    import oracle
    x = np.array([2.0 ** -10, 3 * 2.0 ** -10, 1 + 1 / 16, 1 + 3 / 16, 17.0, 19.0, 464.0],
                 dtype=np.float32)
    got = oracle.e4m3_decode(oracle.e4m3_encode(x))
    assert np.array_equal(got, [0.0, 2.0 ** -8, 1.0, 1.25, 16.0, 20.0, 448.0])


def pin_e4m3_matches_torch(orc):
    """Inside +-448, torch's float8_e4m3fn cast (round to nearest even; an
    independent implementation) gives the same values on random fp32 inputs
    spread over every binade, subnormals included."""
    import oracle
    torch = pytest.importorskip("torch")
    if not hasattr(torch, "float8_e4m3fn"):
        pytest.skip("torch without float8_e4m3fn")
    rng = _rng(41)
    mag = np.ldexp(rng.uniform(1.0, 2.0, 20000), rng.integers(-12, 9, 20000))
    x = (mag * rng.choice([-1.0, 1.0], 20000)).astype(np.float32)
    x = x[np.abs(x) <= 448.0]
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).to(torch.float32).numpy()
    assert np.array_equal(oracle.e4m3_decode(oracle.e4m3_encode(x)), ref.astype(np.float64))


def pin_e4m3_roundtrip_and_order(orc):
    """Every finite code decodes to a value that encodes back to the same
    code (-0 included), and encoding is monotone in the value."""
    import oracle
    codes = np.array([c for c in range(256) if c & 0x7F != 0x7F], dtype=np.uint8)
    vals = oracle.e4m3_decode(codes).astype(np.float32)
    assert np.array_equal(oracle.e4m3_encode(vals), codes)
    x = np.sort(_rng(42).uniform(-500, 500, 5000)).astype(np.float32)
    dec = oracle.e4m3_decode(oracle.e4m3_encode(x))
    assert np.all(np.diff(dec) >= 0)


def pin_s8_rounding(orc):
    """int8 output: half to even (as torch.round), saturation, NaN -> 0."""
    import oracle
    torch = pytest.importorskip("torch")
    x = np.array([0.5, 1.5, 2.5, -0.5, -1.5, -2.5, 126.5, 127.49, 127.6, 1e9, -128.4,
                  -128.6, -1e9, 3.7, -3.7], dtype=np.float32)
    want = np.clip(torch.round(torch.from_numpy(x)).numpy(), -128, 127).astype(np.int8)
    assert np.array_equal(oracle.s8_encode(x), want)
    assert oracle.s8_encode(np.array([np.nan], dtype=np.float32))[0] == 0
    assert np.array_equal(oracle.s8_encode(np.array([126.5, -0.5], dtype=np.float32)), [126, 0])


def _e4m3_table():
    """(value, code) of every non-negative finite E4M3 number, from the OCP
    8-bit floating point definition: exponent field 0 holds m * 2^-9,
    exponent field E > 0 holds (1 + m/8) * 2^(E - 7); S.1111.111 is NaN."""
    out = []
    for ef in range(16):
        for m in range(8):
            if ef == 15 and m == 7:
                continue
            val = Fraction(m, 512) if ef == 0 else (1 + Fraction(m, 8)) * Fraction(2) ** (ef - 7)
            out.append((val, (ef << 3) | m))
    out.sort()
    return out


def _nearest_even(x, grid):
    """The entry of the sorted (value, code) grid nearest to the Fraction
    x >= 0 (ties: the entry whose code is even); x beyond the grid saturates."""
    import bisect
    vals = [g[0] for g in grid]
    i = bisect.bisect_left(vals, x)
    if i == 0:
        return grid[0]
    if i == len(grid):
        return grid[-1]
    lo, hi = grid[i - 1], grid[i]
    dl, dh = x - lo[0], hi[0] - x
    if dl < dh:
        return lo
    if dh < dl:
        return hi
    return lo if lo[1] % 2 == 0 else hi


def _exact_codes_e4m3(vs, s):
    grid = _e4m3_table()
    out = []
    for v in vs:
        x = Fraction(float(np.float32(s))) * Fraction(float(v))
        code = _nearest_even(abs(x), grid)[1]
        out.append(code | (0x80 if x < 0 or (x == 0 and np.signbit(v)) else 0))
    return np.array(out, dtype=np.uint8)


def _exact_s8(vs, s):
    out = []
    for v in vs:
        x = Fraction(float(np.float32(s))) * Fraction(float(v))
        f = x.numerator // x.denominator            # floor
        r = x - f
        n = f + 1 if (r > Fraction(1, 2) or (r == Fraction(1, 2) and f % 2 == 1)) else f
        out.append(min(127, max(-128, n)))
    return np.array(out, dtype=np.int8)


def _exact_f32(vs, s):
    out = []
    for v in vs:
        x = Fraction(float(np.float32(s))) * Fraction(float(v))
        c = np.float32(float(x))
        cands = {c, np.nextafter(c, np.float32(np.inf)), np.nextafter(c, np.float32(-np.inf))}
        best = sorted(cands, key=lambda y: (abs(Fraction(float(y)) - x),
                                            int(np.array(y, np.float32).view(np.uint32)) & 1))
        out.append(best[0])
    return np.array(out, dtype=np.float32)


def _near_ties(ties, scales, rng):
    """fp64 values v whose exact products s * v fall exactly on, or within a
    few fp64 ulps either side of, the given ties."""
    vs, ss = [], []
    for t in ties:
        for s in scales:
            base = float(t) / float(np.float32(s))
            for k in (-3, -1, 0, 1, 3):
                v = base
                for _ in range(abs(k)):
                    v = np.nextafter(v, np.inf if k > 0 else -np.inf)
                sign = rng.choice([-1.0, 1.0])
                vs.append(sign * v)
                ss.append(s)
    return vs, ss


def pin_quantize_single_rounding(orc):
    """The stored code is d_scale * v rounded once: a value just above an
    E4M3 tie goes up even though its nearest fp32 is the tie itself (rounding
    through fp32 first would give the even neighbour below): 1.0625 + 2^-40
    -> 1.125, not 1.0; likewise int8 2.5 + 2^-30 -> 3, not 2; and fp32 output
    1 + 2^-24 + 2^-40 -> 1 + 2^-23.  An exact tie still goes to even."""
    import oracle
    v = np.array([1.0625 + 2.0 ** -40, 1.0625, -(1.0625 + 2.0 ** -40), 17.0 + 2.0 ** -30])
    assert np.array_equal(oracle.e4m3_decode(oracle.quantize(v, "f8e4m3", 1.0)),
                          [1.125, 1.0, -1.125, 18.0])
    assert np.array_equal(oracle.quantize(np.array([2.5 + 2.0 ** -30, 2.5, -2.5 - 2.0 ** -30]),
                                          "s8", 1.0), [3, 2, -3])
    assert oracle.quantize(np.array([1.0 + 2.0 ** -24 + 2.0 ** -40]), "f32", 1.0)[0] == \
        np.float32(1.0 + 2.0 ** -23)
    assert oracle.quantize(np.array([1.0 + 2.0 ** -24]), "f32", 1.0)[0] == np.float32(1.0)


def pin_quantize_exact_rational(orc):
    """quantize against exact rational arithmetic (fractions.Fraction): the
    exact product of the fp32 scale and the fp64 value, rounded to the nearest
    E4M3 value of the format definition (ties to the even code, saturation at
    448), to the nearest integer (ties to even, clamp to [-128, 127]) and to
    the nearest fp32 -- on random values over many binades and on values whose
    exact products sit on, or a few fp64 ulps beside, the formats' ties."""
    import oracle
    rng = _rng(44)
    grid = _e4m3_table()
    e4m3_ties = [(grid[i][0] + grid[i + 1][0]) / 2 for i in range(len(grid) - 1)]
    scales = [1.0, 0.1, 3.0, 40.0, 2.0 ** -5, 0.7]
    vs, ss = _near_ties(e4m3_ties[::3], scales, rng)
    for s in scales:
        mag = np.ldexp(rng.uniform(1.0, 2.0, 150), rng.integers(-14, 10, 150))
        vs += list(mag * rng.choice([-1.0, 1.0], 150) / float(np.float32(s)))
        ss += [s] * 150
    vs, ss = np.array(vs), np.array(ss)
    for s in scales:
        sel = ss == s
        got = oracle.quantize(vs[sel], "f8e4m3", s)
        want = _exact_codes_e4m3(vs[sel], s)
        zero = (want & 0x7F) == 0               # +0 and -0 are both zero
        assert np.array_equal(got[~zero], want[~zero])
        assert np.all((got[zero] & 0x7F) == 0)
    s8_ties = [Fraction(2 * k + 1, 2) for k in range(-130, 130, 7)]
    vs8, ss8 = _near_ties(s8_ties, [1.0, 0.1, 3.0], rng)
    vs8, ss8 = np.array(vs8), np.array(ss8)
    for s in (1.0, 0.1, 3.0):
        sel = ss8 == s
        assert np.array_equal(oracle.quantize(vs8[sel], "s8", s), _exact_s8(vs8[sel], s))
    f32_ties = [Fraction(float(np.float32(x))) + Fraction(2) ** (int(np.floor(np.log2(x))) - 24)
                for x in rng.uniform(0.5, 1000.0, 40)]
    vf, sf = _near_ties(f32_ties, [1.0, 3.0, 0.1], rng)
    vf, sf = np.array(vf), np.array(sf)
    for s in (1.0, 3.0, 0.1):
        sel = sf == s
        assert np.array_equal(oracle.quantize(vf[sel], "f32", s), _exact_f32(vf[sel], s))


def pin_quantize_scale_is_fp32(orc):
    """d_scale enters as the fp32 number the caller passes: 0.1 becomes
    fp32(0.1), so 3 * fp32(0.1) rounds to the fp32 product of the two; and a
    power-of-two scale commutes with the codes."""
    import oracle
    v = np.array([3.0])
    assert oracle.quantize(v, "f32", 0.1)[0] == np.float32(np.float32(0.1) * np.float32(3.0))
    x = _rng(43).uniform(-100, 100, 1000)
    assert np.array_equal(oracle.e4m3_decode(oracle.quantize(x, "f8e4m3", 0.25)),
                          oracle.e4m3_decode(oracle.e4m3_encode(x * 0.25)))


ALL_PINS = [
    pin_identity, pin_identity_right, pin_rank1, pin_k1_outer, pin_alpha_zero,
    pin_beta_zero_nan, pin_beta_one_alpha_zero, pin_k_zero, pin_bruteforce_dyadic,
    pin_bruteforce_float, pin_numpy_matmul, pin_transpose, pin_row_permutation,
    pin_column_permutation, pin_alpha_scaling, pin_leading_dimensions, pin_denominator,
    pin_dims_nonsquare, pin_bf16_definition, pin_bf16_matches_widened_fp32,
    pin_thread_count_invariance, pin_epilogue_relu, pin_epilogue_gelu,
    pin_epilogue_bias_broadcast, pin_epilogue_residual, pin_e4m3_format_values,
    pin_e4m3_ties_to_even, pin_e4m3_matches_torch, pin_e4m3_roundtrip_and_order, pin_s8_rounding,
    pin_quantize_single_rounding, pin_quantize_exact_rational, pin_quantize_scale_is_fp32,
]
