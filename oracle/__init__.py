"""CPU oracle for C <- alpha*(A x B) + beta*C (fp64 triple loop).

TEST INFRASTRUCTURE ONLY.  The CUDA library is checked against this module;
only the tests, the package smoke check and the benchmark's CPU-baseline leg
may import it, and the library never does.  It shares no code with the CUDA
path: the arithmetic lives in ``gemm_oracle.c`` (plain C, fp64, OpenMP over
rows), compiled here with gcc and called through ctypes.

The definition it follows is the GEMM of "GEMM Worklog I: Naive to Tiled"
(opening equation: C = alpha (A x B) + beta C with A M x K, B K x N) and the
SGEMM call of "A GEMM Kernel, Step by Step" ("The ladder we are climbing").
Where the pages are silent (beta == 0, alpha == 0, K == 0, bf16 widening) the
readings are stated in the C file's header.

Every function here is pinned by tests that do not re-type its formula:
identity and rank-1 closed forms, alpha/beta special cases, exact rational
brute force on tiny shapes, numpy's float64 matmul as an independent routine,
and transposition / permutation / linearity invariants.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gemm_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")

_lock = threading.Lock()
_default = None


def compile_library(src: str, out_path: str) -> str:
    """Compile an oracle C source into a shared library at out_path."""
    os.makedirs(os.path.dirname(out_path), exist_ok=True)
    tmp = out_path + ".tmp.%d" % os.getpid()
    cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math",
           "-fopenmp", "-fPIC", "-shared", src, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out_path)
    return out_path


def build(force: bool = False) -> str:
    """Compile gemm_oracle.c into oracle/_build/liboracle.so; return its path."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    return compile_library(_SRC, _LIB_PATH)


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _as_2d(x, dtype, rows, cols, name):
    """Return (array, leading dimension) for a row-major matrix view.

    Accepts a C-contiguous 2-D array, or a 2-D view whose rows are strided
    (a slice of a wider matrix); the leading dimension is the row stride.
    """
    x = np.asarray(x)
    if x.dtype != dtype:
        raise TypeError("%s must be %s, got %s" % (name, dtype, x.dtype))
    if x.ndim != 2 or x.shape != (rows, cols):
        raise ValueError("%s must have shape %s, got %s" % (name, (rows, cols), x.shape))
    item = x.itemsize
    if rows <= 1 and cols <= 1:
        return np.ascontiguousarray(x), max(cols, 1)
    if x.strides[1] != item and cols > 1:
        x = np.ascontiguousarray(x)
    ld = x.strides[0] // item if rows > 1 else max(cols, 1)
    if ld < max(cols, 1) or x.strides[0] % item:
        x = np.ascontiguousarray(x)
        ld = max(cols, 1)
    return x, ld


class OracleLib:
    """ctypes front end of one compiled oracle library."""

    def __init__(self, path: str):
        lib = ctypes.CDLL(path)
        i64, dbl, ptr, cint = (ctypes.c_int64, ctypes.c_double,
                               ctypes.c_void_p, ctypes.c_int)
        for name in ("oracle_sgemm", "oracle_bf16gemm"):
            fn = getattr(lib, name)
            fn.restype = cint
            fn.argtypes = [i64, i64, i64, dbl, ptr, i64, ptr, i64, dbl,
                           ptr, i64, ptr, ptr, ptr, i64, cint]
        lib.oracle_max_threads.restype = cint
        lib.oracle_max_threads.argtypes = []
        self._lib = lib
        self.path = path

    def max_threads(self) -> int:
        return int(self._lib.oracle_max_threads())

    def _run(self, fn_name, M, N, K, alpha, A, B, beta, C, in_dtype, nthreads, want64):
        A2, lda = _as_2d(A, in_dtype, M, K, "A")
        B2, ldb = _as_2d(B, in_dtype, K, N, "B")
        if C is not None:
            C2, ldc = _as_2d(C, np.float32, M, N, "C")
        elif beta == 0.0:
            C2, ldc = None, max(N, 1)
        else:
            raise ValueError("C is required when beta != 0")
        out = np.empty((M, N), dtype=np.float32)
        out64 = np.empty((M, N), dtype=np.float64) if want64 else None
        den = np.empty((M, N), dtype=np.float64)
        rc = getattr(self._lib, fn_name)(M, N, K, float(alpha), _ptr(A2), lda, _ptr(B2),
                                         ldb, float(beta), _ptr(C2), ldc, _ptr(out),
                                         _ptr(out64), _ptr(den), max(N, 1), int(nthreads))
        if rc != 0:
            raise RuntimeError("%s failed with code %d" % (fn_name, rc))
        return out, out64, den

    def sgemm(self, alpha, A, B, beta, C=None, nthreads=0, want64=False):
        """fp32 SGEMM oracle.

        A: (M, K) float32, B: (K, N) float32, C: (M, N) float32 (may be None
        when beta == 0).  Returns (ref_fp32, ref_fp64 or None, den), where den
        is |alpha| * (|A| |B|) + |beta| * |C| in fp64.
        """
        M, K = np.shape(A)
        K2, N = np.shape(B)
        if K2 != K:
            raise ValueError("inner dimensions differ: %d vs %d" % (K, K2))
        return self._run("oracle_sgemm", M, N, K, alpha, A, B, beta, C, np.float32,
                         nthreads, want64)

    def bf16gemm(self, alpha, A_bits, B_bits, beta, C=None, nthreads=0, want64=False):
        """bf16-input / fp32-output oracle.

        A_bits: (M, K) uint16 bf16 bit patterns, B_bits: (K, N) uint16, C
        float32.  The inputs are widened exactly (bf16 is the top half of a
        binary32).
        """
        M, K = np.shape(A_bits)
        K2, N = np.shape(B_bits)
        if K2 != K:
            raise ValueError("inner dimensions differ: %d vs %d" % (K, K2))
        return self._run("oracle_bf16gemm", M, N, K, alpha, A_bits, B_bits, beta, C,
                         np.uint16, nthreads, want64)


def default() -> OracleLib:
    """The oracle built from gemm_oracle.c (compiled on first use)."""
    global _default
    with _lock:
        if _default is None:
            _default = OracleLib(build())
    return _default


def max_threads() -> int:
    """Threads an oracle call with nthreads=0 uses (OpenMP's default)."""
    return default().max_threads()


def sgemm(alpha, A, B, beta, C=None, nthreads=0, want64=False):
    """fp32 SGEMM oracle (see OracleLib.sgemm)."""
    return default().sgemm(alpha, A, B, beta, C, nthreads, want64)


def bf16gemm(alpha, A_bits, B_bits, beta, C=None, nthreads=0, want64=False):
    """bf16-input oracle (see OracleLib.bf16gemm)."""
    return default().bf16gemm(alpha, A_bits, B_bits, beta, C, nthreads, want64)


def _erf(x):
    """erf in fp64, element by element (math.erf: the C library's erf)."""
    import math
    return np.frompyfunc(math.erf, 1, 1)(np.asarray(x, dtype=np.float64)).astype(np.float64)


def activation(x, act):
    """The activations of the fused output stage, in fp64.

    "none": x;  "relu": max(x, 0);  "gelu": x * Phi(x), Phi the standard
    normal CDF, Phi(x) = (1 + erf(x / sqrt(2))) / 2.
    """
    x = np.asarray(x, dtype=np.float64)
    if act == "none":
        return x.copy()
    if act == "relu":
        return np.where(x > 0.0, x, 0.0)
    if act == "gelu":
        return x * 0.5 * (1.0 + _erf(x / np.sqrt(2.0)))
    raise ValueError("unknown activation %r" % (act,))


def epilogue(ref64, bias=None, act="none", residual=None):
    """Fused output stage on the fp64 GEMM result, in fp64:

        v[i][j] = act(ref64[i][j] + bias[j]) + residual[i][j]

    (bias broadcast over rows; either may be None).  ref64 is
    alpha*(A x B) + beta*C from sgemm / bf16gemm (want64=True).  The pages'
    epilogue fusion ("Tiled matrix multiplication", "Implementation notes")
    applies bias, activation, residual, scaling and quantisation, in that
    order, before the tile is stored; scaling and quantisation are
    ``quantize``.
    """
    v = np.asarray(ref64, dtype=np.float64)
    if bias is not None:
        v = v + np.asarray(bias, dtype=np.float64)[None, :]
    v = activation(v, act)
    if residual is not None:
        v = v + np.asarray(residual, dtype=np.float64)
    return v


# ---------------------------------------------------------------- quantise
# The output conversion of the fused stage ("Tiled matrix multiplication",
# "Implementation notes": scaling, then fp8/int8 quantisation).  Reading: the
# value stored is the exact product d_scale * v rounded ONCE to the output
# format (round to nearest, ties to even), with d_scale the fp32 number the
# caller passes.  Nothing in between is rounded to fp32: where a kernel
# rounds d_scale * v to fp32 first, its extra rounding is part of the error
# a test allows, not of the definition.
#
# fp8 E4M3 as the OCP 8-bit floating point format defines it ("E4M3"): sign
# bit, 4 exponent bits with bias 7, 3 mantissa bits; exponent field 0 holds
# the subnormals m * 2^-9; no infinities; S.1111.111 is NaN, so the largest
# finite value is S.1111.110 = 1.75 * 2^8 = 448.
E4M3_MAX = 448.0
_E4M3_MIN_NORMAL = 2.0 ** -6
_E4M3_SUBNORMAL_STEP = 2.0 ** -9


def _exact_product(v, d_scale):
    """d_scale * v as an unevaluated sum hi + lo of two fp64 arrays (exact).

    d_scale is taken as the fp32 number it rounds to (24 significant bits),
    v as fp64.  v is split (Veltkamp) into halves of at most 27 significant
    bits each, so both partial products are exact in fp64; their sum is then
    re-split exactly (Knuth's TwoSum) into hi = fl(hi + lo) and the error lo.
    Exact for |v| between 2^-900 and 2^900 (no underflow or overflow of the
    pieces); outside that only lo may be inexact.
    """
    s = float(np.float32(d_scale))
    v = np.asarray(v, dtype=np.float64)
    with np.errstate(over="ignore", invalid="ignore"):
        c = 134217729.0 * v                     # 2^27 + 1
        vh = c - (c - v)
        vh = np.where(np.isfinite(vh), vh, v)   # huge or non-finite v: no split
        vl = v - vh
        a = s * vh
        b = s * vl
        hi = a + b
        bb = hi - a
        lo = (a - (hi - bb)) + (b - bb)
    lo = np.where(np.isfinite(hi), lo, 0.0)
    return hi, lo


def _round_on_grid(mag, lo, step):
    """Round the exact non-negative value mag + lo to the nearest multiple of
    `step` (a power of two per element), ties to even.

    mag and step are fp64 arrays with mag / step exact and below 2^52; lo is
    the exact value's part below mag's last bit (|lo| <= half an fp64 ulp of
    mag).  A rounding boundary (an odd multiple of step / 2) is itself an fp64
    number, so lo can move the result only when mag lies exactly on one: then
    the sign of lo says on which side the exact value is, and a zero lo is a
    true tie, broken toward the even multiple.
    """
    q = mag / step
    f = np.floor(q)
    r = q - f
    up = (r > 0.5) | ((r == 0.5) & ((lo > 0) | ((lo == 0) & (np.fmod(f, 2.0) == 1.0))))
    return (f + up) * step


def _e4m3_codes(hi, lo):
    """E4M3 codes of the exact values hi + lo (see e4m3_encode)."""
    hi = np.asarray(hi, dtype=np.float64)
    lo = np.broadcast_to(np.asarray(lo, dtype=np.float64), hi.shape)
    sign = np.signbit(hi).astype(np.uint8) << 7
    nan = np.isnan(hi)
    a = np.abs(np.where(nan, 0.0, hi))
    lo_mag = np.where(np.signbit(hi), -lo, lo)
    over = a > E4M3_MAX                     # saturates whatever lo is
    a = np.where(over, E4M3_MAX, a)
    lo_mag = np.where(over, 0.0, lo_mag)
    # spacing of representable values around a: 2^-9 below the smallest
    # normal, 2^(e - 3) in the binade [2^e, 2^(e+1))
    _, E = np.frexp(a)                      # a = f 2^E, f in [0.5, 1)
    e = E.astype(np.int64) - 1
    step = np.where(a < _E4M3_MIN_NORMAL, _E4M3_SUBNORMAL_STEP, np.ldexp(1.0, e - 3))
    y = np.minimum(_round_on_grid(a, lo_mag, step), E4M3_MAX)
    # encode y (0 <= y <= 448, representable)
    _, Ey = np.frexp(y)
    ey = Ey.astype(np.int64) - 1
    normal = y >= _E4M3_MIN_NORMAL
    exp_field = np.where(normal, ey + 7, 0)
    mant = np.where(normal, np.ldexp(y, -ey) * 8.0 - 8.0, y / _E4M3_SUBNORMAL_STEP)
    code = (exp_field.astype(np.uint8) << 3) | mant.astype(np.uint8)
    code = np.where(nan, np.uint8(0x7F), code | sign)
    return code.astype(np.uint8)


def e4m3_encode(x):
    """Values (taken as fp64) -> E4M3 codes (uint8): round to nearest, ties to
    even, finite overflow and infinities saturated to +-448, NaN -> 0x7F."""
    x = np.asarray(x, dtype=np.float64)
    return _e4m3_codes(x, np.zeros_like(x))


def e4m3_decode(code):
    """E4M3 codes (uint8) -> their values as fp64 (NaN for S.1111.111)."""
    c = np.asarray(code, dtype=np.uint8).astype(np.int64)
    s = np.where(c >> 7, -1.0, 1.0)
    ef = (c >> 3) & 0xF
    m = c & 0x7
    mag = np.where(ef == 0, m * _E4M3_SUBNORMAL_STEP, np.ldexp(1.0 + m / 8.0, ef - 7))
    return np.where((ef == 0xF) & (m == 0x7), np.nan, s * mag)


def _s8_codes(hi, lo):
    """int8 of the exact values hi + lo (see s8_encode)."""
    hi = np.asarray(hi, dtype=np.float64)
    lo = np.broadcast_to(np.asarray(lo, dtype=np.float64), hi.shape)
    nan = np.isnan(hi)
    a = np.abs(np.where(nan, 0.0, hi))
    lo_mag = np.where(np.signbit(hi), -lo, lo)
    big = a >= 256.0                        # saturates whatever lo is
    r = _round_on_grid(np.where(big, 256.0, a), np.where(big, 0.0, lo_mag), np.ones_like(a))
    r = np.where(np.signbit(hi), -r, r)
    return np.clip(r, -128.0, 127.0).astype(np.int8)


def s8_encode(x):
    """Values (taken as fp64) -> int8: round half to even, saturate to
    [-128, 127], NaN -> 0."""
    x = np.asarray(x, dtype=np.float64)
    return _s8_codes(x, np.zeros_like(x))


def _f32_of(hi, lo):
    """fp32 nearest to the exact values hi + lo (ties to even), for |hi|
    between the smallest normal fp32 and the largest finite one."""
    hi = np.asarray(hi, dtype=np.float64)
    lo = np.broadcast_to(np.asarray(lo, dtype=np.float64), hi.shape)
    a = np.abs(hi)
    lo_mag = np.where(np.signbit(hi), -lo, lo)
    _, E = np.frexp(np.where(a > 0, a, 1.0))
    step = np.ldexp(1.0, E.astype(np.int64) - 1 - 23)   # fp32 spacing in a's binade
    y = _round_on_grid(a, lo_mag, step)
    y = np.where(np.isfinite(hi), y, a)
    return np.where(np.signbit(hi), -y, y).astype(np.float32)


def quantize(v, d_type, d_scale=1.0):
    """Output conversion of the fused stage: the exact product x = d_scale * v
    (d_scale the fp32 scale argument, v the fp64 value of the stage) rounded
    once to the output format:
    "f32": the nearest fp32;  "f8e4m3": E4M3 codes;  "s8": int8 codes
    (rounding and saturation as in e4m3_encode / s8_encode)."""
    hi, lo = _exact_product(v, d_scale)
    if d_type == "f32":
        return _f32_of(hi, lo)
    if d_type == "f8e4m3":
        return _e4m3_codes(hi, lo)
    if d_type == "s8":
        return _s8_codes(hi, lo)
    raise ValueError("unknown output type %r" % (d_type,))


def error_ratio(C_test, ref, den):
    """max_ij |C_test - ref| / den, with den == 0 entries requiring equality.

    Returns +inf if some entry with den == 0 differs from ref, or if C_test
    holds a NaN where ref does not.
    """
    C_test = np.asarray(C_test, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    den = np.asarray(den, dtype=np.float64)
    diff = np.abs(C_test - ref)
    if np.any(np.isnan(diff)):
        return float("inf")
    zero = den == 0
    if np.any(diff[zero] != 0):
        return float("inf")
    if not np.any(~zero):
        return 0.0
    return float(np.max(diff[~zero] / den[~zero]))
