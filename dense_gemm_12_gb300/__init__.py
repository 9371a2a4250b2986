"""dense_gemm_12_gb300 -- GB300 (sm_103a) dense GEMM, C <- alpha*(A x B) + beta*C.

Python binding of the C ABI in ``include/gemm12.h`` (``libgemm12.so``).  The
functions named like the C entry points take the same arguments (device
pointers as integers, a stream handle as an integer) and only marshal them;
every step of the GEMM runs in the library's CUDA kernels.  The tensor
helpers ``sgemm`` / ``bf16gemm`` derive pointers, leading dimensions and the
current stream from torch tensors and call the same entry points.

There is no fallback: if the compiled library is missing, loading fails with
an error that says how to build it.
"""
from __future__ import annotations

import ctypes
import os
import threading

from . import _build

__all__ = [
    "GemmError", "load_library", "library_path", "gemm_sgemm", "gemm_bf16gemm",
    "gemm_bf16gemm_decode_static", "gemm_bf16gemm_epilogue", "bf16gemm_epilogue", "ACT", "OUT",
    "gemm_bf16gemm_fused", "bf16gemm_fused", "GemmOutput",
    "gemm_sgemm_config", "gemm_bf16gemm_config", "gemm_get_config", "gemm_get_model_config",
    "GemmConfig", "KERNELS", "SPLIT_STREAM",
    "gemm_status_string", "gemm_check_device_error", "gemm_shutdown", "gemm_release_stream",
    "gemm_select_path", "gemm_split_parts", "gemm_split_cluster", "gemm_quantization", "gemm_version", "sgemm", "bf16gemm",
    "STATUS", "PATHS",
]

STATUS = {
    0: "GEMM_OK", 1: "GEMM_ERR_INVALID_VALUE", 2: "GEMM_ERR_MISALIGNED",
    3: "GEMM_ERR_UNSUPPORTED", 4: "GEMM_ERR_LAUNCH", 5: "GEMM_ERR_DEVICE_TIMEOUT",
    6: "GEMM_ERR_NO_MEMORY",
}
PATHS = {
    0: "none", 1: "scale_c", 2: "simt_tma", 3: "simt_generic", 4: "tc_bf16",
    5: "tc_decode", 6: "simt_bf16", 7: "tc_bf16_pair", 8: "simt_staged", 9: "tc_staged",
}


class GemmError(RuntimeError):
    """A C-ABI call returned a status other than GEMM_OK."""

    def __init__(self, status: int, where: str):
        self.status = int(status)
        super().__init__("%s: %s" % (where, gemm_status_string(status)))


class GemmOutput(ctypes.Structure):
    """Mirror of gemm_output_t (include/gemm12.h)."""
    _fields_ = [
        ("beta", ctypes.c_float), ("C", ctypes.c_void_p), ("ldc", ctypes.c_int64),
        ("bias", ctypes.c_void_p), ("act", ctypes.c_int),
        ("residual", ctypes.c_void_p), ("ldr", ctypes.c_int64),
        ("d_scale", ctypes.c_float), ("amax", ctypes.c_void_p),
        ("D", ctypes.c_void_p), ("ldd", ctypes.c_int64), ("d_type", ctypes.c_int),
    ]


class GemmConfig(ctypes.Structure):
    """Mirror of gemm_config_t (include/gemm12.h)."""
    _fields_ = [("kernel", ctypes.c_int), ("split", ctypes.c_int), ("group_m", ctypes.c_int)]


KERNELS = {"auto": 0, "single_cta": 1, "cta_pair": 2, "wide": 3}
# gemm_config_t.split value for the stream-K tail (fp32 only): GEMM_SPLIT_STREAM.
SPLIT_STREAM = -1


class _Quantization(ctypes.Structure):
    _fields_ = [
        ("tiles_m", ctypes.c_int64), ("tiles_n", ctypes.c_int64), ("tiles", ctypes.c_int64),
        ("covered_m", ctypes.c_int64), ("covered_n", ctypes.c_int64),
        ("useful_fraction", ctypes.c_double), ("per_wave", ctypes.c_int64),
        ("waves", ctypes.c_int64), ("wave_efficiency", ctypes.c_double),
    ]


_lock = threading.Lock()
_lib = None


def library_path() -> str:
    return _build.LIB_PATH


def load_library(build_if_missing: bool = False):
    """Load libgemm12.so (optionally compiling it first) and declare signatures."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = _build.LIB_PATH
        if build_if_missing:
            path = _build.build()
        if not os.path.exists(path):
            raise RuntimeError(
                "libgemm12.so is not built (expected at %s); run "
                "`python -c 'import __graft_entry__ as g; g.build()'`" % path)
        lib = ctypes.CDLL(path)
        i64, f32, vp, cint = ctypes.c_int64, ctypes.c_float, ctypes.c_void_p, ctypes.c_int
        gemm_args = [i64, i64, i64, f32, vp, i64, vp, i64, f32, vp, i64, vp]
        lib.gemm_sgemm.argtypes = gemm_args
        lib.gemm_sgemm.restype = cint
        lib.gemm_bf16gemm.argtypes = gemm_args
        lib.gemm_bf16gemm.restype = cint
        lib.gemm_bf16gemm_decode_static.argtypes = gemm_args
        lib.gemm_bf16gemm_decode_static.restype = cint
        lib.gemm_bf16gemm_epilogue.argtypes = [i64, i64, i64, f32, vp, i64, vp, i64, f32, vp, i64,
                                               vp, cint, vp, i64, cint, vp]
        lib.gemm_bf16gemm_epilogue.restype = cint
        lib.gemm_bf16gemm_fused.argtypes = [i64, i64, i64, f32, vp, i64, vp, i64,
                                            ctypes.POINTER(GemmOutput), vp]
        lib.gemm_bf16gemm_fused.restype = cint
        cfg_p = ctypes.POINTER(GemmConfig)
        lib.gemm_sgemm_config.argtypes = gemm_args[:-1] + [cfg_p, vp]
        lib.gemm_sgemm_config.restype = cint
        lib.gemm_bf16gemm_config.argtypes = gemm_args[:-1] + [cfg_p, vp]
        lib.gemm_bf16gemm_config.restype = cint
        lib.gemm_get_config.argtypes = [cint, i64, i64, i64, cfg_p, ctypes.POINTER(cint)]
        lib.gemm_get_config.restype = cint
        lib.gemm_get_model_config.argtypes = [cint, i64, i64, i64, cfg_p]
        lib.gemm_get_model_config.restype = cint
        lib.gemm_status_string.argtypes = [cint]
        lib.gemm_status_string.restype = ctypes.c_char_p
        lib.gemm_check_device_error.argtypes = [vp]
        lib.gemm_check_device_error.restype = cint
        lib.gemm_shutdown.argtypes = []
        lib.gemm_shutdown.restype = cint
        lib.gemm_release_stream.argtypes = [vp]
        lib.gemm_release_stream.restype = cint
        lib.gemm_select_path.argtypes = [cint, i64, i64, i64, f32, vp, i64, vp, i64]
        lib.gemm_select_path.restype = cint
        lib.gemm_quantization.argtypes = [i64, i64, i64, i64, i64, i64,
                                          ctypes.POINTER(_Quantization)]
        lib.gemm_quantization.restype = cint
        lib.gemm_split_parts.argtypes = [cint, i64, i64, i64]
        lib.gemm_split_parts.restype = cint
        lib.gemm_split_cluster.argtypes = [cint, i64, i64, i64, cfg_p]
        lib.gemm_split_cluster.restype = cint
        lib.gemm_version.argtypes = []
        lib.gemm_version.restype = cint
        _lib = lib
        return lib


# ----------------------------------------------------------- C-ABI mirrors
def gemm_sgemm(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream=0) -> int:
    """fp32 SGEMM; pointers are device addresses (int). Returns the status."""
    return load_library().gemm_sgemm(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream)


def gemm_bf16gemm(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream=0) -> int:
    """bf16-in / fp32-out GEMM; pointers are device addresses. Returns the status."""
    return load_library().gemm_bf16gemm(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream)


def gemm_bf16gemm_decode_static(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream=0) -> int:
    """Decode-shaped bf16 GEMM that allocates nothing (scratch in a fixed
    library-owned array); see include/gemm12.h. Returns the status."""
    return load_library().gemm_bf16gemm_decode_static(M, N, K, alpha, A, lda, B, ldb, beta, C,
                                                      ldc, stream)


ACT = {"none": 0, "relu": 1, "gelu": 2}
OUT = {"f32": 0, "bf16": 1, "f8e4m3": 2, "s8": 3}


def gemm_bf16gemm_epilogue(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, bias, act, D, ldd,
                           d_type, stream=0) -> int:
    """bf16 GEMM with fused bias / activation / output type (see include/gemm12.h).
    act and d_type are the C enum values (ACT / OUT). Returns the status."""
    return load_library().gemm_bf16gemm_epilogue(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc,
                                                 bias, act, D, ldd, d_type, stream)


def gemm_bf16gemm_fused(M, N, K, alpha, A, lda, B, ldb, out: "GemmOutput", stream=0) -> int:
    """bf16 GEMM with the general output stage (gemm_output_t). Returns the status."""
    return load_library().gemm_bf16gemm_fused(M, N, K, alpha, A, lda, B, ldb, ctypes.byref(out),
                                              stream)


def _config(cfg):
    if cfg is None:
        return None
    if isinstance(cfg, GemmConfig):
        return ctypes.byref(cfg)
    kernel = cfg.get("kernel", 0)
    split = cfg.get("split", 0)
    c = GemmConfig(KERNELS[kernel] if isinstance(kernel, str) else int(kernel),
                   SPLIT_STREAM if split == "stream" else int(split), int(cfg.get("group_m", 0)))
    return ctypes.byref(c)


def gemm_sgemm_config(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, cfg, stream=0) -> int:
    """gemm_sgemm with a pinned launch configuration (GemmConfig or a dict with
    kernel / split / group_m; None = automatic). Returns the status."""
    return load_library().gemm_sgemm_config(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc,
                                            _config(cfg), stream)


def gemm_bf16gemm_config(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, cfg, stream=0) -> int:
    """gemm_bf16gemm with a pinned launch configuration. Returns the status."""
    return load_library().gemm_bf16gemm_config(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc,
                                               _config(cfg), stream)


def gemm_get_config(is_bf16, M, N, K):
    """(config dict, from_table) automatic dispatch uses for a shape on the current
    device; raises GemmError without a usable device."""
    c = GemmConfig()
    t = ctypes.c_int(0)
    st = load_library().gemm_get_config(int(bool(is_bf16)), M, N, K, ctypes.byref(c),
                                        ctypes.byref(t))
    if st != 0:
        raise GemmError(st, "gemm_get_config")
    names = {v: k for k, v in KERNELS.items()}
    return {"kernel": names[c.kernel], "split": c.split, "group_m": c.group_m}, bool(t.value)


def gemm_get_model_config(is_bf16, M, N, K):
    """The configuration the cost model alone chooses (ignoring the sweep's table)."""
    c = GemmConfig()
    st = load_library().gemm_get_model_config(int(bool(is_bf16)), M, N, K, ctypes.byref(c))
    if st != 0:
        raise GemmError(st, "gemm_get_model_config")
    names = {v: k for k, v in KERNELS.items()}
    return {"kernel": names[c.kernel], "split": c.split, "group_m": c.group_m}


def gemm_status_string(status: int) -> str:
    return load_library().gemm_status_string(int(status)).decode()


def gemm_check_device_error(stream=0) -> int:
    return load_library().gemm_check_device_error(stream)


def gemm_shutdown() -> int:
    return load_library().gemm_shutdown()


def gemm_release_stream(stream=0) -> int:
    """Free the scratch and staging buffers kept for `stream` (stream-ordered)."""
    return load_library().gemm_release_stream(stream)


def gemm_select_path(is_bf16, M, N, K, alpha, A, lda, B, ldb) -> str:
    """Name of the kernel path a call with these arguments takes (host-only):
    "simt_tma" / "simt_generic" / "simt_staged" (fp32 on the CUDA cores, with
    operands loaded by TMA, by generic loads, or from an aligned staging copy),
    "tc_bf16" / "tc_bf16_pair" / "tc_decode" / "tc_staged" (bf16 on the tensor
    cores), "simt_bf16" (bf16 widened on the CUDA cores), "scale_c", "none"."""
    return PATHS[load_library().gemm_select_path(int(bool(is_bf16)), M, N, K, alpha, A, lda,
                                                 B, ldb)]


def gemm_split_parts(is_bf16, M, N, K) -> int:
    """k-ranges per work item of the last round (1 = no split; 0 = no device)."""
    return load_library().gemm_split_parts(int(bool(is_bf16)), M, N, K)


def gemm_split_cluster(is_bf16, M, N, K, config=None) -> int:
    """TMA operands: the cluster size S whose CTAs add a tile's k-parts in
    distributed shared memory, 1 if they meet in global memory or nothing is
    split, 0 for invalid input or no device.  `config` as for the _config calls."""
    return load_library().gemm_split_cluster(int(bool(is_bf16)), M, N, K, _config(config))


def gemm_quantization(M, N, BM, BN, num_sms, ctas_per_sm) -> dict:
    """Tile / wave quantization of a launch (host-only arithmetic)."""
    q = _Quantization()
    st = load_library().gemm_quantization(M, N, BM, BN, num_sms, ctas_per_sm, ctypes.byref(q))
    if st != 0:
        raise GemmError(st, "gemm_quantization")
    return {name: getattr(q, name) for name, _ in _Quantization._fields_}


def gemm_version() -> int:
    return load_library().gemm_version()


# ------------------------------------------------------------ tensor helpers
def _row_major_ld(t, name):
    if t.dim() != 2:
        raise ValueError("%s must be 2-D" % name)
    rows, cols = t.shape
    if cols > 1 and t.stride(1) != 1:
        raise ValueError("%s must be row-major (unit column stride)" % name)
    return t.stride(0) if rows > 1 else max(cols, 1)


def _stream_handle(stream, device):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return stream.cuda_stream


def sgemm(A, B, C, alpha=1.0, beta=0.0, stream=None):
    """C <- alpha*(A @ B) + beta*C in place for fp32 CUDA tensors (row-major views)."""
    import torch
    for t, n in ((A, "A"), (B, "B"), (C, "C")):
        if t.dtype != torch.float32 or not t.is_cuda:
            raise TypeError("%s must be a float32 CUDA tensor" % n)
    M, K = A.shape
    N = B.shape[1]
    if B.shape[0] != K or tuple(C.shape) != (M, N):
        raise ValueError("shape mismatch: A %s, B %s, C %s" % (tuple(A.shape), tuple(B.shape),
                                                               tuple(C.shape)))
    st = gemm_sgemm(M, N, K, float(alpha), A.data_ptr(), _row_major_ld(A, "A"), B.data_ptr(),
                    _row_major_ld(B, "B"), float(beta), C.data_ptr(), _row_major_ld(C, "C"),
                    _stream_handle(stream, C.device))
    if st != 0:
        raise GemmError(st, "gemm_sgemm")
    return C


def bf16gemm(A, B, C, alpha=1.0, beta=0.0, stream=None):
    """C <- alpha*(A @ B) + beta*C in place; A, B bf16 CUDA tensors, C fp32."""
    import torch
    for t, n, dt in ((A, "A", torch.bfloat16), (B, "B", torch.bfloat16), (C, "C", torch.float32)):
        if t.dtype != dt or not t.is_cuda:
            raise TypeError("%s must be a %s CUDA tensor" % (n, dt))
    M, K = A.shape
    N = B.shape[1]
    if B.shape[0] != K or tuple(C.shape) != (M, N):
        raise ValueError("shape mismatch: A %s, B %s, C %s" % (tuple(A.shape), tuple(B.shape),
                                                               tuple(C.shape)))
    st = gemm_bf16gemm(M, N, K, float(alpha), A.data_ptr(), _row_major_ld(A, "A"), B.data_ptr(),
                       _row_major_ld(B, "B"), float(beta), C.data_ptr(), _row_major_ld(C, "C"),
                       _stream_handle(stream, C.device))
    if st != 0:
        raise GemmError(st, "gemm_bf16gemm")
    return C


def bf16gemm_epilogue(A, B, D, C=None, alpha=1.0, beta=0.0, bias=None, act="none", stream=None):
    """D <- act(alpha*(A @ B) + beta*C + bias); A, B bf16, C and bias fp32, D fp32
    or bf16 (all CUDA tensors, row-major)."""
    import torch
    for t, n in ((A, "A"), (B, "B")):
        if t.dtype != torch.bfloat16 or not t.is_cuda:
            raise TypeError("%s must be a bfloat16 CUDA tensor" % n)
    if D.dtype not in (torch.float32, torch.bfloat16) or not D.is_cuda:
        raise TypeError("D must be a float32 or bfloat16 CUDA tensor")
    M, K = A.shape
    N = B.shape[1]
    if B.shape[0] != K or tuple(D.shape) != (M, N):
        raise ValueError("shape mismatch")
    c_ptr, ldc = 0, max(N, 1)
    if C is not None:
        if C.dtype != torch.float32 or tuple(C.shape) != (M, N):
            raise TypeError("C must be a float32 (M, N) tensor")
        c_ptr, ldc = C.data_ptr(), _row_major_ld(C, "C")
    b_ptr = 0
    if bias is not None:
        if bias.dtype != torch.float32 or bias.numel() != N or not bias.is_contiguous():
            raise TypeError("bias must be a contiguous float32 tensor of N values")
        b_ptr = bias.data_ptr()
    st = gemm_bf16gemm_epilogue(M, N, K, float(alpha), A.data_ptr(), _row_major_ld(A, "A"),
                                B.data_ptr(), _row_major_ld(B, "B"), float(beta), c_ptr, ldc,
                                b_ptr, ACT[act], D.data_ptr(), _row_major_ld(D, "D"),
                                OUT["bf16" if D.dtype == torch.bfloat16 else "f32"],
                                _stream_handle(stream, D.device))
    if st != 0:
        raise GemmError(st, "gemm_bf16gemm_epilogue")
    return D


def _out_type(torch, D):
    kinds = {torch.float32: "f32", torch.bfloat16: "bf16", torch.int8: "s8"}
    if hasattr(torch, "float8_e4m3fn"):
        kinds[torch.float8_e4m3fn] = "f8e4m3"
    if D.dtype not in kinds or not D.is_cuda:
        raise TypeError("D must be a float32, bfloat16, float8_e4m3fn or int8 CUDA tensor")
    return OUT[kinds[D.dtype]]


def bf16gemm_fused(A, B, D, C=None, alpha=1.0, beta=0.0, bias=None, act="none", residual=None,
                   d_scale=1.0, amax=None, stream=None):
    """v = act(alpha*(A @ B) + beta*C + bias) + residual; D <- convert(d_scale * v) in D's
    dtype (float32, bfloat16, float8_e4m3fn or int8); amax (a float32 CUDA tensor of one
    element, or None) is raised to max |v|.  A, B bf16; C, bias, residual fp32."""
    import torch
    for t, n in ((A, "A"), (B, "B")):
        if t.dtype != torch.bfloat16 or not t.is_cuda:
            raise TypeError("%s must be a bfloat16 CUDA tensor" % n)
    M, K = A.shape
    N = B.shape[1]
    if B.shape[0] != K or tuple(D.shape) != (M, N):
        raise ValueError("shape mismatch")
    o = GemmOutput()
    o.beta = float(beta)
    o.C, o.ldc = 0, max(N, 1)
    if C is not None:
        if C.dtype != torch.float32 or tuple(C.shape) != (M, N):
            raise TypeError("C must be a float32 (M, N) tensor")
        o.C, o.ldc = C.data_ptr(), _row_major_ld(C, "C")
    o.bias = 0
    if bias is not None:
        if bias.dtype != torch.float32 or bias.numel() != N or not bias.is_contiguous():
            raise TypeError("bias must be a contiguous float32 tensor of N values")
        o.bias = bias.data_ptr()
    o.act = ACT[act]
    o.residual, o.ldr = 0, max(N, 1)
    if residual is not None:
        if residual.dtype != torch.float32 or tuple(residual.shape) != (M, N):
            raise TypeError("residual must be a float32 (M, N) tensor")
        o.residual, o.ldr = residual.data_ptr(), _row_major_ld(residual, "residual")
    o.d_scale = float(d_scale)
    o.amax = 0
    if amax is not None:
        if amax.dtype != torch.float32 or amax.numel() != 1 or not amax.is_cuda:
            raise TypeError("amax must be a float32 CUDA tensor of one element")
        o.amax = amax.data_ptr()
    o.D, o.ldd, o.d_type = D.data_ptr(), _row_major_ld(D, "D"), _out_type(torch, D)
    st = gemm_bf16gemm_fused(M, N, K, float(alpha), A.data_ptr(), _row_major_ld(A, "A"),
                             B.data_ptr(), _row_major_ld(B, "B"), o, _stream_handle(stream, D.device))
    if st != 0:
        raise GemmError(st, "gemm_bf16gemm_fused")
    return D
