"""Host-side checks of the C ABI (no GPU needed, no kernel launched).

* the library loads and exports every function include/gemm12.h declares;
* argument validation returns the documented status before any device work;
* kernel-path selection follows the alignment / shape rules in the header;
* with no usable device the entry points fail loudly (GEMM_ERR_UNSUPPORTED):
  there is no CPU fallback.
"""
import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "gemm12.h")

OK, INVALID, MISALIGNED, UNSUPPORTED = 0, 1, 2, 3


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(gemm_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_entry_points():
    names = declared_functions()
    for required in ("gemm_sgemm", "gemm_bf16gemm", "gemm_status_string",
                     "gemm_check_device_error", "gemm_shutdown"):
        assert required in names


def test_library_exports_every_declared_symbol(gemm_lib):
    path = gemm_lib.library_path()
    out = subprocess.run(["nm", "-D", "--defined-only", path], capture_output=True, text=True,
                         check=True).stdout
    exported = set(line.split()[-1] for line in out.splitlines() if line.strip())
    missing = [n for n in declared_functions() if n not in exported]
    assert not missing, "declared but not exported: %s" % missing
    lib = ctypes.CDLL(path)
    for n in declared_functions():
        assert getattr(lib, n) is not None


def test_status_strings(gemm_lib):
    for code, name in gemm_lib.STATUS.items():
        s = gemm_lib.gemm_status_string(code)
        assert s.startswith(name), (code, s)
    assert "unknown" in gemm_lib.gemm_status_string(99)


def test_version(gemm_lib):
    assert gemm_lib.gemm_version() >= 100


# Fake device addresses: only inspected for alignment by gemm_select_path,
# never dereferenced (no GPU work is issued in this file).
P = 1 << 20


@pytest.mark.parametrize("case,expect", [
    (dict(bf16=0, M=0, N=5, K=5), "none"),
    (dict(bf16=0, M=5, N=0, K=5), "none"),
    (dict(bf16=0, M=5, N=5, K=0), "scale_c"),
    (dict(bf16=0, M=5, N=5, K=5, alpha=0.0), "scale_c"),
    (dict(bf16=0, M=4092, N=4092, K=4092), "simt_tma"),
    # operands TMA cannot describe: staged when the copy is cheap next to the
    # GEMM (fp32: >= 2^31 FLOPs, N >= 256 to copy A, M >= 256 to copy B)
    (dict(bf16=0, M=3000, N=5000, K=1999), "simt_staged"),        # lda*4 = 7996 B
    (dict(bf16=0, M=1000, N=1000, K=999), "simt_generic"),        # 2.0e9 < 2^31 FLOPs
    (dict(bf16=0, M=8192, N=255, K=1023), "simt_generic"),        # A copy too large
    (dict(bf16=0, M=255, N=8192, K=1024, ldb=8193), "simt_generic"),  # B copy too large
    (dict(bf16=0, M=256, N=8192, K=1024, ldb=8193), "simt_staged"),
    (dict(bf16=0, M=2048, N=2048, K=2048, A=P + 4), "simt_staged"),  # A base + 4 B
    (dict(bf16=0, M=64, N=64, K=64, A=P + 4), "simt_generic"),     # A not 16-B aligned
    (dict(bf16=0, M=64, N=64, K=64, ldb=66), "simt_generic"),      # B pitch 264 B
    (dict(bf16=1, M=8192, N=8192, K=8192), "tc_bf16_pair"),
    (dict(bf16=1, M=128, N=8192, K=8192), "tc_decode"),          # two row blocks of 64
    (dict(bf16=1, M=128, N=16392, K=8192), "tc_bf16"),
    (dict(bf16=1, M=129, N=8192, K=8192), "tc_bf16_pair"),        # 64 groups x 3 row blocks
    (dict(bf16=1, M=256, N=4096, K=4096), "tc_decode"),           # 32 groups x 4 row blocks
    (dict(bf16=1, M=512, N=2048, K=1024), "tc_decode"),           # 16 x 8
    (dict(bf16=1, M=320, N=4096, K=4096), "tc_decode"),           # 160, K >= 4096
    (dict(bf16=1, M=320, N=4096, K=1024), "tc_bf16_pair"),        # 160 at small K
    (dict(bf16=1, M=513, N=1024, K=1024), "tc_bf16_pair"),        # beyond eight row blocks
    (dict(bf16=1, M=16, N=12288, K=4096), "tc_decode"),
    (dict(bf16=1, M=1, N=12288, K=4096), "tc_decode"),
    (dict(bf16=1, M=17, N=12288, K=4096), "tc_decode"),
    (dict(bf16=1, M=64, N=4096, K=4096), "tc_decode"),
    (dict(bf16=1, M=65, N=4096, K=4096), "tc_decode"),
    (dict(bf16=1, M=65, N=16384, K=4096), "tc_decode"),
    (dict(bf16=1, M=65, N=16512, K=4096), "tc_bf16"),
    (dict(bf16=1, M=32, N=28672, K=4096), "tc_decode"),
    (dict(bf16=1, M=33, N=16384, K=8192), "tc_decode"),
    (dict(bf16=1, M=33, N=16392, K=4096), "tc_bf16"),            # wide N: tile kernels
    (dict(bf16=1, M=64, N=64, K=60), "simt_bf16"),                 # lda*2 = 120 B
    (dict(bf16=1, M=64, N=64, K=64, B=P + 2), "simt_bf16"),
    # bf16: staged for the tile kernels (M > 16) from 2^24 FLOPs
    (dict(bf16=1, M=256, N=256, K=127), "simt_bf16"),             # 1.66e7 < 2^24
    (dict(bf16=1, M=256, N=256, K=129), "tc_staged"),
    (dict(bf16=1, M=17, N=4096, K=4095), "tc_staged"),
    (dict(bf16=1, M=16, N=4096, K=4095), "simt_bf16"),            # decode shape
    (dict(bf16=1, M=4096, N=4096, K=4096, A=P + 2), "tc_staged"),
    (dict(bf16=0, M=5, N=5, K=5, lda=4), "none"),                  # invalid: lda < K
])
def test_select_path(gemm_lib, case, expect):
    c = dict(alpha=1.0, A=P, B=P, lda=None, ldb=None)
    c.update(case)
    lda = c["lda"] if c["lda"] is not None else max(c["K"], 1)
    ldb = c["ldb"] if c["ldb"] is not None else max(c["N"], 1)
    got = gemm_lib.gemm_select_path(c["bf16"], c["M"], c["N"], c["K"], c["alpha"], c["A"], lda,
                                    c["B"], ldb)
    assert got == expect


@pytest.mark.parametrize("fn", ["gemm_sgemm", "gemm_bf16gemm"])
@pytest.mark.parametrize("args,status", [
    ((-1, 4, 4, 4, 4, 4), INVALID),        # M < 0
    ((4, -1, 4, 4, 4, 4), INVALID),        # N < 0
    ((4, 4, -1, 4, 4, 4), INVALID),        # K < 0
    ((4, 4, 8, 7, 4, 4), INVALID),         # lda < K
    ((4, 8, 4, 4, 7, 8), INVALID),         # ldb < N
    ((4, 8, 4, 4, 8, 7), INVALID),         # ldc < N
    ((1 << 31, 4, 4, 4, 4, 4), INVALID),   # M too large
    ((0, 4, 4, 4, 4, 4), OK),              # empty: nothing launched
    ((4, 0, 4, 4, 4, 4), OK),
])
def test_argument_validation(gemm_lib, fn, args, status):
    M, N, K, lda, ldb, ldc = args
    f = getattr(gemm_lib, fn)
    assert f(M, N, K, 1.0, P, lda, P, ldb, 0.0, P, ldc, 0) == status


def test_null_c_rejected(gemm_lib):
    assert gemm_lib.gemm_sgemm(4, 4, 4, 1.0, P, 4, P, 4, 0.0, 0, 4, 0) == INVALID
    assert gemm_lib.gemm_bf16gemm(4, 4, 4, 1.0, P, 4, P, 4, 0.0, 0, 4, 0) == INVALID


def test_null_operand_rejected(gemm_lib):
    assert gemm_lib.gemm_sgemm(4, 4, 4, 1.0, 0, 4, P, 4, 0.0, P, 4, 0) == INVALID
    assert gemm_lib.gemm_bf16gemm(4, 4, 4, 1.0, P, 4, 0, 4, 0.0, P, 4, 0) == INVALID


def test_misaligned_pointers(gemm_lib):
    assert gemm_lib.gemm_bf16gemm(4, 4, 4, 1.0, P + 1, 4, P, 4, 0.0, P, 4, 0) == MISALIGNED
    assert gemm_lib.gemm_bf16gemm(4, 4, 4, 1.0, P, 4, P + 1, 4, 0.0, P, 4, 0) == MISALIGNED
    # fp32 operands must be at least 4-byte aligned
    assert gemm_lib.gemm_sgemm(4, 4, 4, 1.0, P + 2, 4, P, 4, 0.0, P, 4, 0) == INVALID
    assert gemm_lib.gemm_sgemm(4, 4, 4, 1.0, P, 4, P, 4, 0.0, P + 2, 4, 0) == INVALID


def _no_cuda():
    try:
        import torch
        return not torch.cuda.is_available()
    except Exception:
        return True


@pytest.mark.skipif(not _no_cuda(), reason="checks the no-device path; a GPU is present")
def test_fails_loudly_without_device(gemm_lib):
    # Valid arguments, no device: the library refuses, it does not compute on
    # the host.
    assert gemm_lib.gemm_sgemm(4, 4, 4, 1.0, P, 4, P, 4, 0.0, P, 4, 0) == UNSUPPORTED
    assert gemm_lib.gemm_bf16gemm(4, 4, 4, 1.0, P, 4, P, 4, 0.0, P, 4, 0) == UNSUPPORTED
    assert gemm_lib.gemm_sgemm(4, 4, 0, 1.0, P, 4, P, 4, 2.0, P, 4, 0) == UNSUPPORTED
    # the split plan depends on the device's SM count: no device, no plan
    assert gemm_lib.gemm_split_parts(0, 4096, 4096, 4096) == 0
    assert gemm_lib.gemm_split_parts(1, 8192, 8192, 8192) == 0


def test_split_parts_rejects_negative_sizes(gemm_lib):
    assert gemm_lib.gemm_split_parts(0, -1, 4, 4) == 0
    assert gemm_lib.gemm_split_parts(1, 4, 4, -4) == 0
