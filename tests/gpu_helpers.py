"""Helpers for the GPU parity tests: device buffers with padded leading
dimensions and guard bands, calls through the C ABI, and oracle comparison.

Tolerances (per element, relative to den = |alpha| (|A||B|)_ij + |beta| |C_ij|):
  fp32 path: 2e-6 * sqrt(K)
  bf16 path: 8e-3 (against the oracle on the same bf16-rounded inputs)
"""
from __future__ import annotations

import math

import numpy as np
import torch

import dense_gemm_12_gb300 as g
import oracle

SENTINEL = 1.2345e30  # value planted in padding and guard bands


def tol_fp32(K):
    return 2e-6 * math.sqrt(max(K, 1))


TOL_BF16 = 8e-3


class DeviceMatrix:
    """A row-major matrix inside a larger device buffer.

    The buffer has `guard` rows of sentinel above and below and row pitch
    `ld`; columns past the logical width are sentinel too.  `offset_elems`
    shifts the matrix start (to make the base pointer misaligned).
    """

    def __init__(self, host: torch.Tensor, ld: int | None = None, guard: int = 2,
                 offset_elems: int = 0, device="cuda"):
        rows, cols = host.shape
        self.rows, self.cols = rows, cols
        self.ld = ld if ld is not None else max(cols, 1)
        assert self.ld >= max(cols, 1)
        self.guard = guard
        self.offset = offset_elems
        total = (rows + 2 * guard) * self.ld + offset_elems + 8
        fill = SENTINEL if host.dtype == torch.float32 else 7.0
        self.buf = torch.full((total,), fill, dtype=host.dtype)
        start = guard * self.ld + offset_elems
        if rows > 0 and cols > 0:
            view = self.buf[start:start + rows * self.ld].view(rows, self.ld)[:, :cols]
            view.copy_(host)
        self.buf = self.buf.to(device)
        self.start = start
        self.host_initial = self.buf.cpu().clone()

    @property
    def ptr(self) -> int:
        return self.buf.data_ptr() + self.start * self.buf.element_size()

    def logical(self) -> torch.Tensor:
        b = self.buf.cpu()
        if self.rows == 0 or self.cols == 0:
            return torch.empty((self.rows, self.cols), dtype=b.dtype)
        return b[self.start:self.start + self.rows * self.ld].view(self.rows, self.ld)[:, :self.cols].clone()

    def untouched_outside(self) -> bool:
        """True if every element outside the logical matrix is unchanged."""
        now = self.buf.cpu()
        mask = torch.ones_like(now, dtype=torch.bool)
        if self.rows > 0 and self.cols > 0:
            idx = (self.start + torch.arange(self.rows)[:, None] * self.ld
                   + torch.arange(self.cols)[None, :]).reshape(-1)
            mask[idx] = False
        a = now[mask]
        b = self.host_initial[mask]
        if a.dtype == torch.float32:
            return bool(torch.equal(a.view(torch.int32), b.view(torch.int32)))
        return bool(torch.equal(a, b))


def run_sgemm(A, B, C, alpha, beta, lda=None, ldb=None, ldc=None, offsets=(0, 0, 0),
              stream=0):
    """Run gemm_sgemm on device copies; return (result, status, dA, dB, dC)."""
    dA = DeviceMatrix(A, lda, offset_elems=offsets[0])
    dB = DeviceMatrix(B, ldb, offset_elems=offsets[1])
    dC = DeviceMatrix(C, ldc, offset_elems=offsets[2])
    M, K = A.shape
    N = B.shape[1]
    st = g.gemm_sgemm(M, N, K, alpha, dA.ptr, dA.ld, dB.ptr, dB.ld, beta, dC.ptr, dC.ld, stream)
    torch.cuda.synchronize()
    return dC.logical(), st, dA, dB, dC


def run_bf16gemm(A, B, C, alpha, beta, lda=None, ldb=None, ldc=None, offsets=(0, 0, 0),
                 stream=0):
    dA = DeviceMatrix(A, lda, offset_elems=offsets[0])
    dB = DeviceMatrix(B, ldb, offset_elems=offsets[1])
    dC = DeviceMatrix(C, ldc, offset_elems=offsets[2])
    M, K = A.shape
    N = B.shape[1]
    st = g.gemm_bf16gemm(M, N, K, alpha, dA.ptr, dA.ld, dB.ptr, dB.ld, beta, dC.ptr, dC.ld,
                         stream)
    torch.cuda.synchronize()
    return dC.logical(), st, dA, dB, dC


def oracle_sgemm(A, B, C, alpha, beta, want64=True):
    return oracle.sgemm(alpha, A.numpy(), B.numpy(), beta, C.numpy(), want64=want64)


def bits(t):
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def oracle_bf16(A, B, C, alpha, beta, want64=True):
    return oracle.bf16gemm(alpha, bits(A), bits(B), beta, C.numpy(), want64=want64)


def ratio(C_gpu, ref64, den):
    return oracle.error_ratio(C_gpu.numpy(), ref64, den)


def check_device_error():
    st = g.gemm_check_device_error(0)
    assert st == 0, g.gemm_status_string(st)
