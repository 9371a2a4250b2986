"""Seeded synthetic inputs for the GEMM workloads.

This module draws random matrices and nothing else: it holds none of the
GEMM's arithmetic, so both the CUDA path's tests and the oracle can take their
inputs from it.  Every draw is on the CPU with a ``torch.Generator`` seeded per
workload, in the order A, then B, then C, in fp32, so the inputs do not depend
on the device.  bf16 inputs are the fp32 draws rounded to nearest-even by
``Tensor.to(torch.bfloat16)``.

Distributions:
  * ``uniform``  -- U[-1, 1), drawn as 2*rand - 1
  * ``normal``   -- N(0, sigma^2), drawn as sigma * randn
  * ``int``      -- integers in [-4, 4] inclusive (randint(-4, 5))

The shapes and scalars are those of the workloads this library is measured on:
square fp32 SGEMM at 4092 and 4096 (the sizes used by "A GEMM Kernel, Step by
Step" and "GEMM Worklog I"), a ragged fp32 shape, a bf16 square GEMM and the
decode shape M <= 16 ("Tiled matrix multiplication", "Avoid when").
"""
from __future__ import annotations

from dataclasses import dataclass, field

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    M: int
    N: int
    K: int
    alpha: float
    beta: float
    dtype: str            # "f32" or "bf16" (input type; C is always fp32)
    dist_a: tuple
    dist_b: tuple
    dist_c: tuple
    seed: int
    note: str = field(default="", compare=False)

    @property
    def flops(self) -> int:
        return 2 * self.M * self.N * self.K


# (kind, parameter): ("uniform", None), ("normal", sigma), ("int", None)
U = ("uniform", None)
I4 = ("int", None)


def N_(sigma):
    return ("normal", float(sigma))


WORKLOADS = {
    # 256^3, alpha 1.5, beta -0.5, U[-1,1) from seed 0
    "sgemm_256": Workload("sgemm_256", 256, 256, 256, 1.5, -0.5, "f32", U, U, U, 0),
    # same shape, integers in [-4, 4]: every partial sum is exact in fp32
    "sgemm_256_int": Workload("sgemm_256_int", 256, 256, 256, 1.5, -0.5, "f32",
                              I4, I4, I4, 0),
    # 4092^3 (not a tile multiple), alpha 0.7, beta 0.3, U[-1,1)
    "sgemm_4092": Workload("sgemm_4092", 4092, 4092, 4092, 0.7, 0.3, "f32", U, U, U, 1),
    # 4096^3, alpha 1, beta 0, N(0,1)
    "sgemm_4096": Workload("sgemm_4096", 4096, 4096, 4096, 1.0, 0.0, "f32",
                           N_(1.0), N_(1.0), N_(1.0), 2),
    # ragged 3000 x 5000 x 1999, N(0,1): lda*4 = 7996 B is not 16-B aligned
    "sgemm_ragged": Workload("sgemm_ragged", 3000, 5000, 1999, 1.0, 0.0, "f32",
                             N_(1.0), N_(1.0), N_(1.0), 2),
    # bf16 inputs, fp32 accumulate and output, 8192^3, N(0, 0.02)
    "bf16_8192": Workload("bf16_8192", 8192, 8192, 8192, 1.0, 0.0, "bf16",
                          N_(0.02), N_(0.02), N_(1.0), 3),
    # decode shape: M=16, N=12288, K=4096, beta=1 with C ~ U[-1,1)
    "decode_16": Workload("decode_16", 16, 12288, 4096, 1.0, 1.0, "bf16",
                          N_(1.0), N_(0.02), U, 4),
}


def _draw(gen: torch.Generator, shape, dist) -> torch.Tensor:
    kind, param = dist
    if kind == "uniform":
        return torch.rand(shape, generator=gen, dtype=torch.float32) * 2.0 - 1.0
    if kind == "normal":
        return torch.randn(shape, generator=gen, dtype=torch.float32) * param
    if kind == "int":
        return torch.randint(-4, 5, shape, generator=gen).to(torch.float32)
    raise ValueError("unknown distribution %r" % (kind,))


def make_inputs(M, N, K, dist_a=U, dist_b=U, dist_c=U, seed=0, dtype="f32",
                with_c=True):
    """Return (A, B, C) CPU tensors.

    A is (M, K), B is (K, N), C is (M, N) fp32 (None if ``with_c`` is false).
    For dtype "bf16", A and B are returned as torch.bfloat16 tensors rounded
    to nearest-even from the fp32 draws.
    """
    gen = torch.Generator(device="cpu")
    gen.manual_seed(int(seed))
    A = _draw(gen, (M, K), dist_a)
    B = _draw(gen, (K, N), dist_b)
    C = _draw(gen, (M, N), dist_c) if with_c else None
    if dtype == "bf16":
        A = A.to(torch.bfloat16)
        B = B.to(torch.bfloat16)
    elif dtype != "f32":
        raise ValueError("dtype must be 'f32' or 'bf16'")
    return A, B, C


def workload_inputs(w: Workload, with_c=True):
    """Inputs of a named workload (see WORKLOADS)."""
    return make_inputs(w.M, w.N, w.K, w.dist_a, w.dist_b, w.dist_c, w.seed,
                       w.dtype, with_c=with_c)


def bf16_bits(t: torch.Tensor):
    """The uint16 bit patterns of a bf16 tensor, as a numpy array."""
    if t.dtype != torch.bfloat16:
        raise TypeError("expected a bfloat16 tensor")
    return t.contiguous().view(torch.int16).numpy().view("uint16")


def strided_copy(t: torch.Tensor, ld: int, fill=float("nan")):
    """Copy a 2-D tensor into a wider buffer with row stride ``ld``.

    The padding columns hold ``fill`` (a sentinel the GEMM must neither read
    into its result nor overwrite).  Returns (buffer, view).
    """
    rows, cols = t.shape
    if ld < cols:
        raise ValueError("ld < number of columns")
    buf = torch.full((max(rows, 1), ld), fill, dtype=t.dtype)
    view = buf[:rows, :cols]
    view.copy_(t)
    return buf, view
