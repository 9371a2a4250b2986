"""Roofline arithmetic for GEMM measurements.

The model is the one "A GEMM Kernel, Step by Step" works with ("What the
problem is allowed to cost"): attainable FLOP/s = min(peak, I * bandwidth),
where the arithmetic intensity I is FLOPs per byte moved and the ridge point is
peak / bandwidth.  "GEMM Worklog I" (section 1) and "Tiled matrix
multiplication" ("Efficiency") apply the same model to the A100 and H100.

Work and traffic are counted as the pages count them: 2*M*N*K FLOPs (the
multiply-add of every term; the alpha/beta scaling is not counted -- the pages
differ on it and it is ~3*M*N, under 0.1 % at the sizes measured) and the
algorithmic bytes every GEMM must move: read A and B once, read C once if
beta != 0, write C once.
"""
from __future__ import annotations


def gemm_flops(M: int, N: int, K: int) -> int:
    """2*M*N*K: one multiply and one add per term of every dot product."""
    return 2 * M * N * K


def gemm_bytes(M: int, N: int, K: int, in_bytes: int = 4, out_bytes: int = 4,
               read_c: bool = True) -> int:
    """Minimum DRAM traffic: A and B read once, C read (if beta != 0) and written once."""
    return (M * K + K * N) * in_bytes + (2 if read_c else 1) * M * N * out_bytes


def intensity(flops: float, nbytes: float) -> float:
    return flops / nbytes


def tile_intensity(m: int, n: int, elem_bytes: int = 4) -> float:
    """FLOPs per byte of an m x n output tile fed from memory.

    Per step of k the tile reads m + n elements and does 2*m*n FLOPs, so
    I = 2*m*n / ((m + n) * elem_bytes); for fp32 that is m*n / (2*(m + n)).
    K cancels.
    """
    return 2.0 * m * n / ((m + n) * elem_bytes)


def naive_intensity(elem_bytes: int = 4) -> float:
    """One thread per output element, both operands fetched per multiply-add."""
    return 2.0 / (2 * elem_bytes)


def ceiling(i: float, peak: float, bandwidth: float) -> float:
    """Attainable FLOP/s at intensity i: min(peak, i * bandwidth)."""
    return min(peak, i * bandwidth)


def ridge(peak: float, bandwidth: float) -> float:
    return peak / bandwidth


def fp32_simt_peak(num_sms: int, clock_hz: float, lanes_per_sm: int = 128) -> float:
    """FFMA peak: every fp32 lane retires one fused multiply-add (2 FLOPs) per clock."""
    return num_sms * lanes_per_sm * 2.0 * clock_hz


def blocks_per_sm_by_registers(regs_per_thread: int, threads_per_block: int,
                               register_file: int = 65536) -> int:
    """Resident blocks allowed by the register file alone."""
    return register_file // (regs_per_thread * threads_per_block)


def gemm_roofline(M, N, K, in_bytes, read_c, peak_flops, bandwidth):
    """Roofline summary of one GEMM: flops, bytes, intensity, bound and ceiling."""
    f = gemm_flops(M, N, K)
    b = gemm_bytes(M, N, K, in_bytes=in_bytes, read_c=read_c)
    i = f / b
    c = ceiling(i, peak_flops, bandwidth)
    return {"flops": f, "bytes": b, "intensity": i,
            "bound": "compute" if i * bandwidth >= peak_flops else "hbm",
            "ceiling_flops": c}


def tiled_traffic_bytes(M: int, N: int, K: int, BM: int, BN: int, elem_bytes: int = 4) -> float:
    """Operand traffic of a BM x BN block-tiled GEMM with no cache reuse:
    every A element is fetched once per column of tiles (N/BN times) and every
    B element once per row of tiles (M/BM times): M*N*K*(1/BN + 1/BM) elements."""
    return M * N * K * (1.0 / BN + 1.0 / BM) * elem_bytes


def shared_loads_per_product(tm: int, tn: int) -> float:
    """Register tile tm x tn: per k, tm + tn shared-memory loads feed tm*tn FMAs."""
    return tm * tn / float(tm + tn)
