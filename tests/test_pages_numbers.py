"""Roofline and launch-quantization helpers against the pages' printed numbers.

The fixtures live in tests/golden/pages_numbers.txt, one fact per line with
its citation.  Each test recomputes the fact from the helpers and compares.
The quantization facts go through the C ABI's host-only gemm_quantization.
"""
import math
import os

import pytest

from dense_gemm_12_gb300 import roofline as rf

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "pages_numbers.txt")


def _load():
    facts = {}
    for line in open(GOLDEN):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        key, value, tol, cite = [x.strip() for x in line.split("|")]
        vals = [float(v) for v in value.split(",")]
        facts[key] = (vals if len(vals) > 1 else vals[0], tol, cite)
    return facts


FACTS = _load()


def check(key, got):
    want, tol, cite = FACTS[key]
    if isinstance(want, list):
        assert len(got) == len(want), key
        for g, w in zip(got, want):
            _cmp(key, g, w, tol, cite)
    else:
        _cmp(key, got, want, tol, cite)


def _cmp(key, got, want, tol, cite):
    if tol == "exact":
        assert got == want, "%s: got %r, page says %r (%s)" % (key, got, want, cite)
    else:
        assert math.isclose(got, want, rel_tol=float(tol)), \
            "%s: got %r, page says %r (%s)" % (key, got, want, cite)


PEAK, BW = FACTS["a6000_peak_flops"][0], FACTS["a6000_bw_bytes"][0]


def test_a6000_roofline():
    check("a6000_ridge", rf.ridge(PEAK, BW))
    check("a6000_datasheet_ridge", rf.ridge(38.7e12, BW))
    n = 4092
    f = rf.gemm_flops(n, n, n)
    b = rf.gemm_bytes(n, n, n, read_c=True)
    check("sgemm4092_gflop", f / 1e9)
    check("sgemm4092_read_mb", 3 * n * n * 4 / 1e6)
    check("sgemm4092_write_mb", n * n * 4 / 1e6)
    check("sgemm4092_total_mb", b / 1e6)
    check("sgemm4092_intensity", rf.intensity(f, b))
    check("sgemm4092_mem_ms", b / BW * 1e3)
    check("sgemm4092_compute_ms", f / PEAK * 1e3)
    check("sgemm4092_ratio", (f / PEAK) / (b / BW))


@pytest.mark.parametrize("m,n", [(1, 1), (32, 32), (64, 64), (128, 128), (128, 256)])
def test_ceiling_table(m, n):
    i = rf.tile_intensity(m, n)
    check("tile_%dx%d" % (m, n), [round(i, 2), rf.ceiling(i, PEAK, BW) / 1e9])


def test_rung_one():
    check("naive_floats_per_thread", 2 * 4092)
    check("naive_bytes_per_thread", 2 * 4092 * 4)
    check("naive_ceiling_gflops", rf.ceiling(rf.naive_intensity(), PEAK, BW) / 1e9)
    check("naive_fraction_of_roof", rf.ceiling(rf.naive_intensity(), PEAK, BW) / PEAK)


def test_rungs_three_to_five():
    check("block32_intensity", rf.tile_intensity(32, 32))
    check("column_products_per_load", rf.shared_loads_per_product(8, 1))
    check("square_products_per_load", rf.shared_loads_per_product(8, 8))
    check("regs_64acc_256thr", 64 * 256)
    blocks = rf.blocks_per_sm_by_registers(64, 256)
    check("blocks_per_sm_64acc", blocks)
    check("warps_resident_64acc", blocks * 256 // 32)
    check("occupancy_64acc", blocks * 256 / 32 / 48)


def test_last_rung_hierarchy():
    check("warp_tiles_down", 128 // 32)
    check("warp_tiles_across", 128 // 64)
    check("thread_tiles_per_warp", (32 // 8) * (64 // 8))
    check("double_buffer_bytes", 2 * (128 * 8 + 8 * 128) * 4)


def test_fringe_quantization(gemm_lib):
    q = gemm_lib.gemm_quantization(4092, 4092, 128, 128, 84, 4)
    check("fringe4092_tiles_side", q["tiles_m"])
    check("fringe4092_covered", q["covered_m"])
    check("fringe4092_last_band", 4092 - (q["tiles_m"] - 1) * 128)
    check("fringe4092_extra", 1.0 / q["useful_fraction"] - 1.0)
    q = gemm_lib.gemm_quantization(300, 300, 128, 128, 84, 4)
    check("fringe300_tiles_side", q["tiles_n"])
    check("fringe300_ratio", 300 / 128)
    check("fringe300_covered", q["covered_n"])
    check("fringe300_useful", q["useful_fraction"])


def test_wave_quantization(gemm_lib):
    q = gemm_lib.gemm_quantization(4092, 4092, 128, 128, 84, 4)
    check("wave_a6000_per_wave", q["per_wave"])
    check("wave_a6000_tiles", q["tiles"])
    check("wave_a6000_ratio", q["tiles"] / q["per_wave"])
    check("wave_a6000_waves", q["waves"])
    check("wave_a6000_last_blocks", q["tiles"] - (q["waves"] - 1) * q["per_wave"])
    check("wave_a6000_efficiency", q["wave_efficiency"])
    # 336 and 337 tiles (one row of tiles), 84 x 4 slots
    check("wave_336_waves", gemm_lib.gemm_quantization(128, 336 * 128, 128, 128, 84, 4)["waves"])
    check("wave_337_waves", gemm_lib.gemm_quantization(128, 337 * 128, 128, 128, 84, 4)["waves"])
    check("wave_h100pcie_114", gemm_lib.gemm_quantization(128, 114 * 128, 128, 128, 114, 1)["waves"])
    check("wave_h100pcie_115", gemm_lib.gemm_quantization(128, 115 * 128, 128, 128, 114, 1)["waves"])
    check("wave_two_per_sm", gemm_lib.gemm_quantization(4092, 4092, 128, 128, 84, 2)["per_wave"])
    check("h100_wave_132_133", gemm_lib.gemm_quantization(128, 133 * 128, 128, 128, 132, 1)["waves"])
    # the page's remark: two blocks per SM waste less on the same 1024 tiles
    q2 = gemm_lib.gemm_quantization(4092, 4092, 128, 128, 84, 2)
    assert q2["wave_efficiency"] > q["wave_efficiency"]


def test_quantization_rejects_bad_args(gemm_lib):
    with pytest.raises(gemm_lib.GemmError):
        gemm_lib.gemm_quantization(-1, 4, 128, 128, 1, 1)
    with pytest.raises(gemm_lib.GemmError):
        gemm_lib.gemm_quantization(4, 4, 0, 128, 1, 1)
    q = gemm_lib.gemm_quantization(0, 4, 128, 128, 1, 1)
    assert q["tiles"] == 0 and q["useful_fraction"] == 1.0


def test_a100_worklog():
    n = 4096
    f = rf.gemm_flops(n, n, n)
    check("a100_flops_4096", f)
    check("a100_naive_bytes", rf.tiled_traffic_bytes(n, n, n, 1, 1))
    check("a100_naive_intensity", rf.naive_intensity())
    check("a100_ridge", rf.ridge(19.5e12, 2039e9))
    check("a100_naive_ceiling", rf.ceiling(rf.naive_intensity(), 19.5e12, 2039e9))
    check("a100_naive_ceiling_frac", rf.ceiling(rf.naive_intensity(), 19.5e12, 2039e9) / 19.5e12)
    check("a100_tiled_intensity", rf.naive_intensity() * 32)
    check("a100_tiled_traffic", rf.tiled_traffic_bytes(n, n, n, 32, 32))
    for key, ms in (("a100_table_naive", 528.4), ("a100_table_tiled", 19.3),
                    ("a100_table_cublas", 7.5)):
        t = ms * 1e-3
        check(key, [t, f / t, f / t / 19.5e12])


def test_h100_constants():
    n = 4096
    f = rf.gemm_flops(n, n, n)
    check("h100_gflop_4096", f / 1e9)
    check("h100_ms_4096", f / 989e12 * 1e3)
    check("h100_bf16_operand_mb", 3 * n * n * 2 / 1e6)
    check("h100_ridge", rf.ridge(989e12, 3.35e12))
    check("h100_tile128_intensity", rf.tile_intensity(128, 128))
