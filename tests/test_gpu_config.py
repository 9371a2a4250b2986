"""Pinned launch configurations (gemm_sgemm_config / gemm_bf16gemm_config) and
automatic dispatch's table on the GPU.

Every configuration computes the same GEMM: on small-integer inputs every
partial sum is exact, so each configuration's result must equal the oracle's
bit for bit, whatever kernel, k-split and raster order it uses.
"""
import os
import re

import numpy as np
import pytest
import torch

import dense_gemm_12_gb300 as g
from dense_gemm_12_gb300.workloads import make_inputs
from gpu_helpers import check_device_error, oracle_bf16, oracle_sgemm, ratio, TOL_BF16

pytestmark = pytest.mark.gpu

TABLE = os.path.join(os.path.dirname(__file__), "..", "dense_gemm_12_gb300", "csrc",
                     "dispatch_table.inc")


@pytest.fixture(scope="module", autouse=True)
def _lib(gemm_lib, cuda_device):
    yield


def _run(is_bf16, A, B, C, alpha, beta, cfg):
    M, K = A.shape
    N = B.shape[1]
    dA, dB, dC = A.cuda(), B.cuda(), C.cuda()
    fn = g.gemm_bf16gemm_config if is_bf16 else g.gemm_sgemm_config
    st = fn(M, N, K, alpha, dA.data_ptr(), K, dB.data_ptr(), N, beta, dC.data_ptr(), N, cfg,
            torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    return st, dC.cpu()


BF16_CONFIGS = [
    {"kernel": k, "split": s, "group_m": gm}
    for k in ("single_cta", "cta_pair") for s in (1, 3, 8) for gm in (1, 5)
]


# beta = 0 with a plain fp32 output writes whole tiles through TMA stores (the
# split parts' fix-up keeps the staged output stage); beta != 0 reads C.
@pytest.mark.parametrize("beta", [-0.5, 0.0])
@pytest.mark.parametrize("M,N,K", [(8, 520, 1024), (100, 1000, 1024), (300, 776, 2048),
                                   (1024, 1024, 512)])
def test_bf16_every_config_exact(M, N, K, beta):
    A, B, C = make_inputs(M, N, K, ("int", None), ("int", None), ("int", None), seed=M + N,
                          dtype="bf16")
    ref32, _, _ = oracle_bf16(A, B, C, 1.5, beta)
    for cfg in BF16_CONFIGS + [None, {"split": 2}, {"group_m": 64}]:
        st, out = _run(True, A, B, C, 1.5, beta, cfg)
        assert st == 0, cfg
        assert np.array_equal(out.numpy(), ref32), cfg
    check_device_error()


@pytest.mark.parametrize("cfg", [{"kernel": "single_cta", "split": 1},
                                 {"kernel": "single_cta", "split": 3},
                                 {"kernel": "cta_pair", "split": 1},
                                 {"kernel": "cta_pair", "split": 2},
                                 {"kernel": "cta_pair", "split": -1}])
def test_bf16_tma_output_edges_and_padded_rows(cfg):
    # ragged M and N (the tensor map clips the last tiles), rows of ldc > N
    # whose padding must stay untouched, and a pitch TMA cannot describe
    # (ldc = N + 1: the staged output stage instead); beta = 0
    M, N, K = 1000, 1300, 1500
    A, B, C = make_inputs(M, N, K, ("int", None), ("int", None), ("int", None), seed=31,
                          dtype="bf16")
    ref32, _, _ = oracle_bf16(A, B, C, -2.0, 0.0)
    dA, dB = A.cuda(), B.cuda()
    for ldc in (N, N + 12, N + 1):
        dC = torch.full((M, ldc), -7.0, device="cuda")
        st = g.gemm_bf16gemm_config(M, N, K, -2.0, dA.data_ptr(), K, dB.data_ptr(), N, 0.0,
                                    dC.data_ptr(), ldc, cfg,
                                    torch.cuda.current_stream().cuda_stream)
        torch.cuda.synchronize()
        assert st == 0, (cfg, ldc)
        out = dC.cpu()
        assert torch.all(out[:, N:] == -7.0), (cfg, ldc)
        assert np.array_equal(out[:, :N].numpy().view(np.uint32), ref32.view(np.uint32)), \
            (cfg, ldc)
    check_device_error()


@pytest.mark.parametrize("M,N,K,cfg", [
    (600, 8, 300, None),                                   # one tile column of 8 < the 32-wide box
    (1000, 20, 520, {"kernel": "cta_pair", "split": 1}),
    (700, 36, 1000, {"kernel": "single_cta", "split": 2}),
    (777, 30, 200, None),                                  # ldc * 4 not a multiple of 16: staged
])
def test_bf16_narrow_outputs_beta_zero_exact(M, N, K, cfg):
    # tile kernels (M > 512 keeps these off the decode kernel) with outputs
    # narrower than one TMA store box; beta = 0
    A, B, C = make_inputs(M, N, K, ("int", None), ("int", None), ("int", None), seed=N + K,
                          dtype="bf16")
    ref32, _, _ = oracle_bf16(A, B, C, 1.5, 0.0)
    st, out = _run(True, A, B, C, 1.5, 0.0, cfg)
    assert st == 0
    assert np.array_equal(out.numpy().view(np.uint32), ref32.view(np.uint32))
    check_device_error()


# Stream-K tails of the tensor-core kernels (split = -1).  The tail's k-blocks
# (tail items x k-blocks per item; 128-deep on pairs, 64 on one CTA) must be
# at least the workers -- 76 resident pairs or 152 CTAs on a GB300 -- or the
# equal split runs instead; each shape below has more.
@pytest.mark.parametrize("kernel,M,N,K", [
    ("cta_pair", 1024, 2048, 4096),    # 32 pair tiles, all in the tail: 1024 k-blocks
    ("cta_pair", 2048, 10240, 2048),   # 320 pair tiles: 4 whole rounds + 16 in the tail
    ("cta_pair", 1000, 4100, 1500),    # ragged M, N and K (partial last k-block)
    ("single_cta", 128, 4096, 4096),   # 16 tiles, 1024 k-blocks
    ("single_cta", 200, 3000, 1000),   # 24 tiles, ragged
])
def test_bf16_stream_k_exact_and_repeatable(kernel, M, N, K):
    A, B, C = make_inputs(M, N, K, ("int", None), ("int", None), ("int", None), seed=M + K,
                          dtype="bf16")
    for gm, beta in ((1, -0.5), (8, 0.0)):
        ref32, _, _ = oracle_bf16(A, B, C, 1.5, beta)
        cfg = {"kernel": kernel, "split": -1, "group_m": gm}
        first = None
        for _ in range(2):
            st, out = _run(True, A, B, C, 1.5, beta, cfg)
            assert st == 0, cfg
            assert np.array_equal(out.numpy().view(np.uint32), ref32.view(np.uint32)), cfg
            if first is not None:
                assert torch.equal(out, first)
            first = out
    check_device_error()


@pytest.mark.parametrize("kernel,M,N,K", [("cta_pair", 1000, 4100, 1500),
                                          ("single_cta", 128, 4096, 4096)])
def test_bf16_stream_k_random_within_bound(kernel, M, N, K):
    A, B, C = make_inputs(M, N, K, ("normal", 1.0), ("normal", 0.05), ("uniform", None),
                          seed=7 + M, dtype="bf16")
    _, ref64, den = oracle_bf16(A, B, C, 0.7, 0.3)
    st, out = _run(True, A, B, C, 0.7, 0.3, {"kernel": kernel, "split": -1, "group_m": 0})
    assert st == 0
    assert ratio(out, ref64, den) <= TOL_BF16
    check_device_error()


@pytest.mark.parametrize("M,N,K", [(100, 260, 1024), (1000, 1300, 600), (2048, 1280, 1024),
                                   (2600, 2900, 333)])
def test_fp32_every_config_exact(M, N, K):
    # both tile widths, equal k-splits and the stream-K tail (-1): 2600 x 2900
    # has whole rounds and a tail on either width
    A, B, C = make_inputs(M, N, K, ("int", None), ("int", None), ("int", None), seed=M + K)
    ref32, _, _ = oracle_sgemm(A, B, C, 1.5, -0.5)
    for kernel in ("single_cta", "wide"):
        for s in (1, 2, 7, -1):
            for gm in (1, 3, 16):
                cfg = {"kernel": kernel, "split": s, "group_m": gm}
                st, out = _run(False, A, B, C, 1.5, -0.5, cfg)
                assert st == 0, cfg
                assert np.array_equal(out.numpy().view(np.uint32), ref32.view(np.uint32)), cfg
    check_device_error()


@pytest.mark.parametrize("M,N,K", [(4092, 4092, 4092), (3000, 5000, 1999), (129, 4100, 3000)])
def test_fp32_stream_k_and_wide_within_bound(M, N, K):
    # random inputs at the sizes the planner sends to the stream-K tail; rows
    # sampled against the oracle, and every configuration must agree with the
    # others within the bound (the k order of the sums differs between them)
    A, B, C = make_inputs(M, N, K, ("uniform", None), ("uniform", None), ("uniform", None),
                          seed=M % 97 + K)
    idx = torch.arange(0, M, max(1, M // 23))
    _, ref64, den = oracle_sgemm(A[idx].contiguous(), B, C[idx].contiguous(), 0.7, 0.3)
    tol = 2e-6 * K ** 0.5
    for cfg in ({"kernel": "wide", "split": -1}, {"kernel": "single_cta", "split": -1},
                {"kernel": "wide", "split": 2}, None):
        st, out = _run(False, A, B, C, 0.7, 0.3, cfg)
        assert st == 0, cfg
        assert ratio(out[idx], ref64, den) <= tol, cfg
    check_device_error()


def test_fp32_stream_k_is_reproducible():
    # fixed segment boundaries and a fixed order of the partial sums: two
    # launches give the same bits
    M, N, K = 3000, 5000, 1999
    A, B, C = make_inputs(M, N, K, ("uniform", None), ("uniform", None), ("uniform", None), seed=9)
    cfg = {"kernel": "wide", "split": -1}
    _, a = _run(False, A, B, C, 0.7, 0.3, cfg)
    _, b = _run(False, A, B, C, 0.7, 0.3, cfg)
    assert torch.equal(a.view(torch.int32), b.view(torch.int32))


def test_pinned_split_beyond_k_blocks_is_capped():
    # K = 64: one k-block of the bf16 kernels; a split of 8 runs as 1
    M, N, K = 512, 512, 64
    A, B, C = make_inputs(M, N, K, ("int", None), ("int", None), ("int", None), seed=3,
                          dtype="bf16")
    ref32, _, _ = oracle_bf16(A, B, C, 1.0, 1.0)
    st, out = _run(True, A, B, C, 1.0, 1.0, {"kernel": "cta_pair", "split": 8})
    assert st == 0 and np.array_equal(out.numpy(), ref32)


def test_random_inputs_within_bound_and_auto_matches_its_config():
    M, N, K = 2304, 4296, 2000
    A, B, C = make_inputs(M, N, K, ("normal", 1.0), ("normal", 0.05), ("uniform", None), seed=5,
                          dtype="bf16")
    cfg, _ = g.gemm_get_config(True, M, N, K)
    st, auto = _run(True, A, B, C, 0.7, 0.3, None)
    st2, pinned = _run(True, A, B, C, 0.7, 0.3, cfg)
    assert st == 0 and st2 == 0
    # automatic dispatch is the configuration gemm_get_config reports
    assert torch.equal(auto.view(torch.int32), pinned.view(torch.int32))
    idx = torch.arange(0, M, 97)
    _, ref64, den = oracle_bf16(A[idx].contiguous(), B, C[idx].contiguous(), 0.7, 0.3)
    assert ratio(auto[idx], ref64, den) <= TOL_BF16


def test_invalid_configs_rejected():
    M = N = K = 256
    A = torch.zeros(M, K, dtype=torch.bfloat16, device="cuda")
    B = torch.zeros(K, N, dtype=torch.bfloat16, device="cuda")
    C = torch.zeros(M, N, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    bad = [{"kernel": 3}, {"split": 9}, {"split": -2}, {"group_m": 65}, {"group_m": -2}]
    for cfg in bad:
        assert g.gemm_bf16gemm_config(M, N, K, 1.0, A.data_ptr(), K, B.data_ptr(), N, 0.0,
                                      C.data_ptr(), N, cfg, s) == 1, cfg
    Af, Bf = A.float(), B.float()
    for cfg in ({"kernel": "cta_pair"}, {"kernel": 4}, {"split": -2}, {"split": 9}):
        assert g.gemm_sgemm_config(M, N, K, 1.0, Af.data_ptr(), K, Bf.data_ptr(), N, 0.0,
                                   C.data_ptr(), N, cfg, s) == 1, cfg
    torch.cuda.synchronize()


def _table_rows():
    text = open(TABLE).read()
    sms = int(re.search(r"kTunedSms\s*=\s*(\d+);", text).group(1))
    rows = re.findall(r"^\s*\{(\d+),\s*(\d+),\s*(\d+),\s*(\d+),\s*(\d+),\s*(\d+),\s*(\d+)\}",
                      text, flags=re.M)
    return sms, [tuple(int(x) for x in r) for r in rows]


def test_table_entries_are_what_dispatch_uses():
    sms, rows = _table_rows()
    if torch.cuda.get_device_properties(0).multi_processor_count != sms:
        pytest.skip("table measured on a GPU with another SM count")
    names = {1: "single_cta", 2: "cta_pair", 3: "wide"}
    for is_bf16, lm, ln, lk, kernel, split, group in rows:
        M, N, K = 1 << lm, 1 << ln, 1 << lk
        cfg, from_table = g.gemm_get_config(is_bf16, M, N, K)
        assert from_table, (M, N, K)
        assert cfg["kernel"] == names[kernel] and cfg["group_m"] == group
        # a split is capped by the k-blocks and dropped when no round is partial
        if split == -1:
            assert cfg["split"] in (-1, 1)
        else:
            assert 1 <= cfg["split"] <= split


def test_get_config_for_the_benchmark_shapes():
    cfg, _ = g.gemm_get_config(True, 8192, 8192, 8192)
    assert cfg["kernel"] == "cta_pair"
    cfg, _ = g.gemm_get_config(True, 16, 12288, 4096)
    assert cfg == {"kernel": "auto", "split": 0, "group_m": 0}   # the decode kernel
    cfg, _ = g.gemm_get_config(False, 4092, 4092, 4092)
    assert cfg["kernel"] in ("single_cta", "wide") and cfg["group_m"] >= 1
    assert cfg["split"] >= 1 or cfg["split"] == g.SPLIT_STREAM
