"""The cluster fix-up of the CUDA-core kernel and of the single-CTA tcgen05
kernel: when every tile runs in the first round, cut into S = 2..8 k-ranges,
the S CTAs of a tile form a thread-block cluster and add their partial sums
through distributed shared memory instead of the stream's global workspace.

The partial sums are the same and are added in the same (k) order, so the
result must be bit-identical to the global-memory fix-up, which the
generic-load kernel (an A pitch TMA cannot describe) still takes; on small
integers both must equal the oracle bit for bit.  The mode needs no scratch,
so a first call inside a stream capture keeps its split.
"""
import numpy as np
import pytest
import torch

import dense_gemm_12_gb300 as g
from dense_gemm_12_gb300.workloads import make_inputs
import oracle
from gpu_helpers import TOL_BF16, check_device_error, oracle_bf16, oracle_sgemm, ratio

pytestmark = pytest.mark.gpu

INT = ("int", None)


@pytest.fixture(scope="module", autouse=True)
def _lib(gemm_lib, cuda_device):
    yield


def _call(A, B, C, alpha, beta, cfg, lda=None, ldc=None, stream=None):
    """gemm_sgemm_config on device copies; A is laid out with pitch lda and C
    with pitch ldc (the columns past K / N hold sentinels)."""
    M, K = A.shape
    N = B.shape[1]
    lda = lda or K
    ldc = ldc or N
    dA = torch.full((M, lda), 7.0, device="cuda")
    dA[:, :K] = A.cuda()
    dC = torch.full((M, ldc), -3.0, device="cuda")
    dC[:, :N] = C.cuda()
    dB = B.cuda()
    h = stream.cuda_stream if stream is not None else torch.cuda.current_stream().cuda_stream
    st = g.gemm_sgemm_config(M, N, K, alpha, dA.data_ptr(), lda, dB.data_ptr(), N, beta,
                             dC.data_ptr(), ldc, cfg, h)
    torch.cuda.synchronize()
    assert st == 0, g.gemm_status_string(st)
    out = dC.cpu()
    assert torch.all(out[:, N:] == -3.0), "write past N"
    return out[:, :N].contiguous()


# (M, N, K, S): tiles x S <= 152, ragged M, N and K, S from 2 to 8
CASES = [
    (200, 300, 32 * 2 * 3 + 7, 2),
    (256, 384, 1000, 3),
    (129, 1000, 4 * 32 * 4, 4),
    (100, 520, 1111, 5),
    (384, 256, 6 * 32 * 4 + 31, 6),
    (77, 250, 7 * 32 * 5, 7),
    (300, 260, 2048, 8),
]


@pytest.mark.parametrize("M,N,K,S", CASES)
def test_cluster_fixup_exact_on_integers(M, N, K, S):
    cfg = {"kernel": "single_cta", "split": S, "group_m": 1}
    assert g.gemm_split_cluster(0, M, N, K, cfg) == S
    A, B, C = make_inputs(M, N, K, INT, INT, INT, seed=M + S)
    ref32, _, _ = oracle_sgemm(A, B, C, 1.5, -0.5, want64=False)
    out = _call(A, B, C, 1.5, -0.5, cfg)
    assert np.array_equal(out.numpy().view(np.uint32), ref32.view(np.uint32))
    # an odd C pitch: no float4 rows, the scalar output path
    out = _call(A, B, C, 1.5, -0.5, cfg, ldc=N + 1)
    assert np.array_equal(out.numpy().view(np.uint32), ref32.view(np.uint32))
    check_device_error()


@pytest.mark.parametrize("M,N,K,S", CASES[::2])
def test_cluster_fixup_bits_equal_global_fixup(M, N, K, S):
    # random inputs: the cluster form (TMA operands) against the same split
    # through the workspace (A at an unaligned pitch: generic loads)
    cfg = {"kernel": "single_cta", "split": S, "group_m": 3}
    A, B, C = make_inputs(M, N, K, ("uniform", None), ("uniform", None), ("uniform", None),
                          seed=11 * S)
    lda = K + 1 if (K + 1) % 4 else K + 2   # rows not 16-byte aligned
    assert g.gemm_select_path(0, M, N, K, 0.7, 1 << 20, lda, 1 << 20, N) == "simt_generic"
    a = _call(A, B, C, 0.7, 0.3, cfg)
    b = _call(A, B, C, 0.7, 0.3, cfg, lda=lda)
    assert torch.equal(a.view(torch.int32), b.view(torch.int32))
    _, ref64, den = oracle_sgemm(A, B, C, 0.7, 0.3)
    assert ratio(a, ref64, den) <= 2e-6 * K ** 0.5
    check_device_error()


def test_beta_zero_ignores_nan_c():
    M, N, K, S = 200, 300, 512, 4
    cfg = {"kernel": "single_cta", "split": S}
    assert g.gemm_split_cluster(0, M, N, K, cfg) == S
    A, B, C = make_inputs(M, N, K, INT, INT, INT, seed=5)
    ref32, _, _ = oracle_sgemm(A, B, torch.zeros_like(C), 2.0, 0.0, want64=False)
    out = _call(A, B, torch.full_like(C, float("nan")), 2.0, 0.0, cfg)
    assert np.array_equal(out.numpy().view(np.uint32), ref32.view(np.uint32))


def test_automatic_dispatch_uses_clusters_for_small_shapes():
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    # 256^3: four tiles, each cut along k -- the fix-up runs in clusters
    assert g.gemm_split_parts(0, 256, 256, 256) > 1
    assert g.gemm_split_cluster(0, 256, 256, 256) == g.gemm_split_parts(0, 256, 256, 256)
    # the 4092^3 plan has whole rounds: no clusters
    assert g.gemm_split_cluster(0, 4092, 4092, 4092) == 1
    # more tiles than SMs: the split tail meets in global memory
    assert g.gemm_split_cluster(0, 128 * 13, 128 * 13, 2048) == 1
    # pinned: the wide tile, stream-K and no split never use clusters
    assert g.gemm_split_cluster(0, 256, 256, 256, {"kernel": "wide", "split": 4}) == 1
    assert g.gemm_split_cluster(0, 256, 256, 256, {"split": -1}) == 1
    assert g.gemm_split_cluster(0, 256, 256, 256, {"split": 1}) == 1
    # tiles x S above the SM count cannot all run at once
    tiles = sms // 2 + 1
    assert g.gemm_split_cluster(0, 128 * tiles, 128, 4096, {"kernel": "single_cta", "split": 2}) == 1
    assert g.gemm_split_cluster(0, -1, 256, 256) == 0
    assert g.gemm_split_cluster(0, 256, 256, 256, {"split": 9}) == 0
    A, B, C = make_inputs(256, 256, 256, INT, INT, INT, seed=8)
    ref32, _, _ = oracle_sgemm(A, B, C, 1.0, 1.0, want64=False)
    dA, dB, dC = A.cuda(), B.cuda(), C.cuda()
    assert g.gemm_sgemm(256, 256, 256, 1.0, dA.data_ptr(), 256, dB.data_ptr(), 256, 1.0,
                        dC.data_ptr(), 256, torch.cuda.current_stream().cuda_stream) == 0
    assert np.array_equal(dC.cpu().numpy().view(np.uint32), ref32.view(np.uint32))


def test_first_call_inside_capture_keeps_its_split():
    # a new stream has no scratch, and a capture allocates none: the global
    # fix-up would fall back to whole tiles (other sums, other bits on random
    # inputs); the cluster fix-up needs none and gives the eager call's bits
    # the first shape whose automatic plan splits in clusters (the plan comes
    # from the cost model or the sweep's table)
    shapes = [(256, 256, 512), (256, 256, 256), (384, 384, 1024), (640, 384, 768)]
    M, N, K = next((m, n, k) for m, n, k in shapes if g.gemm_split_cluster(0, m, n, k) > 1)
    S = g.gemm_split_parts(0, M, N, K)
    assert S > 1 and g.gemm_split_cluster(0, M, N, K) == S
    A, B, C = make_inputs(M, N, K, ("uniform", None), ("uniform", None), ("uniform", None),
                          seed=21)
    dA, dB, dC = A.cuda(), B.cuda(), C.cuda()
    out = torch.empty_like(dC)
    s = torch.cuda.Stream()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(graph, stream=s):
            out.copy_(dC)
            assert g.gemm_sgemm(M, N, K, 0.7, dA.data_ptr(), K, dB.data_ptr(), N, 0.3,
                                out.data_ptr(), N, s.cuda_stream) == 0
        out.fill_(float("nan"))
        graph.replay()
        s.synchronize()
        captured = out.clone()
        out.copy_(dC)
        assert g.gemm_sgemm(M, N, K, 0.7, dA.data_ptr(), K, dB.data_ptr(), N, 0.3,
                            out.data_ptr(), N, s.cuda_stream) == 0
        s.synchronize()
    assert torch.equal(captured.view(torch.int32), out.view(torch.int32))
    assert g.gemm_release_stream(s.cuda_stream) == 0
    check_device_error()


def test_two_streams_at_once():
    # no shared scratch: two cluster launches on two streams overlap freely
    M, N, K, S = 512, 512, 2048, 4
    cfg = {"kernel": "single_cta", "split": S}
    assert g.gemm_split_cluster(0, M, N, K, cfg) == S
    ins = [make_inputs(M, N, K, INT, INT, INT, seed=30 + i) for i in range(2)]
    dev = [[t.cuda() for t in x] for x in ins]
    streams = [torch.cuda.Stream() for _ in range(2)]
    torch.cuda.synchronize()
    for _ in range(3):
        for (dA, dB, dC), s in zip(dev, streams):
            assert g.gemm_sgemm_config(M, N, K, 1.0, dA.data_ptr(), K, dB.data_ptr(), N, 1.0,
                                       dC.data_ptr(), N, cfg, s.cuda_stream) == 0
    torch.cuda.synchronize()
    for (A, B, C), (_, _, dC) in zip(ins, dev):
        # C <- A B + C three times over
        ref = C
        for _ in range(3):
            ref32, _, _ = oracle_sgemm(A, B, ref, 1.0, 1.0, want64=False)
            ref = torch.from_numpy(ref32)
        assert np.array_equal(dC.cpu().numpy().view(np.uint32), ref32.view(np.uint32))
    check_device_error()


# ------------------------------------------------------------------ bf16
# The single-CTA tcgen05 kernel (128 x 256 tiles): the parts' partial sums go
# from tensor memory into each CTA's shared memory, and CTA r of a cluster
# adds, for its share of the tile's 32-column chunks, the S partials in k
# order and runs them through the output stage.  Pinned configurations run
# the tile kernels even where automatic dispatch would take the decode
# kernel.  bf16 pitches are multiples of 8 elements (TMA).
BF16_CASES = [
    (200, 600, 1000, 2),    # 2 x 3 tiles, ragged M, N and K (partial last k-block)
    (300, 520, 2048, 3),    # 3 x 3 tiles
    (129, 1000, 4096, 4),   # 2 x 4 tiles, one row in the second tile row
    (100, 520, 1112, 5),    # 1 x 3 tiles
    (384, 256, 1592, 6),    # 3 x 1 tiles
    (77, 248, 2240, 7),     # 1 x 1 tile
    (300, 264, 2048, 8),    # 3 x 2 tiles
]


def _bf16_call(A, B, C, alpha, beta, cfg, ldc=None):
    M, K = A.shape
    N = B.shape[1]
    ldc = ldc or N
    dA, dB = A.cuda(), B.cuda()
    dC = torch.full((M, ldc), -3.0, device="cuda")
    dC[:, :N] = C.cuda()
    st = g.gemm_bf16gemm_config(M, N, K, alpha, dA.data_ptr(), K, dB.data_ptr(), N, beta,
                                dC.data_ptr(), ldc, cfg, torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    assert st == 0, g.gemm_status_string(st)
    out = dC.cpu()
    assert torch.all(out[:, N:] == -3.0), "write past N"
    return out[:, :N].contiguous()


@pytest.mark.parametrize("M,N,K,S", BF16_CASES)
def test_bf16_cluster_fixup_exact_on_integers(M, N, K, S):
    cfg = {"kernel": "single_cta", "split": S, "group_m": 1}
    assert g.gemm_split_cluster(1, M, N, K, cfg) == S
    A, B, C = make_inputs(M, N, K, INT, INT, INT, seed=M + S, dtype="bf16")
    ref32, _, _ = oracle_bf16(A, B, C, 1.5, -0.5, want64=False)
    for ldc in (None, N + 1):
        out = _bf16_call(A, B, C, 1.5, -0.5, cfg, ldc=ldc)
        assert np.array_equal(out.numpy().view(np.uint32), ref32.view(np.uint32))
    check_device_error()


@pytest.mark.parametrize("M,N,K,S", BF16_CASES[::2])
def test_bf16_cluster_tma_output_exact_on_integers(M, N, K, S):
    # beta = 0: each CTA's share of the reduced tile leaves through TMA stores,
    # clipped at the ragged edges; padded rows keep their padding
    cfg = {"kernel": "single_cta", "split": S, "group_m": 1}
    assert g.gemm_split_cluster(1, M, N, K, cfg) == S
    A, B, C = make_inputs(M, N, K, INT, INT, INT, seed=M + 3 * S, dtype="bf16")
    ref32, _, _ = oracle_bf16(A, B, C, 1.5, 0.0, want64=False)
    for ldc in (None, N + 4, N + 1):
        out = _bf16_call(A, B, C, 1.5, 0.0, cfg, ldc=ldc)
        assert np.array_equal(out.numpy().view(np.uint32), ref32.view(np.uint32))
    check_device_error()


@pytest.mark.parametrize("M,N,K,S", BF16_CASES[1::2])
def test_bf16_cluster_fixup_random_within_bound_and_repeatable(M, N, K, S):
    cfg = {"kernel": "single_cta", "split": S}
    A, B, C = make_inputs(M, N, K, ("normal", 1.0), ("normal", 0.05), ("uniform", None),
                          seed=13 * S, dtype="bf16")
    a = _bf16_call(A, B, C, 0.7, 0.3, cfg)
    b = _bf16_call(A, B, C, 0.7, 0.3, cfg)
    assert torch.equal(a.view(torch.int32), b.view(torch.int32))
    _, ref64, den = oracle_bf16(A, B, C, 0.7, 0.3)
    assert ratio(a, ref64, den) <= TOL_BF16
    check_device_error()


def test_bf16_cluster_choice():
    # the single-CTA kernel only (CTA pairs are clusters already); all tiles
    # in one round; every cluster resident at once (15 of 8 on a GB300)
    assert g.gemm_split_cluster(1, 300, 264, 2048, {"kernel": "cta_pair", "split": 4}) == 1
    assert g.gemm_split_cluster(1, 300, 264, 2048, {"kernel": "single_cta", "split": 1}) == 1
    assert g.gemm_split_cluster(1, 300, 264, 2048, {"kernel": "single_cta", "split": -1}) == 1
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    tiles = sms // 2 + 1     # x 2 parts > SMs
    assert g.gemm_split_cluster(1, 128, 256 * tiles, 4096, {"kernel": "single_cta",
                                                             "split": 2}) == 1
    # automatic dispatch: the decode kernel plans its own clusters
    assert g.gemm_split_cluster(1, 16, 12288, 4096) == 1
    # M <= 128 beyond the decode kernel's N: single-CTA tiles split in two
    assert g.gemm_split_cluster(1, 100, 16640, 4096) == g.gemm_split_parts(1, 100, 16640, 4096)


def test_bf16_cluster_fused_output_exact():
    # bias + ReLU + residual, int8 output and amax through the cluster form
    # (automatic dispatch: 65 single-CTA tiles of 128 x 256, each split in two)
    M, N, K = 100, 16640, 4096
    assert g.gemm_split_cluster(1, M, N, K) > 1
    gen = torch.Generator().manual_seed(4)
    A, B, C = make_inputs(M, N, K, INT, INT, INT, seed=4, dtype="bf16")
    bias = torch.randint(-64, 65, (N,), generator=gen).float()
    res = torch.randint(-32, 33, (M, N), generator=gen).float()
    D = torch.empty(M, N, dtype=torch.int8, device="cuda")
    amax = torch.zeros(1, device="cuda")
    g.bf16gemm_fused(A.cuda(), B.cuda(), D, C=C.cuda(), alpha=1.0, beta=-0.5, bias=bias.cuda(),
                     act="relu", residual=res.cuda(), d_scale=2.0 ** -4, amax=amax)
    torch.cuda.synchronize()
    _, ref64, _ = oracle_bf16(A, B, C, 1.0, -0.5)
    v = oracle.epilogue(ref64, bias=bias.numpy(), act="relu", residual=res.numpy())
    assert np.array_equal(D.cpu().numpy(), oracle.quantize(v, "s8", 2.0 ** -4))
    assert float(amax.item()) == float(np.max(np.abs(v)))
    check_device_error()
