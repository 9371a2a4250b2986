"""Library calls captured into a CUDA graph and replayed.

After one eager call of each shape on the capturing stream (which creates
that stream's split-K scratch), every launch path -- the CUDA-core kernel
with a split tail, the CTA-pair kernel with a split tail, the fused output
stage with fp8 output and amax, the decode kernel in clusters, all of them
launched with programmatic dependent launch -- must capture, and every
replay must reproduce the eager results bit for bit.

Inside a capture the library allocates nothing: a first call on a new
stream whose plan needs scratch runs whole tiles instead (the decode kernel's
runs of column groups fall back to the single-CTA tile kernel, an operand
that would be staged is read by the generic loads).  Those captures must
succeed and their replays must match the oracle -- bit for bit on small
integers, where every order of summation is exact.  Growing a stream's
scratch outside a capture is stream-ordered and must not wait for the work
already queued on the stream.
"""
import time

import numpy as np
import pytest
import torch

import dense_gemm_12_gb300 as g
from dense_gemm_12_gb300.workloads import make_inputs
from gpu_helpers import check_device_error, oracle_bf16, oracle_sgemm

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib(gemm_lib, cuda_device):
    yield


def test_capture_and_replay_matches_eager():
    if not hasattr(torch, "float8_e4m3fn"):
        pytest.skip("torch without float8_e4m3fn")
    A1, B1, C1 = make_inputs(1024, 1024, 2048, seed=51)
    A2, B2, C2 = make_inputs(512, 10240, 4096, ("normal", 1.0), ("normal", 0.05),
                             ("uniform", None), seed=52, dtype="bf16")
    A3, B3, C3 = make_inputs(16, 4096, 4096, ("normal", 1.0), ("normal", 0.05),
                             ("uniform", None), seed=53, dtype="bf16")
    assert g.gemm_split_parts(0, 1024, 1024, 2048) > 1
    assert g.gemm_split_parts(1, 512, 10240, 4096) > 1
    dev = [t.cuda() for t in (A1, B1, C1, A2, B2, C2, A3, B3, C3)]
    dA1, dB1, dC1, dA2, dB2, dC2, dA3, dB3, dC3 = dev
    bias = torch.randn(10240, generator=torch.Generator().manual_seed(5)).cuda()
    out1 = torch.empty(1024, 1024, device="cuda")
    out2 = torch.empty(512, 10240, device="cuda")
    out3 = torch.empty(16, 4096, device="cuda")
    d8 = torch.empty(512, 10240, dtype=torch.float8_e4m3fn, device="cuda")
    amax = torch.zeros(1, device="cuda")

    def work(stream):
        h = stream.cuda_stream
        out1.copy_(dC1)
        assert g.gemm_sgemm(1024, 1024, 2048, 0.7, dA1.data_ptr(), 2048, dB1.data_ptr(), 1024,
                            0.3, out1.data_ptr(), 1024, h) == 0
        out2.copy_(dC2)
        assert g.gemm_bf16gemm(512, 10240, 4096, 1.0, dA2.data_ptr(), 4096, dB2.data_ptr(),
                               10240, 0.5, out2.data_ptr(), 10240, h) == 0
        amax.zero_()
        g.bf16gemm_fused(dA2, dB2, d8, bias=bias, act="gelu", d_scale=32.0, amax=amax,
                         stream=stream)
        out3.copy_(dC3)
        assert g.gemm_bf16gemm(16, 4096, 4096, 1.0, dA3.data_ptr(), 4096, dB3.data_ptr(), 4096,
                               1.0, out3.data_ptr(), 4096, h) == 0

    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        work(s)                       # warm-up: this stream's scratch is created here
        s.synchronize()
        eager = [t.clone() for t in (out1, out2, out3, d8.view(torch.uint8), amax)]
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=s):
            work(s)
        for _ in range(3):
            for t in (out1, out2, out3, amax):
                t.fill_(float("nan"))
            d8.view(torch.uint8).fill_(0x7F)
            graph.replay()
            s.synchronize()
            for got, want in zip((out1, out2, out3, d8.view(torch.uint8), amax), eager):
                assert torch.equal(got.view(torch.uint8), want.view(torch.uint8))
    check_device_error()


INT = ("int", None)


def _sms():
    return torch.cuda.get_device_properties(0).multi_processor_count


def _first_call_cases():
    sms = _sms()
    return [
        # (name, is_bf16, M, N, K, lda): each plan needs scratch or staging
        ("fp32_split_tail", False, 128 * 13, 128 * 13, 2048, 2048),
        ("fp32_staged_A", False, 1024, 1024, 1025, 1025),   # 2^31 FLOPs: staged
        ("bf16_pair_split_tail", True, 512, 10240, 4096, 4096),
        ("decode_runs_of_groups", True, 16, 128 * (sms + 10), 1024, 1024),
    ]


@pytest.mark.parametrize("case", range(4))
def test_first_call_inside_capture_allocates_nothing(case):
    name, bf16, M, N, K, lda = _first_call_cases()[case]
    if bf16:
        A, B, C = make_inputs(M, N, K, INT, INT, INT, seed=60 + case, dtype="bf16")
    else:
        A, B, C = make_inputs(M, N, K, INT, INT, INT, seed=60 + case)
    dA, dB, dC0 = A.cuda(), B.cuda(), C.cuda()
    out = torch.empty_like(dC0)
    fn = g.gemm_bf16gemm if bf16 else g.gemm_sgemm
    s = torch.cuda.Stream()            # new: the library holds nothing for it
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(graph, stream=s):
            out.copy_(dC0)
            st = fn(M, N, K, 1.5, dA.data_ptr(), lda, dB.data_ptr(), N, -0.5, out.data_ptr(), N,
                    s.cuda_stream)
        assert st == 0, (name, g.gemm_status_string(st))
        ref32, _, _ = (oracle_bf16 if bf16 else oracle_sgemm)(A, B, C, 1.5, -0.5, want64=False)
        for _ in range(2):
            out.fill_(float("nan"))
            graph.replay()
            s.synchronize()
            assert np.array_equal(out.cpu().numpy().view(np.uint32), ref32.view(np.uint32)), name
        # the same call eager afterwards creates the scratch and takes the
        # planned path; on integers it gives the same bits
        out.copy_(dC0)
        assert fn(M, N, K, 1.5, dA.data_ptr(), lda, dB.data_ptr(), N, -0.5, out.data_ptr(), N,
                  s.cuda_stream) == 0
        s.synchronize()
        assert np.array_equal(out.cpu().numpy().view(np.uint32), ref32.view(np.uint32)), name
        assert g.gemm_release_stream(s.cuda_stream) == 0
    check_device_error()


def test_scratch_growth_does_not_wait_for_queued_work():
    # a long GEMM queued first; then a call on the same new stream whose plan
    # needs scratch.  Growing the scratch is stream-ordered, so the call
    # returns while the long GEMM still runs.
    big = 6144
    A0, B0, _ = make_inputs(big, big, big, seed=70, with_c=False)
    dA0, dB0 = A0.cuda(), B0.cuda()
    dC0 = torch.empty(big, big, device="cuda")
    M, N, K = 128 * 13, 128 * 13, 2048
    A, B, C = make_inputs(M, N, K, INT, INT, INT, seed=71)
    dA, dB, dC = A.cuda(), B.cuda(), C.cuda()
    assert g.gemm_split_parts(0, M, N, K) > 1
    s = torch.cuda.Stream()
    done = torch.cuda.Event()
    torch.cuda.synchronize()
    assert g.gemm_sgemm(big, big, big, 1.0, dA0.data_ptr(), big, dB0.data_ptr(), big, 0.0,
                        dC0.data_ptr(), big, s.cuda_stream) == 0
    t0 = time.perf_counter()
    assert g.gemm_sgemm(M, N, K, 1.5, dA.data_ptr(), K, dB.data_ptr(), N, -0.5, dC.data_ptr(),
                        N, s.cuda_stream) == 0
    host_s = time.perf_counter() - t0
    done.record(s)
    still_running = not done.query()
    s.synchronize()
    # 6144^3 fp32 takes ~7 ms on the GPU; the second call must not have waited for it
    assert still_running and host_s < 3e-3, host_s
    ref32, _, _ = oracle_sgemm(A, B, C, 1.5, -0.5, want64=False)
    assert np.array_equal(dC.cpu().numpy().view(np.uint32), ref32.view(np.uint32))
    assert g.gemm_release_stream(s.cuda_stream) == 0
    assert g.gemm_release_stream(s.cuda_stream) == 0   # nothing left: still fine
    check_device_error()
