"""Library calls captured into a CUDA graph and replayed.

The header's rule: a stream's first call that needs split-K scratch must
come before that stream is captured (growing scratch synchronises the
stream).  After such a warm-up, every launch path -- the CUDA-core kernel
with a split tail, the CTA-pair kernel with a split tail, the fused output
stage with fp8 output and amax, the decode kernel split over all SMs, all of
them launched with programmatic dependent launch -- must capture, and every
replay must reproduce the eager results bit for bit.
"""
import pytest
import torch

import dense_gemm_12_gb300 as g
from dense_gemm_12_gb300.workloads import make_inputs
from gpu_helpers import check_device_error

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
