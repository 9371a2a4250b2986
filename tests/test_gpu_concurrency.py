"""Several host threads, each on its own stream, calling the library at once.

The header allows calls from several host threads on different streams; the
split-K paths then need each stream's own scratch (partial sums, arrival
counters), created and grown on first use under a lock.  Each thread runs
GEMMs whose work is split along k -- the CUDA-core kernel with a pinned
split, the CTA-pair kernel's split tail and a pinned stream-K tail, the
decode kernel's runs of column groups combined through scratch (one row
block, and two), and its cluster split, which needs none --
in a different order and with scratch growing at different times, and
every result must equal, bit for bit, the same call run alone beforehand
(fixed plans sum their parts in a fixed order, so results are reproducible).
"""
import threading

import pytest
import torch

import dense_gemm_12_gb300 as g
from dense_gemm_12_gb300.workloads import make_inputs
from gpu_helpers import check_device_error

pytestmark = pytest.mark.gpu

THREADS = 4
ROUNDS = 6


@pytest.fixture(scope="module", autouse=True)
def _lib(gemm_lib, cuda_device):
    yield


def _cases():
    """(name, launcher) pairs; each launcher(stream) writes its own output."""
    cases = []
    # fp32, 16 tiles split 6 ways (pinned)
    A, B, C = make_inputs(512, 512, 2048, seed=41)
    dA, dB = A.cuda(), B.cuda()
    C0 = C.cuda()

    def fp32(stream, out):
        out.copy_(C0)
        st = g.gemm_sgemm_config(512, 512, 2048, 0.7, dA.data_ptr(), 2048, dB.data_ptr(), 512,
                                 0.3, out.data_ptr(), 512, {"split": 6}, stream.cuda_stream)
        assert st == 0
    cases.append(("fp32_split", fp32, (512, 512)))
    # bf16 CTA-pair kernel with its last round split (automatic)
    A2, B2, C2 = make_inputs(512, 10240, 4096, ("normal", 1.0), ("normal", 0.05),
                             ("uniform", None), seed=42, dtype="bf16")
    assert g.gemm_split_parts(1, 512, 10240, 4096) > 1
    dA2, dB2, C20 = A2.cuda(), B2.cuda(), C2.cuda()

    def pair(stream, out):
        out.copy_(C20)
        st = g.gemm_bf16gemm(512, 10240, 4096, 1.0, dA2.data_ptr(), 4096, dB2.data_ptr(), 10240,
                             0.5, out.data_ptr(), 10240, stream.cuda_stream)
        assert st == 0
    cases.append(("bf16_pair_split", pair, (512, 10240)))
    # decode kernel: 160 column groups, more than SMs, so CTAs take runs of
    # groups and combine the split ones through the stream's scratch
    A3, B3, C3 = make_inputs(16, 20480, 2048, ("normal", 1.0), ("normal", 0.05),
                             ("uniform", None), seed=43, dtype="bf16")
    dA3, dB3, C30 = A3.cuda(), B3.cuda(), C3.cuda()

    def decode(stream, out):
        out.copy_(C30)
        st = g.gemm_bf16gemm(16, 20480, 2048, 1.0, dA3.data_ptr(), 2048, dB3.data_ptr(), 20480,
                             1.0, out.data_ptr(), 20480, stream.cuda_stream)
        assert st == 0
    cases.append(("decode_split", decode, (16, 20480)))
    # decode kernel, 32 groups: clusters of 4 add their partial sums in
    # shared memory (no scratch)
    A4, B4, C4 = make_inputs(40, 4096, 4096, ("normal", 1.0), ("normal", 0.05),
                             ("uniform", None), seed=44, dtype="bf16")
    dA4, dB4, C40 = A4.cuda(), B4.cuda(), C4.cuda()

    def decode_cluster(stream, out):
        out.copy_(C40)
        st = g.gemm_bf16gemm(40, 4096, 4096, 1.0, dA4.data_ptr(), 4096, dB4.data_ptr(), 4096,
                             1.0, out.data_ptr(), 4096, stream.cuda_stream)
        assert st == 0
    cases.append(("decode_cluster", decode_cluster, (40, 4096)))
    # bf16 CTA-pair kernel with a pinned stream-K tail: partial sums of every
    # worker's segments in the stream's scratch
    def pair_stream_k(stream, out):
        out.copy_(C20)
        st = g.gemm_bf16gemm_config(512, 10240, 4096, 1.0, dA2.data_ptr(), 4096, dB2.data_ptr(),
                                    10240, 0.5, out.data_ptr(), 10240,
                                    {"kernel": "cta_pair", "split": -1}, stream.cuda_stream)
        assert st == 0
    cases.append(("bf16_pair_stream_k", pair_stream_k, (512, 10240)))
    # decode kernel, two row blocks of 64 with more column groups than SMs per
    # block: each block's runs of groups meet in its own part of the scratch
    A5, B5, C5 = make_inputs(100, 16384, 1024, ("normal", 1.0), ("normal", 0.05),
                             ("uniform", None), seed=45, dtype="bf16")
    dA5, dB5, C50 = A5.cuda(), B5.cuda(), C5.cuda()

    def decode_rows(stream, out):
        out.copy_(C50)
        st = g.gemm_bf16gemm(100, 16384, 1024, 1.0, dA5.data_ptr(), 1024, dB5.data_ptr(), 16384,
                             1.0, out.data_ptr(), 16384, stream.cuda_stream)
        assert st == 0
    cases.append(("decode_two_row_blocks", decode_rows, (100, 16384)))
    return cases


def test_threads_on_their_own_streams_match_serial_results():
    cases = _cases()
    # serial references, on one fresh stream
    ref = {}
    s0 = torch.cuda.Stream()
    with torch.cuda.stream(s0):
        for name, fn, shape in cases:
            out = torch.empty(shape, device="cuda")
            fn(s0, out)
            s0.synchronize()
            ref[name] = out.clone()
    check_device_error()

    errors = []
    start = threading.Barrier(THREADS)

    def worker(t):
        try:
            stream = torch.cuda.Stream()
            outs = {name: torch.empty(shape, device="cuda") for name, _, shape in cases}
            order = cases[t % len(cases):] + cases[:t % len(cases)]   # different orders
            start.wait()
            with torch.cuda.stream(stream):
                for _ in range(ROUNDS):
                    for name, fn, _ in order:
                        fn(stream, outs[name])
                    stream.synchronize()
                    for name in outs:
                        if not torch.equal(outs[name].view(torch.int32),
                                           ref[name].view(torch.int32)):
                            errors.append((t, name))
        except Exception as exc:  # reported below, on the main thread
            errors.append((t, repr(exc)))

    threads = [threading.Thread(target=worker, args=(t,)) for t in range(THREADS)]
    for th in threads:
        th.start()
    for th in threads:
        th.join(timeout=300)
    assert not any(th.is_alive() for th in threads), "a worker did not finish"
    torch.cuda.synchronize()
    assert not errors, errors[:5]
    check_device_error()
