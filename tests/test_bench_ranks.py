"""The multi-rank bookkeeping of bench.py on two CPU ranks (gloo).

bench.py runs one independent replica per GPU; the only cross-rank steps are
the barrier, the max of the timed durations and the whole-job throughput.
This runs those helpers in a world of two processes on the CPU.
"""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank), BENCH_BACKEND="gloo")
    import bench
    r, local, w, pg = bench.dist_setup(world)
    assert (r, local, w) == (rank, rank, world)
    bench.barrier(pg, "cpu")
    local_ms = 10.0 + 5.0 * rank             # rank 1 is the slow one
    max_ms = bench.max_over_ranks(pg, local_ms, "cpu")
    value = bench.whole_job_gflops(w, 2.0e9, 4, max_ms)
    out[rank] = (max_ms, value)
    pg.destroy_process_group()


def test_two_gloo_ranks_agree_on_max_time_and_value():
    world = 2
    port = _free_port()
    manager = mp.Manager()
    out = manager.dict()
    ctx = mp.get_context("spawn")
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, out)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    # both ranks see the slowest rank's time; value counts both ranks' work
    assert out[0] == out[1]
    max_ms, value = out[0]
    assert max_ms == 15.0
    assert value == pytest.approx(2 * 2.0e9 * 4 / 15e-3 / 1e9)


def test_single_rank_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(None, 3.5, "cpu") == 3.5
    assert bench.whole_job_gflops(1, 1e9, 10, 1000.0) == pytest.approx(10.0)
