"""Benchmark of the GEMM library on the GPU, printing one JSON line.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Headline workload (one "step"): fp32 SGEMM C = 0.7*A*B + 0.3*C at
M = N = K = 4092 through gemm_sgemm, inputs resident in HBM.  Two input sets
of 201 MB each are used in turn, so every step starts from operands that are
not in the 129 MB L2 (no flush needed between steps).  ``value`` is
GFLOP/s = 2*M*N*K*steps / time (the alpha/beta scaling is not counted).

The same run also measures the other two kernels the metric names, each with
its own warm-up and timed launches, under ``parts``:
  * bf16 8192^3 (alpha 1, beta 0) on the tcgen05 kernel -- operands and C
    total 768 MB, larger than L2;
  * decode M=16, N=12288, K=4096, beta=1 on the split-K decode kernel -- B
    is 100.7 MB, so three copies are cycled (302 MB) and each launch reads a
    B not touched by the previous two launches; launches are replayed from a
    CUDA graph.

Kernel durations come from CUDA events on the launching stream.  ``e2e`` times
the same SGEMM through the C ABI with host buffers: per step the pinned host
A, B, C are copied in and C is copied back inside the timed region.
``cpu_baseline`` times the CPU oracle on a bounded sample of rows of the same
workload on the host cores.  N > 1 (torchrun): every rank runs an independent
replica on its own GPU (no data exchange), the time is the max over ranks and
``value`` is the sum of all ranks' FLOPs over that time.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "GFLOP/s and % of roofline: fp32 4092^3 SIMT, bf16 8192^3 tcgen05, M=16 HBM GB/s"
SM_LANES_FP32 = 128        # fp32 FFMA lanes per SM (4 partitions x 32)
MAX_SM_CLOCK_HZ = 2.07e9   # GB300 maximum SM clock


def parse_args():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=200)
    p.add_argument("--warmup", type=int, default=3)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--no-parts", action="store_true", help="headline workload only")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--only", choices=["sgemm", "bf16", "decode"], default=None,
                   help="time one kernel's workload alone (profiling runs); prints its part")
    p.add_argument("--cpu-seconds", type=float, default=12.0,
                   help="target duration of the CPU-oracle sample")
    return p.parse_args()


# ------------------------------------------------------------------ helpers
def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained", d["bf16_tflops"]),
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "source": "fallback"}


def recorded_traffic(kernel):
    """DRAM bytes of one launch of `kernel` from the committed ncu record, or
    None if the kernel's sources changed since the capture."""
    import hashlib
    path = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)[kernel]
        h = hashlib.sha256()
        for src in (rec["source"], "dense_gemm_12_gb300/csrc/ptx.cuh",
                    "dense_gemm_12_gb300/csrc/internal.h",
                    "dense_gemm_12_gb300/csrc/epilogue.cuh"):
            with open(os.path.join(ROOT, src), "rb") as f:
                h.update(f.read())
        if h.hexdigest() != rec["source_sha256"]:
            return None
        return rec["dram_read_bytes"] + rec["dram_write_bytes"]
    except (OSError, KeyError, ValueError):
        return None


class ClockSampler:
    """nvidia-smi clock / throttle-reason sampling while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu_index = gpu_index
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu_index), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, FileNotFoundError):
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)
        sm, smax, power, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
                power.append(float(parts[3]))
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        loaded = [s for s, p in zip(sm, power) if p > 0.4 * max(power)] or sm
        return {"sm_mhz": statistics.median(loaded), "sm_max_mhz": max(smax),
                "reasons": sorted(reasons), "samples": len(sm),
                "power_w_max": max(power)}


def dist_setup(n_gpus):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    pg = None
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if os.environ.get("BENCH_BACKEND", "nccl") == "nccl" else "gloo"
        dist.init_process_group(backend=backend)
        pg = dist
    return rank, local, world, pg


def barrier(pg, device):
    import torch
    if pg is not None:
        pg.barrier()
    if torch.device(device).type == "cuda":
        torch.cuda.synchronize(device)


def max_over_ranks(pg, value, device):
    """The largest `value` over all ranks (every rank gets it)."""
    import torch
    if pg is None:
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    pg.all_reduce(t, op=pg.ReduceOp.MAX)
    return float(t.item())


def whole_job_gflops(world, flops_per_step_per_rank, steps, max_ms):
    """Whole-job throughput: every rank's FLOPs over the slowest rank's time."""
    return world * flops_per_step_per_rank * steps / (max_ms * 1e-3) / 1e9


# ------------------------------------------------------------------ workloads
def sgemm_step_fn(g, sets, w, stream):
    """Return a callable that runs gemm_sgemm on input set i (in place on C)."""
    def step(i):
        A, B, C = sets[i % len(sets)]
        st = g.gemm_sgemm(w.M, w.N, w.K, w.alpha, A.data_ptr(), w.K, B.data_ptr(), w.N,
                          w.beta, C.data_ptr(), w.N, stream)
        if st != 0:
            raise RuntimeError("gemm_sgemm: " + g.gemm_status_string(st))
    return step


def time_launches(torch, step, n, stream_obj):
    """Per-launch CUDA-event durations (ms) on the launching stream."""
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(n)]
    for i, (a, b) in enumerate(evs):
        a.record(stream_obj)
        step(i)
        b.record(stream_obj)
    torch.cuda.synchronize()
    return [a.elapsed_time(b) for a, b in evs]


def bench_sgemm_shape(torch, g, wl, name, fp32_peak, device, stream_obj):
    """Another fp32 workload on the CUDA-core kernel (4096^3, or the ragged
    3000x5000x1999 whose K = 1999 rows are not 16-byte multiples, so A is
    loaded by the generic cp.async producers).  Two input sets in turn, each
    larger than L2."""
    w = wl.WORKLOADS[name]
    w2 = wl.Workload(**{**w.__dict__, "seed": w.seed + 100, "name": name + "_b"})
    sets = [tuple(t.to(device) for t in wl.workload_inputs(x)) for x in (w, w2)]
    step = sgemm_step_fn(g, sets, w, stream_obj.cuda_stream)
    for i in range(3):
        step(i)
    torch.cuda.synchronize()
    times = time_launches(torch, step, 20, stream_obj)
    ms = statistics.median(times)
    tflops = w.flops / (ms * 1e-3) / 1e12
    del sets
    torch.cuda.empty_cache()
    return {
        "workload": "fp32 SGEMM M=%d N=%d K=%d, alpha=%g, beta=%g" % (w.M, w.N, w.K, w.alpha,
                                                                      w.beta),
        "kernel": "simt_gemm_kernel (CUDA cores, fma.rn.f32x2)",
        "value": tflops * 1e3, "unit": "GFLOP/s", "ms_per_launch_median": ms,
        "launches_timed": len(times),
        "roofline": {"bound": "alu", "achieved": tflops, "peak": fp32_peak, "unit": "TFLOP/s",
                     "frac": tflops / fp32_peak, "traffic": None,
                     "peak_note": "derived fp32 FFMA peak, as the headline"},
        "l2": "two input sets used in turn, each larger than L2",
    }


def bench_bf16_8192(torch, g, wl, peaks, device, stream_obj):
    w = wl.WORKLOADS["bf16_8192"]
    A, B, _ = wl.workload_inputs(w, with_c=False)
    A, B = A.to(device), B.to(device)
    C = torch.empty((w.M, w.N), dtype=torch.float32, device=device)
    s = stream_obj.cuda_stream

    def step(i):
        st = g.gemm_bf16gemm(w.M, w.N, w.K, w.alpha, A.data_ptr(), w.K, B.data_ptr(), w.N,
                             w.beta, C.data_ptr(), w.N, s)
        if st != 0:
            raise RuntimeError("gemm_bf16gemm: " + g.gemm_status_string(st))
    for i in range(3):
        step(i)
    torch.cuda.synchronize()
    times = time_launches(torch, step, 10, stream_obj)
    ms = statistics.median(times)
    flops = w.flops
    tflops = flops / (ms * 1e-3) / 1e12
    peak = peaks["bf16_tflops"]
    del A, B, C
    torch.cuda.empty_cache()
    return {
        "workload": "bf16 in / fp32 out GEMM M=N=K=8192, alpha=1, beta=0, N(0,0.02)",
        "kernel": "tc_bf16_pair_kernel (tcgen05 cta_group::2: CTA pairs on 256x256 tiles, TMEM accumulators)",
        "value": tflops * 1e3, "unit": "GFLOP/s", "ms_per_launch_median": ms,
        "ms_per_launch_min": min(times), "launches_timed": len(times),
        "roofline": {"bound": "tensor", "achieved": tflops, "peak": peak, "unit": "TFLOP/s",
                     "frac": tflops / peak, "traffic": recorded_traffic("tc_bf16_pair_kernel"),
                     "peak_note": "%s dense bf16 burst (cuBLAS); sustained %.1f" % (
                         peaks["source"], peaks["bf16_tflops_sustained"])},
        "l2": "operands 256 MB + C 256 MB per launch exceed the 129 MB L2",
    }


def bench_bf16_8192_fused(torch, g, wl, peaks, device, stream_obj):
    """The bf16 8192^3 GEMM with the fused output stage: bias + GELU, bf16 D."""
    w = wl.WORKLOADS["bf16_8192"]
    A, B, _ = wl.workload_inputs(w, with_c=False)
    A, B = A.to(device), B.to(device)
    bias = (torch.randn(w.N, generator=torch.Generator().manual_seed(9)) * 0.1).to(device)
    D = torch.empty((w.M, w.N), dtype=torch.bfloat16, device=device)
    s = stream_obj.cuda_stream

    def step(i):
        st = g.gemm_bf16gemm_epilogue(w.M, w.N, w.K, w.alpha, A.data_ptr(), w.K, B.data_ptr(), w.N,
                                      0.0, 0, w.N, bias.data_ptr(), g.ACT["gelu"], D.data_ptr(),
                                      w.N, g.OUT["bf16"], s)
        if st != 0:
            raise RuntimeError("gemm_bf16gemm_epilogue: " + g.gemm_status_string(st))
    for i in range(3):
        step(i)
    torch.cuda.synchronize()
    times = time_launches(torch, step, 10, stream_obj)
    ms = statistics.median(times)
    tflops = w.flops / (ms * 1e-3) / 1e12
    peak = peaks["bf16_tflops"]
    del A, B, D, bias
    torch.cuda.empty_cache()
    return {
        "workload": "bf16 GEMM M=N=K=8192 with fused bias + GELU, bf16 output",
        "kernel": "tc_bf16_pair_kernel (same kernel, fused output stage)",
        "value": tflops * 1e3, "unit": "GFLOP/s", "ms_per_launch_median": ms,
        "launches_timed": len(times),
        "roofline": {"bound": "tensor", "achieved": tflops, "peak": peak, "unit": "TFLOP/s",
                     "frac": tflops / peak, "traffic": None,
                     "peak_note": "%s dense bf16 burst (cuBLAS)" % peaks["source"]},
    }


def bench_bf16_8192_fp8(torch, g, wl, peaks, device, stream_obj):
    """The bf16 8192^3 GEMM quantised in its output stage: bias + GELU, fp8 E4M3
    D scaled by d_scale, and the amax of the unscaled values."""
    w = wl.WORKLOADS["bf16_8192"]
    A, B, _ = wl.workload_inputs(w, with_c=False)
    A, B = A.to(device), B.to(device)
    bias = (torch.randn(w.N, generator=torch.Generator().manual_seed(9)) * 0.1).to(device)
    D = torch.empty((w.M, w.N), dtype=torch.uint8, device=device)
    amax = torch.zeros(1, dtype=torch.float32, device=device)
    s = stream_obj.cuda_stream
    o = g.GemmOutput()
    o.beta, o.C, o.ldc = 0.0, 0, w.N
    o.bias, o.act = bias.data_ptr(), g.ACT["gelu"]
    o.residual, o.ldr = 0, w.N
    o.d_scale, o.amax = 64.0, amax.data_ptr()
    o.D, o.ldd, o.d_type = D.data_ptr(), w.N, g.OUT["f8e4m3"]

    def step(i):
        st = g.gemm_bf16gemm_fused(w.M, w.N, w.K, w.alpha, A.data_ptr(), w.K, B.data_ptr(), w.N,
                                   o, s)
        if st != 0:
            raise RuntimeError("gemm_bf16gemm_fused: " + g.gemm_status_string(st))
    for i in range(3):
        step(i)
    torch.cuda.synchronize()
    times = time_launches(torch, step, 10, stream_obj)
    ms = statistics.median(times)
    tflops = w.flops / (ms * 1e-3) / 1e12
    peak = peaks["bf16_tflops"]
    del A, B, D, bias, amax
    torch.cuda.empty_cache()
    return {
        "workload": "bf16 GEMM M=N=K=8192 with fused bias + GELU, fp8 E4M3 output (scale 64) + amax",
        "kernel": "tc_bf16_pair_kernel (same kernel, fused output stage)",
        "value": tflops * 1e3, "unit": "GFLOP/s", "ms_per_launch_median": ms,
        "launches_timed": len(times),
        "roofline": {"bound": "tensor", "achieved": tflops, "peak": peak, "unit": "TFLOP/s",
                     "frac": tflops / peak, "traffic": None,
                     "peak_note": "%s dense bf16 burst (cuBLAS)" % peaks["source"]},
    }


def bench_decode(torch, g, wl, peaks, device, stream_obj):
    w = wl.WORKLOADS["decode_16"]
    A, B, C0 = wl.workload_inputs(w)
    A = A.to(device)
    Bs = [B.to(device) for _ in range(3)]  # 3 x 100.7 MB, cycled: each launch reads a cold B
    C = C0.to(device)
    bytes_alg = (w.M * w.K + w.K * w.N) * 2 + 2 * w.M * w.N * 4
    s = stream_obj

    def step(i, stream_handle):
        Bi = Bs[i % 3]
        st = g.gemm_bf16gemm(w.M, w.N, w.K, w.alpha, A.data_ptr(), w.K, Bi.data_ptr(), w.N,
                             w.beta, C.data_ptr(), w.N, stream_handle)
        if st != 0:
            raise RuntimeError("gemm_bf16gemm (decode): " + g.gemm_status_string(st))
    # warm-up (also allocates the split-K workspace before capture)
    for i in range(6):
        step(i, s.cuda_stream)
    torch.cuda.synchronize()
    reps = 60
    graph = torch.cuda.CUDAGraph()
    cap = torch.cuda.Stream()
    step(0, cap.cuda_stream)   # any per-stream set-up happens before capture
    torch.cuda.synchronize()
    with torch.cuda.stream(cap):
        graph.capture_begin()
        for i in range(reps):
            step(i, cap.cuda_stream)
        graph.capture_end()
    torch.cuda.synchronize()
    trial_ms = []
    with torch.cuda.stream(cap):   # replay() launches on the current stream
        graph.replay()
        torch.cuda.synchronize()
        for _ in range(5):
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record(cap)
            graph.replay()
            b.record(cap)
            torch.cuda.synchronize()
            trial_ms.append(a.elapsed_time(b) / reps)
    ms = statistics.median(trial_ms)
    gbs = bytes_alg / (ms * 1e-3) / 1e9
    peak = peaks["hbm_gbs"]
    del A, Bs, C, graph
    torch.cuda.empty_cache()
    return {
        "workload": "decode bf16 GEMM M=16, N=12288, K=4096, alpha=1, beta=1",
        "kernel": "tc_decode_kernel (tcgen05 swap-AB, split-K, fixed-order fix-up)",
        "value": gbs, "unit": "GB/s", "gflops": w.flops / (ms * 1e-3) / 1e9,
        "us_per_launch_median": ms * 1e3, "launches_timed": reps * 5,
        "algorithmic_bytes": bytes_alg,
        "roofline": {"bound": "hbm", "achieved": gbs, "peak": peak, "unit": "GB/s",
                     "frac": gbs / peak, "traffic": recorded_traffic("tc_decode_kernel"),
                     "peak_note": "%s STREAM-style copy" % peaks["source"]},
        "l2": "3 copies of B (302 MB) cycled; launches replayed from a CUDA graph",
    }


class OracleSampler:
    """Times the oracle on whole rows of the 4092^3 workload: the inputs are
    drawn and the rate calibrated once, then each sample runs as many rows as
    fit its time budget."""

    def __init__(self, wl):
        import oracle
        self.w = wl.WORKLOADS["sgemm_4092"]
        A, B, C = wl.workload_inputs(self.w)
        self.A, self.B, self.C = A.numpy(), B.numpy(), C.numpy()
        self.threads = oracle.max_threads()
        rows = 4 * self.threads  # calibration: a few rows per thread
        t0 = time.perf_counter()
        oracle.sgemm(self.w.alpha, self.A[:rows], self.B, self.w.beta, self.C[:rows])
        self.sec_per_row = max(time.perf_counter() - t0, 1e-6) / rows

    def sample(self, target_seconds):
        import oracle
        w = self.w
        rows = int(max(1, min(w.M, target_seconds / self.sec_per_row)))
        t0 = time.perf_counter()
        oracle.sgemm(w.alpha, self.A[:rows], self.B, w.beta, self.C[:rows])
        t = time.perf_counter() - t0
        flops = 2.0 * rows * w.N * w.K
        return {"value": flops / t / 1e9, "unit": "GFLOP/s", "cores": self.threads,
                "kind": "oracle",
                "sample": "%d of 4092 rows of the fp32 4092^3 workload (fp64 triple loop, "
                          "%.2f s, %s)" % (rows, t, os.uname().machine),
                "seconds": t}


def cpu_oracle_sample(wl, target_seconds):
    """One oracle sample of about `target_seconds` on the 4092^3 workload."""
    return OracleSampler(wl).sample(target_seconds)


# ------------------------------------------------------------------ main arms
def run_reference(args):
    """The oracle timed on the host cores, on the headline workload's config."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    from dense_gemm_12_gb300 import workloads as wl
    w = wl.WORKLOADS["sgemm_4092"]
    # About 150 s of oracle time for the whole run, whatever --steps is.
    per_step = max(0.05, min(20.0, 150.0 / max(args.steps + args.warmup, 1)))
    sampler = OracleSampler(wl)
    for _ in range(args.warmup):
        sampler.sample(per_step / 4)
    samples = [sampler.sample(per_step) for _ in range(args.steps)]
    total_flops = sum(s["value"] * 1e9 * s["seconds"] for s in samples)
    total_t = sum(s["seconds"] for s in samples)
    value = total_flops / total_t / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "GFLOP/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": total_t / args.steps * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": "fp32 SGEMM M=N=K=4092, alpha=0.7, beta=0.3, U[-1,1)",
                   "step": "a bounded sample of whole rows of the workload per step",
                   "l2": "n/a (CPU)"},
        "cpu_baseline": {"value": value, "unit": "GFLOP/s", "cores": samples[0]["cores"],
                         "kind": "oracle", "sample": samples[0]["sample"]},
        "e2e": {"value": value, "unit": "GFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)


def run_ours(args):
    import torch

    import dense_gemm_12_gb300 as g
    from dense_gemm_12_gb300 import workloads as wl

    rank, local, world, pg = dist_setup(args.gpus)
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    g.load_library(build_if_missing=True)
    peaks = load_peaks()
    num_sms = torch.cuda.get_device_properties(device).multi_processor_count
    fp32_peak = num_sms * SM_LANES_FP32 * 2 * MAX_SM_CLOCK_HZ / 1e12  # TFLOP/s

    w = wl.WORKLOADS["sgemm_4092"]
    stream_obj = torch.cuda.current_stream(device)
    stream = stream_obj.cuda_stream
    host_sets = [wl.workload_inputs(w)]
    w2 = wl.Workload(**{**w.__dict__, "seed": w.seed + 100, "name": "sgemm_4092_b"})
    host_sets.append(wl.workload_inputs(w2))
    sets = [tuple(t.to(device) for t in hs) for hs in host_sets]
    step = sgemm_step_fn(g, sets, w, stream)

    for i in range(args.warmup):
        step(i)
    barrier(pg, device)

    sampler = ClockSampler(local) if rank == 0 else None
    if sampler:
        sampler.start()
        time.sleep(0.3)
    # timed region: exactly K steps between barriers, events on the launching stream
    barrier(pg, device)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_start.record(stream_obj)
    for i in range(args.steps):
        ev[i][0].record(stream_obj)
        step(i)
        ev[i][1].record(stream_obj)
    t_end.record(stream_obj)
    barrier(pg, device)
    clocks = sampler.stop() if sampler else None
    total_ms = max_over_ranks(pg, t_start.elapsed_time(t_end), device)
    launch_ms = [a.elapsed_time(b) for a, b in ev]
    st = g.gemm_check_device_error(stream)
    if st != 0:
        raise RuntimeError("device error: " + g.gemm_status_string(st))

    flops_step = w.flops
    value = whole_job_gflops(world, flops_step, args.steps, total_ms)
    kernel_ms = statistics.mean(launch_ms)
    achieved = flops_step / (kernel_ms * 1e-3) / 1e12

    # e2e: host buffers through the C ABI, copies inside the timed region.
    # Every step copies its A, B, C in from pinned host memory and its C out.
    # The copies are pipelined with the GEMMs on separate streams over the two
    # device buffer sets: while step i computes on set i % 2, the inputs of
    # step i + 1 are copied into the other set and the result of step i - 1 is
    # copied out.
    e2e = None
    if not args.no_e2e:
        pinned = [tuple(t.pin_memory() for t in hs) for hs in host_sets]
        outs = [torch.empty((w.M, w.N), dtype=torch.float32).pin_memory() for _ in range(2)]
        dev_bufs = sets
        s_in, s_out = torch.cuda.Stream(device), torch.cuda.Stream(device)
        loaded = [torch.cuda.Event() for _ in range(2)]
        computed = [torch.cuda.Event() for _ in range(2)]
        freed = [None, None]

        def e2e_step(i):
            k = i % 2
            hA, hB, hC = pinned[k]
            dA, dB, dC = dev_bufs[k]
            with torch.cuda.stream(s_in):
                if freed[k] is not None:
                    s_in.wait_event(freed[k])      # step i-2 is done with set k
                dA.copy_(hA, non_blocking=True)
                dB.copy_(hB, non_blocking=True)
                dC.copy_(hC, non_blocking=True)
                loaded[k].record(s_in)
            stream_obj.wait_event(loaded[k])
            s_ = g.gemm_sgemm(w.M, w.N, w.K, w.alpha, dA.data_ptr(), w.K, dB.data_ptr(), w.N,
                              w.beta, dC.data_ptr(), w.N, stream)
            if s_ != 0:
                raise RuntimeError(g.gemm_status_string(s_))
            computed[k].record(stream_obj)
            with torch.cuda.stream(s_out):
                s_out.wait_event(computed[k])
                outs[k].copy_(dC, non_blocking=True)
                ev = torch.cuda.Event()
                ev.record(s_out)
                freed[k] = ev
        e2e_step(0)
        e2e_step(1)
        torch.cuda.synchronize(device)
        barrier(pg, device)
        # Enough steps that the pipeline's fill (the first step's input copy)
        # and drain (the last step's output copy) are a small part of the time.
        n_e2e = max(3, min(args.steps, 40))
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(s_in)
        for i in range(n_e2e):
            e2e_step(i)
        b.record(s_out)
        torch.cuda.synchronize(device)
        barrier(pg, device)
        e2e_ms = max_over_ranks(pg, a.elapsed_time(b), device)
        e2e = {"value": whole_job_gflops(world, flops_step, n_e2e, e2e_ms), "unit": "GFLOP/s",
               "h2d_bytes_per_step": (w.M * w.K + w.K * w.N + w.M * w.N) * 4,
               "d2h_bytes_per_step": w.M * w.N * 4, "steps": n_e2e,
               "pipelined": "copies of step i+1 and i-1 overlap the GEMM of step i"}
        del pinned, outs

    parts = {}
    if not args.no_parts and rank == 0:
        del sets
        torch.cuda.empty_cache()
        for name in ("sgemm_4096", "sgemm_ragged"):
            w_ = wl.WORKLOADS[name]
            parts["sgemm_%dx%dx%d" % (w_.M, w_.N, w_.K)] = bench_sgemm_shape(
                torch, g, wl, name, fp32_peak, device, stream_obj)
        parts["bf16_8192"] = bench_bf16_8192(torch, g, wl, peaks, device, stream_obj)
        parts["bf16_8192_bias_gelu_bf16out"] = bench_bf16_8192_fused(torch, g, wl, peaks, device,
                                                                      stream_obj)
        parts["bf16_8192_bias_gelu_fp8out_amax"] = bench_bf16_8192_fp8(torch, g, wl, peaks,
                                                                        device, stream_obj)
        parts["decode_16x12288x4096"] = bench_decode(torch, g, wl, peaks, device, stream_obj)

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        cpu = cpu_oracle_sample(wl, args.cpu_seconds)
        cpu.pop("seconds", None)

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "GFLOP/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": total_ms / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": "fp32 SGEMM M=N=K=4092, alpha=0.7, beta=0.3, "
                                   "A,B,C ~ U[-1,1), row-major",
                       "l2": "two 201 MB input sets used in turn (inputs larger than L2)",
                       "parallelism": "replicas" if world > 1 else "single GPU"},
            "roofline": {"bound": "alu", "achieved": achieved, "peak": fp32_peak,
                         "unit": "TFLOP/s", "frac": achieved / fp32_peak,
                         "traffic": recorded_traffic("simt_gemm_kernel"),
                         "peak_note": "%d SMs x 128 fp32 lanes x 2 FLOP x 2.07 GHz max clock "
                                      "(derived)" % num_sms,
                         "kernel_ms_mean": kernel_ms, "kernel_ms_min": min(launch_ms)},
            "clocks": clocks,
            "e2e": e2e,
            "gpu_launches": args.steps,
            "cpu_baseline": cpu,
            "parts": parts,
        }
        print(json.dumps(line), flush=True)
    if pg is not None:
        pg.destroy_process_group()


def run_only(args):
    """One kernel's workload alone, for profiler captures (not the contract line)."""
    import torch

    import dense_gemm_12_gb300 as g
    from dense_gemm_12_gb300 import workloads as wl
    device = torch.device("cuda", 0)
    torch.cuda.set_device(device)
    g.load_library(build_if_missing=True)
    peaks = load_peaks()
    stream_obj = torch.cuda.current_stream(device)
    if args.only == "bf16":
        out = bench_bf16_8192(torch, g, wl, peaks, device, stream_obj)
    elif args.only == "decode":
        out = bench_decode(torch, g, wl, peaks, device, stream_obj)
    else:
        w = wl.WORKLOADS["sgemm_4092"]
        w2 = wl.Workload(**{**w.__dict__, "seed": w.seed + 100, "name": "sgemm_4092_b"})
        sets = [tuple(t.to(device) for t in wl.workload_inputs(x)) for x in (w, w2)]
        step = sgemm_step_fn(g, sets, w, stream_obj.cuda_stream)
        for i in range(args.warmup):
            step(i)
        ms = time_launches(torch, step, args.steps, stream_obj)
        out = {"workload": "fp32 SGEMM 4092^3", "ms_per_launch": ms,
               "gflops_median": w.flops / (statistics.median(ms) * 1e-3) / 1e9}
    st = g.gemm_check_device_error(stream_obj.cuda_stream)
    if st != 0:
        raise RuntimeError("device error: " + g.gemm_status_string(st))
    print(json.dumps({"only": args.only, **out}), flush=True)


def main():
    args = parse_args()
    if args.only:
        run_only(args)
        return
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
