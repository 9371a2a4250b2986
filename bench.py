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
MIN_TRIAL_MS = 200.0       # each timed trial of a part lasts at least this long
TRIALS = 5                 # trials per part; the median is reported
E2E_TRIALS = 5             # end-to-end trials (median reported)
SUSTAINED_MS = 2000.0      # the sustained bf16 part runs back to back this long


def parse_args():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=200)
    p.add_argument("--warmup", type=int, default=3)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--no-parts", action="store_true", help="headline workload only")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--brief-parts", action="store_true",
                   help="profiler runs: one short trial per part (not bench values)")
    p.add_argument("--only", choices=["sgemm", "sgemm4096", "sgemm256", "ragged", "bf16",
                                      "decode", "decode_graph"],
                   default=None,
                   help="time one kernel's workload alone (profiling runs); prints its part")
    p.add_argument("--cpu-seconds", type=float, default=12.0,
                   help="target duration of the CPU-oracle sample")
    return p.parse_args()


# ------------------------------------------------------------------ helpers
def _smi_max_sm_mhz():
    try:
        out = subprocess.run(["nvidia-smi", "-i", "0", "--query-gpu=clocks.max.sm",
                              "--format=csv,noheader,nounits"], capture_output=True, text=True,
                             timeout=30).stdout.split()
        return float(out[0]) if out else None
    except (OSError, ValueError, subprocess.TimeoutExpired):
        return None


def load_peaks():
    """Roofline denominators: HBM GB/s and dense bf16 TFLOP/s (burst and
    sustained) measured on this machine (MEASURED_PEAKS.json), and the maximum
    SM clock the fp32 FFMA peak is derived from (the same file, else the
    device's own clocks.max.sm)."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    d = {}
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
    if "hbm_gbs" in d and "bf16_tflops" in d:
        peaks = {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                 "bf16_tflops_sustained": d.get("bf16_tflops_sustained", d["bf16_tflops"]),
                 "source": "measured"}
    else:
        peaks = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
                 "source": "fallback"}
    # median SM clock sampled under load during those measurements (mostly
    # the seconds-long loop behind the sustained bf16 figure)
    peaks["sustained_sm_mhz"] = (d.get("clocks_under_load") or {}).get("sm_mhz_median")
    if d.get("sm_max_mhz"):
        peaks["sm_max_mhz"], peaks["sm_clock_source"] = float(d["sm_max_mhz"]), "MEASURED_PEAKS.json"
    else:
        mhz = _smi_max_sm_mhz()
        peaks["sm_max_mhz"], peaks["sm_clock_source"] = (
            (mhz, "nvidia-smi clocks.max.sm") if mhz else (2070.0, "fallback (GB300 maximum)"))
    return peaks


def fp32_ffma_peak(num_sms, peaks):
    """Derived fp32 FFMA peak in TFLOP/s: SMs x 128 lanes x 2 FLOP x max SM clock."""
    return num_sms * SM_LANES_FP32 * 2 * peaks["sm_max_mhz"] * 1e6 / 1e12


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


def time_window(torch, step, reps, stream_obj, first=0):
    """Duration (ms) of `reps` back-to-back calls of step(first..), between two
    CUDA events on the launching stream."""
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record(stream_obj)
    for i in range(reps):
        step(first + i)
    b.record(stream_obj)
    torch.cuda.synchronize()
    return a.elapsed_time(b)


# --brief-parts (profiler runs only: a launch list of the whole command):
# one short trial per part instead of the protocol's; its numbers are not
# bench values.
BRIEF = {"on": False}


def measure_part(torch, step, stream_obj, gpu_index, units_per_call=1, warmup=3,
                 min_trial_ms=MIN_TRIAL_MS, trials=TRIALS):
    """The timing protocol of every part: `warmup` untimed calls, then
    `trials` trials of R back-to-back calls each, R chosen so that a trial
    lasts at least `min_trial_ms`; nvidia-smi samples the clocks over the
    trials.  A call may run several launches (`units_per_call`, e.g. a CUDA
    graph); times are reported per launch.  Returns the per-launch median,
    the spread over trials, R and the clock record."""
    if BRIEF["on"]:
        min_trial_ms, trials = 1.0, 1
    for i in range(warmup):
        step(i)
    torch.cuda.synchronize()
    est = time_window(torch, step, 3, stream_obj, first=warmup) / 3
    reps = max(1, int(math.ceil(min_trial_ms / max(est, 1e-3))))
    sampler = ClockSampler(gpu_index)
    sampler.start()
    time.sleep(0.3)
    per = []
    first = warmup + 3
    for _ in range(trials):
        per.append(time_window(torch, step, reps, stream_obj, first) / (reps * units_per_call))
        first += reps
    clocks = sampler.stop()
    med = statistics.median(per)
    return {"ms_per_launch_median": med, "ms_per_launch_min": min(per),
            "ms_per_launch_max": max(per), "trial_spread": (max(per) - min(per)) / med,
            "trials": trials, "launches_per_trial": reps * units_per_call,
            "trial_ms_median": med * reps * units_per_call, "clocks": clocks}


def bench_sgemm_shape(torch, g, wl, name, fp32_peak, device, stream_obj, gpu_index):
    """Another fp32 workload on the CUDA-core kernel (4096^3, or the ragged
    3000x5000x1999 whose K = 1999 rows are not 16-byte multiples, so A is
    first copied to a 16-byte pitch; the copy is inside the timed launch).
    Two input sets in turn, each larger than L2."""
    w = wl.WORKLOADS[name]
    w2 = wl.Workload(**{**w.__dict__, "seed": w.seed + 100, "name": name + "_b"})
    sets = [tuple(t.to(device) for t in wl.workload_inputs(x)) for x in (w, w2)]
    step = sgemm_step_fn(g, sets, w, stream_obj.cuda_stream)
    t = measure_part(torch, step, stream_obj, gpu_index)
    tflops = w.flops / (t["ms_per_launch_median"] * 1e-3) / 1e12
    del sets
    torch.cuda.empty_cache()
    return {
        "workload": "fp32 SGEMM M=%d N=%d K=%d, alpha=%g, beta=%g" % (w.M, w.N, w.K, w.alpha,
                                                                      w.beta),
        "kernel": "simt_gemm_kernel (CUDA cores, fma.rn.f32x2)",
        "value": tflops * 1e3, "unit": "GFLOP/s", **t,
        "roofline": {"bound": "alu", "achieved": tflops, "peak": fp32_peak, "unit": "TFLOP/s",
                     "frac": tflops / fp32_peak, "traffic": None,
                     "peak_note": "derived fp32 FFMA peak, as the headline"},
        "l2": "two input sets used in turn, each larger than L2",
    }


def _bf16_8192_operands(torch, wl, device):
    w = wl.WORKLOADS["bf16_8192"]
    A, B, _ = wl.workload_inputs(w, with_c=False)
    return w, A.to(device), B.to(device)


def per_clock(tflops, clocks, peaks):
    """A power-capped bf16 part's rate per GHz of its median SM clock, against
    the sustained cuBLAS figure per GHz of the clock it was measured at: the
    comparison without the box-to-box spread of the power-capped clock."""
    mhz, ref_mhz = (clocks or {}).get("sm_mhz"), peaks.get("sustained_sm_mhz")
    if not mhz or not ref_mhz:
        return None
    ours, ref = tflops / (mhz / 1e3), peaks["bf16_tflops_sustained"] / (ref_mhz / 1e3)
    return {"tflops_per_ghz": ours, "sm_mhz": mhz, "sustained_tflops_per_ghz": ref,
            "sustained_sm_mhz": ref_mhz, "ratio": ours / ref}


def bench_bf16_8192(torch, g, wl, peaks, device, stream_obj, gpu_index):
    w, A, B = _bf16_8192_operands(torch, wl, device)
    C = torch.empty((w.M, w.N), dtype=torch.float32, device=device)
    s = stream_obj.cuda_stream

    def step(i):
        st = g.gemm_bf16gemm(w.M, w.N, w.K, w.alpha, A.data_ptr(), w.K, B.data_ptr(), w.N,
                             w.beta, C.data_ptr(), w.N, s)
        if st != 0:
            raise RuntimeError("gemm_bf16gemm: " + g.gemm_status_string(st))
    t = measure_part(torch, step, stream_obj, gpu_index)
    tflops = w.flops / (t["ms_per_launch_median"] * 1e-3) / 1e12
    # the same kernel back to back for seconds, against the sustained peak
    sustained = measure_part(torch, step, stream_obj, gpu_index, warmup=0,
                             min_trial_ms=SUSTAINED_MS, trials=1)
    s_tflops = w.flops / (sustained["ms_per_launch_median"] * 1e-3) / 1e12
    del A, B, C
    torch.cuda.empty_cache()
    burst, sus = peaks["bf16_tflops"], peaks["bf16_tflops_sustained"]
    return {
        "workload": "bf16 in / fp32 out GEMM M=N=K=8192, alpha=1, beta=0, N(0,0.02)",
        "kernel": "tc_bf16_pair_kernel (tcgen05 cta_group::2: CTA pairs on 256x256 tiles, TMEM accumulators)",
        "value": tflops * 1e3, "unit": "GFLOP/s", **t,
        "roofline": {"bound": "tensor", "achieved": tflops, "peak": sus, "unit": "TFLOP/s",
                     "frac": tflops / sus, "frac_of_burst": tflops / burst,
                     "traffic": recorded_traffic("tc_bf16_pair_kernel"),
                     "peak_note": BF16_PEAK_NOTE % (peaks["source"], sus, burst)},
        "per_clock": per_clock(tflops, t["clocks"], peaks),
        "sustained": {"value": s_tflops * 1e3, "unit": "GFLOP/s",
                      "seconds": sustained["trial_ms_median"] / 1e3,
                      "launches": sustained["launches_per_trial"],
                      "ms_per_launch": sustained["ms_per_launch_median"],
                      "roofline": {"bound": "tensor", "achieved": s_tflops, "peak": sus,
                                   "unit": "TFLOP/s", "frac": s_tflops / sus,
                                   "peak_note": "%s dense bf16 sustained (cuBLAS, 4 s back to "
                                                "back)" % peaks["source"]},
                      "clocks": sustained["clocks"]},
        "l2": "operands 256 MB + C 256 MB per launch exceed the 129 MB L2",
    }


def bench_bf16_8192_fused(torch, g, wl, peaks, device, stream_obj, gpu_index):
    """The bf16 8192^3 GEMM with the fused output stage: bias + GELU, bf16 D."""
    w, A, B = _bf16_8192_operands(torch, wl, device)
    bias = (torch.randn(w.N, generator=torch.Generator().manual_seed(9)) * 0.1).to(device)
    D = torch.empty((w.M, w.N), dtype=torch.bfloat16, device=device)
    s = stream_obj.cuda_stream

    def step(i):
        st = g.gemm_bf16gemm_epilogue(w.M, w.N, w.K, w.alpha, A.data_ptr(), w.K, B.data_ptr(), w.N,
                                      0.0, 0, w.N, bias.data_ptr(), g.ACT["gelu"], D.data_ptr(),
                                      w.N, g.OUT["bf16"], s)
        if st != 0:
            raise RuntimeError("gemm_bf16gemm_epilogue: " + g.gemm_status_string(st))
    t = measure_part(torch, step, stream_obj, gpu_index)
    tflops = w.flops / (t["ms_per_launch_median"] * 1e-3) / 1e12
    peak, sus = peaks["bf16_tflops"], peaks["bf16_tflops_sustained"]
    del A, B, D, bias
    torch.cuda.empty_cache()
    return {
        "workload": "bf16 GEMM M=N=K=8192 with fused bias + GELU, bf16 output",
        "kernel": "tc_bf16_pair_kernel (same kernel, fused output stage)",
        "value": tflops * 1e3, "unit": "GFLOP/s", **t,
        "roofline": {"bound": "tensor", "achieved": tflops, "peak": sus, "unit": "TFLOP/s",
                     "frac": tflops / sus, "frac_of_burst": tflops / peak, "traffic": None,
                     "peak_note": BF16_PEAK_NOTE % (peaks["source"], sus, peak)},
    }


def bench_bf16_8192_fp8(torch, g, wl, peaks, device, stream_obj, gpu_index):
    """The bf16 8192^3 GEMM quantised in its output stage: bias + GELU, fp8 E4M3
    D scaled by d_scale, and the amax of the unscaled values."""
    w, A, B = _bf16_8192_operands(torch, wl, device)
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
    t = measure_part(torch, step, stream_obj, gpu_index)
    tflops = w.flops / (t["ms_per_launch_median"] * 1e-3) / 1e12
    peak, sus = peaks["bf16_tflops"], peaks["bf16_tflops_sustained"]
    del A, B, D, bias, amax
    torch.cuda.empty_cache()
    return {
        "workload": "bf16 GEMM M=N=K=8192 with fused bias + GELU, fp8 E4M3 output (scale 64) + amax",
        "kernel": "tc_bf16_pair_kernel (same kernel, fused output stage)",
        "value": tflops * 1e3, "unit": "GFLOP/s", **t,
        "roofline": {"bound": "tensor", "achieved": tflops, "peak": sus, "unit": "TFLOP/s",
                     "frac": tflops / sus, "frac_of_burst": tflops / peak, "traffic": None,
                     "peak_note": BF16_PEAK_NOTE % (peaks["source"], sus, peak)},
    }


DECODE_GRAPH_LAUNCHES = 200
# Trials of >= 200 ms of back-to-back 8192^3 launches run at the power cap
# (clocks ~1.5 GHz), the regime of the sustained cuBLAS figure, not of its
# best-of-10 burst.
BF16_PEAK_NOTE = ("%s dense bf16 sustained (cuBLAS back to back for 4 s: %.1f); the burst "
                  "figure (best of 10 launches: %.1f) is frac_of_burst's denominator")


def bench_decode(torch, g, wl, peaks, device, stream_obj, gpu_index):
    w = wl.WORKLOADS["decode_16"]
    A, B, C0 = wl.workload_inputs(w)
    A = A.to(device)
    Bs = [B.to(device) for _ in range(3)]  # 3 x 100.7 MB, cycled: each launch reads a cold B
    C = C0.to(device)
    bytes_alg = (w.M * w.K + w.K * w.N) * 2 + 2 * w.M * w.N * 4

    def launch(i, stream_handle):
        Bi = Bs[i % 3]
        st = g.gemm_bf16gemm(w.M, w.N, w.K, w.alpha, A.data_ptr(), w.K, Bi.data_ptr(), w.N,
                             w.beta, C.data_ptr(), w.N, stream_handle)
        if st != 0:
            raise RuntimeError("gemm_bf16gemm (decode): " + g.gemm_status_string(st))
    reps = DECODE_GRAPH_LAUNCHES   # a multiple of 3: the graph ends on the B it began with
    graph = torch.cuda.CUDAGraph()
    cap = torch.cuda.Stream()
    for i in range(6):
        launch(i, cap.cuda_stream)   # any per-stream set-up happens before capture
    torch.cuda.synchronize()
    with torch.cuda.stream(cap):
        graph.capture_begin()
        for i in range(reps):
            launch(i, cap.cuda_stream)
        graph.capture_end()
    torch.cuda.synchronize()
    with torch.cuda.stream(cap):   # replay() launches on the current stream
        t = measure_part(torch, lambda i: graph.replay(), cap, gpu_index, units_per_call=reps)
    ms = t["ms_per_launch_median"]
    gbs = bytes_alg / (ms * 1e-3) / 1e9
    peak = peaks["hbm_gbs"]
    del A, Bs, C, graph
    torch.cuda.empty_cache()
    return {
        "workload": "decode bf16 GEMM M=16, N=12288, K=4096, alpha=1, beta=1",
        "kernel": "tc_decode_kernel (tcgen05 swap-AB, one CTA per 128-column group)",
        "value": gbs, "unit": "GB/s", "gflops": w.flops / (ms * 1e-3) / 1e9,
        "us_per_launch_median": ms * 1e3, **t,
        "algorithmic_bytes": bytes_alg,
        "roofline": {"bound": "hbm", "achieved": gbs, "peak": peak, "unit": "GB/s",
                     "frac": gbs / peak, "traffic": recorded_traffic("tc_decode_kernel"),
                     "peak_note": "%s STREAM-style copy" % peaks["source"]},
        "l2": "3 copies of B (302 MB) cycled; launches replayed from a CUDA graph of %d" % reps,
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
        """Whole rows of the workload for about target_seconds: a leading block
        of rows, or -- when the whole matrix takes less -- the whole matrix
        as many times as fit."""
        import oracle
        w = self.w
        rows = int(max(1, min(w.M, target_seconds / self.sec_per_row)))
        passes = 1
        if rows == w.M:
            passes = max(1, int(round(target_seconds / (self.sec_per_row * w.M))))
        t0 = time.perf_counter()
        for _ in range(passes):
            oracle.sgemm(w.alpha, self.A[:rows], self.B, w.beta, self.C[:rows])
        t = time.perf_counter() - t0
        flops = 2.0 * rows * w.N * w.K * passes
        what = ("%d of 4092 rows" % rows if passes == 1 else
                "all 4092 rows, %d times" % passes)
        return {"value": flops / t / 1e9, "unit": "GFLOP/s", "cores": self.threads,
                "kind": "oracle",
                "sample": "%s of the fp32 4092^3 workload (fp64 triple loop, %.2f s, %s)"
                          % (what, t, os.uname().machine),
                "seconds": t}


def cpu_oracle_sample(wl, target_seconds):
    """One oracle sample of about `target_seconds` on the 4092^3 workload."""
    return OracleSampler(wl).sample(target_seconds)


# ------------------------------------------------------------------ main arms
# The pages' own measurements of this path (other hardware; context, not
# targets): "A GEMM Kernel, Step by Step" on an RTX A6000 at 4092^3 fp32, and
# "GEMM Worklog I: Naive to Tiled" ("4. Benchmark Results on NVIDIA A100") at
# 4096^3 fp32.
PAGES_CONTEXT = {
    "note": "figures the pages report on other GPUs; context only, not targets",
    "rtx_a6000_fp32_4092": {"cublas_gflops": 23249.6, "naive_gflops": 309.0,
                            "warptiling_gflops": 21779.3},
    "a100_fp32_4096": {"naive_tflops": 0.26, "naive_frac_of_peak": 0.013,
                       "tiled_32x32_tflops": 7.12, "tiled_32x32_frac_of_peak": 0.365,
                       "cublas_tflops": 18.32, "cublas_frac_of_peak": 0.939},
}


def headline_config(world):
    """The `config` of the JSON line, identical in both arms."""
    return {"workload": "fp32 SGEMM M=N=K=4092, alpha=0.7, beta=0.3, A,B,C ~ U[-1,1), row-major",
            "l2": "two 201 MB input sets used in turn (inputs larger than L2)",
            "parallelism": "replicas" if world > 1 else "single GPU"}


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
        "config": headline_config(int(os.environ.get("WORLD_SIZE", "1"))),
        "step": "the CPU oracle on a bounded sample of whole rows of the workload per step "
                "(host cores; L2 flushing does not apply)",
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
    fp32_peak = fp32_ffma_peak(num_sms, peaks)  # TFLOP/s

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
        # Warm-up: every pinned buffer through the copies a few times (the
        # first steps after pinning ran ~1 ms slower each).
        for i in range(2 * max(3, args.warmup)):
            e2e_step(i)
        torch.cuda.synchronize(device)
        barrier(pg, device)
        # Enough steps that the pipeline's fill (the first step's input copy,
        # ~1 ms) and drain (the last step's output copy, ~0.35 ms) are a small
        # part of the time: at 20 steps they were 3 % of it.
        n_e2e = min(max(args.steps, 60), 200)
        # Five trials, the median reported: the host link is shared with the
        # machine's other work, and a trial can run ~1 ms per step slower on the
        # copies alone (the GEMM's own time does not move).
        trial_ms = []
        for _ in range(E2E_TRIALS):
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record(s_in)
            for i in range(n_e2e):
                e2e_step(i)
            b.record(s_out)
            torch.cuda.synchronize(device)
            barrier(pg, device)
            trial_ms.append(max_over_ranks(pg, a.elapsed_time(b), device))
        e2e_ms = statistics.median(trial_ms)
        e2e = {"value": whole_job_gflops(world, flops_step, n_e2e, e2e_ms), "unit": "GFLOP/s",
               "h2d_bytes_per_step": (w.M * w.K + w.K * w.N + w.M * w.N) * 4,
               "d2h_bytes_per_step": w.M * w.N * 4, "steps": n_e2e,
               "trials": len(trial_ms),
               "trial_values": [whole_job_gflops(world, flops_step, n_e2e, t) for t in trial_ms],
               "pipelined": "copies of step i+1 and i-1 overlap the GEMM of step i; "
                            "the first step's input copy and the last step's output "
                            "copy are not overlapped"}
        del pinned, outs

    parts = {}
    if not args.no_parts and rank == 0:
        del sets
        torch.cuda.empty_cache()
        for name in ("sgemm_4096", "sgemm_ragged"):
            w_ = wl.WORKLOADS[name]
            parts["sgemm_%dx%dx%d" % (w_.M, w_.N, w_.K)] = bench_sgemm_shape(
                torch, g, wl, name, fp32_peak, device, stream_obj, local)
        parts["bf16_8192"] = bench_bf16_8192(torch, g, wl, peaks, device, stream_obj, local)
        parts["bf16_8192_bias_gelu_bf16out"] = bench_bf16_8192_fused(
            torch, g, wl, peaks, device, stream_obj, local)
        parts["bf16_8192_bias_gelu_fp8out_amax"] = bench_bf16_8192_fp8(
            torch, g, wl, peaks, device, stream_obj, local)
        parts["decode_16x12288x4096"] = bench_decode(torch, g, wl, peaks, device, stream_obj,
                                                     local)
        parts["protocol"] = ("every part: 3 warm-up launches, then %d trials of back-to-back "
                             "launches lasting >= %d ms each between CUDA events on the "
                             "launching stream; median per launch reported with the spread; "
                             "clocks sampled by nvidia-smi over the trials"
                             % (TRIALS, MIN_TRIAL_MS))

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:   # N = 1 only
        cpu = cpu_oracle_sample(wl, args.cpu_seconds)
        cpu.pop("seconds", None)

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "GFLOP/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": total_ms / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": headline_config(world),
            "roofline": {"bound": "alu", "achieved": achieved, "peak": fp32_peak,
                         "unit": "TFLOP/s", "frac": achieved / fp32_peak,
                         "traffic": recorded_traffic("simt_gemm_kernel"),
                         "peak_note": "%d SMs x 128 fp32 lanes x 2 FLOP x %.0f MHz max SM clock "
                                      "(%s; derived)" % (num_sms, peaks["sm_max_mhz"],
                                                         peaks["sm_clock_source"]),
                         "kernel_ms_mean": kernel_ms, "kernel_ms_min": min(launch_ms)},
            "clocks": clocks,
            "context": PAGES_CONTEXT,
            "e2e": e2e,
            "gpu_launches": args.steps,
            "cpu_baseline": cpu,
            "parts": parts,
        }
        print(json.dumps(line), flush=True)
    if pg is not None:
        pg.destroy_process_group()


def run_only(args):
    """One kernel's workload alone, `--warmup` then `--steps` launches, for
    profiler captures (not the contract line; numbers taken under a profiler
    are not bench values)."""
    import torch

    import dense_gemm_12_gb300 as g
    from dense_gemm_12_gb300 import workloads as wl
    device = torch.device("cuda", 0)
    torch.cuda.set_device(device)
    g.load_library(build_if_missing=True)
    stream_obj = torch.cuda.current_stream(device)
    s = stream_obj.cuda_stream
    if args.only == "bf16":
        w, A, B = _bf16_8192_operands(torch, wl, device)
        C = torch.empty((w.M, w.N), dtype=torch.float32, device=device)

        def step(i):
            g.gemm_bf16gemm(w.M, w.N, w.K, w.alpha, A.data_ptr(), w.K, B.data_ptr(), w.N,
                            w.beta, C.data_ptr(), w.N, s)
    elif args.only in ("decode", "decode_graph"):
        w = wl.WORKLOADS["decode_16"]
        A, B, C = (t.to(device) for t in wl.workload_inputs(w))
        Bs = [B, B.clone(), B.clone()]

        def launch(i, stream):
            g.gemm_bf16gemm(w.M, w.N, w.K, w.alpha, A.data_ptr(), w.K, Bs[i % 3].data_ptr(),
                            w.N, w.beta, C.data_ptr(), w.N, stream)
        step = lambda i: launch(i, s)
        if args.only == "decode_graph":
            # `steps` launches captured once and replayed as one graph per step
            for i in range(3):
                step(i)
            torch.cuda.synchronize()
            graph = torch.cuda.CUDAGraph()
            cap = torch.cuda.Stream()
            with torch.cuda.stream(cap):
                graph.capture_begin()
                for i in range(args.steps):
                    launch(i, cap.cuda_stream)
                graph.capture_end()
            torch.cuda.synchronize()
            stream_obj = cap

            def step(i):
                with torch.cuda.stream(cap):   # replay() launches on the current stream
                    graph.replay()
    else:
        name = {"sgemm": "sgemm_4092", "sgemm4096": "sgemm_4096", "sgemm256": "sgemm_256",
                "ragged": "sgemm_ragged"}[args.only]
        w = wl.WORKLOADS[name]
        w2 = wl.Workload(**{**w.__dict__, "seed": w.seed + 100, "name": name + "_b"})
        sets = [tuple(t.to(device) for t in wl.workload_inputs(x)) for x in (w, w2)]
        step = sgemm_step_fn(g, sets, w, s)
    for i in range(args.warmup):
        step(i)
    ms = time_launches(torch, step, args.steps, stream_obj)
    if args.only == "decode_graph":     # each step replayed a graph of `steps` launches
        ms = [x / args.steps for x in ms]
    st = g.gemm_check_device_error(s)
    if st != 0:
        raise RuntimeError("device error: " + g.gemm_status_string(st))
    print(json.dumps({"only": args.only, "workload": w.name, "ms_per_launch": ms,
                      "gflops_median": w.flops / (statistics.median(ms) * 1e-3) / 1e9}),
          flush=True)


def main():
    args = parse_args()
    BRIEF["on"] = args.brief_parts
    if args.only:
        run_only(args)
        return
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
