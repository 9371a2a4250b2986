"""Offline launch-configuration sweep for the tile kernels (run on the GPU).

"A GEMM Kernel, Step by Step" ("Six parameters, found by search"): the best
tiling depends on the card and the shape, so it is searched for.  The tile
sizes, stages and warp layouts of this library are fixed per kernel at build
time (chosen by earlier sweeps); what varies per call is which kernel runs
(bf16: one CTA per 128 x 256 tile or a CTA pair per 256 x 256 tile), how the
last round's work items are cut along k, and the raster group height.  This
script times every such configuration on one representative shape per class
(class = ceil(log2) of M, N, K), keeps the configurations that beat the cost
model's own choice (gemm_get_model_config, not the table being replaced) by
a margin on a second timing that alternates the two, and writes

  * the table automatic dispatch reads (``csrc/dispatch_table.inc``; rebuild
    the library afterwards), and
  * a summary of every class (markdown).

Every candidate's result is compared with the cost model's configuration's
before it is timed; a configuration whose result differs beyond the GEMM's
error bound is reported and never enters the table.

    python -m dense_gemm_12_gb300.tune --table dense_gemm_12_gb300/csrc/dispatch_table.inc \\
        --summary sweep.md
"""
from __future__ import annotations

import argparse
import datetime
import itertools
import math
import os
import re
import statistics
import sys

# (bf16 shapes that automatic dispatch sends to the decode kernel -- M <= 32,
# and larger M with few column groups -- have no class: see main)
BF16_M = [256, 512, 1024, 2048, 4096, 8192]
BF16_NK = [256, 512, 1024, 2048, 4096, 8192]
FP32_M = [128, 256, 512, 1024, 2048, 4092]
FP32_NK = [256, 512, 1024, 2048, 4092, 8192]
# Every k-split up to 8: with the cluster fix-up (the CUDA-core kernel's
# 128-wide tiles, the single-CTA tcgen05 kernel) the largest split whose
# thread-block clusters all fit at once is often 5 or 7.
SPLITS = [1, 2, 3, 4, 5, 6, 7, 8]
GROUPS = [4, 8, 16]


def ceil_log2(x: int) -> int:
    b = 0
    while (1 << b) < x:
        b += 1
    return b


def bf16_stream_k_runs(kernel: str, M: int, N: int, K: int, num_sms: int) -> bool:
    """Whether a pinned stream-K tail really runs for this bf16 shape: the
    tail items' k-blocks must be at least the workers (CTAs, or about half as
    many CTA pairs); otherwise the library runs the equal split instead, the
    same launch as another candidate."""
    pair = kernel == "cta_pair"
    tiles_m, tiles_n = -(-M // 128), -(-N // 256)
    items = (-(-tiles_m // 2) if pair else tiles_m) * tiles_n
    workers = num_sms // 2 if pair else num_sms
    num_kb = -(-K // (128 if pair else 64))
    tail = items % workers if items >= workers else items
    return tail > 0 and tail * num_kb >= workers


def candidates(is_bf16: bool, M: int, N: int, K: int, num_sms: int = 152):
    """Every pinned configuration worth timing for a shape."""
    kernels = ["single_cta"] if is_bf16 else ["single_cta", "wide"]
    if is_bf16 and M > 128:
        kernels = ["cta_pair", "single_cta"]
    splits = SPLITS + [-1]   # -1: the stream-K tail
    num_kb = -(-K // (64 if is_bf16 else 32))
    for kernel, split, group in itertools.product(kernels, splits, GROUPS):
        if split > num_kb:
            continue
        if split == -1 and is_bf16 and not bf16_stream_k_runs(kernel, M, N, K, num_sms):
            continue
        yield {"kernel": kernel, "split": split, "group_m": group}


def table_lines(entries, num_sms: int, gpu: str, date: str):
    """Text of dispatch_table.inc for `entries` (dicts with is_bf16, M, N, K,
    kernel, split, group_m and the timings)."""
    kid = {"single_cta": 1, "cta_pair": 2, "wide": 3}
    out = [
        "// dispatch_table.inc -- launch configurations chosen by the offline sweep",
        "// (dense_gemm_12_gb300/tune.py) for the tile kernels, keyed by ceil(log2) of",
        "// M, N and K.  Written by that script; edit by re-running it.",
        "//",
        "// Measured on %s (%d SMs), %s.  Shapes whose class has no entry use" % (gpu, num_sms, date),
        "// the cost model.",
        "constexpr int kTunedSms = %d;" % num_sms,
        "constexpr TunedEntry kTuned[] = {",
        "    // {is_bf16, log2 M, log2 N, log2 K, kernel, split, group_m}",
    ]
    for e in sorted(entries, key=lambda e: (e["is_bf16"], e["M"], e["N"], e["K"])):
        out.append("    {%d, %d, %d, %d, %d, %d, %d},  // %dx%dx%d: %.4f ms, cost model %.4f ms" % (
            e["is_bf16"], ceil_log2(e["M"]), ceil_log2(e["N"]), ceil_log2(e["K"]),
            kid[e["kernel"]], e["split"], e["group_m"], e["M"], e["N"], e["K"],
            e["best_ms"], e["auto_ms"]))
    out.append("    {-1, 0, 0, 0, 0, 0, 0},  // end")
    out.append("};")
    return "\n".join(out) + "\n"


def choose(results, margin: float):
    """Table entries: shapes whose confirmed best configuration beats the cost
    model's configuration by more than `margin` (relative)."""
    return [r for r in results
            if r.get("best") is not None and r["best"] != r["auto"]
            and r["best_ms"] < r["auto_ms"] * (1.0 - margin)]


def _run(torch, g, is_bf16, M, N, K, tensors, cfg, stream):
    A, B, C = tensors
    fn = g.gemm_bf16gemm_config if is_bf16 else g.gemm_sgemm_config
    st = fn(M, N, K, 1.0, A.data_ptr(), K, B.data_ptr(), N, 0.0, C.data_ptr(), N, cfg,
            stream.cuda_stream)
    if st != 0:
        raise RuntimeError("%s: %s" % (cfg, g.gemm_status_string(st)))


def _time(torch, g, is_bf16, M, N, K, tensors, cfg, stream, reps):
    """Milliseconds per launch of `reps` launches queued back to back between two
    events (per-launch events would time the host's launch latency too on
    short kernels, and leave nothing for launches to overlap with)."""
    for _ in range(2):
        _run(torch, g, is_bf16, M, N, K, tensors, cfg, stream)
    torch.cuda.synchronize()
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(reps):
        _run(torch, g, is_bf16, M, N, K, tensors, cfg, stream)
    b.record(stream)
    torch.cuda.synchronize()
    return a.elapsed_time(b) / reps


def sweep_shape(torch, g, is_bf16, M, N, K, stream, reps=5, confirm_reps=20):
    dev = torch.device("cuda", torch.cuda.current_device())
    num_sms = torch.cuda.get_device_properties(dev).multi_processor_count
    gen = torch.Generator(device=dev).manual_seed(M * 131 + N * 17 + K)
    dt = torch.bfloat16 if is_bf16 else torch.float32
    A = torch.randn(M, K, device=dev, generator=gen).to(dt)
    B = (torch.randn(K, N, device=dev, generator=gen) * 0.05).to(dt)
    C = torch.empty(M, N, device=dev, dtype=torch.float32)
    tensors = (A, B, C)
    # the baseline is the cost model's own choice, pinned, so that the table
    # being replaced does not take part
    auto_cfg = g.gemm_get_model_config(is_bf16, M, N, K)
    _run(torch, g, is_bf16, M, N, K, tensors, auto_cfg, stream)
    torch.cuda.synchronize()
    ref = C.clone()
    # error scale of this GEMM: |A||B| per element bounds every order's error
    den = (A.float().abs() @ B.float().abs())
    tol = (8e-3 if is_bf16 else 2e-6 * math.sqrt(K)) * den
    timed, rejected = [], []
    for cfg in candidates(is_bf16, M, N, K, num_sms):
        _run(torch, g, is_bf16, M, N, K, tensors, cfg, stream)
        torch.cuda.synchronize()
        if not bool(((C - ref).abs() <= tol).all()):
            rejected.append(cfg)
            continue
        timed.append((_time(torch, g, is_bf16, M, N, K, tensors, cfg, stream, reps), cfg))
    timed.sort(key=lambda t: t[0])
    best = timed[0][1] if timed else None
    # confirm: model and best timed in turn, four times each
    a_ms, b_ms = [], []
    for _ in range(4):
        a_ms.append(_time(torch, g, is_bf16, M, N, K, tensors, auto_cfg, stream,
                          confirm_reps // 4))
        if best is not None:
            b_ms.append(_time(torch, g, is_bf16, M, N, K, tensors, best, stream,
                              confirm_reps // 4))
    auto_ms = statistics.median(a_ms)
    best_ms = statistics.median(b_ms) if b_ms else None
    del A, B, C, ref, den, tol
    torch.cuda.empty_cache()
    return {"is_bf16": int(is_bf16), "M": M, "N": N, "K": K, "auto": auto_cfg,
            "auto_ms": auto_ms, "best": best, "best_ms": best_ms,
            "kernel": best["kernel"] if best else None, "split": best["split"] if best else None,
            "group_m": best["group_m"] if best else None, "rejected": rejected,
            "candidates": len(timed)}


TABLE_ENTRY = re.compile(r"^\s*\{(\d+), (\d+), (\d+), (\d+), (\d+), (-?\d+), (\d+)\},\s*//\s*"
                         r"(\d+)x(\d+)x(\d+): ([\d.]+) ms, cost model ([\d.]+) ms")


def kept_entries(table_text: str, is_bf16: int):
    """Entries of one type in an existing table (what a sweep of the other
    type alone keeps), as table_lines takes them."""
    names = {1: "single_cta", 2: "cta_pair", 3: "wide"}
    out = []
    for line in table_text.splitlines():
        m = TABLE_ENTRY.match(line)
        if m is None or int(m.group(1)) != is_bf16:
            continue
        v = m.groups()
        out.append({"is_bf16": is_bf16, "M": int(v[7]), "N": int(v[8]), "K": int(v[9]),
                    "kernel": names[int(v[4])], "split": int(v[5]), "group_m": int(v[6]),
                    "best_ms": float(v[10]), "auto_ms": float(v[11])})
    return out


def kept_rows(summary_text: str, is_bf16: int):
    """Class rows of one type in an existing summary."""
    tag = "| bf16 |" if is_bf16 else "| fp32 |"
    return [line for line in summary_text.splitlines() if line.startswith(tag)]


def summary_lines(results, chosen, gpu, num_sms, command, kept=(), kept_after=()):
    """Markdown summary; `kept` / `kept_after`: class rows of the other type,
    kept from the previous summary, placed before / after the new rows."""
    flops = lambda r: 2.0 * r["M"] * r["N"] * r["K"]
    lines = ["# Launch-configuration sweep of the tile kernels", "",
             "Command (%s, %d SMs):" % (gpu, num_sms), "", "    " + command, "",
             "Per class (ceil(log2) of M, N, K), one representative shape; model = "
             "the cost model's choice without the table (split of the last round, -1 = "
             "stream-K; bf16 CTA pairs on large problems, single CTAs otherwise; fp32 tile width single_cta = "
             "128x128 or wide = 128x256; raster groups of 8); best = fastest pinned "
             "configuration; both re-timed in turn (4 x 5 back-to-back launches, median).  Entries "
             "marked `table` beat the model by more than the margin and were written "
             "to `csrc/dispatch_table.inc`.", "",
             "| type | M x N x K | model (kernel, split, group) | ms | TFLOP/s | best | ms "
             "| TFLOP/s | gain | |", "|---|---|---|---:|---:|---|---:|---:|---:|---|"]
    if kept or kept_after:
        lines[-2:-2] = ["Rows of the other type are kept from the previous sweep that wrote "
                        "this file (a sweep of one type, --only).", ""]
    lines += list(kept)
    chosen_keys = {(c["is_bf16"], c["M"], c["N"], c["K"]) for c in chosen}
    for r in results:
        a = r["auto"]
        b = r["best"] or {}
        gain = r["auto_ms"] / r["best_ms"] - 1.0 if r["best_ms"] else 0.0
        lines.append("| %s | %dx%dx%d | %s, %d, %d | %.4f | %.1f | %s, %s, %s | %.4f | %.1f | "
                     "%+.1f %% | %s |" % (
                         "bf16" if r["is_bf16"] else "fp32", r["M"], r["N"], r["K"],
                         a["kernel"], a["split"], a["group_m"], r["auto_ms"],
                         flops(r) / r["auto_ms"] / 1e9, b.get("kernel"), b.get("split"),
                         b.get("group_m"), r["best_ms"] or 0.0,
                         flops(r) / r["best_ms"] / 1e9 if r["best_ms"] else 0.0, 100 * gain,
                         "table" if (r["is_bf16"], r["M"], r["N"], r["K"]) in chosen_keys
                         else ""))
    lines += list(kept_after)
    bad = [(r, c) for r in results for c in r["rejected"]]
    lines += ["", "Configurations rejected by the result check: %d." % len(bad)]
    for r, c in bad:
        lines.append("- %dx%dx%d %s" % (r["M"], r["N"], r["K"], c))
    return "\n".join(lines) + "\n"


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--table", required=True, help="where to write dispatch_table.inc")
    ap.add_argument("--summary", required=True, help="where to write the markdown summary")
    ap.add_argument("--margin", type=float, default=0.03,
                    help="relative gain over automatic dispatch a table entry needs")
    ap.add_argument("--only", choices=["bf16", "fp32"], default=None)
    args = ap.parse_args(argv)

    import torch

    import dense_gemm_12_gb300 as g
    g.load_library(build_if_missing=True)
    dev = torch.cuda.current_device()
    props = torch.cuda.get_device_properties(dev)
    num_sms = props.multi_processor_count
    stream = torch.cuda.current_stream(dev)
    shapes = []
    if args.only in (None, "bf16"):
        shapes += [(True, M, N, K) for M in BF16_M for N in BF16_NK for K in BF16_NK]
    if args.only in (None, "fp32"):
        shapes += [(False, M, N, K) for M in FP32_M for N in FP32_NK for K in FP32_NK]
    # shapes automatic dispatch sends to the decode kernel (which plans itself
    # and never reads the table) have no class
    shapes = [s for s in shapes if not (s[0] and g.gemm_select_path(
        1, s[1], s[2], s[3], 1.0, 1 << 20, s[3], 1 << 20, s[2]) == "tc_decode")]
    results = []
    for is_bf16, M, N, K in shapes:
        r = sweep_shape(torch, g, is_bf16, M, N, K, stream)
        results.append(r)
        print("%s %dx%dx%d model %.4f best %s %.4f" % ("bf16" if is_bf16 else "fp32", M, N, K,
                                                     r["auto_ms"], r["best"], r["best_ms"] or 0),
              flush=True)
    st = g.gemm_check_device_error(stream.cuda_stream)
    if st != 0:
        raise RuntimeError("device error during the sweep: " + g.gemm_status_string(st))
    chosen = choose(results, args.margin)
    # a sweep of one type keeps the other type's entries and summary rows
    kept_table, kept_summary = [], []
    if args.only is not None:
        other = 0 if args.only == "bf16" else 1
        if os.path.exists(args.table):
            kept_table = kept_entries(open(args.table).read(), other)
        if os.path.exists(args.summary):
            kept_summary = kept_rows(open(args.summary).read(), other)
    date = datetime.date.today().isoformat()
    with open(args.table, "w") as f:
        f.write(table_lines(kept_table + chosen, num_sms, props.name, date))
    command = "python -m dense_gemm_12_gb300.tune " + " ".join(argv or sys.argv[1:])
    with open(args.summary, "w") as f:
        f.write(summary_lines(results, chosen, props.name, num_sms, command,
                              kept_summary if args.only == "fp32" else (),
                              kept_summary if args.only == "bf16" else ()))
    print("%d of %d classes written to the table" % (len(chosen), len(results)))


if __name__ == "__main__":
    main()
