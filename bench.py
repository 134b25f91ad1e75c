#!/usr/bin/env python
"""Benchmark of the GB300 TRSM library (L X = alpha B, left/lower/no-trans/
non-unit, in place of B).

Default workload ("square64"): m = n = 64, column-major, lda = ldb = 64,
alpha = 1, strided batch of 4096 systems in each of f32, f64, complex64 and
complex128 -- one step solves the four batches (four launches of the
small-regime kernel).  Metric: GFLOPS counted as m^2 n real flops per system
(x4 for complex), summed over the step.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl gb300|reference]
                    [--no-configs] [--nb-sweep] [--no-cpu-baseline]

With N > 1 (torchrun, one rank per GPU) every rank solves its own batches
(independent systems, no collective on the data path): weak scaling.

--impl reference times the CPU oracle (plain forward substitution, f64
accumulation, all host cores) on a bounded sample of the same workload.
By default the line also carries, under "configs", the rest of the metric:
the small-regime sweep at batch 16384 (m = n in {8..64} x four types, f32
m = 64 with n in {1, 6, 10, 32}; GB/s) and the large blocked solves (f32 /
complex64 m = n = 16384, f64 / complex128 m = n = 8192; GFLOPS against the
pipe their products run on), each with its roofline fraction and the oracle
timed on a sample (--no-configs skips them).
--nb-sweep times the blocked path for NB in {128, 256, 512} over m in
{1024, 2048, 4096, 8192, 16384} and the four types, and prints the table.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import trsm_inputs as ti  # noqa: E402

DTYPES = ("f32", "f64", "c64", "c128")
TORCH_NAME = {"f32": "float32", "f64": "float64", "c64": "complex64", "c128": "complex128"}
SQUARE = dict(m=64, n=64, batch=4096)
# the kernel that solves the square64 batch of each type, and its key in
# profiles/traffic.json
SQUARE_KERNEL = {"f32": "small_tma_f32_kernel<64, 2>", "f64": "small_fast_kernel<double, 64, 64, 1, 32, 1>",
                 "c64": "small_fast_kernel<float2, 64, 64, 1, 16, 2>",
                 "c128": "small_fast_kernel<double2, 64, 64, 1, 16, 1>"}
SQUARE_TRAFFIC_KEY = {"f32": "small_tma_f32_kernel", "f64": "small_fast_kernel<f64>",
                      "c64": "small_tma_c64_kernel", "c128": "small_fast_kernel<c128>"}
FLUSH_BYTES = 256 << 20          # > 129 MB L2, written between timed launches
FP64_PEAK_TFLOPS = 1.25          # nominal GB300 FP64 rate (DFMA and FP64 MMA alike); no measured figure
# nominal dense tensor rates of one GB300 (TFLOP/s): their ratio scales the
# measured bf16 GEMM rate to the TF32 rate the f32 / c64 products run at
NOMINAL_BF16_TFLOPS, NOMINAL_TF32_TFLOPS = 2250.0, 1100.0
SM_COUNT, FP32_LANES, SM_MAX_GHZ = 152, 128, 2.07


def fp32_alu_peak_tflops():
    """FFMA peak from unit counts and the maximum SM clock: 152 SMs x 128
    FP32 lanes x 2 flops x 2.07 GHz."""
    return SM_COUNT * FP32_LANES * 2 * SM_MAX_GHZ / 1e3


def tf32_peaks(peaks, src):
    """TF32 tensor rate: measured bf16 GEMM rate x the nominal TF32 / bf16
    ratio (1100 / 2250), burst and sustained; a 3xTF32 (f32-accurate)
    product costs three TF32 products, so its ceiling is a third of that."""
    ratio = NOMINAL_TF32_TFLOPS / NOMINAL_BF16_TFLOPS
    burst = peaks["bf16_tflops"] * ratio
    sustained = peaks.get("bf16_tflops_sustained", peaks["bf16_tflops"]) * ratio
    how = (f"bf16_tflops ({src}) x {NOMINAL_TF32_TFLOPS:.0f}/{NOMINAL_BF16_TFLOPS:.0f} (nominal TF32/bf16) "
           f"/ 3 (3xTF32 = three TF32 products)")
    return burst, sustained, how


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0}, "fallback"


# --------------------------------------------------------------------------- ranks
def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def init_dist(ws, backend):
    import torch.distributed as dist
    if ws > 1 and not dist.is_initialized():
        dist.init_process_group(backend=backend)
    return dist if ws > 1 else None


def reduce_max(dist, value, device=None):
    """Max of a float over ranks (identity on one rank)."""
    if dist is None:
        return value
    import torch
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(dist):
    if dist is not None:
        dist.barrier()


def weak_scaling_value(world_size, flops_per_rank_step, steps, max_rank_ms):
    """Whole-job GFLOPS: every rank solves its own batches (no exchange), so
    the work is world_size times one rank's, over the slowest rank's time."""
    return world_size * flops_per_rank_step * steps / (max_rank_ms * 1e-3) / 1e9


# --------------------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi clock / throttle-reason samples during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except (FileNotFoundError, OSError):
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.thread.join(timeout=2)

    def summary(self):
        if self.proc is None:
            return None
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(nm)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# --------------------------------------------------------------------------- helpers
def source_closure(tu):
    """A CUDA translation unit under csrc/ and every file it includes with
    quotes, transitively (resolved beside the including file, in csrc/ or in
    include/)."""
    import re
    csrc = os.path.join(ROOT, "triangular_solve_gb300", "csrc")
    inc = os.path.join(ROOT, "include")
    seen, stack = [], [os.path.join(csrc, tu)]
    while stack:
        p = os.path.normpath(stack.pop())
        if p in seen or not os.path.exists(p):
            continue
        seen.append(p)
        with open(p) as f:
            for line in f:
                mm = re.match(r'\s*#include\s+"([^"]+)"', line)
                if not mm:
                    continue
                for base in (os.path.dirname(p), csrc, inc):
                    q = os.path.join(base, mm.group(1))
                    if os.path.exists(q):
                        stack.append(q)
                        break
    return sorted(seen)


def kernel_source_hash(tu=None):
    """Hash of the sources a kernel is built from (its translation unit's
    include closure; all CUDA sources when none is named): ncu traffic
    figures are only valid for the kernels they were captured on."""
    h = hashlib.sha256()
    if tu is None:
        csrc = os.path.join(ROOT, "triangular_solve_gb300", "csrc")
        files = [os.path.join(csrc, n) for n in sorted(os.listdir(csrc)) if n.endswith((".cu", ".cuh", ".h"))]
        for p in files:
            with open(p, "rb") as f:
                h.update(os.path.basename(p).encode())
                h.update(f.read())
        return h.hexdigest()[:16]
    for p in source_closure(tu):
        with open(p, "rb") as f:
            h.update(os.path.relpath(p, ROOT).encode())
            h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic(kernel_key):
    """dram bytes per launch from the committed ncu summary, or None when the
    kernel's sources changed since the capture."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    e = d.get(kernel_key)
    if not e or e.get("source_hash") != kernel_source_hash(e.get("translation_unit")):
        return None
    return e.get("dram_bytes_per_launch")


def make_square_inputs(dtype, m, n, batch):
    L, B = ti.generate(dtype, m, n, batch, kind="dd64")
    return ti.to_storage(L, "col"), ti.to_storage(B, "col")


# --------------------------------------------------------------------------- gb300 arm
def run_gb300(args, ws, rank, local):
    import torch

    import triangular_solve_gb300 as tg
    from triangular_solve_gb300 import build as tgb
    torch.cuda.set_device(local)
    dist = init_dist(ws, "nccl")
    dev = torch.device("cuda", local)
    if rank == 0:
        tgb.build()
    barrier(dist)
    tg.load_library()
    m, n, batch = SQUARE["m"], SQUARE["n"], SQUARE["batch"]
    stream = torch.cuda.current_stream()

    bufs = {}
    for d in DTYPES:
        a_np, b_np = make_square_inputs(d, m, n, batch)
        bufs[d] = dict(
            a=torch.from_numpy(a_np).to(dev),
            b0=torch.from_numpy(b_np).to(dev),
            b=torch.empty(b_np.shape, dtype=getattr(torch, TORCH_NAME[d]), device=dev),
            a_host=torch.from_numpy(a_np).pin_memory(),
            b_host=torch.from_numpy(b_np).pin_memory(),
            io_host=torch.from_numpy(b_np).pin_memory(),  # B in, X out of the host entry point
        )
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)

    def solve(d):
        bb = bufs[d]
        tg.trsm_llnn_strided_batched(d, "col", m, n, 1.0, bb["a"], m, m * m, bb["b"], m, m * n, batch,
                                     stream)

    def step(evs=None):
        for i, d in enumerate(DTYPES):
            bufs[d]["b"].copy_(bufs[d]["b0"])
            flush.fill_(i + 1)
            if evs is not None:
                evs[i][0].record(stream)
            solve(d)
            if evs is not None:
                evs[i][1].record(stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()

    events = [[[torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)]
               for _ in DTYPES] for _ in range(args.steps)]
    barrier(dist)
    torch.cuda.synchronize()
    with ClockSampler(local) as clocks:
        t0 = time.perf_counter()
        for s in range(args.steps):
            step(events[s])
        torch.cuda.synchronize()
        wall = time.perf_counter() - t0
    barrier(dist)
    per_dtype_ms = {d: [events[s][i][0].elapsed_time(events[s][i][1]) for s in range(args.steps)]
                    for i, d in enumerate(DTYPES)}
    kernel_ms_total = sum(sum(v) for v in per_dtype_ms.values())
    kernel_ms_max = reduce_max(dist, kernel_ms_total, dev)
    step_flops = sum(ti.flops(d, m, n, batch) for d in DTYPES)
    value = weak_scaling_value(ws, step_flops, args.steps, kernel_ms_max)

    # end to end through the public API: the C-ABI entry point on host
    # buffers (pinned), its copies in both directions inside the timed region
    # (it pipelines them against the solves of other chunks)
    h2d = sum(bufs[d]["a_host"].numel() * bufs[d]["a_host"].element_size()
              + bufs[d]["io_host"].numel() * bufs[d]["io_host"].element_size() for d in DTYPES)
    d2h = sum(bufs[d]["io_host"].numel() * bufs[d]["io_host"].element_size() for d in DTYPES)

    # the four types are independent batches: one stream each, as a caller
    # with independent problems would issue them
    e2e_streams = {d: torch.cuda.Stream() for d in DTYPES}

    def e2e_step():
        for d in DTYPES:
            bb = bufs[d]
            tg.trsm_llnn_strided_batched_host(d, "col", m, n, 1.0, bb["a_host"], m, m * m, bb["io_host"], m,
                                              m * n, batch, e2e_streams[d])
        torch.cuda.synchronize()

    e2e_steps = max(3, min(args.steps, 20))
    for _ in range(2):
        e2e_step()
    barrier(dist)
    t0 = time.perf_counter()
    for _ in range(e2e_steps):
        e2e_step()
    e2e_wall = reduce_max(dist, time.perf_counter() - t0, dev)
    barrier(dist)
    e2e_value = ws * step_flops * e2e_steps / e2e_wall / 1e9
    # the host path gives the device path's X on the same inputs (chunks of the
    # batch may take a different kernel, so up to rounding)
    for d in DTYPES:
        bufs[d]["io_host"].copy_(bufs[d]["b_host"])
    e2e_step()
    for d in DTYPES:
        tol = 1e-5 if d in ("f32", "c64") else 1e-12
        if not torch.allclose(bufs[d]["io_host"], bufs[d]["b"].cpu(), rtol=tol, atol=tol):
            raise RuntimeError(f"host entry point and device entry point differ for {d}")

    detail = {}
    for d in DTYPES:
        ms = statistics.mean(per_dtype_ms[d])
        detail[d] = {
            "ms_per_launch": round(ms, 5),
            "gflops": round(ti.flops(d, m, n, batch) / (ms * 1e-3) / 1e9, 2),
            "gbs": round(ti.algorithmic_bytes(d, m, n, batch) / (ms * 1e-3) / 1e9, 1),
        }
    # batch-1 latency (one system per launch), the pages' small-regime figure
    for d in DTYPES:
        a1, b1 = bufs[d]["a"][: m * m], bufs[d]["b"][: m * n]
        for _ in range(5):
            tg.trsm_llnn(d, m, n, 1.0, a1, m, b1, m, stream)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        reps = 200
        for _ in range(reps):
            tg.trsm_llnn(d, m, n, 1.0, a1, m, b1, m, stream)
        e1.record(stream)
        torch.cuda.synchronize()
        us = e0.elapsed_time(e1) * 1e3 / reps
        detail[d]["batch1_us"] = round(us, 2)
        detail[d]["batch1_gflops"] = round(ti.flops(d, m, n, 1) / (us * 1e-6) / 1e9, 2)

    peaks, peak_src = measured_peaks()
    dom = max(DTYPES, key=lambda d: statistics.mean(per_dtype_ms[d]))
    dom_ms = statistics.mean(per_dtype_ms[dom])
    if dom in ("f64", "c128"):
        roof = {"bound": "alu", "achieved": ti.flops(dom, m, n, batch) / (dom_ms * 1e-3) / 1e12,
                "peak": FP64_PEAK_TFLOPS, "unit": "TFLOP/s",
                "peak_source": "nominal GB300 FP64 rate (recipe table)"}
    else:
        roof = {"bound": "hbm", "achieved": ti.algorithmic_bytes(dom, m, n, batch) / (dom_ms * 1e-3) / 1e9,
                "peak": peaks["hbm_gbs"], "unit": "GB/s", "peak_source": f"hbm_gbs ({peak_src})"}
    roof["frac"] = roof["achieved"] / roof["peak"]
    roof["kernel"] = f"{SQUARE_KERNEL[dom]} (square64, batch 4096)"
    roof["algorithmic_per_launch"] = (ti.flops(dom, m, n, batch) if roof["bound"] == "alu"
                                      else ti.algorithmic_bytes(dom, m, n, batch))
    roof["traffic"] = recorded_traffic(f"{SQUARE_TRAFFIC_KEY[dom]}/square64x4096")
    roof["achieved"] = round(roof["achieved"], 3)
    roof["frac"] = round(roof["frac"], 4)

    out = {
        "metric": "TRSM GFLOPS (m^2 n real flops, x4 complex), m=n=64 strided batch 4096, "
                  "f32+f64+c64+c128 per step",
        "value": round(value, 2), "unit": "GFLOPS", "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(kernel_ms_max / args.steps, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32+f64+c64+c128",
        "data": "synthetic (seeded: L strictly lower U(-1,1)/64, diag 1+U(0,1); B U(-1,1))",
        "config": {"workload": "square64: m=n=64 column-major lda=ldb=64 alpha=1, strided batch 4096 "
                               "per type, one launch per type", "m": m, "n": n, "batch_per_gpu": batch,
                   "l2": "flushed (256 MB write) before every timed launch; B restored from a pristine copy",
                   "parallelism": f"independent batches per GPU x{ws}"},
        "e2e": {"value": round(e2e_value, 2), "unit": "GFLOPS", "h2d_bytes_per_step": int(h2d),
                "d2h_bytes_per_step": int(d2h)},
        "gpu_launches": len(DTYPES) * args.steps,
        "roofline": roof,
        "clocks": clocks.summary(),
        "wall_s_timed_region": round(wall, 4),
        "detail": detail,
    }
    if rank == 0 and not args.no_configs:
        # the rest of the metric: the batch-16384 small sweep (GB/s) and the
        # large blocked solves, each with its roofline and oracle baseline
        out["configs"] = {
            "small_sweep_b16384": config_small_sweep(torch, tg, dev, stream, flush, peaks, peak_src),
            "large_blocked": config_large(torch, tg, dev, stream, peaks, peak_src),
        }
    if rank == 0 and not args.no_cpu_baseline:
        out["cpu_baseline"] = cpu_baseline(seconds=args.cpu_seconds)
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(out), flush=True)


def _events(torch):
    return torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)


def fp32_roof(d):
    """Arithmetic ceiling (TFLOP/s) of a small-regime type and its source."""
    if d in ("f64", "c128"):
        return FP64_PEAK_TFLOPS, "nominal GB300 FP64 rate (recipe table)"
    return fp32_alu_peak_tflops(), "FP32 FMA: 152 SMs x 128 lanes x 2 flops x 2.07 GHz (unit counts, max clock)"


def config_small_sweep(torch, tg, dev, stream, flush, peaks, peak_src, reps=5, sample=1024):
    """The small-regime sweep: m = n in {8, 16, 32, 48, 64} x four types and
    f32 m = 64 with n in {1, 6, 10, 32}, strided batch 16384 (column-major,
    lda = ldb = m, L strictly lower U(-1,1)/64, diagonal 1 + U(0,1), B
    U(-1,1), alpha = 1).  Per point: CUDA-event time of one launch (L2
    flushed and B restored before each), GB/s of the algorithmic bytes,
    GFLOPS, the roofline time max(bytes / HBM, flops / pipe) over the measured
    time, and the oracle on a sample of the same batch."""
    import oracle
    batch = 16384
    points = [(d, mm, mm) for d in DTYPES for mm in (8, 16, 32, 48, 64)]
    points += [("f32", 64, nn) for nn in (1, 6, 10, 32) if "f32" in DTYPES]
    res = {}
    for d, mm, nn in points:
        L, B = ti.generate(d, mm, nn, batch, kind="dd64")
        a = torch.from_numpy(ti.to_storage(L, "col")).to(dev)
        b0 = torch.from_numpy(ti.to_storage(B, "col")).to(dev)
        b = torch.empty_like(b0)

        def launch():
            tg.trsm_llnn_strided_batched(d, "col", mm, nn, 1.0, a, mm, mm * mm, b, mm, mm * nn, batch, stream)

        for _ in range(2):
            b.copy_(b0)
            launch()
        times = []
        for _ in range(reps):
            b.copy_(b0)
            flush.fill_(len(times) + 1)
            e0, e1 = _events(torch)
            e0.record(stream)
            launch()
            e1.record(stream)
            torch.cuda.synchronize()
            times.append(e0.elapsed_time(e1))
        ms = statistics.mean(times)
        q, f = ti.algorithmic_bytes(d, mm, nn, batch), ti.flops(d, mm, nn, batch)
        p_tf, p_src = fp32_roof(d)
        t_hbm = q / (peaks["hbm_gbs"] * 1e9) * 1e3
        t_alu = f / (p_tf * 1e12) * 1e3
        if t_hbm >= t_alu:
            roof = {"bound": "hbm", "achieved": round(q / (ms * 1e-3) / 1e9, 1), "peak": peaks["hbm_gbs"],
                    "unit": "GB/s", "peak_source": f"hbm_gbs ({peak_src})"}
        else:
            roof = {"bound": "alu", "achieved": round(f / (ms * 1e-3) / 1e12, 3), "peak": round(p_tf, 2),
                    "unit": "TFLOP/s", "peak_source": p_src}
        roof["frac"] = round(max(t_hbm, t_alu) / ms, 4)
        # the oracle on the first `sample` systems of the batch
        a_h = ti.to_storage(L[:sample], "col")
        b_h = ti.to_storage(B[:sample], "col")
        t0 = time.perf_counter()
        oracle.trsm_llnn(d, mm, nn, 1.0, a_h, mm, b_h, mm, stride_a=mm * mm, stride_b=mm * nn, batch=sample)
        el = time.perf_counter() - t0
        res[f"{d}_m{mm}_n{nn}"] = {
            "dtype": d, "m": mm, "n": nn, "batch": batch, "ms": round(ms, 5),
            "gbs": round(q / (ms * 1e-3) / 1e9, 1), "gflops": round(f / (ms * 1e-3) / 1e9, 1),
            "roofline": roof,
            "cpu_baseline": {"value": round(ti.flops(d, mm, nn, sample) / el / 1e9, 3), "unit": "GFLOPS",
                             "cores": oracle.max_threads(), "kind": "oracle",
                             "sample": f"{sample} of the {batch} systems, {el * 1e3:.1f} ms"},
        }
        del a, b0, b, L, B
    torch.cuda.empty_cache()
    return res


def config_large(torch, tg, dev, stream, peaks, peak_src, which=None, reps=2):
    """The blocked path on the large workloads, table NB: f32 and complex64
    at m = n = 16384 (alpha = 1), f64 and complex128 at m = n = 8192
    (alpha = 1.5); L strictly lower U(-1,1)/m, diagonal 1 + U(0,1), B U(-1,1),
    column-major.  Per workload: CUDA-event time of one solve (after a
    warm-up solve), GFLOPS (m^3, x4 complex), the fraction of the pipe the
    products run on, the inversion / apply / update split, and the oracle on
    64 sampled right-hand-side columns -- timed (the CPU baseline) and
    compared with the GPU's X on those columns."""
    import oracle
    tf_burst, tf_sus, tf_how = tf32_peaks(peaks, peak_src)
    res = {}
    work = [("f32", 16384, 1.0), ("c64", 16384, 1.0), ("f64", 8192, 1.5), ("c128", 8192, 1.5)]
    for d, mm, alpha in work:
        if d not in DTYPES or (which and d not in which):
            continue
        L, B = ti.generate(d, mm, mm, 1, kind="ddm")
        # the logical (row-major) arrays are the column-major storage of the
        # transposes; transposing on the device gives column-major L and B
        a = torch.from_numpy(L[0]).to(dev).t().contiguous().t()
        b0 = torch.from_numpy(B[0]).to(dev).t().contiguous().t()
        cols = ti.sample_columns(mm)
        b = torch.empty_like(b0)
        nb = tg.trsm_llnn_select_nb(d, mm, mm)
        wsb = tg.trsm_llnn_workspace_bytes(d, mm, mm, nb)
        wsp = torch.empty(wsb, dtype=torch.uint8, device=dev)
        b.copy_(b0)
        tg.trsm_llnn_ex(d, mm, mm, alpha, a, mm, b, mm, nb, wsp, wsb, stream)  # warm-up
        times = []
        for _ in range(reps):
            b.copy_(b0)
            e0, e1 = _events(torch)
            e0.record(stream)
            tg.trsm_llnn_ex(d, mm, mm, alpha, a, mm, b, mm, nb, wsp, wsb, stream)
            e1.record(stream)
            torch.cuda.synchronize()
            times.append(e0.elapsed_time(e1))
        x_cols = b[:, torch.from_numpy(cols).to(dev)].cpu().numpy()
        b.copy_(b0)
        phases = tg.trsm_llnn_profile(d, mm, mm, alpha, a, mm, b, mm, nb, wsp, wsb, stream)
        del a, b0, b, wsp
        torch.cuda.empty_cache()
        # the oracle on the sampled columns (row-major storage of the same values)
        bs = np.ascontiguousarray(B[0][:, cols])
        t0 = time.perf_counter()
        oracle.trsm_llnn(d, mm, len(cols), alpha, L[0], mm, bs, len(cols), layout="row")
        el = time.perf_counter() - t0
        t = np.complex128 if ti.IS_COMPLEX[d] else np.float64
        err = float(np.linalg.norm((x_cols.astype(t) - bs.astype(t)).ravel()) / np.linalg.norm(bs.astype(t).ravel()))
        tol = 1e-5 if d in ("f32", "c64") else 1e-12
        del L, B
        ms = statistics.mean(times)
        fl = ti.flops(d, mm, mm)
        tfs = fl / (ms * 1e-3) / 1e12
        tot = sum(phases) or 1.0
        if d in ("f64", "c128"):
            roof = {"bound": "alu", "achieved": round(tfs, 3), "peak": FP64_PEAK_TFLOPS, "unit": "TFLOP/s",
                    "frac": round(tfs / FP64_PEAK_TFLOPS, 4), "pipe": "FP64 (DFMA)",
                    "peak_source": "nominal GB300 FP64 rate (recipe table); no measured FP64 peak"}
        else:
            roof = {"bound": "tensor", "achieved": round(tfs, 2), "peak": round(tf_burst / 3, 1),
                    "unit": "TFLOP/s", "frac": round(tfs / (tf_burst / 3), 4),
                    "frac_of_sustained": round(tfs / (tf_sus / 3), 4),
                    "pipe": "tensor (tcgen05 kind::tf32, 3xTF32 split)", "peak_source": tf_how,
                    "frac_of_fp32_fma_peak": round(tfs / fp32_alu_peak_tflops(), 3)}
        res[f"{d}_m{mm}"] = {
            "dtype": d, "m": mm, "n": mm, "alpha": alpha, "nb": nb, "ms": round(ms, 3),
            "gflops": round(fl / (ms * 1e-3) / 1e9, 1), "roofline": roof,
            "phase_share": {"diag_inversion": round(phases[0] / tot, 4), "block_apply": round(phases[1] / tot, 4),
                            "gemm_update": round(phases[2] / tot, 4)},
            "parity": {"rel_fro_sampled_cols": err, "tol": tol, "ok": bool(err <= tol),
                       "columns": "default_rng(1).choice(n, 64, replace=False), sorted"},
            "cpu_baseline": {"value": round(ti.flops(d, mm, len(cols)) / el / 1e9, 3), "unit": "GFLOPS",
                             "cores": oracle.max_threads(), "kind": "oracle",
                             "sample": f"the 64 sampled right-hand-side columns of this system, {el:.1f} s"},
        }
    return res


def variants_bench(args):
    """One JSON line per (type, m, variant): trsm_general on a square system
    (m = n; side, triangle, op, diagonal as in BLAS), CUDA events on the
    launching stream, inputs resident, B restored before every run; GFLOPS
    credit m^2 n (x4 complex) and `vs_llnn` is the native left-lower time
    over this variant's (the mapped variants add the copies of A and B)."""
    import itertools

    import torch

    import triangular_solve_gb300 as tg
    from triangular_solve_gb300 import build as tgb
    tgb.build()
    dev = torch.device("cuda", 0)
    stream = torch.cuda.current_stream()
    for d in args.sweep_dtypes.split(","):
        for mm in [int(x) for x in args.sweep_ms.split(",")]:
            rng = np.random.default_rng(0)
            cplx = d in ("c64", "c128")

            def u(shape):
                x = rng.uniform(-1, 1, shape)
                return x + 1j * rng.uniform(-1, 1, shape) if cplx else x

            A = u((mm, mm)) / mm
            A[np.diag_indices(mm)] = 1 + rng.uniform(0, 1, mm)
            a = torch.from_numpy(ti.to_storage(A.astype(ti.NUMPY[d])[None], "col")).to(dev)
            b0 = torch.from_numpy(ti.to_storage(u((mm, mm)).astype(ti.NUMPY[d])[None], "col")).to(dev)
            del A
            b = torch.empty_like(b0)
            base = None
            for v in ["LLNN"] + ["".join(x) for x in itertools.product("LR", "LU", "NTC", "NU")
                                 if "".join(x) != "LLNN"]:
                b.copy_(b0)
                tg.trsm_general(d, v[0], v[1], v[2], v[3], mm, mm, 1.0, a, mm, b, mm, stream)  # warm-up
                times = []
                for _ in range(max(args.sweep_reps, 1)):
                    b.copy_(b0)
                    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                    e0.record(stream)
                    tg.trsm_general(d, v[0], v[1], v[2], v[3], mm, mm, 1.0, a, mm, b, mm, stream)
                    e1.record(stream)
                    torch.cuda.synchronize()
                    times.append(e0.elapsed_time(e1))
                ms = statistics.mean(times)
                base = ms if base is None else base
                print(json.dumps({"op": "trsm_general", "dtype": d, "m": mm, "n": mm, "variant": v,
                                  "ms": round(ms, 3), "gflops": round(ti.flops(d, mm, mm) / (ms * 1e-3) / 1e9, 1),
                                  "vs_llnn": round(base / ms, 3)}), flush=True)
            del a, b0, b
            torch.cuda.empty_cache()


def medium_bench(args):
    """One JSON line per (type, m): a strided batch of --batch systems of
    order m (n = m, column-major, contiguous, L strictly lower U(-1,1)/m,
    diagonal 1 + U(0,1), B U(-1,1), alpha = 1) through
    trsm_llnn_strided_batched; CUDA events on the launching stream after a
    warm-up call, inputs resident, B restored before every run; GFLOPS credit
    m^2 n per system (x4 complex)."""
    import torch

    import triangular_solve_gb300 as tg
    from triangular_solve_gb300 import build as tgb
    tgb.build()
    dev = torch.device("cuda", 0)
    stream = torch.cuda.current_stream()
    batch = args.batch
    for d in args.sweep_dtypes.split(","):
        for mm in [int(x) for x in args.sweep_ms.split(",")]:
            L, B = ti.generate(d, mm, mm, batch, kind="ddm")
            a = torch.from_numpy(ti.to_storage(L, "col")).to(dev)
            b0 = torch.from_numpy(ti.to_storage(B, "col")).to(dev)
            del L, B
            b = b0.clone()
            tg.trsm_llnn_strided_batched(d, "col", mm, mm, 1.0, a, mm, mm * mm, b, mm, mm * mm, batch, stream)
            times = []
            for _ in range(max(args.sweep_reps, 1)):
                b.copy_(b0)
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                tg.trsm_llnn_strided_batched(d, "col", mm, mm, 1.0, a, mm, mm * mm, b, mm, mm * mm, batch, stream)
                e1.record(stream)
                torch.cuda.synchronize()
                times.append(e0.elapsed_time(e1))
            ms = statistics.mean(times)
            print(json.dumps({"op": "strided_batched", "dtype": d, "m": mm, "n": mm, "batch": batch,
                              "ms": round(ms, 4),
                              "gflops": round(ti.flops(d, mm, mm, batch) / (ms * 1e-3) / 1e9, 1),
                              "gbs": round(ti.algorithmic_bytes(d, mm, mm, batch) / (ms * 1e-3) / 1e9, 1)}),
                  flush=True)
            del a, b0, b
            torch.cuda.empty_cache()


def few_rhs_bench(args):
    """One JSON line per (type, m, n) for few right-hand sides, n in
    --few-ns: one system of order m (column-major, L strictly lower
    U(-1,1)/m, diagonal 1 + U(0,1), B U(-1,1), alpha = 1; generated on the
    device: timing only) through trsm_llnn_ex with the table's block size;
    CUDA events after a warm-up solve, B restored before every run; GB/s
    counts the algorithmic bytes (L's lower triangle once, B read, X written),
    beside the phase split of trsm_llnn_profile."""
    import torch

    import triangular_solve_gb300 as tg
    from triangular_solve_gb300 import build as tgb
    tgb.build()
    dev = torch.device("cuda", 0)
    stream = torch.cuda.current_stream()
    for d in args.sweep_dtypes.split(","):
        t = getattr(torch, TORCH_NAME[d])
        real_t = torch.float32 if d in ("f32", "c64") else torch.float64
        for mm in [int(x) for x in args.sweep_ms.split(",")]:
            g = torch.Generator(device=dev).manual_seed(0)
            lv = (torch.rand((mm, mm), generator=g, device=dev, dtype=real_t) * 2 - 1) / mm
            lv.diagonal().copy_(1 + torch.rand(mm, generator=g, device=dev, dtype=real_t))
            a = lv.to(t).t().contiguous().t()
            del lv
            for nn in [int(x) for x in args.few_ns.split(",")]:
                b0 = (torch.rand((mm, nn), generator=g, device=dev, dtype=real_t) * 2 - 1).to(t).t().contiguous().t()
                b = b0.clone()
                wsb = tg.trsm_llnn_workspace_bytes(d, mm, nn, 0)
                wsp = torch.empty(max(wsb, 1), dtype=torch.uint8, device=dev)
                tg.trsm_llnn_ex(d, mm, nn, 1.0, a, mm, b, mm, 0, wsp, wsb, stream)
                times = []
                for _ in range(max(args.sweep_reps, 1)):
                    b.copy_(b0)
                    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                    e0.record(stream)
                    tg.trsm_llnn_ex(d, mm, nn, 1.0, a, mm, b, mm, 0, wsp, wsb, stream)
                    e1.record(stream)
                    torch.cuda.synchronize()
                    times.append(e0.elapsed_time(e1))
                b.copy_(b0)
                ph = tg.trsm_llnn_profile(d, mm, nn, 1.0, a, mm, b, mm, 0, wsp, wsb, stream)
                ms = statistics.mean(times)
                print(json.dumps({"op": "few_rhs", "dtype": d, "m": mm, "n": nn, "ms": round(ms, 4),
                                  "gbs": round(ti.algorithmic_bytes(d, mm, nn) / (ms * 1e-3) / 1e9, 1),
                                  "gflops": round(ti.flops(d, mm, nn) / (ms * 1e-3) / 1e9, 1),
                                  "phases_ms": [round(x, 4) for x in ph],
                                  "device_status": tg.trsm_device_status()}), flush=True)
                del b0, b, wsp
            del a
            torch.cuda.empty_cache()


def trtri_bench(args):
    """One JSON line per (type, m): the triangular inverse L^-1 through
    trsm_trtri_lower (set to I, then the L X = I solve), CUDA events on the
    launching stream, inputs resident; GFLOPS credit TRTRI's m^3/3 real flops
    (x4 complex) and, beside it, the m^3 of the solve it runs."""
    import torch

    import triangular_solve_gb300 as tg
    from triangular_solve_gb300 import build as tgb
    tgb.build()
    dev = torch.device("cuda", 0)
    stream = torch.cuda.current_stream()
    for d in args.sweep_dtypes.split(","):
        for mm in [int(x) for x in args.sweep_ms.split(",")]:
            L, _ = ti.generate(d, mm, 1, 1, kind="ddm")
            a = torch.from_numpy(ti.to_storage(L, "col")).to(dev)
            del L
            x = torch.empty_like(a)
            tg.trsm_trtri_lower(d, mm, a, mm, x, mm, stream)  # warm-up (and workspace pool)
            times = []
            for _ in range(max(args.sweep_reps, 1)):
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                tg.trsm_trtri_lower(d, mm, a, mm, x, mm, stream)
                e1.record(stream)
                torch.cuda.synchronize()
                times.append(e0.elapsed_time(e1))
            ms = statistics.mean(times)
            cplx = 4 if d in ("c64", "c128") else 1
            print(json.dumps({"op": "trtri", "dtype": d, "m": mm, "ms": round(ms, 3),
                              "gflops_trtri": round(cplx * mm ** 3 / 3 / (ms * 1e-3) / 1e9, 1),
                              "gflops_solve": round(cplx * mm ** 3 / (ms * 1e-3) / 1e9, 1)}), flush=True)
            del a, x
            torch.cuda.empty_cache()


def nb_sweep(args):
    import torch

    import triangular_solve_gb300 as tg
    from triangular_solve_gb300 import build as tgb
    tgb.build()
    dev = torch.device("cuda", 0)
    stream = torch.cuda.current_stream()
    rows = []
    for d in args.sweep_dtypes.split(","):
        for mm in [int(x) for x in args.sweep_ms.split(",")]:
            g = torch.Generator(device=dev).manual_seed(0)
            t = getattr(torch, TORCH_NAME[d])
            real_t = torch.float32 if d in ("f32", "c64") else torch.float64
            # device-side synthetic inputs of the same distribution (timing only)
            shape = (mm, mm)
            if d in ("c64", "c128"):
                lv = torch.complex(torch.rand(shape, generator=g, device=dev, dtype=real_t),
                                   torch.rand(shape, generator=g, device=dev, dtype=real_t))
                bv = torch.complex(torch.rand(shape, generator=g, device=dev, dtype=real_t),
                                   torch.rand(shape, generator=g, device=dev, dtype=real_t)) * 2 - (1 + 1j)
            else:
                lv = torch.rand(shape, generator=g, device=dev, dtype=real_t)
                bv = torch.rand(shape, generator=g, device=dev, dtype=real_t) * 2 - 1
            lv = (lv * 2 - 1) / mm
            lv.diagonal().copy_(1 + torch.rand(mm, generator=g, device=dev, dtype=real_t))
            a = lv.to(t).t().contiguous().t()  # column-major
            b0 = bv.to(t).t().contiguous().t()
            del lv, bv
            best = None
            for nb in [int(x) for x in args.sweep_nbs.split(",")]:
                wsb = tg.trsm_llnn_workspace_bytes(d, mm, mm, nb)
                wsp = torch.empty(wsb, dtype=torch.uint8, device=dev)
                b = b0.clone()
                tg.trsm_llnn_ex(d, mm, mm, 1.0, a, mm, b, mm, nb, wsp, wsb, stream)
                ts = []
                for _ in range(args.sweep_reps):
                    b.copy_(b0)
                    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                    e0.record(stream)
                    tg.trsm_llnn_ex(d, mm, mm, 1.0, a, mm, b, mm, nb, wsp, wsb, stream)
                    e1.record(stream)
                    torch.cuda.synchronize()
                    ts.append(e0.elapsed_time(e1))
                ms = statistics.mean(ts)
                gf = ti.flops(d, mm, mm) / (ms * 1e-3) / 1e9
                b.copy_(b0)
                ph = tg.trsm_llnn_profile(d, mm, mm, 1.0, a, mm, b, mm, nb, wsp, wsb, stream)
                tot = sum(ph) or 1.0
                rows.append({"dtype": d, "m": mm, "nb": nb, "ms": round(ms, 3), "gflops": round(gf, 1),
                             "phase_share": [round(v / tot, 4) for v in ph]})
                print(json.dumps(rows[-1]), flush=True)
                if best is None or gf > best[1]:
                    best = (nb, gf)
                del wsp, b
            rows.append({"dtype": d, "m": mm, "best_nb": best[0]})
            print(json.dumps(rows[-1]), flush=True)
            del a, b0
            torch.cuda.empty_cache()
    return rows


# --------------------------------------------------------------------------- oracle arm
def cpu_baseline(seconds=15.0):
    """The oracle, as it stands, on the host cores: square64 systems of the
    four types, a bounded sample of each batch, repeated for ~`seconds`."""
    import oracle
    oracle.build()
    m, n = SQUARE["m"], SQUARE["n"]
    sample = 512
    data = {}
    for d in DTYPES:
        a, b = make_square_inputs(d, m, n, SQUARE["batch"])
        data[d] = (a[: sample * m * m].copy(), b[: sample * m * n].copy())
    flops_rep = sum(ti.flops(d, m, n, sample) for d in DTYPES)

    def rep():
        for d in DTYPES:
            a, b = data[d]
            bb = b.copy()
            oracle.trsm_llnn(d, m, n, 1.0, a, m, bb, m, stride_a=m * m, stride_b=m * n, batch=sample)

    rep()
    t0 = time.perf_counter()
    reps = 0
    while True:
        rep()
        reps += 1
        if time.perf_counter() - t0 >= seconds:
            break
    el = time.perf_counter() - t0
    return {"value": round(flops_rep * reps / el / 1e9, 3), "unit": "GFLOPS", "cores": oracle.max_threads(),
            "kind": "oracle",
            "sample": f"{sample} of the 4096 systems per type (m=n=64, four types), x{reps} repetitions, "
                      f"{el:.1f} s"}


def run_reference(args, ws, rank):
    if rank != 0:
        return
    import oracle
    oracle.build()
    m, n = SQUARE["m"], SQUARE["n"]
    sample = 256
    data = {}
    for d in DTYPES:
        a, b = make_square_inputs(d, m, n, SQUARE["batch"])
        data[d] = (a[: sample * m * m].copy(), b[: sample * m * n].copy())

    def step():
        for d in DTYPES:
            a, b = data[d]
            bb = b.copy()
            oracle.trsm_llnn(d, m, n, 1.0, a, m, bb, m, stride_a=m * m, stride_b=m * n, batch=sample)

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    el = time.perf_counter() - t0
    step_flops = sum(ti.flops(d, m, n, sample) for d in DTYPES)
    value = step_flops * args.steps / el / 1e9
    cores = oracle.max_threads()
    sample_txt = f"{sample} of the 4096 systems per type (m=n=64, four types) per step"
    print(json.dumps({
        "impl": "reference",
        "metric": "TRSM GFLOPS (m^2 n real flops, x4 complex), m=n=64 strided batch 4096, "
                  "f32+f64+c64+c128 per step",
        "value": round(value, 3), "unit": "GFLOPS", "n_gpus": 0, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(el / args.steps * 1e3, 3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64 accumulation (f32+f64+c64+c128 storage)", "data": "synthetic",
        "n_gpus_requested": ws,
        "config": {"workload": "square64: m=n=64 column-major, batch sample per type", "sample": sample_txt},
        "cpu_baseline": {"value": round(value, 3), "unit": "GFLOPS", "cores": cores, "kind": "oracle",
                         "sample": sample_txt},
        "e2e": {"value": round(value, 3), "unit": "GFLOPS", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


def main():
    global DTYPES
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=("gb300", "reference"), default="gb300")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the small sweep (batch 16384) and the large blocked solves")
    ap.add_argument("--nb-sweep", action="store_true")
    ap.add_argument("--sweep-dtypes", default="f32,f64,c64,c128")
    ap.add_argument("--sweep-ms", default="1024,2048,4096,8192,16384")
    ap.add_argument("--sweep-reps", type=int, default=3)
    ap.add_argument("--sweep-nbs", default="128,256,512", help="block sizes of the sweep")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--dtypes", default="f32,f64,c64,c128",
                    help="subset of the step's types (profiling a single kernel)")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--variants", action="store_true",
                    help="time every TRSM variant (trsm_general) at m = n = --sweep-ms per --sweep-dtypes")
    ap.add_argument("--few-rhs", action="store_true",
                    help="time few right-hand sides (--few-ns) at m = --sweep-ms per --sweep-dtypes")
    ap.add_argument("--few-ns", default="1,8")
    ap.add_argument("--medium", action="store_true",
                    help="time strided batches (--batch) of m = n = --sweep-ms systems per --sweep-dtypes")
    ap.add_argument("--batch", type=int, default=1024)
    ap.add_argument("--trtri", action="store_true",
                    help="time the exported triangular inverse (trsm_trtri_lower) at --sweep-ms per --sweep-dtypes")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    ws, rank, local = dist_env()
    DTYPES = tuple(d for d in DTYPES if d in args.dtypes.split(","))
    if args.impl == "reference":
        run_reference(args, ws, rank)
        return
    if args.nb_sweep:
        nb_sweep(args)
        return
    if args.trtri:
        trtri_bench(args)
        return
    if args.medium:
        medium_bench(args)
        return
    if args.few_rhs:
        few_rhs_bench(args)
        return
    if args.variants:
        variants_bench(args)
        return
    run_gb300(args, ws, rank, local)


if __name__ == "__main__":
    main()
