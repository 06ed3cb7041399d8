#!/usr/bin/env python3
"""Benchmark of the block-quantised decode GEMV on one GB300.

Default workload (one "step" = one call on every shape, each on its next
rotated weight copy):  Q4_0 GEMV, M = 1 token, Llama-3-8B-style tables
4096x4096, 6144x4096, 4096x14336, 14336x4096, 28672x4096, 128256x4096 (the
shapes of sm8x-bench's summary table), codes uniform 0..15, per-32 fp16 scale
uniform in [0.005, 0.02], fp16 N(0,1) activations, seeded.  Every shape cycles
through enough copies of its weights to exceed 4x the L2 so each call streams
from HBM ("cycles through enough copies of its weights" -- volta-kernel-bakeoff,
"Making it fair").

Metric: HBM GB/s of algorithmic bytes (weights + activations + outputs) over
the timed steps, plus per-shape us/call, GB/s and the fraction of the measured
HBM copy bandwidth.  Other workloads (--workload q4_0_mlp_up | q8_0 | moe |
prefill) print their own line.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
Under torchrun each rank runs the same workload on its own GPU (independent
problems, no collective on the data path): scaling "weak".
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from weight_quantized_decode_gb300 import synth  # noqa: E402

SPEC_HBM_GBS = 8000.0        # nominal HBM3e figure the target is quoted against
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0

WORKLOADS = {
    # name: (fmt, [(N, K)], [M values])
    "q4_0_m1_sweep": ("q4_0", [(4096, 4096), (6144, 4096), (4096, 14336), (14336, 4096), (28672, 4096),
                               (128256, 4096)], [1]),
    "q4_0_mlp_up": ("q4_0", [(6144, 2048)], [1]),
    "q8_0": ("q8_0", [(12288, 2560), (2560, 6144), (8192, 2048)], [1, 2, 4, 8]),
}


# ---------------------------------------------------------------------------------
def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return {"hbm_gbs": d.get("hbm_gbs", FALLBACK_HBM_GBS), "bf16_tflops": d.get("bf16_tflops"),
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained"), "source": "measured"}
    return {"hbm_gbs": FALLBACK_HBM_GBS, "bf16_tflops": FALLBACK_BF16_TFLOPS,
            "bf16_tflops_sustained": 1700.0, "source": "fallback"}


def algo_bytes(fmt, N, K, M):
    bb = 18 if fmt == "q4_0" else 34
    return N * (K // 32) * bb + 2 * M * K + 4 * M * N


class ClockSampler:
    """nvidia-smi sampling of SM clock and throttle reasons during the timed region."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [v.strip() for v in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
            except ValueError:
                continue
            for nm, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def traffic_record(kernel_name):
    """ncu DRAM traffic per launch for a kernel, if recorded for the current source."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    try:
        rec = json.load(open(p)).get(kernel_name)
    except (ValueError, OSError):
        return None
    if not rec or rec.get("source_sha") != source_sha():
        return None
    return rec


def source_sha():
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "weight_quantized_decode_gb300", "csrc")
    for fn in sorted(os.listdir(csrc)):
        if fn.endswith((".cu", ".cuh", ".h")):
            h.update(open(os.path.join(csrc, fn), "rb").read())
    return h.hexdigest()[:16]


# ---------------------------------------------------------------------------------
def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if args.impl == "ours" else "gloo"
        dist.init_process_group(backend=backend)
        return dist, rank, local, world
    return None, rank, local, world


def run_ours(args, dist, rank, local, world):
    import torch
    import weight_quantized_decode_gb300 as q

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    q.lib()
    fmt, shapes, Ms = WORKLOADS[args.workload]
    prop = torch.cuda.get_device_properties(dev)
    l2 = int(getattr(prop, "L2_cache_size", 128 * 1024 * 1024) or 128 * 1024 * 1024)

    # ---- inputs: rotated weight copies per shape, activations, outputs ----------
    # Copies per shape: a power of two >= 4 x L2 / table bytes, so every shape's
    # rotation divides the longest one and a single CUDA graph of `period`
    # steps replays the exact call sequence.
    calls = []   # one entry per (shape, M): the call made once per step
    for (N, K) in shapes:
        wbytes = N * (K // 32) * (18 if fmt == "q4_0" else 34)
        copies = 1 << max(1, math.ceil(math.log2(max(2.0, 4.0 * l2 / wbytes))))
        base = synth.weights(fmt, N, K, synth.seed_for(f"{fmt}_{N}x{K}"))
        bb = 18 if fmt == "q4_0" else 34
        Wd = torch.empty((copies, N, base.shape[1]), dtype=torch.uint8, device=dev)
        Wd[0].copy_(torch.from_numpy(base))
        for c in range(1, copies):
            # Distinct bytes per copy: XOR the code bytes with a per-copy
            # constant (any byte is a valid code); scales stay as generated.
            Wd[c].copy_(Wd[0])
            codes = Wd[c].view(N, K // 32, bb)[:, :, 2:]
            codes.bitwise_xor_(c & 0xFF)
        for M in Ms:
            x = synth.activations(M, K, synth.seed_for(f"x_{K}_{M}"))
            xd = torch.from_numpy(x).to(dev)
            yd = torch.empty((M, N), dtype=torch.float32, device=dev)
            calls.append({"N": N, "K": K, "M": M, "W": Wd, "copies": copies, "x": xd, "y": yd,
                          "x_host": torch.from_numpy(x).pin_memory(),
                          "y_host": torch.empty((M, N), dtype=torch.float32).pin_memory(),
                          "bytes": algo_bytes(fmt, N, K, M)})
    fn_ptr = q.qmv_q4_0_ptr if fmt == "q4_0" else q.qmv_q8_0_ptr
    stream = torch.cuda.Stream(dev)
    sh = int(stream.cuda_stream)
    period = max(c["copies"] for c in calls)

    def enqueue_step(s):
        for c in calls:
            W = c["W"][s % c["copies"]]
            fn_ptr(W.data_ptr(), c["x"].data_ptr(), c["y"].data_ptr(), c["N"], c["K"], c["M"], sh)

    step_bytes = sum(c["bytes"] for c in calls)
    launches_per_step = len(calls)

    # one eager pass (module loading, shared-memory opt-in) before any capture
    with torch.cuda.stream(stream):
        enqueue_step(0)
    torch.cuda.synchronize()

    # ---- CUDA graphs covering the exact step sequence ---------------------------
    def capture(count):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(stream):
            with torch.cuda.graph(g, stream=stream):
                for s in range(count):
                    enqueue_step(s)
        return g

    g_period = capture(period)
    rem_graphs = {}

    def run_steps(n):
        for _ in range(n // period):
            g_period.replay()
        r = n % period
        if r:
            if r not in rem_graphs:
                rem_graphs[r] = capture(r)
            rem_graphs[r].replay()

    # capture the remainder graphs outside the timed region
    for n in (args.warmup, args.steps):
        if n % period and (n % period) not in rem_graphs:
            rem_graphs[n % period] = capture(n % period)
    torch.cuda.synchronize()

    run_steps(args.warmup)
    torch.cuda.synchronize()

    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        run_steps(args.steps)
        e1.record(stream)
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    ms = e0.elapsed_time(e1)

    # ---- per-shape us/call (graph of R back-to-back calls cycling copies) -------
    sweep = []
    pk = peaks()
    def event_time_us(g, reps=1):
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            a.record(stream)
            for _ in range(reps):
                g.replay()
            b.record(stream)
        torch.cuda.synchronize()
        return a.elapsed_time(b) * 1e3

    for c in calls:
        R = max(64, 2 * c["copies"])

        def one_shape(first, count, c=c):
            for s in range(first, first + count):
                W = c["W"][s % c["copies"]]
                fn_ptr(W.data_ptr(), c["x"].data_ptr(), c["y"].data_ptr(), c["N"], c["K"], c["M"], sh)

        def cap(count):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.stream(stream):
                with torch.cuda.graph(g, stream=stream):
                    one_shape(0, count)
            return g

        g = cap(R)
        g1 = cap(1)
        event_time_us(g)
        best = min(event_time_us(g) / R for _ in range(5))
        # one call on its own (graph launch + ramp + drain), median of 20
        iso = statistics.median(event_time_us(g1) for _ in range(20))
        gbs = c["bytes"] / (best * 1e-6) / 1e9
        sweep.append({"N": c["N"], "K": c["K"], "M": c["M"], "copies": c["copies"],
                      "us_per_call": round(best, 3), "us_isolated_call": round(iso, 3),
                      "GBps": round(gbs, 1), "frac_of_measured_hbm": round(gbs / pk["hbm_gbs"], 4),
                      "frac_of_8TBps_spec": round(gbs / SPEC_HBM_GBS, 4)})

    clock_info = clocks.stop()

    # ---- end to end through the public API with host buffers --------------------
    e2e = None
    if not args.no_e2e:
        def e2e_step(s):
            for c in calls:
                c["x"].copy_(c["x_host"], non_blocking=True)
                W = c["W"][s % c["copies"]]
                fn_ptr(W.data_ptr(), c["x"].data_ptr(), c["y"].data_ptr(), c["N"], c["K"], c["M"], sh)
                c["y_host"].copy_(c["y"], non_blocking=True)

        with torch.cuda.stream(stream):
            for s in range(args.warmup):
                e2e_step(s)
            torch.cuda.synchronize()
            t0 = time.perf_counter()
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record(stream)
            for s in range(args.steps):
                e2e_step(args.warmup + s)
            b.record(stream)
            stream.synchronize()
            wall = time.perf_counter() - t0
        e2e_ms = max(a.elapsed_time(b), wall * 1e3)
        h2d = sum(2 * c["M"] * c["K"] for c in calls)
        d2h = sum(4 * c["M"] * c["N"] for c in calls)
        e2e = {"value": step_bytes * args.steps / (e2e_ms * 1e-3) / 1e9 * world, "unit": "GB/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "note": "weights resident in HBM (model state); per step each call's x is copied from pinned "
                       "host memory and its y read back; host-launched calls through the C ABI"}

    # ---- cross-rank timing -----------------------------------------------------
    if dist:
        t = torch.tensor([ms], dtype=torch.float64, device=dev)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        ms = float(t.item())
    value = step_bytes * args.steps * world / (ms * 1e-3) / 1e9

    out = None
    if rank == 0:
        kname = "gemv_stream_kernel"
        tr = traffic_record(f"{fmt}:{shapes[-1][0]}x{shapes[-1][1]}")
        roof = {"bound": "hbm", "achieved": round(value / world, 1), "peak": pk["hbm_gbs"], "unit": "GB/s",
                "frac": round(value / world / pk["hbm_gbs"], 4),
                "traffic": (tr or {}).get("bytes_per_launch"),
                "peak_source": f"{pk['source']} (MEASURED_PEAKS.json hbm_gbs, STREAM-style copy)",
                "kernel": kname,
                "achieved_basis": "algorithmic bytes of all launches in the timed region / CUDA-event time on "
                                  "the launching stream"}
        out = {
            "metric": f"{fmt.upper()} GEMV HBM GB/s (algorithmic bytes; us/call per shape in 'sweep')",
            "value": round(value, 1), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(ms / args.steps, 4), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f16", "data": "synthetic",
            "config": {"workload": args.workload, "format": fmt,
                       "shapes": [f"{N}x{K}" for (N, K) in shapes], "M": Ms,
                       "values": "Q4_0 codes uniform 0..15, d~U[0.005,0.02]; Q8_0 codes U[-127,127], "
                                 "d~U[0.001,0.01]; x fp16 N(0,1); seeded",
                       "l2": "inputs larger than L2: each shape cycles >= 4x L2 bytes of weight copies",
                       "timing": "CUDA graphs of back-to-back calls (programmatic dependent launch), "
                                 "CUDA events on the launching stream",
                       "parallelism": f"replica x{world} (independent problems per GPU)"},
            "sweep": sweep,
            "roofline": roof,
            "clocks": clock_info,
            "gpu_launches": launches_per_step * args.steps,
            "e2e": e2e,
            "impl": "ours",
        }
    return out, step_bytes, calls


# ---------------------------------------------------------------------------------
def oracle_sample(fmt, shapes, Ms, budget_s):
    """Time the CPU oracle (as it stands) on a bounded row sample of the workload."""
    from oracle import oracle as O
    orc = O.default()
    threads = os.cpu_count() or 1
    fid = 0 if fmt == "q4_0" else 1
    data = []
    for (N, K) in shapes:
        W = synth.weights(fmt, N, K, synth.seed_for(f"{fmt}_{N}x{K}"))
        for M in Ms:
            x = synth.activations(M, K, synth.seed_for(f"x_{K}_{M}"))
            data.append((W, x, N, K, M))
    # calibrate: 1 % of each table's rows
    done_bytes, t_total = 0, 0.0
    frac = 0.01
    while True:
        t0 = time.perf_counter()
        b = 0
        for (W, x, N, K, M) in data:
            nrows = max(1, int(N * frac))
            rows = np.linspace(0, N - 1, nrows).astype(np.int64)
            orc.qmv_rows(fid, W, x, N, K, rows, nthreads=threads)
            b += nrows * (K // 32) * (18 if fmt == "q4_0" else 34) + 2 * M * K + 4 * M * nrows
        dt = time.perf_counter() - t0
        done_bytes += b
        t_total += dt
        if t_total >= budget_s or frac >= 1.0:
            break
        frac = min(1.0, frac * max(1.5, min(8.0, budget_s / max(dt, 1e-3) / 4)))
    return {"value": round(done_bytes / t_total / 1e9, 4), "unit": "GB/s", "cores": threads, "kind": "oracle",
            "sample": f"row samples (growing to {frac:.0%} of rows) of every table of the workload, "
                      f"{t_total:.1f} s of fp64 oracle work, OpenMP over rows"}


def run_reference(args, rank, world):
    """The oracle arm: the CPU fp64 oracle timed on this host's cores."""
    if rank != 0:
        return None
    fmt, shapes, Ms = WORKLOADS[args.workload]
    from oracle import oracle as O
    orc = O.default()
    threads = os.cpu_count() or 1
    fid = 0 if fmt == "q4_0" else 1
    data = []
    for (N, K) in shapes:
        W = synth.weights(fmt, N, K, synth.seed_for(f"{fmt}_{N}x{K}"))
        for M in Ms:
            x = synth.activations(M, K, synth.seed_for(f"x_{K}_{M}"))
            data.append((W, x, N, K, M))
    # Per step: the same fixed row sample of every table, sized so that the
    # whole run stays within about two minutes.
    per_step_budget = min(1.0, 120.0 / max(1, args.steps + args.warmup))
    frac = 0.002
    while True:
        t0 = time.perf_counter()
        for (W, x, N, K, M) in data:
            rows = np.linspace(0, N - 1, max(1, int(N * frac))).astype(np.int64)
            orc.qmv_rows(fid, W, x, N, K, rows, nthreads=threads)
        dt = time.perf_counter() - t0
        if dt >= per_step_budget / 2 or frac >= 1.0:
            break
        frac = min(1.0, frac * 2)
    samples = [(W, x, N, K, M, np.linspace(0, N - 1, max(1, int(N * frac))).astype(np.int64))
               for (W, x, N, K, M) in data]
    bb = 18 if fmt == "q4_0" else 34
    step_bytes = sum(r.size * (K // 32) * bb + 2 * M * K + 4 * M * r.size for (_, _, _, K, M, r) in samples)

    def step():
        for (W, x, N, K, M, rows) in samples:
            orc.qmv_rows(fid, W, x, N, K, rows, nthreads=threads)

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    dt = time.perf_counter() - t0
    value = step_bytes * args.steps / dt / 1e9
    sample = (f"{frac:.2%} of the rows of every table per step (evenly spaced), fp64 oracle, "
              f"OpenMP over rows")
    return {
        "metric": f"{fmt.upper()} GEMV HBM GB/s (algorithmic bytes; us/call per shape in 'sweep')",
        "value": round(value, 4), "unit": "GB/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(dt * 1e3 / args.steps, 3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": args.workload, "format": fmt, "shapes": [f"{N}x{K}" for (N, K) in shapes],
                   "M": Ms},
        "impl": "reference",
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": threads, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


# ---------------------------------------------------------------------------------
def ncu_case(spec):
    """A handful of eager calls of one shape over rotated copies larger than L2
    (a small, bounded program for an Nsight Compute capture)."""
    import torch
    import weight_quantized_decode_gb300 as q
    fmt, shape, M = spec.split(":")
    N, K = (int(v) for v in shape.split("x"))
    M = int(M)
    dev = torch.device("cuda", 0)
    bb = 18 if fmt == "q4_0" else 34
    wbytes = N * (K // 32) * bb
    copies = max(2, math.ceil(2.5 * 128e6 / wbytes))
    base = torch.from_numpy(synth.weights(fmt, N, K, synth.seed_for(f"{fmt}_{N}x{K}"))).to(dev)
    W = base.unsqueeze(0).repeat(copies, 1, 1)
    x = torch.from_numpy(synth.activations(M, K, 1)).to(dev)
    y = torch.empty((M, N), dtype=torch.float32, device=dev)
    fn = {"q4_0": q.qmv_q4_0_ptr, "q8_0": q.qmv_q8_0_ptr}[fmt]
    s = torch.cuda.current_stream().cuda_stream
    for i in range(8):
        fn(W[i % copies].data_ptr(), x.data_ptr(), y.data_ptr(), N, K, M, s)
    torch.cuda.synchronize()
    print(f"ncu case {spec}: {copies} copies, 8 calls, ok")


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=200)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default="q4_0_m1_sweep")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-budget", type=float, default=12.0, help="seconds of oracle work for cpu_baseline")
    ap.add_argument("--ncu-case", default=None,
                    help="FMT:NxK:M -- only run a few eager calls of one shape (for Nsight Compute captures)")
    args = ap.parse_args()
    if args.ncu_case:
        ncu_case(args.ncu_case)
        return
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")

    dist, rank, local, world = dist_setup(args)
    if args.impl == "reference":
        out = run_reference(args, rank, world)
        if out is not None:
            print(json.dumps(out), flush=True)
        if dist:
            dist.destroy_process_group()
        return

    out, _, _ = run_ours(args, dist, rank, local, world)
    if rank == 0:
        if not args.no_cpu_baseline:
            fmt, shapes, Ms = WORKLOADS[args.workload]
            out["cpu_baseline"] = oracle_sample(fmt, shapes, Ms, args.cpu_budget)
        else:
            out["cpu_baseline"] = None
        print(json.dumps(out), flush=True)
    if dist:
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
