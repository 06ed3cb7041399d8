#!/usr/bin/env python3
"""Benchmark of the block-quantised decode GEMV on one GB300.

Default workload (one "step" = one call on every shape, each on its next
rotated weight copy):  Q4_0 GEMV, M = 1 token, Llama-3-8B-style tables
4096x4096, 6144x4096, 4096x14336, 14336x4096, 28672x4096, 128256x4096 (the
shapes of sm8x-bench's summary table), codes uniform 0..15, per-32 fp16 scale
uniform in [0.005, 0.02], fp16 N(0,1) activations, seeded.  Every shape rotates
over enough copies of its weights to exceed 4x the L2 so each call streams
from HBM (the bakeoff rotates weight copies for the same reason --
volta-kernel-bakeoff, "Making it fair").

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

BLOCK_BYTES = {"q4_0": 18, "q8_0": 34, "q2w": 10}
FMT_ID = {"q4_0": 0, "q8_0": 1, "q2w": 2}
SPEC_HBM_GBS = 8000.0        # nominal HBM3e figure the target is quoted against
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0

WORKLOADS = {
    # The configuration the headline metric is quoted on: Q4_0, one token,
    # Llama-3-8B-style tables (sm8x-bench summary table).
    "q4_0_m1_sweep": {"kind": "gemv", "fmt": "q4_0", "M": [1],
                      "shapes": [(4096, 4096), (6144, 4096), (4096, 14336), (14336, 4096), (28672, 4096),
                                 (128256, 4096)]},
    # Qwen3-1.7B MLP up (volta-kernel-bakeoff, "What's in the race").
    "q4_0_mlp_up": {"kind": "gemv", "fmt": "q4_0", "M": [1], "shapes": [(6144, 2048)]},
    # Q8_0 attention / output tables at a few tokens.
    "q8_0": {"kind": "gemv", "fmt": "q8_0", "M": [1, 2, 4, 8],
             "shapes": [(12288, 2560), (2560, 6144), (8192, 2048)]},
    # Experts in one launch: (pool size, slots, N, K).
    "moe": {"kind": "moe", "fmt": "q4_0", "configs": [(128, 10, 640, 2560), (128, 8, 512, 2048)]},
    # The MLP's gate + up + SwiGLU in one call: Llama-3-8B (gate and up 14336x4096
    # each) and Qwen3-1.7B (6144x2048 each, the fused MLP table the bakeoff times
    # -- volta-kernel-bakeoff, "A few tokens at once"), one token and eight.
    "q4_0_swiglu": {"kind": "swiglu", "fmt": "q4_0", "M": [1, 8], "shapes": [(14336, 4096), (6144, 2048)]},
    # fp32 activations in, narrowed to fp16 inside the kernel (the bakeoff's
    # like-for-like fp32in comparison: its six one-token tables -- volta-kernel-
    # bakeoff, "Results (one token, microseconds, lower is better)" -- at one
    # token and eight; and Qwen3-1.7B's fused gate + up + SwiGLU).
    "q4_0_f32in": {"kind": "gemv", "fmt": "q4_0", "x": "f32", "M": [1, 8],
                   "shapes": [(12288, 2560), (8192, 2048), (6144, 2048), (640, 2560), (512, 2048), (2048, 512)]},
    "q4_0_swiglu_f32in": {"kind": "swiglu", "fmt": "q4_0", "x": "f32", "M": [1, 8], "shapes": [(6144, 2048)]},
    # Q4_0 against activations quantised to Q8_1 in the kernel, integer dots
    # (sm8x-bench, "Our kernel does what llama.cpp does"): the Llama-3-8B
    # tables at one token and eight.
    "q4_0_q8_1": {"kind": "gemv", "fmt": "q4_0", "x": "q8_1", "M": [1, 8], "dtype": "i8",
                  "shapes": [(4096, 4096), (6144, 4096), (4096, 14336), (14336, 4096), (28672, 4096),
                             (128256, 4096)]},
    # The same tables in the two steps of the sm8x kernel and llama.cpp: the
    # activations to Q8_1 (one launch), then the int8 product on them (another).
    "q4_0_q8_1_pre": {"kind": "gemv", "fmt": "q4_0", "x": "q8_1_pre", "M": [1, 8], "dtype": "i8",
                      "shapes": [(4096, 4096), (6144, 4096), (4096, 14336), (14336, 4096), (28672, 4096),
                                 (128256, 4096)]},
    # The Q8_0 tables against activations quantised to Q8_1, signed int8 dots
    # (the Q8_1 form carried from Q4_0 to Q8_0): fused, and in two launches.
    "q8_0_q8_1": {"kind": "gemv", "fmt": "q8_0", "x": "q8_1", "M": [1, 2, 4, 8], "dtype": "i8",
                  "shapes": [(12288, 2560), (2560, 6144), (8192, 2048)]},
    "q8_0_q8_1_pre": {"kind": "gemv", "fmt": "q8_0", "x": "q8_1_pre", "M": [1, 2, 4, 8], "dtype": "i8",
                      "shapes": [(12288, 2560), (2560, 6144), (8192, 2048)]},
    # Plain 2-bit (codes -2..1, fp16 scale per 32): the bakeoff's six one-token
    # tables (volta-kernel-bakeoff, "Results (one token, microseconds, lower is
    # better)", its 2-bit column).
    "q2w": {"kind": "gemv", "fmt": "q2w", "M": [1],
            "shapes": [(12288, 2560), (8192, 2048), (6144, 2048), (640, 2560), (512, 2048), (2048, 512)]},
    # Prompt (prefill) on the tensor cores.
    "prefill": {"kind": "prefill", "fmt": "q4_0", "M": [64, 512], "shapes": [(12288, 2560), (8192, 2048)]},
}


def call_names(workload):
    """The calls of one step of a workload, in order (as build_calls names them)."""
    wl = WORKLOADS[workload]
    if wl["kind"] == "moe":
        return [f"{slots}x({N}x{K}) of {E}" for (E, slots, N, K) in wl["configs"]]
    return [f"{N}x{K}/M{M}" for (N, K) in wl["shapes"] for M in wl["M"]]


VALUES = ("Q4_0 codes uniform 0..15, d~U[0.005,0.02]; Q8_0 codes U[-127,127], d~U[0.001,0.01]; "
          "x fp16 N(0,1); seeded")


def metric_name(workload):
    wl = WORKLOADS[workload]
    if wl["kind"] == "prefill":
        return "Q4_0 prefill GEMM TFLOP/s (fp16 tensor cores; us/call per table in 'sweep')"
    if wl["kind"] == "moe":
        return "Q4_0 multi-expert GEMV (one launch) HBM GB/s (algorithmic bytes; us/call per config in 'sweep')"
    xin = {"f32": " (fp32 activations in)", "q8_1": " (activations quantised to Q8_1 in the kernel, int8 dots)",
           "q8_1_pre": " (activations quantised to Q8_1 by a launch of their own, then int8 dots)"}.get(wl.get("x"), "")
    if wl["kind"] == "swiglu":
        return (f"Q4_0 fused gate+up+SwiGLU{xin} HBM GB/s (algorithmic bytes of both tables; "
                "us/call per table in 'sweep')")
    return f"{wl['fmt'].upper()} GEMV{xin} HBM GB/s (algorithmic bytes; us/call per table in 'sweep')"


# ---------------------------------------------------------------------------------
def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return {"hbm_gbs": d.get("hbm_gbs", FALLBACK_HBM_GBS), "bf16_tflops": d.get("bf16_tflops"),
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained"), "source": "measured"}
    return {"hbm_gbs": FALLBACK_HBM_GBS, "bf16_tflops": FALLBACK_BF16_TFLOPS,
            "bf16_tflops_sustained": 1700.0, "source": "fallback"}


def algo_bytes(fmt, N, K, M, x_bytes=2):
    """The table once, the activations once (x_bytes each), y once."""
    bb = BLOCK_BYTES[fmt]
    return N * (K // 32) * bb + x_bytes * M * K + 4 * M * N


def algo_bytes_swiglu(N, K, M, x_bytes=2):
    """Both Q4_0 tables once, the activations once, y once."""
    return 2 * N * (K // 32) * 18 + x_bytes * M * K + 4 * M * N


def x_dtype(wl):
    """(numpy dtype, bytes) of a workload's activations."""
    return (np.float32, 4) if wl.get("x") == "f32" else (np.float16, 2)


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


def traffic_record(workload):
    """ncu DRAM traffic per launch for a workload, if recorded for the current
    sources of the kernels it runs."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    try:
        rec = json.load(open(p)).get(workload)
    except (ValueError, OSError):
        return None
    if not rec or rec.get("source_sha") != source_sha(source_family(workload)):
        return None
    return rec


def source_family(workload):
    """Which kernel sources a workload's launches come from: the prefill
    kernel alone, the decode kernels alone, or both (fp16-activation Q4_0 /
    Q8_0 GEMVs with four tokens or more, whose calls may run on the prefill
    kernel's 16-token tiles)."""
    wl = WORKLOADS.get(workload, {})
    if wl.get("kind") == "prefill":
        return "prefill"
    if (wl.get("kind") == "gemv" and wl.get("fmt") in ("q4_0", "q8_0") and "x" not in wl
            and max(wl.get("M", [1])) >= 4):
        return "all"
    return "decode"


PREFILL_SOURCES = ("qmv_prefill.cu", "qmv_prefill.h", "qmv_prefill_plan.h", "qmv_common.cuh", "qmv_launch.h")


def source_sha(family="decode"):
    """Hash of the kernel sources a traffic record depends on: the prefill
    kernel's files, (decode) every other source of the library, or (all)
    every source."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "weight_quantized_decode_gb300", "csrc")
    for fn in sorted(os.listdir(csrc)):
        if not fn.endswith((".cu", ".cuh", ".h")):
            continue
        if family == "prefill":
            if fn not in PREFILL_SOURCES:
                continue
        elif fn == "qmv_probe.cu" or (family == "decode" and fn in ("qmv_prefill.cu", "qmv_prefill_plan.h")):
            continue
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


def cross_rank_max_ms(dist, ms, device):
    """The slowest rank's duration of a timed region (every rank calls this)."""
    if not dist:
        return ms
    import torch
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(units_per_step, steps, world, ms):
    """Units per second of the whole job: every rank processes units_per_step
    per step (weak scaling), over the slowest rank's time."""
    return units_per_step * steps * world / (ms * 1e-3)


def build_calls(workload, q, torch, dev, l2, sh):
    """The calls one step of `workload` makes, each on its own rotated weight
    copies, and the rotation period (steps after which the sequence repeats)."""
    wl = WORKLOADS[workload]
    kind, fmt = wl["kind"], wl["fmt"]
    bb = BLOCK_BYTES[fmt]

    def rotated_copies(rows, K, seed_name):
        """A power of two of weight copies, >= 4x L2 in total, each with distinct
        bytes (codes XOR a per-copy constant; scales as generated)."""
        wbytes = rows * (K // 32) * bb
        copies = 1 << max(1, math.ceil(math.log2(max(2.0, 4.0 * l2 / wbytes))))
        base = synth.weights(fmt, rows, K, synth.seed_for(seed_name))
        Wd = torch.empty((copies, rows, base.shape[1]), dtype=torch.uint8, device=dev)
        Wd[0].copy_(torch.from_numpy(base))
        for c in range(1, copies):
            Wd[c].copy_(Wd[0])
            Wd[c].view(rows, K // 32, bb)[:, :, 2:].bitwise_xor_(c & 0xFF)
        return Wd, copies

    # Copies per table are powers of two, so every table's rotation divides the
    # longest one and a single CUDA graph of `period` steps replays the exact
    # call sequence.
    calls = []
    xdt, xb = x_dtype(wl)
    if kind in ("gemv", "prefill"):
        fn_ptr = {"gemv": {"q4_0": q.qmv_q4_0_ptr, "q8_0": q.qmv_q8_0_ptr, "q2w": q.qmv_q2w_ptr}[fmt],
                  "prefill": q.qmm_q4_0_prefill_ptr}[kind]
        if xb == 4:
            fn_ptr = q.qmv_q4_0_f32_ptr
        if wl.get("x") == "q8_1":
            fn_ptr = {"q4_0": q.qmv_q4_0_q8_1_ptr, "q8_0": q.qmv_q8_0_q8_1_ptr}[fmt]
        pre = wl.get("x") == "q8_1_pre"
        for (N, K) in wl["shapes"]:
            Wd, copies = rotated_copies(N, K, f"{fmt}_{N}x{K}")
            for M in wl["M"]:
                x = synth.activations(M, K, synth.seed_for(f"x_{K}_{M}"), dtype=xdt)
                c = {"name": f"{N}x{K}/M{M}", "N": N, "K": K, "M": M, "W": Wd, "copies": copies,
                     "x": torch.from_numpy(x).to(dev), "y": torch.empty((M, N), dtype=torch.float32, device=dev),
                     "x_host": torch.from_numpy(x).pin_memory(),
                     "y_host": torch.empty((M, N), dtype=torch.float32).pin_memory(),
                     "bytes": algo_bytes(fmt, N, K, M, xb), "flops": 2 * M * N * K}

                if pre:   # Q8_1 buffers for the activations, written by the quantisation launch
                    c["xq"] = torch.empty((M, K), dtype=torch.int8, device=dev)
                    c["xq_d"] = torch.empty((M, K // 32), dtype=torch.int16, device=dev)
                    c["xq_s"] = torch.empty((M, K // 32), dtype=torch.int32, device=dev)
                    c["launches"] = 2

                    def call(s, c=c):
                        W = c["W"][s % c["copies"]]
                        q.qmv_quantize_q8_1_ptr(c["x"].data_ptr(), c["xq"].data_ptr(), c["xq_d"].data_ptr(),
                                                c["xq_s"].data_ptr(), c["M"], c["K"], sh)
                        if fmt == "q8_0":   # Q8_0 codes carry no offset: no code sums
                            q.qmv_q8_0_q8_1_pre_ptr(W.data_ptr(), c["xq"].data_ptr(), c["xq_d"].data_ptr(),
                                                    c["y"].data_ptr(), c["N"], c["K"], c["M"], sh)
                        else:
                            q.qmv_q4_0_q8_1_pre_ptr(W.data_ptr(), c["xq"].data_ptr(), c["xq_d"].data_ptr(),
                                                    c["xq_s"].data_ptr(), c["y"].data_ptr(), c["N"], c["K"], c["M"],
                                                    sh)
                else:
                    def call(s, c=c):
                        W = c["W"][s % c["copies"]]
                        fn_ptr(W.data_ptr(), c["x"].data_ptr(), c["y"].data_ptr(), c["N"], c["K"], c["M"], sh)
                c["call"] = call
                calls.append(c)
    elif kind == "swiglu":
        for (N, K) in wl["shapes"]:
            # gate rows 0..N-1 and up rows N..2N-1 of one rotated allocation
            Wd, copies = rotated_copies(2 * N, K, f"swiglu_{N}x{K}")
            sw_ptr = q.qmv_q4_0_swiglu_f32_ptr if xb == 4 else q.qmv_q4_0_swiglu_ptr
            for M in wl["M"]:
                x = synth.activations(M, K, synth.seed_for(f"x_{K}_{M}"), dtype=xdt)
                c = {"name": f"{N}x{K}/M{M}", "N": N, "K": K, "M": M, "W": Wd, "copies": copies,
                     "x": torch.from_numpy(x).to(dev), "y": torch.empty((M, N), dtype=torch.float32, device=dev),
                     "x_host": torch.from_numpy(x).pin_memory(),
                     "y_host": torch.empty((M, N), dtype=torch.float32).pin_memory(),
                     "bytes": algo_bytes_swiglu(N, K, M, xb), "flops": 4 * M * N * K}

                def call(s, c=c, sw_ptr=sw_ptr):
                    W = c["W"][s % c["copies"]]
                    sw_ptr(W[:c["N"]].data_ptr(), W[c["N"]:].data_ptr(), c["x"].data_ptr(),
                           c["y"].data_ptr(), c["N"], c["K"], c["M"], sh)
                c["call"] = call
                calls.append(c)
    else:  # moe: a pool of experts, distinct indices drawn per step
        for (E, slots, N, K) in wl["configs"]:
            Wd, copies = rotated_copies(E * N, K, f"moe_{E}x{N}x{K}")
            period_idx = 64
            idx = synth.expert_indices(period_idx, slots, E, synth.seed_for(f"moe_idx_{E}_{slots}"))
            x = synth.activations(slots, K, synth.seed_for(f"moe_x_{K}_{slots}"))
            c = {"name": f"{slots}x({N}x{K}) of {E}", "N": N, "K": K, "M": slots, "E": E, "W": Wd,
                 "copies": copies, "idx": torch.from_numpy(idx).to(dev), "idx_period": period_idx,
                 "x": torch.from_numpy(x).to(dev), "y": torch.empty((slots, N), dtype=torch.float32, device=dev),
                 "x_host": torch.from_numpy(x).pin_memory(),
                 "y_host": torch.empty((slots, N), dtype=torch.float32).pin_memory(),
                 "bytes": slots * algo_bytes(fmt, N, K, 1) + 4 * slots, "flops": 2 * slots * N * K}

            def call(s, c=c):
                W = c["W"][s % c["copies"]]
                ix = c["idx"][s % c["idx_period"]]
                q.qmv_moe_ptr(W.data_ptr(), ix.data_ptr(), c["E"], c["x"].data_ptr(), c["y"].data_ptr(),
                              c["N"], c["K"], c["M"], sh)
            c["call"] = call
            calls.append(c)
    period = max(max(c["copies"] for c in calls), max(c.get("idx_period", 1) for c in calls))
    return calls, period


class StepRunner:
    """CUDA graphs that replay the exact call sequence of any number of steps."""

    def __init__(self, torch, stream, calls, period):
        self.torch, self.stream, self.calls, self.period = torch, stream, calls, period
        self.rem = {}
        self.g_period = self.capture(period)

    def enqueue(self, s):
        for c in self.calls:
            c["call"](s)

    def capture(self, count):
        torch = self.torch
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(self.stream):
            with torch.cuda.graph(g, stream=self.stream):
                for s in range(count):
                    self.enqueue(s)
        return g

    def prepare(self, n):
        """Capture the remainder graph for n steps (outside any timed region)."""
        r = n % self.period
        if r and r not in self.rem:
            self.rem[r] = self.capture(r)

    def run(self, n):
        for _ in range(n // self.period):
            self.g_period.replay()
        r = n % self.period
        if r:
            self.prepare(n)
            self.rem[r].replay()

    def time_ms(self, n):
        torch = self.torch
        self.prepare(n)
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(self.stream):
            e0.record(self.stream)
            self.run(n)
            e1.record(self.stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1)


def per_call_sweep(torch, stream, calls, kind, pk):
    """Per call: us/call over a graph of R back-to-back calls cycling copies
    (best of 5) and one call alone in its own graph (median of 20)."""
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

    sweep = []
    for c in calls:
        R = max(64, 2 * c["copies"])

        def cap(count, c=c):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.stream(stream):
                with torch.cuda.graph(g, stream=stream):
                    for s_ in range(count):
                        c["call"](s_)
            return g

        g = cap(R)
        g1 = cap(1)
        event_time_us(g)
        best = min(event_time_us(g) / R for _ in range(5))
        # one call on its own (graph launch + ramp + drain), median of 20
        iso = statistics.median(event_time_us(g1) for _ in range(20))
        gbs = c["bytes"] / (best * 1e-6) / 1e9
        row = {"call": c["name"], "copies": c["copies"], "us_per_call": round(best, 3),
               "us_isolated_call": round(iso, 3), "GBps": round(gbs, 1),
               "frac_of_measured_hbm": round(gbs / pk["hbm_gbs"], 4),
               "frac_of_8TBps_spec": round(gbs / SPEC_HBM_GBS, 4)}
        if pk.get("read_probe_gbs"):
            row["frac_of_read_probe"] = round(gbs / pk["read_probe_gbs"], 4)
        if kind == "prefill":
            tf = c["flops"] / (best * 1e-6) / 1e12
            row["TFLOPs"] = round(tf, 1)
            row["frac_of_measured_tensor"] = round(tf / pk["bf16_tflops"], 4)
        sweep.append(row)
    return sweep


def read_probe_gbs(q, torch, dev, stream, l2):
    """The read-only bandwidth probe (the decode kernels' bulk-copy streaming
    with no arithmetic) over 16x L2: best of 5 runs of 10 back-to-back launches."""
    nbytes = (16 * l2 + 255) // 256 * 256
    buf = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    buf.random_(0, 256)
    out = torch.empty(1, dtype=torch.int32, device=dev)
    sh = int(stream.cuda_stream)
    with torch.cuda.stream(stream):
        for _ in range(3):
            q.qmv_read_probe_ptr(buf.data_ptr(), nbytes, out.data_ptr(), sh)
        torch.cuda.synchronize()
        best = None
        for _ in range(5):
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record(stream)
            for _ in range(10):
                q.qmv_read_probe_ptr(buf.data_ptr(), nbytes, out.data_ptr(), sh)
            b.record(stream)
            torch.cuda.synchronize()
            ms = a.elapsed_time(b)
            best = ms if best is None else min(best, ms)
    del buf
    return 10 * nbytes / (best * 1e-3) / 1e9, nbytes


# Other configurations of the metric, timed by the default run after the
# headline workload: Q8_0 at 1..8 tokens, the multi-expert call, prefill.
EXTRA_SWEEPS = {"sweep_q8_0": "q8_0", "sweep_moe": "moe", "sweep_prefill": "prefill"}


def run_ours(args, dist, rank, local, world):
    import torch
    import weight_quantized_decode_gb300 as q

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    q.lib()
    wl = WORKLOADS[args.workload]
    kind, fmt = wl["kind"], wl["fmt"]
    prop = torch.cuda.get_device_properties(dev)
    l2 = int(getattr(prop, "L2_cache_size", 128 * 1024 * 1024) or 128 * 1024 * 1024)
    stream = torch.cuda.Stream(dev)
    sh = int(stream.cuda_stream)
    pk = peaks()

    calls, period = build_calls(args.workload, q, torch, dev, l2, sh)

    def one_buffer(key_dev, key_host):
        """Lay the calls' device tensors `key_dev` out in one device buffer (pieces
        256-byte aligned) with a pinned host twin holding `key_host`, so that a
        step's activations go host->device in one copy and its outputs come back
        in one.  Returns (device buffer, host buffer)."""
        sizes = [c[key_dev].numel() * c[key_dev].element_size() for c in calls]
        offs, o = [], 0
        for sz in sizes:
            offs.append(o)
            o += (sz + 255) // 256 * 256
        dbuf = torch.zeros(o, dtype=torch.uint8, device=dev)
        hbuf = torch.zeros(o, dtype=torch.uint8).pin_memory()
        for c, off, sz in zip(calls, offs, sizes):
            t = c[key_dev]
            view = dbuf[off:off + sz].view(t.dtype).view(t.shape)
            view.copy_(t)
            hbuf[off:off + sz].view(t.dtype).view(t.shape).copy_(c[key_host])
            c[key_dev] = view
        return dbuf, hbuf

    x_dev_all, x_host_all = one_buffer("x", "x_host")
    y_dev_all, y_host_all = one_buffer("y", "y_host")

    step_bytes = sum(c["bytes"] for c in calls)
    step_flops = sum(c["flops"] for c in calls)
    launches_per_step = sum(c.get("launches", 1) for c in calls)

    # one eager pass (module loading, shared-memory opt-in) before any capture
    with torch.cuda.stream(stream):
        for c in calls:
            c["call"](0)
    torch.cuda.synchronize()

    # ---- CUDA graphs covering the exact step sequence ---------------------------
    runner = StepRunner(torch, stream, calls, period)
    runner.prepare(args.warmup)
    runner.prepare(args.steps)
    torch.cuda.synchronize()

    runner.run(args.warmup)
    torch.cuda.synchronize()

    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    if dist:
        dist.barrier()
    ms = runner.time_ms(args.steps)
    if dist:
        dist.barrier()

    # ---- the read roofline, then per-shape us/call ------------------------------
    probe_gbs, probe_bytes = read_probe_gbs(q, torch, dev, stream, l2)
    pk["read_probe_gbs"] = probe_gbs
    sweep = per_call_sweep(torch, stream, calls, kind, pk)

    # ---- the rest of the metric's configurations (default run only) -------------
    extras = {}
    if args.workload == "q4_0_m1_sweep" and not args.no_extra:
        for key, ewl in EXTRA_SWEEPS.items():
            ecalls, eperiod = build_calls(ewl, q, torch, dev, l2, sh)
            with torch.cuda.stream(stream):
                for c in ecalls:
                    c["call"](0)
            torch.cuda.synchronize()
            er = StepRunner(torch, stream, ecalls, eperiod)
            n_steps = max(3 * eperiod, 96)
            er.run(max(eperiod, 8))
            e_ms = er.time_ms(n_steps)
            ekind = WORKLOADS[ewl]["kind"]
            eb = sum(c["bytes"] for c in ecalls) * n_steps
            ef = sum(c["flops"] for c in ecalls) * n_steps
            entry = {"workload": ewl, "steps": n_steps, "ms_per_step": round(e_ms / n_steps, 4),
                     "calls_per_step": [c["name"] for c in ecalls],
                     "launches_per_step": sum(c.get("launches", 1) for c in ecalls)}
            if ekind == "prefill":
                tf = ef / (e_ms * 1e-3) / 1e12
                entry.update({"value": round(tf, 1), "unit": "TFLOP/s",
                              "frac_of_measured_tensor": round(tf / pk["bf16_tflops"], 4)})
            else:
                gb = eb / (e_ms * 1e-3) / 1e9
                entry.update({"value": round(gb, 1), "unit": "GB/s",
                              "frac_of_measured_hbm": round(gb / pk["hbm_gbs"], 4),
                              "frac_of_read_probe": round(gb / probe_gbs, 4)})
            entry["sweep"] = per_call_sweep(torch, stream, ecalls, ekind, pk)
            extras[key] = entry
            del er, ecalls
            torch.cuda.synchronize()
            torch.cuda.empty_cache()

    clock_info = clocks.stop()

    # ---- end to end through the public API with host buffers --------------------
    e2e = None
    if not args.no_e2e:
        def e2e_step(s):
            # the step's activations in, every call, the step's outputs out
            x_dev_all.copy_(x_host_all, non_blocking=True)
            for c in calls:
                c["call"](s)
            y_host_all.copy_(y_dev_all, non_blocking=True)

        with torch.cuda.stream(stream):
            for s in range(args.warmup):
                e2e_step(s)
            torch.cuda.synchronize()
            if dist:
                dist.barrier()
            t0 = time.perf_counter()
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record(stream)
            for s in range(args.steps):
                e2e_step(args.warmup + s)
            b.record(stream)
            stream.synchronize()
            wall = time.perf_counter() - t0
        e2e_ms = cross_rank_max_ms(dist, max(a.elapsed_time(b), wall * 1e3), dev)
        h2d = x_host_all.numel()
        d2h = y_host_all.numel()
        e2e_val = whole_job_rate(step_flops / 1e12 if kind == "prefill" else step_bytes / 1e9, args.steps, world, e2e_ms)
        e2e = {"value": round(e2e_val, 3), "unit": "TFLOP/s" if kind == "prefill" else "GB/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "note": "weights resident in HBM (model state); per step all calls' activations are copied from "
                       "pinned host memory in one transfer and all outputs read back in one; host-launched calls "
                       "through the C ABI"}

    # ---- cross-rank timing -----------------------------------------------------
    ms = cross_rank_max_ms(dist, ms, dev)
    gbs_total = whole_job_rate(step_bytes, args.steps, world, ms) / 1e9
    tflops_total = whole_job_rate(step_flops, args.steps, world, ms) / 1e12

    out = None
    if rank == 0:
        if kind == "prefill":
            value, unit = tflops_total, "TFLOP/s"
            roof = {"bound": "tensor", "achieved": round(tflops_total / world, 1), "peak": pk["bf16_tflops"],
                    "unit": "TFLOP/s", "frac": round(tflops_total / world / pk["bf16_tflops"], 4),
                    "peak_source": f"{pk['source']} (MEASURED_PEAKS.json bf16_tflops burst; fp16 has the same "
                                   f"nominal dense rate)",
                    "hbm_frac": round(gbs_total / world / pk["hbm_gbs"], 4), "kernel": "prefill_kernel"}
        else:
            value, unit = gbs_total, "GB/s"
            roof = {"bound": "hbm", "achieved": round(gbs_total / world, 1), "peak": pk["hbm_gbs"], "unit": "GB/s",
                    "frac": round(gbs_total / world / pk["hbm_gbs"], 4),
                    "peak_source": f"{pk['source']} (MEASURED_PEAKS.json hbm_gbs, STREAM-style copy)",
                    "kernel": "qmv_stream_kernel"}
        roof["peak_read_probe"] = round(probe_gbs, 1)
        roof["frac_of_read_probe"] = None if kind == "prefill" else round(gbs_total / world / probe_gbs, 4)
        roof["read_probe"] = (f"qmv_read_probe: {probe_bytes / 2**30:.2f} GiB (16x L2) streamed by bulk copies "
                              f"into per-warp rings, no arithmetic; best of 5 x 10 launches on this GPU")
        tr = traffic_record(args.workload)
        roof["traffic"] = (tr or {}).get("bytes_per_launch")
        if tr:
            roof["traffic_launch"] = tr.get("launch")
        roof["achieved_basis"] = ("algorithmic work of all launches in the timed region / CUDA-event time on the "
                                  "launching stream (per-launch figures in 'sweep')")
        cfg = {"workload": args.workload, "format": fmt, "calls_per_step": [c["name"] for c in calls],
               "values": VALUES,
               "l2": "inputs larger than L2: each table cycles >= 4x L2 bytes of weight copies",
               "timing": "CUDA graphs of back-to-back calls (programmatic dependent launch for the decode "
                         "kernels), CUDA events on the launching stream",
               "parallelism": f"replica x{world} (independent problems per GPU)"}
        out = {
            "metric": metric_name(args.workload), "value": round(value, 2), "unit": unit, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(ms / args.steps, 4), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": wl.get("dtype", "f16"), "data": "synthetic",
            "config": cfg,
            "sweep": sweep,
            "roofline": roof,
            "clocks": clock_info,
            "gpu_launches": launches_per_step * args.steps,
            "e2e": e2e,
            "impl": "ours",
        }
        out.update(extras)
    return out, step_bytes, calls


# ---------------------------------------------------------------------------------
def oracle_tasks(workload):
    """The workload's tables as oracle jobs: run(frac) evaluates an evenly
    spaced `frac` of each table's rows and returns (bytes, flops) of that work."""
    from oracle import oracle as O
    orc = O.default()
    threads = os.cpu_count() or 1
    wl = WORKLOADS[workload]
    fmt = wl["fmt"]
    fid = FMT_ID[fmt]
    bb = BLOCK_BYTES[fmt]
    xdt, xb = x_dtype(wl)
    jobs = []
    if wl["kind"] == "swiglu":
        sjobs = []
        for (N, K) in wl["shapes"]:
            W2 = synth.weights(fmt, 2 * N, K, synth.seed_for(f"swiglu_{N}x{K}"))
            for M in wl["M"]:
                x = synth.activations(M, K, synth.seed_for(f"x_{K}_{M}"), dtype=xdt)
                sjobs.append((W2[:N], W2[N:], x, N, K, M))

        def run_swiglu(frac):
            b = f = 0
            for (Wg, Wu, x, N, K, M) in sjobs:
                rows = np.linspace(0, N - 1, max(1, int(N * frac))).astype(np.int64)
                orc.swiglu(fid, Wg, Wu, x, N, K, rows=rows, nthreads=threads)
                b += 2 * rows.size * (K // 32) * bb + xb * M * K + 4 * M * rows.size
                f += 4 * M * rows.size * K
            return b, f
        return run_swiglu, threads, wl["kind"]
    if wl["kind"] in ("gemv", "prefill"):
        for (N, K) in wl["shapes"]:
            W = synth.weights(fmt, N, K, synth.seed_for(f"{fmt}_{N}x{K}"))
            for M in wl["M"]:
                x = synth.activations(M, K, synth.seed_for(f"x_{K}_{M}"), dtype=xdt)
                jobs.append((W, x, N, K, M))
    else:
        for (E, slots, N, K) in wl["configs"]:
            pool = synth.weights(fmt, E * N, K, synth.seed_for(f"moe_{E}x{N}x{K}"))
            idx = synth.expert_indices(1, slots, E, synth.seed_for(f"moe_idx_{E}_{slots}"))[0]
            x = synth.activations(slots, K, synth.seed_for(f"moe_x_{K}_{slots}"))
            for sl in range(slots):
                e = int(idx[sl])
                jobs.append((pool[e * N:(e + 1) * N], x[sl:sl + 1], N, K, 1))

    q81 = wl.get("x") in ("q8_1", "q8_1_pre")

    def run(frac):
        b = f = 0
        for (W, x, N, K, M) in jobs:
            rows = np.linspace(0, N - 1, max(1, int(N * frac))).astype(np.int64)
            if q81:   # the activations to Q8_1, then the product on them
                qx, dx, _ = orc.quantize_q8_1(x)
                orc.qmv_q8_1(fid, W, qx, dx, N, K, rows=rows, nthreads=threads)
                b += rows.size * (K // 32) * bb + xb * M * K + 4 * M * rows.size
                f += 2 * M * rows.size * K
                continue
            orc.qmv_rows(fid, W, x, N, K, rows, nthreads=threads)
            b += rows.size * (K // 32) * bb + xb * M * K + 4 * M * rows.size
            f += 2 * M * rows.size * K
        return b, f
    return run, threads, wl["kind"]


def oracle_sample(workload, budget_s):
    """Time the CPU oracle (as it stands) on a bounded row sample of the workload."""
    run, threads, kind = oracle_tasks(workload)
    done_b = done_f = 0
    t_total = 0.0
    frac = 0.001
    full_passes = 0
    # Row samples grow until the budget is spent; a workload the oracle covers
    # whole in less than the budget is then repeated in full passes.
    while True:
        t0 = time.perf_counter()
        b, f = run(frac)
        dt = time.perf_counter() - t0
        done_b += b
        done_f += f
        t_total += dt
        full_passes += frac >= 1.0
        if t_total >= budget_s:
            break
        frac = min(1.0, frac * max(1.5, min(8.0, budget_s / max(dt, 1e-3) / 4)))
    val = done_f / t_total / 1e12 if kind == "prefill" else done_b / t_total / 1e9
    extent = (f"growing evenly spaced row samples, then {full_passes} passes over every row"
              if full_passes else f"evenly spaced row samples (up to {frac:.2%} of the rows)")
    return {"value": round(val, 5), "unit": "TFLOP/s" if kind == "prefill" else "GB/s", "cores": threads,
            "kind": "oracle",
            "sample": f"{extent} of every table of the workload, {t_total:.1f} s of fp64 oracle work, "
                      f"OpenMP over rows"}


def run_reference(args, rank, world):
    """The oracle arm: the CPU fp64 oracle timed on this host's cores."""
    if rank != 0:
        return None
    run, threads, kind = oracle_tasks(args.workload)
    # Per step: the same fixed row sample of every table, sized so that the
    # whole run stays within about two minutes.
    per_step_budget = min(1.0, 120.0 / max(1, args.steps + args.warmup))
    frac = 0.0005
    while True:
        t0 = time.perf_counter()
        run(frac)
        dt = time.perf_counter() - t0
        if dt >= per_step_budget / 2 or frac >= 1.0:
            break
        frac = min(1.0, frac * 2)
    for _ in range(args.warmup):
        run(frac)
    t0 = time.perf_counter()
    b = f = 0
    for _ in range(args.steps):
        bb_, ff_ = run(frac)
        b += bb_
        f += ff_
    dt = time.perf_counter() - t0
    value = f / dt / 1e12 if kind == "prefill" else b / dt / 1e9
    unit = "TFLOP/s" if kind == "prefill" else "GB/s"
    wl = WORKLOADS[args.workload]
    sample = f"{frac:.3%} of the rows of every table per step (evenly spaced), fp64 oracle, OpenMP over rows"
    return {
        "metric": metric_name(args.workload), "value": round(value, 5), "unit": unit, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt * 1e3 / args.steps, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": args.workload, "format": wl["fmt"], "calls_per_step": call_names(args.workload),
                   "values": VALUES, "parallelism": f"replica x{world} (independent problems per GPU)"},
        "impl": "reference",
        "cpu_baseline": {"value": round(value, 5), "unit": unit, "cores": threads, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(value, 5), "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


# ---------------------------------------------------------------------------------
def phase_timeline(workload, out_json=None):
    """Per-phase timeline of one workload's calls replayed back to back from
    CUDA graphs, read from global-timer stamps that a build with
    -DQMV_PHASE_STAMPS records per CTA (a separate library variant; the product
    build has no stamps).  Run under QMV_LIB pointing at that variant.

    Decode calls (per CTA: entry, griddepcontrol.wait returned, activations
    staged, first and last warp done) and prefill calls (entry, set-up done,
    first MMA, last commit, accumulator ready, exit, SM cycles of the MMA span)
    are summarised per call as medians over the CTAs of each launch and then
    over steps (ns)."""
    import ctypes
    import torch
    import weight_quantized_decode_gb300 as q
    L = q.lib()
    prefill = WORKLOADS[workload]["kind"] == "prefill"
    words = 8 if prefill else 7
    fn = L.qmv_prefill_phase_stamps if prefill else L.qmv_phase_stamps
    fn.restype = ctypes.c_int64
    fn.argtypes = [ctypes.c_void_p, ctypes.c_int64]
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    l2 = int(torch.cuda.get_device_properties(dev).L2_cache_size)
    stream = torch.cuda.Stream(dev)
    calls, period = build_calls(workload, q, torch, dev, l2, int(stream.cuda_stream))
    with torch.cuda.stream(stream):
        for c in calls:
            c["call"](0)
    torch.cuda.synchronize()
    runner = StepRunner(torch, stream, calls, period)
    runner.run(2 * period)
    cap = 1 << 18
    buf = (ctypes.c_ulonglong * (cap * words))()
    fn(buf, cap)                      # discard the warm-up records
    ms = runner.time_ms(period)       # one replay of the period graph: every launch once
    n = fn(buf, cap)
    a = np.frombuffer(buf, dtype=np.uint64, count=n * words).reshape(n, words).astype(np.int64)
    # launches in replay order; a call split into token subsets has several
    seqs = sorted(set((a[:, 0] >> 32).tolist()))
    launches = [a[(a[:, 0] >> 32) == s] for s in seqs]
    per_step = len(launches) // period
    names = []
    for c in calls:
        names.append(c["name"])
    if per_step != len(names):     # token-split calls: label the extra launches
        names = [f"launch{i}" for i in range(per_step)]
    rows = {}
    for i, r in enumerate(launches):
        nm = names[i % per_step]
        d = rows.setdefault(nm, {})
        def put(k, v):
            d.setdefault(k, []).append(float(v))
        put("grid", len(r))
        prev_end = launches[i - 1][:, 6 if prefill else 5].max() if i else None
        if prefill:
            e, su, f, lc, acc, ex, clk = (r[:, j] for j in range(1, 8))
            put("setup", np.median(su - e))
            put("to_first_mma", np.median(f - su))
            put("mma_span", np.median(lc - f))
            put("sm_mhz", np.median(clk / np.maximum(lc - f, 1) * 1e3))
            put("acc_ready_after_last_commit", np.median(acc - lc))
            put("epilogue", np.median(ex - acc))
            if prev_end is not None:
                put("call_period", ex.max() - prev_end)
                put("entry_after_prev_end", np.median(e) - prev_end)
        else:
            e, w, st, first, last = (r[:, j] for j in range(1, 6))
            put("wait_minus_entry", np.median(w - e))
            put("stage_activations", np.median(st - w))
            put("main_loop", np.median(last - st))
            put("tail", last.max() - np.median(last))
            if prev_end is not None:
                put("call_period", last.max() - prev_end)
                put("wait_after_prev_end", np.median(w) - prev_end)
    summary = {nm: {k: round(statistics.median(v), 1) for k, v in d.items()} for nm, d in rows.items()}
    out = {"workload": workload, "us_per_step": round(ms / period * 1e3, 2), "steps": period,
           "unit": "ns (medians over the CTAs of a launch, then over steps)", "calls": summary}
    print(json.dumps(out, indent=1))
    if out_json:
        with open(out_json, "w") as f:
            json.dump(out, f, indent=1)
    return out


# ---------------------------------------------------------------------------------
def ncu_case(spec):
    """A handful of eager calls of one table over rotated copies larger than L2
    (a small, bounded program for an Nsight Compute capture).
    spec: q4_0:NxK:M | q8_0:NxK:M | prefill:NxK:M | moe:NxK:SLOTS (pool of 128) |
    swiglu:NxK:M (gate and up tables of N rows each) | q4_0_f32:NxK:M | swiglu_f32:NxK:M
    (fp32 activations) | q2w:NxK:M (plain 2-bit) | q4_0_q81:NxK:M (Q8_1 activations)."""
    import torch
    import weight_quantized_decode_gb300 as q
    kind, shape, M = spec.split(":")
    f32 = kind.endswith("_f32")
    kind = kind[:-4] if f32 else kind
    q81 = kind == "q4_0_q81"
    kind = "q4_0" if q81 else kind
    N, K = (int(v) for v in shape.split("x"))
    M = int(M)
    dev = torch.device("cuda", 0)
    fmt = kind if kind in ("q8_0", "q2w") else "q4_0"
    bb = BLOCK_BYTES[fmt]
    rows = 128 * N if kind == "moe" else (2 * N if kind == "swiglu" else N)
    wbytes = rows * (K // 32) * bb
    copies = max(2, math.ceil(2.5 * 128e6 / wbytes))
    base = torch.from_numpy(synth.weights(fmt, rows, K, synth.seed_for(f"{fmt}_{rows}x{K}"))).to(dev)
    W = base.unsqueeze(0).repeat(copies, 1, 1)
    x = torch.from_numpy(synth.activations(M, K, 1, dtype=np.float32 if f32 else np.float16)).to(dev)
    y = torch.empty((M, N), dtype=torch.float32, device=dev)
    s = torch.cuda.current_stream().cuda_stream
    idx = torch.from_numpy(synth.expert_indices(8, M, 128, 3)).to(dev) if kind == "moe" else None
    for i in range(8):
        Wi = W[i % copies].data_ptr()
        if kind == "moe":
            q.qmv_moe_ptr(Wi, idx[i].data_ptr(), 128, x.data_ptr(), y.data_ptr(), N, K, M, s)
        elif kind == "swiglu":
            Wc = W[i % copies]
            fn = q.qmv_q4_0_swiglu_f32_ptr if f32 else q.qmv_q4_0_swiglu_ptr
            fn(Wc[:N].data_ptr(), Wc[N:].data_ptr(), x.data_ptr(), y.data_ptr(), N, K, M, s)
        else:
            fn = {"q4_0": q.qmv_q4_0_q8_1_ptr if q81 else (q.qmv_q4_0_f32_ptr if f32 else q.qmv_q4_0_ptr),
                  "q8_0": q.qmv_q8_0_ptr,
                  "q2w": q.qmv_q2w_ptr, "prefill": q.qmm_q4_0_prefill_ptr}[kind]
            fn(Wi, x.data_ptr(), y.data_ptr(), N, K, M, s)
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
    ap.add_argument("--no-extra", action="store_true",
                    help="default workload only: skip the Q8_0, multi-expert and prefill sweeps")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-budget", type=float, default=12.0, help="seconds of oracle work for cpu_baseline")
    ap.add_argument("--phase-timeline", default=None, metavar="WORKLOAD",
                    help="build the phase-stamp variant of the library and print the per-phase timeline of "
                         "WORKLOAD's calls back to back (no bench line)")
    ap.add_argument("--ncu-case", default=None,
                    help="FMT:NxK:M -- only run a few eager calls of one shape (for Nsight Compute captures)")
    args = ap.parse_args()
    if args.phase_timeline:
        if not os.environ.get("QMV_LIB"):
            from weight_quantized_decode_gb300 import build as _b
            lib = _b.build(extra=["-DQMV_PHASE_STAMPS"], variant="phase")
            env = dict(os.environ, QMV_LIB=lib)
            sys.exit(subprocess.run([sys.executable] + sys.argv, env=env).returncode)
        phase_timeline(args.phase_timeline)
        return
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
            out["cpu_baseline"] = oracle_sample(args.workload, args.cpu_budget)
        else:
            out["cpu_baseline"] = None
        print(json.dumps(out), flush=True)
    if dist:
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
