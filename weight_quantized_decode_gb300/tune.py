"""Launch-shape sweep for the streaming decode kernel.

For every candidate launch shape (warps per CTA, ring stages, lanes per row,
passes per stage, CTAs per SM) a child process sets QMV_GEMV_TUNE, times each
table with a CUDA graph of back-to-back calls over weight copies larger than 4x
the L2, and reports us/call.  The parent prints the fastest shape per table.

    python -m weight_quantized_decode_gb300.tune --fmt q4_0 --shapes 4096x4096,128256x4096 --M 1
"""
from __future__ import annotations

import argparse
import itertools
import json
import math
import os
import subprocess
import sys


def child(fmt, shapes, Ms, reps):
    import torch

    import weight_quantized_decode_gb300 as q
    dev = torch.device("cuda", 0)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    bb = 18 if fmt == "q4_0" else 34
    fn = q.qmv_q4_0_ptr if fmt == "q4_0" else q.qmv_q8_0_ptr
    stream = torch.cuda.Stream(dev)
    sh = int(stream.cuda_stream)
    out = []
    for (N, K) in shapes:
        rb = (K // 32) * bb
        copies = max(2, math.ceil(4 * l2 / (N * rb)))
        W = torch.randint(0, 256, (copies, N, K // 32, bb), dtype=torch.uint8, device=dev)
        W[..., 0] = 0x00
        W[..., 1] = 0x20            # d = 2^-7, a valid fp16 scale
        W = W.view(copies, N, rb)
        for M in Ms:
            x = torch.randn((M, K), device=dev).half()
            y = torch.empty((M, N), device=dev)
            R = max(reps, 2 * copies)
            with torch.cuda.stream(stream):
                fn(W[0].data_ptr(), x.data_ptr(), y.data_ptr(), N, K, M, sh)
            torch.cuda.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.stream(stream):
                with torch.cuda.graph(g, stream=stream):
                    for i in range(R):
                        fn(W[i % copies].data_ptr(), x.data_ptr(), y.data_ptr(), N, K, M, sh)
            best = None
            for _ in range(5):
                a = torch.cuda.Event(enable_timing=True)
                b = torch.cuda.Event(enable_timing=True)
                with torch.cuda.stream(stream):
                    a.record(stream)
                    g.replay()
                    b.record(stream)
                torch.cuda.synchronize()
                t = a.elapsed_time(b) * 1e3 / R
                best = t if best is None else min(best, t)
            nbytes = N * rb + 2 * M * K + 4 * M * N
            out.append({"N": N, "K": K, "M": M, "us": round(best, 3), "GBps": round(nbytes / best / 1e3, 1)})
        del W
        torch.cuda.empty_cache()
    print(json.dumps(out))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--fmt", default="q4_0")
    ap.add_argument("--shapes", default="4096x4096,6144x4096,4096x14336,14336x4096,28672x4096,128256x4096")
    ap.add_argument("--M", default="1")
    ap.add_argument("--reps", type=int, default=64)
    ap.add_argument("--warps", default="4,8,16")
    ap.add_argument("--stages", default="2,3,4,6")
    ap.add_argument("--G", default="0")
    ap.add_argument("--SP", default="1")
    ap.add_argument("--ctas", default="1")
    ap.add_argument("--share", default="1")
    ap.add_argument("--child", action="store_true")
    ap.add_argument("--out", default=None)
    args = ap.parse_args()
    shapes = [tuple(int(v) for v in s.split("x")) for s in args.shapes.split(",")]
    Ms = [int(v) for v in args.M.split(",")]
    if args.child:
        child(args.fmt, shapes, Ms, args.reps)
        return
    grid = itertools.product(*[[int(v) for v in getattr(args, k).split(",")]
                               for k in ("warps", "stages", "G", "SP", "ctas", "share")])
    results = []
    for warps, stages, G, SP, ctas, share in grid:
        cfg = f"warps={warps},stages={stages},G={G},SP={SP},ctas={ctas},share={share}"
        env = dict(os.environ, QMV_GEMV_TUNE=cfg)
        r = subprocess.run([sys.executable, "-m", "weight_quantized_decode_gb300.tune", "--child",
                            "--fmt", args.fmt, "--shapes", args.shapes, "--M", args.M, "--reps", str(args.reps)],
                           env=env, capture_output=True, text=True, timeout=600)
        if r.returncode != 0:
            print(f"{cfg}: failed\n{r.stderr[-800:]}", flush=True)
            continue
        rows = json.loads(r.stdout.strip().splitlines()[-1])
        for row in rows:
            row["cfg"] = cfg
        results += rows
        print(cfg, " ".join(f"{row['N']}x{row['K']}/M{row['M']}:{row['us']}us" for row in rows), flush=True)
    best = {}
    for row in results:
        key = (row["N"], row["K"], row["M"])
        if key not in best or row["us"] < best[key]["us"]:
            best[key] = row
    print("BEST")
    for key, row in sorted(best.items()):
        print(json.dumps(row))
    if args.out:
        json.dump({"all": results, "best": list(best.values())}, open(args.out, "w"), indent=1)


if __name__ == "__main__":
    main()
