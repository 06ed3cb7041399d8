"""The N > 1 path of bench.py on the CPU with the gloo backend: cross-rank
timing (max over ranks, whole-job throughput over all ranks' work) and the
reference arm under torchrun (rank 0 alone runs and prints one line)."""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    ms = bench.cross_rank_max_ms(dist, 10.0 + 5.0 * rank, "cpu")
    rate = bench.whole_job_rate(100.0, 2, world, ms)
    dist.barrier()
    dist.destroy_process_group()
    with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
        json.dump({"ms": ms, "rate": rate}, f)


def test_cross_rank_timing_gloo(tmp_path):
    torch = pytest.importorskip("torch")
    import torch.multiprocessing as mp
    world = 2
    mp.start_processes(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True,
                       start_method="spawn")
    got = [json.load(open(tmp_path / f"rank{r}.json")) for r in range(world)]
    for g in got:
        assert g["ms"] == 15.0                      # the slowest rank's time, on every rank
        assert g["rate"] == pytest.approx(100.0 * 2 * world / 0.015)   # all ranks' units / that time


def test_single_process_timing_is_local():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.cross_rank_max_ms(None, 12.5, "cpu") == 12.5
    assert bench.whole_job_rate(10.0, 4, 1, 2.0) == pytest.approx(20000.0)


def test_reference_arm_under_torchrun():
    pytest.importorskip("torch")
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()),
           "bench.py", "--impl", "reference", "--workload", "q4_0_mlp_up", "--steps", "1", "--warmup", "3"]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600,
                       env=dict(os.environ, OMP_NUM_THREADS="2"))
    assert r.returncode == 0, r.stderr[-3000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout           # rank 0 alone prints
    out = json.loads(lines[0])
    assert out["impl"] == "reference" and out["n_gpus"] == 2
    assert out["cpu_baseline"]["kind"] == "oracle"
    assert out["e2e"]["h2d_bytes_per_step"] == 0 and out["e2e"]["d2h_bytes_per_step"] == 0
    assert out["value"] > 0
    # the same workload description as the GPU arm's line
    assert out["config"]["workload"] == "q4_0_mlp_up" and out["config"]["calls_per_step"] == ["6144x2048/M1"]
