"""Which kernel sources a workload's DRAM-traffic record is keyed to (bench.py
source_family / source_sha): a record stays valid only while the sources of
every kernel the workload can launch are unchanged."""
import os
import shutil
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def test_families():
    fam = {w: bench.source_family(w) for w in bench.WORKLOADS}
    assert fam["prefill"] == "prefill"
    # fp16 Q4_0 / Q8_0 calls of four or more tokens may run on the prefill kernel
    assert fam["q8_0"] == "all"
    # one-token, fp32-activation, Q8_1, fused, multi-expert and 2-bit workloads never do
    for w in ("q4_0_m1_sweep", "q4_0_mlp_up", "moe", "q4_0_swiglu", "q4_0_f32in", "q4_0_swiglu_f32in",
              "q4_0_q8_1", "q4_0_q8_1_pre", "q8_0_q8_1", "q8_0_q8_1_pre", "q2w"):
        assert fam[w] == "decode", w


def _hashes(root):
    old = bench.ROOT
    bench.ROOT = root
    try:
        return {f: bench.source_sha(f) for f in ("decode", "prefill", "all")}
    finally:
        bench.ROOT = old


def test_hash_covers_the_right_files(tmp_path):
    src = os.path.join(ROOT, "weight_quantized_decode_gb300", "csrc")
    dst = tmp_path / "weight_quantized_decode_gb300" / "csrc"
    shutil.copytree(src, dst, ignore=shutil.ignore_patterns("*.o", "*.so", "__pycache__"))
    base = _hashes(str(tmp_path))

    def touched(fn):
        p = dst / fn
        orig = p.read_bytes()
        p.write_bytes(orig + b"\n// edit\n")
        try:
            h = _hashes(str(tmp_path))
        finally:
            p.write_bytes(orig)
        return {f: h[f] != base[f] for f in h}

    # the prefill kernel: prefill and all change, decode does not
    assert touched("qmv_prefill.cu") == {"decode": False, "prefill": True, "all": True}
    # a decode kernel: decode and all change, prefill does not
    assert touched("qmv_gemv.cuh") == {"decode": True, "prefill": False, "all": True}
    # shared device code: every family
    assert touched("qmv_common.cuh") == {"decode": True, "prefill": True, "all": True}
    # the probe kernel is in no record's family
    assert touched("qmv_probe.cu") == {"decode": False, "prefill": False, "all": False}
    assert _hashes(str(tmp_path)) == base
