"""Child process for test_gpu_give_up: QMV_TEST_SKIP_COPY (read once per
process) arms one launch of the decode or prefill kernel to skip a copy whose
bytes a barrier expects.  Runs that call on a sentinel-filled output, reads the
status word, then repeats the call normally and reads the status again.
Usage: python -m tests._give_up_child OUT.npz decode|prefill"""
import sys

import numpy as np
import torch

import weight_quantized_decode_gb300 as q
from weight_quantized_decode_gb300 import synth

SENTINEL = 1234.5


def main():
    out, kind = sys.argv[1], sys.argv[2]
    if kind == "decode":
        N, K, M = 4096, 4096, 1
        fn = q.qmv_q4_0
    else:
        N, K, M = 256, 512, 64
        fn = q.qmm_q4_0_prefill
    W = torch.from_numpy(synth.q4_0_weights(N, K, synth.seed_for(f"giveup_{kind}"))).cuda()
    x = torch.from_numpy(synth.activations(M, K, synth.seed_for(f"giveup_x_{kind}"))).cuda()
    y1 = torch.full((M, N), SENTINEL, dtype=torch.float32, device="cuda")
    fn(W, x, y1)
    torch.cuda.synchronize()
    s1 = q.qmv_device_status()
    y2 = torch.full((M, N), SENTINEL, dtype=torch.float32, device="cuda")
    fn(W, x, y2)
    torch.cuda.synchronize()
    s2 = q.qmv_device_status()
    np.savez(out, y1=y1.cpu().numpy(), y2=y2.cpu().numpy(), s1=np.array([s1]), s2=np.array([s2]),
             N=np.array([N]), K=np.array([K]), M=np.array([M]))


if __name__ == "__main__":
    main()
