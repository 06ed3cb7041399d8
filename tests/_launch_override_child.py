"""Child process for test_launch_overrides: runs decode calls with the launch
shape forced through QMV_GEMV_TUNE (read once per process) and saves the
outputs.  Usage: python -m tests._launch_override_child OUT.npz CASE..."""
import sys

import numpy as np
import torch

import weight_quantized_decode_gb300 as q
from weight_quantized_decode_gb300 import synth


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def main():
    out = sys.argv[1]
    res = {}
    for case in sys.argv[2:]:
        kind, fmt, n, k, m = case.split(":")
        N, K, M = int(n), int(k), int(m)
        if kind == "pfrep":   # the same prefill call repeated: outputs must be bit-identical
            W = dev(synth.weights(fmt, N, K, synth.seed_for(f"ovr_pf_{N}x{K}")))
            x = dev(synth.activations(M, K, synth.seed_for(f"ovr_pf_x_{K}_{M}")))
            fn = {"q4_0": q.qmm_q4_0_prefill, "q8_0": q.qmm_q8_0_prefill}[fmt]
            ys = [fn(W, x) for _ in range(4)]
            torch.cuda.synchronize()
            res[case] = ys[0].cpu().numpy()
            res[case + ":identical"] = np.array([all(torch.equal(ys[0], v) for v in ys[1:])])
        elif kind == "swiglu":
            Wg = synth.q4_0_weights(N, K, synth.seed_for(f"ovr_sg_{N}x{K}"))
            Wu = synth.q4_0_weights(N, K, synth.seed_for(f"ovr_su_{N}x{K}"))
            x = synth.activations(M, K, synth.seed_for(f"ovr_x_{K}_{M}"))
            y = q.qmv_q4_0_swiglu(dev(Wg), dev(Wu), dev(x))
            torch.cuda.synchronize()
            res[case] = y.cpu().numpy()
        elif kind == "q81":
            W = synth.q4_0_weights(N, K, synth.seed_for(f"ovr_q81_{N}x{K}"))
            x = synth.activations(M, K, synth.seed_for(f"ovr_x_{K}_{M}"))
            y = q.qmv_q4_0_q8_1(dev(W), dev(x))
            torch.cuda.synchronize()
            res[case] = y.cpu().numpy()
        elif kind == "gemv":
            W = synth.weights(fmt, N, K, synth.seed_for(f"ovr_{fmt}_{N}x{K}"))
            x = synth.activations(M, K, synth.seed_for(f"ovr_x_{K}_{M}"))
            fn = {"q4_0": q.qmv_q4_0, "q8_0": q.qmv_q8_0, "q2w": q.qmv_q2w}[fmt]
            y = fn(dev(W), dev(x))
            torch.cuda.synchronize()
            res[case] = y.cpu().numpy()
        else:   # moe: M = slots over a pool of 2 * M experts; also every slot as a single call
            E = 2 * M
            pool = synth.q4_0_weights(E * N, K, synth.seed_for(f"ovr_pool_{N}x{K}"))
            idx = synth.expert_indices(1, M, E, 7)[0]
            x = synth.activations(M, K, synth.seed_for(f"ovr_moe_x_{K}"))
            pd, xd = dev(pool), dev(x)
            y = q.qmv_moe(pd, dev(idx), E, xd, N)
            rb = (K // 32) * 18
            singles = [q.qmv_q4_0(pd.view(E * N, rb)[int(e) * N:(int(e) + 1) * N], xd[s:s + 1])[0]
                       for s, e in enumerate(idx)]
            torch.cuda.synchronize()
            res[case] = y.cpu().numpy()
            res[case + ":single"] = torch.stack(singles).cpu().numpy()
            res[case + ":idx"] = idx
    res["status"] = np.array([q.qmv_device_status()])
    np.savez(out, **res)


if __name__ == "__main__":
    main()
