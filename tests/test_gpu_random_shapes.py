"""Seeded random shapes through every decode entry point, against the oracle.

Each case draws a format (Q4_0, Q8_0, plain 2-bit, Q4_0 with fp32 or Q8_1
activations, Q8_0 with Q8_1 activations), N in 1..3000, K a multiple of 32 up to 8192 (mostly multiples of
256, so the streaming kernel runs; the rest take the generic kernel) and M in
1..8.  The launch plan, the lanes-per-row rule, ragged row groups and token
splits are then exercised on shapes no fixed list names.
"""
import numpy as np
import pytest

from tests import helpers as H
from weight_quantized_decode_gb300 import synth

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

KINDS = ["q4_0", "q8_0", "q2w", "q4_0_f32", "q4_0_q8_1"]


def _cases(n=40, seed=20261202, kinds=KINDS):
    rng = np.random.default_rng(seed)
    out = []
    for i in range(n):
        kind = kinds[i % len(kinds)]
        N = int(rng.integers(1, 3001))
        if rng.random() < 0.8:
            K = 256 * int(rng.integers(1, 33))
        else:
            K = 32 * int(rng.integers(1, 97))
        M = int(rng.integers(1, 9))
        out.append((kind, N, K, M, int(rng.integers(0, 2 ** 31))))
    return out


@pytest.fixture(scope="module", autouse=True)
def cuda_lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import weight_quantized_decode_gb300 as q
    q.lib()
    yield q
    torch.cuda.synchronize()


@pytest.mark.parametrize("kind,N,K,M,seed", _cases() + _cases(8, 20261203, ["q8_0_q8_1"]), ids=lambda v: str(v))
def test_random_shape(cuda_lib, orc, kind, N, K, M, seed):
    q = cuda_lib
    fmt = "q4_0" if kind.startswith("q4_0") else ("q8_0" if kind.startswith("q8_0") else kind)
    W = synth.weights(fmt, N, K, seed)
    x = synth.activations(M, K, seed + 1, dtype=np.float32 if kind == "q4_0_f32" else np.float16)
    Wd = torch.from_numpy(W).cuda()
    xd = torch.from_numpy(x).cuda()
    fn = {"q4_0": q.qmv_q4_0, "q8_0": q.qmv_q8_0, "q2w": q.qmv_q2w, "q4_0_f32": q.qmv_q4_0_f32,
          "q4_0_q8_1": q.qmv_q4_0_q8_1, "q8_0_q8_1": q.qmv_q8_0_q8_1}[kind]
    y = fn(Wd, xd)
    torch.cuda.synchronize()
    yn = y.cpu().numpy().astype(np.float64)
    if kind.endswith("_q8_1"):
        qo, do, _ = orc.quantize_q8_1(x)
        y_ref, S = orc.qmv_q8_1(H.FMT[fmt], W, qo, do, N, K, nthreads=8)
        tol = 5e-5
    else:
        y_ref, S = orc.qmv(H.FMT[fmt], W, x, N, K, nthreads=8)
        tol = H.TOL
    err = H.normalised_error(yn, y_ref, S)
    assert err <= tol, (kind, N, K, M, err)
    assert q.qmv_device_status() == 0
