"""Dense blocks of the largest fp16 activations against the extreme codes.

The decode kernels sum eight products in each half of a half2 chain before the
chain goes to fp32; the weights are pre-scaled so that no such partial sum can
overflow fp16 for any finite activation (volta-kernel-bakeoff, "A few tokens at
once": the centred code is divided by 64 where a lane sums two words).  The
pages' own "large" plant (1 % of the activations at 20000..60000) almost never
puts eight large values into one chain, so these cases fill whole blocks with
+-65504 and +-40000, signed to agree with rows whose codes are all at one
extreme (every product of a chain then has the same sign), and also put one
such block among N(0,1) activations.  Every entry point that takes fp16 or fp32
activations is checked, on the streaming kernel (K = 4096) and on the generic
kernel (K = 640), at one token and at eight: every output must be finite and
within the per-output bound of the fp64 oracle.
"""
import numpy as np
import pytest

from tests import helpers as H
from weight_quantized_decode_gb300 import synth

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

BIG = 65504.0          # largest finite fp16
MID = 40000.0


@pytest.fixture(scope="module", autouse=True)
def cuda_lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import weight_quantized_decode_gb300 as q
    q.lib()
    yield q
    torch.cuda.synchronize()


@pytest.fixture(autouse=True)
def clean_status(cuda_lib):
    cuda_lib.qmv_device_status()
    yield
    assert cuda_lib.qmv_device_status() == 0


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


# Per format: code bytes that put every weight of a block at one extreme.
EXTREME_BYTES = {
    "q4_0": [0x00, 0xFF],            # all codes 0 (w = -8d) / all codes 15 (w = 7d)
    "q8_0": [0x7F, 0x81, 0x80],      # all +127 / all -127 / all -128
    "q2w": [0x00, 0xFF],             # all codes 0 (w = -2d) / all codes 3 (w = d)
}


def edge_table(fmt, N, K, seed):
    """Seeded table whose rows cycle through: each extreme code byte with the
    generated (positive) scales, the first extreme again with negated scales,
    and one row of random codes."""
    W = synth.weights(fmt, N, K, seed).copy()
    bb = H.BLOCK_BYTES[fmt]
    Wv = W.reshape(N, K // 32, bb)
    kinds = EXTREME_BYTES[fmt]
    period = len(kinds) + 2
    for r in range(N):
        k = r % period
        if k < len(kinds):
            Wv[r, :, 2:] = kinds[k]
        elif k == len(kinds):
            Wv[r, :, 2:] = kinds[0]
            Wv[r, :, 1] ^= 0x80        # sign bit of the little-endian fp16 scale
    return W


def edge_tokens(K, dtype=np.float16):
    """Eight tokens: dense +-65504 and +-40000, alternating-sign blocks, and
    single extreme blocks (aligned to a 32-block, hence to a chain) among
    N(0,1) values.  With fp32 activations one token holds 65519, which fp16
    rounds to 65504."""
    base = synth.activations(8, K, seed=77).astype(np.float64)
    x = np.empty((8, K))
    x[0] = BIG
    x[1] = -BIG
    x[2] = MID
    x[3] = -MID
    blk = np.arange(K) // 32
    x[4] = np.where(blk % 2 == 0, BIG, -BIG)
    x[5] = base[5]
    x[5][32:64] = BIG
    x[6] = base[6]
    x[6][64:96] = -BIG
    x[6][160:192] = MID
    x[7] = base[7]
    x[7][K - 32:] = -MID
    if dtype == np.float32:
        x[2][::7] = 65519.0
    return x.astype(dtype)


def assert_close(y, y_ref, S, what):
    assert np.all(np.isfinite(y)), f"{what}: non-finite outputs"
    err = H.normalised_error(y, y_ref, S)
    assert err <= H.TOL, (what, err)


def token_sets(M, K, dtype=np.float16):
    xs = edge_tokens(K, dtype)
    if M == 8:
        return [xs]
    return [xs[t:t + 1] for t in range(8)]


KS = [4096, 640]   # streaming kernel, generic kernel


@pytest.mark.parametrize("fmt", ["q4_0", "q8_0", "q2w"])
@pytest.mark.parametrize("K", KS)
@pytest.mark.parametrize("M", [1, 8])
def test_plain_dense_extremes(cuda_lib, orc, fmt, K, M):
    q = cuda_lib
    N = 67
    W = edge_table(fmt, N, K, seed=500 + K)
    fn = {"q4_0": q.qmv_q4_0, "q8_0": q.qmv_q8_0, "q2w": q.qmv_q2w}[fmt]
    Wd = dev(W)
    for x in token_sets(M, K):
        y = fn(Wd, dev(x))
        torch.cuda.synchronize()
        y_ref, S = orc.qmv(H.FMT[fmt], W, x, N, K, nthreads=8)
        assert_close(y.cpu().numpy().astype(np.float64), y_ref, S, (fmt, K, x.shape[0]))


@pytest.mark.parametrize("K", KS)
@pytest.mark.parametrize("M", [1, 8])
def test_fp32_activations_dense_extremes(cuda_lib, orc, K, M):
    q = cuda_lib
    N = 67
    W = edge_table("q4_0", N, K, seed=510 + K)
    Wd = dev(W)
    for x in token_sets(M, K, np.float32):
        y = q.qmv_q4_0_f32(Wd, dev(x))
        torch.cuda.synchronize()
        y_ref, S = orc.qmv(0, W, x, N, K, nthreads=8)
        assert_close(y.cpu().numpy().astype(np.float64), y_ref, S, ("f32", K, x.shape[0]))


@pytest.mark.parametrize("K", KS)
@pytest.mark.parametrize("M", [1, 8])
@pytest.mark.parametrize("xin", ["f16", "f32"])
def test_swiglu_dense_extremes(cuda_lib, orc, K, M, xin):
    q = cuda_lib
    N = 45
    Wg, Wu = edge_table("q4_0", N, K, seed=520 + K), edge_table("q4_0", N, K, seed=530 + K)
    Wgd, Wud = dev(Wg), dev(Wu)
    fn = q.qmv_q4_0_swiglu if xin == "f16" else q.qmv_q4_0_swiglu_f32
    for x in token_sets(M, K, np.float16 if xin == "f16" else np.float32):
        y = fn(Wgd, Wud, dev(x))
        torch.cuda.synchronize()
        yn = y.cpu().numpy().astype(np.float64)
        assert np.all(np.isfinite(yn)), ("swiglu", xin, K)
        ref = orc.swiglu(0, Wg, Wu, x, N, K, nthreads=8)
        err = H.swiglu_normalised_error(yn, ref)
        assert err <= H.TOL, ("swiglu", xin, K, x.shape[0], err)


@pytest.mark.parametrize("K", KS)
def test_multi_expert_dense_extremes(cuda_lib, orc, K):
    q = cuda_lib
    E, N, slots = 6, 40, 8
    pool = edge_table("q4_0", E * N, K, seed=540 + K)
    # slot s takes expert s % E: experts start at rows 0, 40, 80, ... so their
    # first rows cycle through the extreme kinds
    idx = (np.arange(slots) % E).astype(np.int32)
    x = edge_tokens(K)
    y = q.qmv_moe(dev(pool), dev(idx), E, dev(x), N)
    torch.cuda.synchronize()
    y_ref, S = orc.moe(0, pool, idx, E, x, N, K, nthreads=8)
    assert_close(y.cpu().numpy().astype(np.float64), y_ref, S, ("moe", K))


def test_tiny_activations_keep_their_precision(cuda_lib, orc):
    """The pre-scale moves small products toward fp16's subnormal range; the
    pages' tiny plant (activations x 1e-4) at the streaming kernel's shortest
    rows (K = 256, where the fewest products average out the rounding) must
    still meet the bound, for both formats the pre-scale changed."""
    q = cuda_lib
    N, K = 999, 256
    for fmt, fn in (("q4_0", q.qmv_q4_0), ("q8_0", q.qmv_q8_0)):
        W = synth.weights(fmt, N, K, seed=550)
        x = synth.activations(8, K, seed=551, plant="tiny")
        y = fn(dev(W), dev(x))
        torch.cuda.synchronize()
        y_ref, S = orc.qmv(H.FMT[fmt], W, x, N, K, nthreads=8)
        err = H.normalised_error(y.cpu().numpy().astype(np.float64), y_ref, S)
        assert err <= H.TOL, (fmt, err)
