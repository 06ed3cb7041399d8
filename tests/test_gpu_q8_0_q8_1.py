"""Q8_0 weights against activations quantised to Q8_1 (qmv_q8_0_q8_1, and
qmv_q8_0_q8_1_pre on activations quantised beforehand), compared through the C
ABI with the CPU fp64 oracle's product on the same Q8_1 activations."""
import numpy as np
import pytest

from tests import helpers as H
from weight_quantized_decode_gb300 import synth

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

TIGHT = 5e-5     # against the oracle's Q8_1 product: only the fp32 sums of the block terms differ


@pytest.fixture(scope="module", autouse=True)
def cuda_lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import weight_quantized_decode_gb300 as q
    q.lib()
    return q


@pytest.fixture(autouse=True)
def clean_status(cuda_lib):
    cuda_lib.qmv_device_status()
    yield
    assert cuda_lib.qmv_device_status() == 0


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def sample_rows(N, k=96, seed=0):
    rng = np.random.default_rng(seed)
    return np.unique(np.concatenate([[0, N - 1], rng.integers(0, N, size=k)])).astype(np.int64)


def check(q, orc, W, x, N, K, rows=None):
    y = q.qmv_q8_0_q8_1(dev(W), dev(x))
    torch.cuda.synchronize()
    yn = y.cpu().numpy().astype(np.float64)
    qo, do, _ = orc.quantize_q8_1(x)
    yr, S = orc.qmv_q8_1(1, W, qo, do, N, K, rows=rows, nthreads=8)
    got = yn if rows is None else yn[:, rows]
    err = H.normalised_error(got, yr, S)
    assert err <= H.TOL and err <= TIGHT, (N, K, x.shape[0], err)
    return yn


@pytest.mark.parametrize("N,K", [(1, 256), (7, 512), (33, 768), (1000, 2048), (333, 4096), (4133, 1024),
                                 (64, 14336), (130, 2560), (77, 6144)])
def test_m1(cuda_lib, orc, N, K):
    check(cuda_lib, orc, synth.q8_0_weights(N, K, 900 + N + K), synth.activations(1, K, 901 + K), N, K)


@pytest.mark.parametrize("M", [2, 3, 4, 5, 6, 7, 8])
def test_tokens(cuda_lib, orc, M):
    N, K = 515, 2560
    check(cuda_lib, orc, synth.q8_0_weights(N, K, 910 + M), synth.activations(M, K, 911 + M), N, K)


@pytest.mark.parametrize("M", [1, 8])
def test_planted_activations(cuda_lib, orc, M):
    N, K = 300, 4096
    for plant in ("large", "tiny"):
        y = check(cuda_lib, orc, synth.q8_0_weights(N, K, 920), synth.activations(M, K, 921 + M, plant=plant), N, K)
        assert np.all(np.isfinite(y))


@pytest.mark.parametrize("K", [96, 640])
def test_generic_kernel(cuda_lib, orc, K):
    N = 45
    check(cuda_lib, orc, synth.q8_0_weights(N, K, 930 + K), synth.activations(3, K, 931 + K), N, K)


@pytest.mark.parametrize("K,M", [(2560, 1), (4096, 8), (96, 2)])
def test_integer_case_is_exact(cuda_lib, K, M):
    # d = 1 and activations whose every block holds +-127: the Q8_1 codes are
    # the activations themselves with scale 1, so y is the integer matmul of
    # the codes, exactly (every partial sum is an integer below 2^24)
    rng = np.random.default_rng(940 + K + M)
    N = 131
    codes = rng.integers(-128, 128, size=(N, K))
    W = H.encode_q8_0(codes, np.full((N, K // 32), 0x3C00, dtype=np.uint16))
    x = rng.integers(-127, 128, size=(M, K))
    x.reshape(M, K // 32, 32)[:, :, 7] = 127
    y = cuda_lib.qmv_q8_0_q8_1(dev(W), dev(x.astype(np.float16)))
    torch.cuda.synchronize()
    assert np.array_equal(y.cpu().numpy().astype(np.float64), x.astype(np.float64) @ codes.astype(np.float64).T)


@pytest.mark.parametrize("N,K,M", [(12288, 2560, 1), (2560, 6144, 8), (8192, 2048, 4), (128256, 4096, 1),
                                   (4096, 14336, 8)])
def test_full_size_sampled(cuda_lib, orc, N, K, M):
    W = synth.q8_0_weights(N, K, synth.seed_for(f"q8_0_{N}x{K}"))
    x = synth.activations(M, K, synth.seed_for(f"x_{K}_{M}"))
    check(cuda_lib, orc, W, x, N, K, rows=sample_rows(N))


def test_within_the_quantisation_bound_of_the_exact_product(cuda_lib, orc):
    N, K, M = 200, 2048, 3
    W = synth.q8_0_weights(N, K, 950)
    x = synth.activations(M, K, 951, plant="large")
    y = cuda_lib.qmv_q8_0_q8_1(dev(W), dev(x))
    torch.cuda.synchronize()
    yn = y.cpu().numpy().astype(np.float64)
    ye, S = orc.qmv(1, W, x, N, K, nthreads=8)
    qo, do, _ = orc.quantize_q8_1(x)
    wabs = np.abs(np.stack([orc.dequant_row(1, W, n, K) for n in range(N)]))
    xf = x.astype(np.float64).reshape(M, K // 32, 32)
    dd = np.abs(xf).max(axis=2) / 127
    dq = do.view(np.float16).astype(np.float64)
    per_x = (dd[:, :, None] / 2 + np.abs(qo.reshape(M, K // 32, 32)) * np.abs(dq - dd)[:, :, None]).reshape(M, K)
    assert np.all(np.abs(yn - ye) <= per_x @ wabs.T + TIGHT * S)
    y16 = cuda_lib.qmv_q8_0(dev(W), dev(x)).cpu().numpy()
    assert not np.array_equal(y16, y.cpu().numpy())


def test_unaligned_x_empty_and_sabotage(cuda_lib, orc):
    q = cuda_lib
    N, K = 70, 512
    W = synth.q8_0_weights(N, K, 960)
    x = synth.activations(2, K, 961)
    # x only 2-byte aligned: the generic kernel runs, same contract
    buf = torch.zeros(2 * K + 1, dtype=torch.float16, device="cuda")
    buf[1:].copy_(dev(x).reshape(-1))
    y = torch.empty((2, N), dtype=torch.float32, device="cuda")
    Wd = dev(W)
    q.qmv_q8_0_q8_1_ptr(Wd.data_ptr(), buf.data_ptr() + 2, y.data_ptr(), N, K, 2)
    torch.cuda.synchronize()
    qo, do, _ = orc.quantize_q8_1(x)
    yr, S = orc.qmv_q8_1(1, W, qo, do, N, K)
    assert H.normalised_error(y.cpu().numpy().astype(np.float64), yr, S) <= TIGHT
    # K = 0 gives y = 0; N = 0 and M = 0 do nothing
    y0 = torch.full((2, 5), 7.0, device="cuda")
    q.qmv_q8_0_q8_1_ptr(0, torch.empty(0, dtype=torch.float16, device="cuda").data_ptr(), y0.data_ptr(), 5, 0, 2)
    q.qmv_q8_0_q8_1_ptr(0, 0, 0, 0, 256, 1)
    torch.cuda.synchronize()
    assert torch.all(y0 == 0)
    # corrupted weights fail the check against the intact ones
    N, K = 512, 2048
    W = synth.q8_0_weights(N, K, 962)
    x = synth.activations(2, K, 963)
    yb = q.qmv_q8_0_q8_1(dev(H.sabotage(W, "q8_0")), dev(x)).cpu().numpy().astype(np.float64)
    qo, do, _ = orc.quantize_q8_1(x)
    yr, S = orc.qmv_q8_1(1, W, qo, do, N, K, nthreads=8)
    assert H.normalised_error(yb, yr, S) > 20 * H.TOL


@pytest.mark.parametrize("N,K,M", [(1000, 2048, 1), (515, 2560, 5), (4096, 4096, 8), (45, 640, 3), (300, 14336, 8),
                                   (77, 96, 2)])
def test_prequantised_equals_fused(cuda_lib, N, K, M):
    q = cuda_lib
    W = dev(synth.q8_0_weights(N, K, 970 + K))
    x = dev(synth.activations(M, K, 971 + N, plant="large"))
    qc, qd, _ = q.qmv_quantize_q8_1(x)
    y_pre = q.qmv_q8_0_q8_1_pre(W, qc, qd)
    y_fused = q.qmv_q8_0_q8_1(W, x)
    torch.cuda.synchronize()
    assert torch.equal(y_pre, y_fused)
