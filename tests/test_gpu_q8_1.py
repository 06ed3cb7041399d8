"""Q4_0 against Q8_1-quantised activations (qmv_q4_0_q8_1) and the Q8_1
quantisation itself (qmv_quantize_q8_1) on the GPU.

The quantisation is integer work decided in fp32: the codes, the fp16 scales'
bits and the code sums must equal the oracle's bit for bit.  The product is then
compared with the oracle's product on the same Q8_1 activations (the north-star
bar, 2e-3 of S per output, and a much tighter 5e-5: the kernel's integer dots are
exact and only the fp32 accumulation of per-block terms rounds), and with the
exact product on the unquantised activations within the quantisation bound
sum_k |w| (d/2 + |q| |fp16(d) - d|) (sm8x-bench, "Our kernel does what llama.cpp
does": activations to Q8_1 once, int8 dot).
"""
import numpy as np
import pytest

from tests import helpers as H
from weight_quantized_decode_gb300 import synth

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

TIGHT = 5e-5


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


def sample_rows(N, k=96, seed=0):
    rng = np.random.default_rng(seed)
    return sorted(set(rng.choice(N, size=min(k, N), replace=False).tolist()) | {0, N - 1, N // 2})


def special_activations(M, K, seed):
    """N(0,1) blocks mixed with blocks that exercise the rounding: all zeros,
    exact integers with max 127 (codes = values), values on ties (x = (k + 1/2) d),
    a single non-zero, large plants and tiny values."""
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((M, K)).astype(np.float16).astype(np.float64)
    xb = x.reshape(M, K // 32, 32)
    for m in range(M):
        for b in range(K // 32):
            kind = (m * 7 + b) % 7
            if kind == 1:
                xb[m, b] = 0.0
            elif kind == 2:
                xb[m, b] = rng.integers(-127, 128, 32); xb[m, b, 0] = 127
            elif kind == 3:
                xb[m, b] = (rng.integers(-120, 120, 32) + 0.5) * 2.0; xb[m, b, 5] = 254.0
            elif kind == 4:
                xb[m, b] = 0.0; xb[m, b, rng.integers(0, 32)] = rng.standard_normal()
            elif kind == 5:
                xb[m, b, rng.integers(0, 32)] = 40000.0 * (1 if rng.random() < 0.5 else -1)
            elif kind == 6:
                xb[m, b] *= 1e-4
    out = x.astype(np.float16)
    assert np.all(np.isfinite(out))
    return out


# -- the quantisation, bit for bit ------------------------------------------------------

@pytest.mark.parametrize("M,K", [(1, 32), (3, 256), (8, 4096), (5, 2560), (2, 14336), (1, 96)])
def test_quantize_bit_exact(cuda_lib, orc, M, K):
    x = special_activations(M, K, M * 1000 + K)
    q, d, s = cuda_lib.qmv_quantize_q8_1(dev(x))
    torch.cuda.synchronize()
    qo, do, so = orc.quantize_q8_1(x)
    assert np.array_equal(q.cpu().numpy(), qo)
    assert np.array_equal(d.cpu().numpy().view(np.uint16), do)
    assert np.array_equal(s.cpu().numpy(), so)


def test_quantize_plain_activations(cuda_lib, orc):
    for plant in (None, "large", "tiny"):
        x = synth.activations(4, 4096, 901, plant=plant)
        q, d, s = cuda_lib.qmv_quantize_q8_1(dev(x))
        torch.cuda.synchronize()
        qo, do, so = orc.quantize_q8_1(x)
        assert np.array_equal(q.cpu().numpy(), qo) and np.array_equal(d.cpu().numpy().view(np.uint16), do)
        assert np.array_equal(s.cpu().numpy(), so)


# -- the product ------------------------------------------------------------------------

def q81_check(q, orc, W, x, N, K, rows=None):
    y = q.qmv_q4_0_q8_1(dev(W), dev(x))
    torch.cuda.synchronize()
    yn = y.cpu().numpy().astype(np.float64)
    qo, do, _ = orc.quantize_q8_1(x)
    yr, S = orc.qmv_q8_1(0, W, qo, do, N, K, rows=rows, nthreads=8)
    got = yn if rows is None else yn[:, rows]
    err = H.normalised_error(got, yr, S)
    assert err <= H.TOL and err <= TIGHT, (N, K, x.shape[0], err)
    return yn


@pytest.mark.parametrize("N,K", [(1, 256), (7, 512), (33, 768), (1000, 2048), (333, 4096), (4133, 1024),
                                 (64, 14336), (130, 2560), (77, 6144)])
def test_q8_1_m1(cuda_lib, orc, N, K):
    q81_check(cuda_lib, orc, synth.q4_0_weights(N, K, 700 + N + K), synth.activations(1, K, 701 + K), N, K)


@pytest.mark.parametrize("M", [2, 3, 4, 5, 6, 7, 8])
def test_q8_1_tokens(cuda_lib, orc, M):
    N, K = 515, 2560
    q81_check(cuda_lib, orc, synth.q4_0_weights(N, K, 710 + M), synth.activations(M, K, 711 + M), N, K)


@pytest.mark.parametrize("M", [1, 8])
def test_q8_1_special_activations(cuda_lib, orc, M):
    N, K = 300, 4096
    y = q81_check(cuda_lib, orc, synth.q4_0_weights(N, K, 720), special_activations(M, K, 721 + M), N, K)
    assert np.all(np.isfinite(y))


@pytest.mark.parametrize("K", [96, 640])
def test_q8_1_generic_kernel(cuda_lib, orc, K):
    N = 45
    q81_check(cuda_lib, orc, synth.q4_0_weights(N, K, 730 + K), special_activations(3, K, 731 + K), N, K)


@pytest.mark.parametrize("N,K,M", [(4096, 4096, 1), (14336, 4096, 1), (128256, 4096, 1), (4096, 14336, 8),
                                   (28672, 4096, 4), (6144, 4096, 2)])
def test_q8_1_full_size_sampled(cuda_lib, orc, N, K, M):
    W = synth.q4_0_weights(N, K, synth.seed_for(f"q4_0_{N}x{K}"))
    x = synth.activations(M, K, synth.seed_for(f"x_{K}_{M}"))
    q81_check(cuda_lib, orc, W, x, N, K, rows=sample_rows(N))


def test_q8_1_within_the_quantisation_bound_of_the_exact_product(cuda_lib, orc):
    N, K, M = 200, 2048, 3
    W = synth.q4_0_weights(N, K, 740)
    x = synth.activations(M, K, 741, plant="large")
    y = cuda_lib.qmv_q4_0_q8_1(dev(W), dev(x))
    torch.cuda.synchronize()
    yn = y.cpu().numpy().astype(np.float64)
    ye, S = orc.qmv(0, W, x, N, K, nthreads=8)
    qo, do, _ = orc.quantize_q8_1(x)
    wabs = np.abs(np.stack([orc.dequant_row(0, W, n, K) for n in range(N)]))
    xf = x.astype(np.float64).reshape(M, K // 32, 32)
    dd = np.abs(xf).max(axis=2) / 127
    dq = do.view(np.float16).astype(np.float64)
    per_x = (dd[:, :, None] / 2 + np.abs(qo.reshape(M, K // 32, 32)) * np.abs(dq - dd)[:, :, None]).reshape(M, K)
    bound = per_x @ wabs.T + TIGHT * S
    assert np.all(np.abs(yn - ye) <= bound)
    # and the quantisation is really there: the result is not the fp16 product
    y16 = cuda_lib.qmv_q4_0(dev(W), dev(x)).cpu().numpy()
    assert not np.array_equal(y16, y.cpu().numpy())


def test_q8_1_unaligned_x_empty_and_sabotage(cuda_lib, orc):
    q = cuda_lib
    N, K = 70, 512
    W = synth.q4_0_weights(N, K, 750)
    x = synth.activations(2, K, 751)
    # x only 2-byte aligned: the generic kernel runs, same contract
    buf = torch.zeros(2 * K + 1, dtype=torch.float16, device="cuda")
    buf[1:].copy_(dev(x).reshape(-1))
    y = torch.empty((2, N), dtype=torch.float32, device="cuda")
    Wd = dev(W)
    q.qmv_q4_0_q8_1_ptr(Wd.data_ptr(), buf.data_ptr() + 2, y.data_ptr(), N, K, 2)
    torch.cuda.synchronize()
    qo, do, _ = orc.quantize_q8_1(x)
    yr, S = orc.qmv_q8_1(0, W, qo, do, N, K)
    assert H.normalised_error(y.cpu().numpy().astype(np.float64), yr, S) <= TIGHT
    # K = 0 gives y = 0; N = 0 and M = 0 do nothing
    y0 = torch.full((2, 5), 7.0, device="cuda")
    q.qmv_q4_0_q8_1_ptr(0, torch.empty(0, dtype=torch.float16, device="cuda").data_ptr(), y0.data_ptr(), 5, 0, 2)
    q.qmv_q4_0_q8_1_ptr(0, 0, 0, 0, 256, 1)
    torch.cuda.synchronize()
    assert torch.all(y0 == 0)
    # corrupted weights fail the check against the intact ones
    N, K = 512, 2048
    W = synth.q4_0_weights(N, K, 752)
    x = synth.activations(2, K, 753)
    yb = q.qmv_q4_0_q8_1(dev(H.sabotage(W, "q4_0")), dev(x)).cpu().numpy().astype(np.float64)
    qo, do, _ = orc.quantize_q8_1(x)
    yr, S = orc.qmv_q8_1(0, W, qo, do, N, K, nthreads=8)
    assert H.normalised_error(yb, yr, S) > 20 * H.TOL


# -- activations quantised once, then the product (qmv_q4_0_q8_1_pre) ---------------------

@pytest.mark.parametrize("N,K,M", [(1000, 2048, 1), (515, 2560, 5), (4096, 4096, 8), (45, 640, 3), (300, 14336, 8),
                                   (77, 96, 2)])
def test_prequantised_equals_fused(cuda_lib, orc, N, K, M):
    q = cuda_lib
    W = dev(synth.q4_0_weights(N, K, 760 + K))
    x = dev(special_activations(M, K, 761 + N))
    qc, qd, qs = q.qmv_quantize_q8_1(x)
    y_pre = q.qmv_q4_0_q8_1_pre(W, qc, qd, qs)
    y_fused = q.qmv_q4_0_q8_1(W, x)
    torch.cuda.synchronize()
    assert torch.equal(y_pre, y_fused)


def test_prequantised_two_tables_share_one_quantisation(cuda_lib, orc):
    q = cuda_lib
    K, M = 4096, 4
    x = synth.activations(M, K, 770)
    qc, qd, qs = q.qmv_quantize_q8_1(dev(x))
    qo, do, _ = orc.quantize_q8_1(x)
    for N, seed in ((6144, 771), (1024, 772)):
        W = synth.q4_0_weights(N, K, seed)
        y = q.qmv_q4_0_q8_1_pre(dev(W), qc, qd, qs)
        torch.cuda.synchronize()
        rows = sample_rows(N)
        yr, S = orc.qmv_q8_1(0, W, qo, do, N, K, rows=rows, nthreads=8)
        assert H.normalised_error(y.cpu().numpy().astype(np.float64)[:, rows], yr, S) <= TIGHT
