"""fp32-activation entry points (qmv_q4_0_f32, qmv_q4_0_swiglu_f32) on the GPU.

Two bars.  Against the fp64 oracle on the fp32 values themselves: the same
per-output tolerance as the fp16 calls (max |y - y_ref| / (S + 1e-6) <= 2e-3;
rounding x to fp16 adds at most 2^-11 of each |x w| to the error).  Against
the fp16 calls on the activations rounded to fp16 (nearest even, as
torch.Tensor.half rounds): bit-identical, since the kernels round while
staging and then run the fp16 product unchanged (the bakeoff's fp32in kernels
take fp32 in -- volta-kernel-bakeoff, "Results (one token, microseconds, lower
is better)" and "A few tokens at once").
"""
import numpy as np
import pytest

from tests import helpers as H
from weight_quantized_decode_gb300 import synth

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


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


def x32(M, K, seed, plant=None):
    return synth.activations(M, K, seed, plant=plant, dtype=np.float32)


def sample_rows(N, k=96, seed=0):
    rng = np.random.default_rng(seed)
    return sorted(set(rng.choice(N, size=min(k, N), replace=False).tolist()) | {0, N - 1, N // 2})


def gemv_check(q, W, x, N, K, orc, rows=None):
    y = q.qmv_q4_0_f32(dev(W), dev(x))
    torch.cuda.synchronize()
    yn = y.cpu().numpy().astype(np.float64)
    if rows is None:
        y_ref, S = orc.qmv(0, W, x, N, K, nthreads=8)
        err = H.normalised_error(yn, y_ref, S)
    else:
        y_ref, S = orc.qmv_rows(0, W, x, N, K, rows, nthreads=8)
        err = H.normalised_error(yn[:, rows], y_ref, S)
    assert err <= H.TOL, (N, K, x.shape[0], err)
    return y


def swiglu_check(q, Wg, Wu, x, N, K, orc, rows=None):
    y = q.qmv_q4_0_swiglu_f32(dev(Wg), dev(Wu), dev(x))
    torch.cuda.synchronize()
    yn = y.cpu().numpy().astype(np.float64)
    ref = orc.swiglu(0, Wg, Wu, x, N, K, rows=rows, nthreads=8)
    err = H.swiglu_normalised_error(yn if rows is None else yn[:, rows], ref)
    assert err <= H.TOL, (N, K, x.shape[0], err)
    return y


# -- against the oracle on the fp32 values ----------------------------------------------

@pytest.mark.parametrize("N,K", [(1, 256), (7, 512), (33, 768), (1000, 2048), (300, 4096), (64, 14336),
                                 (130, 2560), (4133, 1024)])
def test_f32_m1(cuda_lib, orc, N, K):
    gemv_check(cuda_lib, synth.q4_0_weights(N, K, 500 + N + K), x32(1, K, 501 + K), N, K, orc)


@pytest.mark.parametrize("M", [2, 3, 4, 5, 8])
def test_f32_tokens(cuda_lib, orc, M):
    N, K = 515, 2560
    gemv_check(cuda_lib, synth.q4_0_weights(N, K, 510 + M), x32(M, K, 511 + M), N, K, orc)


@pytest.mark.parametrize("plant", ["large", "tiny"])
@pytest.mark.parametrize("M", [1, 8])
def test_f32_planted(cuda_lib, orc, plant, M):
    N, K = 300, 4096
    y = gemv_check(cuda_lib, synth.q4_0_weights(N, K, 520), x32(M, K, 521, plant), N, K, orc)
    assert torch.isfinite(y).all()


@pytest.mark.parametrize("K", [96, 640])
def test_f32_generic_kernel(cuda_lib, orc, K):
    N = 45
    gemv_check(cuda_lib, synth.q4_0_weights(N, K, 530 + K), x32(3, K, 531), N, K, orc)


@pytest.mark.parametrize("N,K,M", [(4096, 4096, 1), (14336, 4096, 1), (128256, 4096, 1), (4096, 14336, 8),
                                   (12288, 2560, 4), (640, 2560, 1), (2048, 512, 8)])
def test_f32_full_size_sampled(cuda_lib, orc, N, K, M):
    W = synth.q4_0_weights(N, K, synth.seed_for(f"q4_0_{N}x{K}"))
    gemv_check(cuda_lib, W, x32(M, K, synth.seed_for(f"f32_x_{K}_{M}")), N, K, orc, rows=sample_rows(N))


@pytest.mark.parametrize("N,K,M", [(333, 4096, 1), (515, 2560, 5), (45, 640, 3), (6144, 2048, 8)])
def test_f32_swiglu(cuda_lib, orc, N, K, M):
    Wg, Wu = synth.q4_0_weights(N, K, 540 + N), synth.q4_0_weights(N, K, 541 + N)
    swiglu_check(cuda_lib, Wg, Wu, x32(M, K, 542 + M), N, K, orc, rows=None if N < 1000 else sample_rows(N))


@pytest.mark.parametrize("M", [1, 8])
def test_f32_swiglu_full_size_sampled(cuda_lib, orc, M):
    N, K = 14336, 4096
    Wg = synth.q4_0_weights(N, K, synth.seed_for(f"swiglu_{N}x{K}"))
    Wu = synth.q4_0_weights(N, K, synth.seed_for(f"swiglu_{N}x{K}") + 7919)
    swiglu_check(cuda_lib, Wg, Wu, x32(M, K, synth.seed_for(f"f32_swiglu_x_{K}_{M}")), N, K, orc,
                 rows=sample_rows(N))


# -- bit-identity with the fp16 calls on x rounded to fp16 --------------------------------

@pytest.mark.parametrize("N,K,M", [(1000, 2048, 1), (515, 2560, 3), (4096, 4096, 8), (45, 640, 2), (7, 96, 1)])
def test_f32_equals_fp16_call_on_rounded_x(cuda_lib, orc, N, K, M):
    q = cuda_lib
    W_host = synth.q4_0_weights(N, K, 550 + K)
    x_host = x32(M, K, 551 + M, plant="large")
    W = dev(W_host)
    x = dev(x_host)
    y32 = q.qmv_q4_0_f32(W, x)
    y16 = q.qmv_q4_0(W, x.half())
    Wu = dev(synth.q4_0_weights(N, K, 552 + K))
    s32 = q.qmv_q4_0_swiglu_f32(W, Wu, x)
    s16 = q.qmv_q4_0_swiglu(W, Wu, x.half())
    torch.cuda.synchronize()
    assert torch.equal(s32, s16)
    if M >= 4 and K % 256 == 0:
        # qmv_q4_0 may take the tensor cores at several tokens (the header's
        # rule); the fp32 call always streams: both within the bound of the
        # exact product on the rounded x
        y_ref, S = orc.qmv(0, W_host, x_host.astype(np.float16), N, K, nthreads=8)
        assert H.normalised_error(y32.cpu().numpy(), y_ref, S) <= H.TOL
        assert H.normalised_error(y16.cpu().numpy(), y_ref, S) <= H.TOL
    else:
        assert torch.equal(y32, y16)


# -- edges ----------------------------------------------------------------------------

def test_f32_alignment_and_empty(cuda_lib, orc):
    q = cuda_lib
    N, K = 70, 512
    W = synth.q4_0_weights(N, K, 560)
    x = x32(2, K, 561)
    # fp32 x only 4-byte aligned: the generic kernel runs, same contract
    buf = torch.zeros(2 * K + 1, dtype=torch.float32, device="cuda")
    buf[1:].copy_(dev(x).reshape(-1))
    y = torch.empty((2, N), dtype=torch.float32, device="cuda")
    Wd = dev(W)
    q.qmv_q4_0_f32_ptr(Wd.data_ptr(), buf.data_ptr() + 4, y.data_ptr(), N, K, 2)
    torch.cuda.synchronize()
    y_ref, S = orc.qmv(0, W, x, N, K)
    assert H.normalised_error(y.cpu().numpy().astype(np.float64), y_ref, S) <= H.TOL
    # a 2-byte offset is refused on the host
    with pytest.raises(q.QmvError):
        q.qmv_q4_0_f32_ptr(Wd.data_ptr(), buf.data_ptr() + 2, y.data_ptr(), N, K, 2)
    # K = 0: y = 0; N = 0 and M = 0: nothing to do
    y0 = torch.full((2, 5), 7.0, device="cuda")
    q.qmv_q4_0_f32_ptr(0, torch.empty(0, dtype=torch.float32, device="cuda").data_ptr(), y0.data_ptr(), 5, 0, 2)
    q.qmv_q4_0_swiglu_f32_ptr(0, 0, 0, 0, 0, 256, 1)
    q.qmv_q4_0_swiglu_f32_ptr(0, 0, 0, 0, 4, 256, 0)
    torch.cuda.synchronize()
    assert torch.all(y0 == 0)


def test_f32_rejects_wrong_dtype(cuda_lib):
    q = cuda_lib
    W = torch.zeros((4, 144), dtype=torch.uint8, device="cuda")
    with pytest.raises(TypeError):
        q.qmv_q4_0_f32(W, torch.zeros((1, 256), dtype=torch.float16, device="cuda"))
    with pytest.raises(TypeError):
        q.qmv_q4_0(W, torch.zeros((1, 256), dtype=torch.float32, device="cuda"))
