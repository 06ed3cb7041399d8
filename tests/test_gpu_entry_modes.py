"""Every entry point gives bit-identical results whether it runs eagerly, with
programmatic dependent launch switched off, or replayed from a CUDA graph
captured on a side stream (the way a decode loop would capture it).  Launch
mode changes only when a kernel may start, never what it computes."""
import numpy as np
import pytest

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
    q.qmv_set_pdl(True)
    torch.cuda.synchronize()


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def _calls(q):
    """name -> (function of a stream returning the output tensor)."""
    N, K = 1000, 2048
    W4 = dev(synth.q4_0_weights(N, K, 1))
    Wu = dev(synth.q4_0_weights(N, K, 2))
    W8 = dev(synth.q8_0_weights(N, K, 3))
    W2 = dev(synth.q2w_weights(N, K, 4))
    x = dev(synth.activations(3, K, 5))
    xf = dev(synth.activations(3, K, 6, dtype=np.float32))
    pool = dev(synth.q4_0_weights(16 * 128, 512, 7))
    idx = dev(synth.expert_indices(1, 5, 16, 8)[0])
    xe = dev(synth.activations(5, 512, 9))
    Wp = dev(synth.q4_0_weights(256, 512, 10))
    xp = dev(synth.activations(64, 512, 11))
    qc, qd, qs = q.qmv_quantize_q8_1(x)
    torch.cuda.synchronize()
    return {
        "q4_0": lambda s: q.qmv_q4_0(W4, x, stream=s),
        "q8_0": lambda s: q.qmv_q8_0(W8, x, stream=s),
        "q2w": lambda s: q.qmv_q2w(W2, x, stream=s),
        "q4_0_f32": lambda s: q.qmv_q4_0_f32(W4, xf, stream=s),
        "swiglu": lambda s: q.qmv_q4_0_swiglu(W4, Wu, x, stream=s),
        "swiglu_f32": lambda s: q.qmv_q4_0_swiglu_f32(W4, Wu, xf, stream=s),
        "q8_1": lambda s: q.qmv_q4_0_q8_1(W4, x, stream=s),
        "q8_1_pre": lambda s: q.qmv_q4_0_q8_1_pre(W4, qc, qd, qs, stream=s),
        "q8_0_q8_1": lambda s: q.qmv_q8_0_q8_1(W8, x, stream=s),
        "q8_0_q8_1_pre": lambda s: q.qmv_q8_0_q8_1_pre(W8, qc, qd, stream=s),
        "moe": lambda s: q.qmv_moe(pool, idx, 16, xe, 128, stream=s),
        "prefill": lambda s: q.qmm_q4_0_prefill(Wp, xp, stream=s),
    }


NAMES = ["q4_0", "q8_0", "q2w", "q4_0_f32", "swiglu", "swiglu_f32", "q8_1", "q8_1_pre", "q8_0_q8_1", "q8_0_q8_1_pre",
         "moe", "prefill"]


@pytest.mark.parametrize("name", NAMES)
def test_eager_pdl_off_and_graph_agree(cuda_lib, name):
    q = cuda_lib
    fn = _calls(q)[name]
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        y_eager = fn(s).clone()
    s.synchronize()
    q.qmv_set_pdl(False)
    try:
        with torch.cuda.stream(s):
            y_plain = fn(s).clone()
        s.synchronize()
    finally:
        q.qmv_set_pdl(True)
    # capture twice back to back in one graph (the second call depends on the first's stream order)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        fn(s)                                  # warm the lazy attribute setup outside the capture
        s.synchronize()
        with torch.cuda.graph(g, stream=s):
            y1 = fn(s)
            y2 = fn(s)
    g.replay()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(y_eager, y_plain)
    assert torch.equal(y_eager, y1) and torch.equal(y_eager, y2)
    assert q.qmv_device_status() == 0


def test_binding_refuses_bad_arguments(cuda_lib):
    """The Python binding refuses, before any launch, arguments the kernels
    would read with the wrong layout or size."""
    q = cuda_lib
    N, K = 64, 512
    W = dev(synth.q4_0_weights(N, K, 11))
    x = dev(synth.activations(2, K, 12))
    pool = dev(synth.q4_0_weights(4 * N, K, 13))
    idx = torch.tensor([1, 3], dtype=torch.int32, device="cuda")
    qc, qd, qs = q.qmv_quantize_q8_1(x)
    wide = dev(synth.activations(2, 2 * K, 14))
    with pytest.raises(ValueError):          # strided activations
        q.qmv_moe(pool, idx, 4, wide[:, ::2], N)
    with pytest.raises(ValueError):          # output of the wrong size
        q.qmv_moe(pool, idx, 4, x, N, y=torch.empty((2, N + 1), dtype=torch.float32, device="cuda"))
    with pytest.raises(ValueError):          # W not a whole number of rows
        q.qmv_q4_0_q8_1_pre(W.view(-1)[:-18 * 3], qc, qd, qs)
    with pytest.raises(ValueError):
        q.qmv_q4_0_q8_1_pre(W, qc, qd, qs, y=torch.empty((2, N), dtype=torch.float16, device="cuda"))
    with pytest.raises(ValueError):
        q.qmv_q4_0(W, x, y=torch.empty((3, N), dtype=torch.float32, device="cuda"))
    # the accepted forms still agree with each other
    y_pre = q.qmv_q4_0_q8_1_pre(W, qc, qd, qs)
    y_one = q.qmv_q4_0_q8_1(W, x)
    torch.cuda.synchronize()
    assert torch.equal(y_pre, y_one)
    assert q.qmv_device_status() == 0
