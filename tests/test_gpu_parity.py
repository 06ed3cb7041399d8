"""Parity of the CUDA path (through the C ABI) with the CPU fp64 oracle.

Bar: max |y - y_ref| / (S + 1e-6) <= 2e-3 per output, S = sum_k |x w|
(volta-kernel-bakeoff, "Making it fair" and "A few tokens at once").  Expert
routing is checked bit for bit.  Inputs are seeded synthetic GGUF bytes shaped
like the pages' workloads (weight_quantized_decode_gb300.synth).
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
    # No test may leave a device-side error behind unless it expects one.


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def gpu_call(fmt, W, x):
    import weight_quantized_decode_gb300 as q
    fn = {"q4_0": q.qmv_q4_0, "q8_0": q.qmv_q8_0, "q2w": q.qmv_q2w}[fmt]
    y = fn(dev(W), dev(x))
    torch.cuda.synchronize()
    return y.cpu().numpy().astype(np.float64)


def check(fmt, W, x, N, K, orc, rows=None):
    y = gpu_call(fmt, W, x)
    if rows is None:
        y_ref, S = orc.qmv(H.FMT[fmt], W, x, N, K, nthreads=8)
        err = H.normalised_error(y, y_ref, S)
    else:
        y_ref, S = orc.qmv_rows(H.FMT[fmt], W, x, N, K, rows, nthreads=8)
        err = H.normalised_error(y[:, rows], y_ref, S)
    assert err <= H.TOL, (fmt, N, K, x.shape[0], err)
    return y


# -- decode GEMV: tiles, ragged tails, token counts -----------------------------------

SHAPES = [(1, 256), (7, 512), (33, 768), (1000, 2048), (333, 4096), (4133, 1024), (64, 14336), (130, 2560),
          (77, 6144)]


@pytest.mark.parametrize("fmt", ["q4_0", "q8_0", "q2w"])
@pytest.mark.parametrize("N,K", SHAPES)
def test_decode_m1(orc, fmt, N, K):
    W = synth.weights(fmt, N, K, seed=N * 7 + K)
    x = synth.activations(1, K, seed=N + K)
    check(fmt, W, x, N, K, orc)


@pytest.mark.parametrize("fmt", ["q4_0", "q8_0", "q2w"])
@pytest.mark.parametrize("M", [2, 3, 4, 5, 6, 7, 8])
def test_decode_tokens(orc, fmt, M):
    N, K = 515, 2560
    W = synth.weights(fmt, N, K, seed=M)
    x = synth.activations(M, K, seed=100 + M)
    check(fmt, W, x, N, K, orc)


# Shapes whose built-in launch rule takes a lane count that is not a power of
# two (rows of 9..15 units at one or two tokens: one unit per lane) or more
# lanes than the row has units (short tables at several tokens).
RULE_SHAPES = [(37, 2304, 1), (300, 2816, 2), (200, 3072, 1), (64, 3328, 2), (129, 3584, 1), (41, 3840, 1),
               (640, 2560, 8), (512, 2048, 8), (2048, 512, 8), (100, 2560, 5), (1000, 3584, 8), (96, 768, 3)]


@pytest.mark.parametrize("fmt", ["q4_0", "q8_0", "q2w"])
@pytest.mark.parametrize("N,K,M", RULE_SHAPES)
def test_decode_rule_lane_counts(orc, fmt, N, K, M):
    W = synth.weights(fmt, N, K, seed=N * 3 + K + M)
    x = synth.activations(M, K, seed=N + 2 * K + M)
    check(fmt, W, x, N, K, orc)


# Eight tokens of K = 14336 in fp16 (235 KB) do not fit in shared memory beside
# a weight ring: the call is split into launches over token subsets.
@pytest.mark.parametrize("fmt", ["q4_0", "q8_0", "q2w"])
@pytest.mark.parametrize("N,M", [(100, 8), (1029, 7), (37, 8)])
def test_decode_token_split(orc, fmt, N, M):
    K = 14336
    W = synth.weights(fmt, N, K, seed=N + M)
    x = synth.activations(M, K, seed=2 * N + M)
    check(fmt, W, x, N, K, orc)


def test_token_split_swiglu_and_fp32(cuda_lib, orc):
    q = cuda_lib
    N, K, M = 90, 14336, 8
    Wg, Wu = _swiglu_tables(N, K, 360)
    x = synth.activations(M, K, 361)
    swiglu_check(Wg, Wu, x, N, K, orc)
    xf = synth.activations(M, K, 362, dtype=np.float32)
    y = q.qmv_q4_0_f32(dev(Wg), dev(xf))
    torch.cuda.synchronize()
    y_ref, S = orc.qmv(0, Wg, xf, N, K, nthreads=8)
    assert H.normalised_error(y.cpu().numpy().astype(np.float64), y_ref, S) <= H.TOL


@pytest.mark.parametrize("fmt", ["q4_0", "q8_0", "q2w"])
@pytest.mark.parametrize("plant", ["large", "tiny"])
@pytest.mark.parametrize("M", [1, 8])
def test_planted_activations(orc, fmt, plant, M):
    N, K = 300, 4096
    W = synth.weights(fmt, N, K, seed=5)
    x = synth.activations(M, K, seed=9, plant=plant)
    y = check(fmt, W, x, N, K, orc)
    assert np.all(np.isfinite(y))


@pytest.mark.parametrize("fmt", ["q4_0", "q8_0", "q2w"])
@pytest.mark.parametrize("K", [32, 96, 640, 1056])
def test_generic_kernel_k_not_multiple_of_256(orc, fmt, K):
    N, M = 45, 3
    W = synth.weights(fmt, N, K, seed=K)
    x = synth.activations(M, K, seed=K + 1)
    check(fmt, W, x, N, K, orc)


def test_all_code8_gives_exact_zero():
    N, K = 257, 4096
    W = synth.q4_0_weights(N, K, 3)
    W.reshape(N, -1, 18)[:, :, 2:] = 0x88
    x = synth.activations(4, K, 3)
    assert np.all(gpu_call("q4_0", W, x) == 0.0)


def test_empty_and_degenerate(cuda_lib):
    q = cuda_lib
    x = torch.zeros((2, 0), dtype=torch.float16, device="cuda")
    W = torch.zeros((5, 0), dtype=torch.uint8, device="cuda")
    y = torch.full((2, 5), 7.0, device="cuda")
    q.qmv_q4_0(W, x, y)                      # K == 0: an empty sum
    torch.cuda.synchronize()
    assert torch.all(y == 0)
    xN = torch.zeros((1, 256), dtype=torch.float16, device="cuda")
    y0 = q.qmv_q4_0(torch.zeros((0, 144), dtype=torch.uint8, device="cuda"), xN)   # N == 0
    assert y0.shape == (1, 0)


def test_deterministic_and_pdl_independent(cuda_lib):
    q = cuda_lib
    N, K = 2048, 4096
    W = dev(synth.q4_0_weights(N, K, 21))
    x = dev(synth.activations(3, K, 22))
    a = q.qmv_q4_0(W, x).clone()
    b = q.qmv_q4_0(W, x).clone()
    q.qmv_set_pdl(False)
    try:
        c = q.qmv_q4_0(W, x).clone()
    finally:
        q.qmv_set_pdl(True)
    torch.cuda.synchronize()
    assert torch.equal(a, b) and torch.equal(a, c)


def test_back_to_back_calls_keep_dependencies(cuda_lib, orc):
    """With programmatic dependent launch a call may start streaming W early;
    its x must still be the value written by the kernel before it."""
    q = cuda_lib
    N, K = 4096, 4096
    W1 = synth.q4_0_weights(K, K, 31)
    W2 = synth.q4_0_weights(N, K, 32)
    x0 = synth.activations(1, K, 33)
    Wd1, Wd2, xd = dev(W1), dev(W2), dev(x0)
    h = torch.empty((1, K), dtype=torch.float32, device="cuda")
    q.qmv_q4_0(Wd1, xd, h)                          # h = x0 @ W1^T  (K outputs)
    hx = h.to(torch.float16)                          # a torch kernel between the two calls
    y = q.qmv_q4_0(Wd2, hx)                          # consumes h
    torch.cuda.synchronize()
    y_ref, S = orc.qmv(0, W2, hx.cpu().numpy(), N, K, nthreads=8)
    assert H.normalised_error(y.cpu().numpy(), y_ref, S) <= H.TOL


def test_prefill_back_to_back_keeps_dependencies(cuda_lib, orc):
    """The prefill kernel also starts streaming and dequantising W before the
    kernel ahead of it finishes; the activations it multiplies must still be
    the ones that kernel wrote."""
    q = cuda_lib
    M, K, N = 96, 1024, 384
    W1 = synth.q4_0_weights(K, K, 34)
    W2 = synth.q4_0_weights(N, K, 35)
    x0 = synth.activations(M, K, 36)
    Wd1, Wd2 = dev(W1), dev(W2)
    h = torch.empty((M, K), dtype=torch.float32, device="cuda")
    q.qmm_q4_0_prefill(Wd1, dev(x0), h)              # h = x0 @ W1^T
    hx = (h * 0.25).to(torch.float16)                 # a torch kernel between the calls
    y = q.qmm_q4_0_prefill(Wd2, hx)                   # consumes hx
    y2 = q.qmm_q4_0_prefill(Wd2, hx)                  # straight after another prefill
    torch.cuda.synchronize()
    y_ref, S = orc.qmv(0, W2, hx.cpu().numpy(), N, K, nthreads=8)
    assert H.normalised_error(y.cpu().numpy(), y_ref, S) <= H.TOL
    assert torch.equal(y, y2)


# -- full-size configurations (sampled outputs) ----------------------------------------

def _sample_rows(N, k=96, seed=0):
    rng = np.random.default_rng(seed)
    rows = set(rng.choice(N, size=min(k, N), replace=False).tolist())
    rows |= {0, N - 1, N // 2}
    return sorted(rows)


FULL_Q4 = [(6144, 2048), (4096, 4096), (6144, 4096), (4096, 14336), (14336, 4096), (28672, 4096),
           (128256, 4096)]


@pytest.mark.parametrize("N,K", FULL_Q4)
def test_full_size_q4_0_m1(orc, N, K):
    W = synth.q4_0_weights(N, K, synth.seed_for(f"q4_0_{N}x{K}"))
    x = synth.activations(1, K, synth.seed_for(f"x_{K}"))
    check("q4_0", W, x, N, K, orc, rows=_sample_rows(N))


@pytest.mark.parametrize("N,K", [(12288, 2560), (2560, 6144), (8192, 2048)])
@pytest.mark.parametrize("M", [1, 2, 4, 8])
def test_full_size_q8_0(orc, N, K, M):
    W = synth.q8_0_weights(N, K, synth.seed_for(f"q8_0_{N}x{K}"))
    x = synth.activations(M, K, synth.seed_for(f"x_{K}_{M}"))
    check("q8_0", W, x, N, K, orc, rows=_sample_rows(N))


# The bakeoff's six one-token tables in the plain 2-bit format, plus a large
# one, at one and eight tokens (sampled rows).
@pytest.mark.parametrize("N,K", [(12288, 2560), (8192, 2048), (6144, 2048), (640, 2560), (512, 2048), (2048, 512),
                                 (128256, 4096)])
@pytest.mark.parametrize("M", [1, 8])
def test_full_size_q2w(orc, N, K, M):
    W = synth.q2w_weights(N, K, synth.seed_for(f"q2w_{N}x{K}"))
    x = synth.activations(M, K, synth.seed_for(f"x_{K}_{M}"))
    check("q2w", W, x, N, K, orc, rows=_sample_rows(N))


# -- fused gate + up + SwiGLU -----------------------------------------------------------

def swiglu_check(Wg, Wu, x, N, K, orc, rows=None):
    import weight_quantized_decode_gb300 as q
    y = q.qmv_q4_0_swiglu(dev(Wg), dev(Wu), dev(x))
    torch.cuda.synchronize()
    yn = y.cpu().numpy().astype(np.float64)
    ref = orc.swiglu(0, Wg, Wu, x, N, K, rows=rows, nthreads=8)
    err = H.swiglu_normalised_error(yn if rows is None else yn[:, rows], ref)
    assert err <= H.TOL, (N, K, x.shape[0], err)
    return yn


def _swiglu_tables(N, K, seed):
    return synth.q4_0_weights(N, K, seed), synth.q4_0_weights(N, K, seed + 7919)


@pytest.mark.parametrize("N,K", [(1, 256), (7, 512), (33, 768), (1000, 2048), (333, 4096), (64, 14336),
                                 (130, 2560), (4133, 1024)])
def test_swiglu_m1(orc, N, K):
    Wg, Wu = _swiglu_tables(N, K, 300 + N + K)
    swiglu_check(Wg, Wu, synth.activations(1, K, 301 + K), N, K, orc)


@pytest.mark.parametrize("M", [2, 3, 5, 8])
def test_swiglu_tokens(orc, M):
    N, K = 515, 2560
    Wg, Wu = _swiglu_tables(N, K, 310 + M)
    swiglu_check(Wg, Wu, synth.activations(M, K, 311 + M), N, K, orc)


@pytest.mark.parametrize("plant", ["large", "tiny"])
@pytest.mark.parametrize("M", [1, 8])
def test_swiglu_planted(orc, plant, M):
    N, K = 300, 4096
    Wg, Wu = _swiglu_tables(N, K, 320)
    y = swiglu_check(Wg, Wu, synth.activations(M, K, 321, plant=plant), N, K, orc)
    assert np.all(np.isfinite(y))


@pytest.mark.parametrize("K", [96, 640])
def test_swiglu_generic_kernel(orc, K):
    N = 45
    Wg, Wu = _swiglu_tables(N, K, 330 + K)
    swiglu_check(Wg, Wu, synth.activations(3, K, 331), N, K, orc)


@pytest.mark.parametrize("N,K", [(14336, 4096), (6144, 2048)])
@pytest.mark.parametrize("M", [1, 8])
def test_swiglu_full_size_sampled(orc, N, K, M):
    Wg, Wu = _swiglu_tables(N, K, synth.seed_for(f"swiglu_{N}x{K}"))
    x = synth.activations(M, K, synth.seed_for(f"swiglu_x_{K}_{M}"))
    swiglu_check(Wg, Wu, x, N, K, orc, rows=_sample_rows(N))


def test_swiglu_empty_and_sabotage(cuda_lib, orc):
    q = cuda_lib
    # K = 0: silu(0) * 0 = 0 everywhere
    y = torch.full((2, 5), 7.0, device="cuda")
    q.qmv_q4_0_swiglu_ptr(0, 0, torch.empty(0, dtype=torch.float16, device="cuda").data_ptr(), y.data_ptr(), 5, 0, 2, 0)
    torch.cuda.synchronize()
    assert torch.all(y == 0)
    # N = 0 and M = 0: nothing to do
    q.qmv_q4_0_swiglu_ptr(0, 0, 0, 0, 0, 256, 1, 0)
    q.qmv_q4_0_swiglu_ptr(0, 0, 0, 0, 4, 256, 0, 0)
    # corrupted tables: most outputs fail (outputs whose gate is near zero or
    # far negative are small either way and may pass)
    N, K = 256, 2048
    Wg, Wu = _swiglu_tables(N, K, 340)
    x = synth.activations(1, K, 341)
    y = q.qmv_q4_0_swiglu(dev(H.sabotage(Wg, "q4_0")), dev(H.sabotage(Wu, "q4_0")), dev(x))
    torch.cuda.synchronize()
    ref = orc.swiglu(0, Wg, Wu, x, N, K, nthreads=8)
    yn = y.cpu().numpy().astype(np.float64)
    silu = ref["g"] / (1 + np.exp(-ref["g"]))
    scale = H.SILU_SLOPE_MAX * ref["Sg"] * (np.abs(ref["u"]) + H.TOL * ref["Su"]) + np.abs(silu) * ref["Su"]
    err = np.abs(yn - ref["y"]) / (scale + 1e-6)
    assert (err > H.TOL).mean() > 0.75 and err.max() > 20 * H.TOL, ((err > H.TOL).mean(), err.max())


# -- multi-expert decode --------------------------------------------------------------

@pytest.mark.parametrize("E,slots,N,K", [(128, 10, 640, 2560), (128, 8, 512, 2048), (5, 5, 64, 512),
                                         (3, 7, 33, 256)])
def test_moe_matches_oracle_and_single_calls(cuda_lib, orc, E, slots, N, K):
    q = cuda_lib
    pool = synth.q4_0_weights(E * N, K, 40 + E)
    idx = synth.expert_indices(1, min(slots, E), E, 41)[0]
    if slots > E:      # more slots than experts: duplicates
        idx = np.resize(idx, slots).astype(np.int32)
    x = synth.activations(slots, K, 42)
    pd, xd = dev(pool), dev(x)
    y = q.qmv_moe(pd, dev(idx), E, xd, N)
    torch.cuda.synchronize()
    yn = y.cpu().numpy().astype(np.float64)
    y_ref, S = orc.moe(0, pool, idx, E, x, N, K, nthreads=8)
    assert H.normalised_error(yn, y_ref, S) <= H.TOL
    rb = (K // 32) * 18
    for s in range(slots):
        e = int(idx[s])
        ys = q.qmv_q4_0(pd.view(E * N, rb)[e * N:(e + 1) * N], xd[s:s + 1])
        torch.cuda.synchronize()
        assert torch.equal(ys[0], y[s]), f"slot {s} is not bit-identical to the single call"
        # every other expert fails this slot's check (a wrong index fails)
        if s == 0:
            for other in range(min(E, 6)):
                if other == e:
                    continue
                yo, So = orc.qmv(0, pool[other * N:(other + 1) * N], x[s:s + 1], N, K)
                assert H.normalised_error(yn[s:s + 1], yo, So) > H.TOL
    assert q.qmv_device_status() == 0


def test_moe_bad_index_sets_status_and_nans(cuda_lib):
    q = cuda_lib
    E, N, K = 4, 96, 512
    pool = dev(synth.q4_0_weights(E * N, K, 50))
    x = dev(synth.activations(3, K, 51))
    idx = dev(np.array([1, 9, 2], dtype=np.int32))
    y = q.qmv_moe(pool, idx, E, x, N)
    st = q.qmv_device_status()
    assert st & q.QMV_DEV_BAD_EXPERT
    assert torch.all(torch.isnan(y[1]))
    assert torch.all(torch.isfinite(y[0])) and torch.all(torch.isfinite(y[2]))
    ok = q.qmv_moe(pool, dev(np.array([1, 3, 2], dtype=np.int32)), E, x, N)
    assert torch.equal(ok[0], y[0]) and torch.equal(ok[2], y[2])
    assert q.qmv_device_status() == 0


# -- launch shapes forced through the tuning override ----------------------------------

OVERRIDES = {
    # Launch shapes the measured table and the rule do not pick: lanes per row
    # from 1 to 32 (also ones that do not divide 32), odd passes per stage, deep
    # rings, two CTAs per SM; the multi-expert form must still equal the single
    # calls bit for bit.
    "G=4,SP=3": ["gemv:q4_0:77:6144:1", "gemv:q8_0:130:2560:2", "moe:q4_0:64:2560:5", "gemv:q2w:77:6144:3",
                 "q81:q4_0:77:6144:3"],
    "G=32,warps=4": ["gemv:q4_0:40:8192:1", "gemv:q8_0:130:2560:4", "moe:q4_0:96:4096:6"],
    "G=1,SP=5,stages=3": ["gemv:q4_0:16:14336:1", "gemv:q4_0:33:2048:3", "moe:q4_0:20:2048:3", "gemv:q2w:16:14336:1"],
    "warps=16,stages=4,G=2": ["gemv:q4_0:100:4096:2", "gemv:q8_0:9:3072:1", "gemv:q2w:100:4096:1",
                              "q81:q4_0:100:4096:2"],
    "ctas=2,share=2": ["gemv:q4_0:1000:4096:1", "gemv:q8_0:600:2048:1", "moe:q4_0:33:1024:7",
                       "q81:q4_0:1000:4096:8"],
    # lanes per row that do not divide 32 (idle lanes, lane-order reduction)
    "G=10": ["gemv:q4_0:130:2560:1", "gemv:q8_0:77:2560:2", "moe:q4_0:64:2560:5", "gemv:q2w:130:2560:2",
             "q81:q4_0:130:2560:1"],
    "G=3,SP=3": ["gemv:q4_0:41:2304:1", "gemv:q8_0:50:1536:4", "moe:q4_0:20:2304:3"],
    "G=12,warps=16": ["gemv:q4_0:90:3072:2", "gemv:q8_0:33:6144:1", "swiglu:q4_0:90:3072:2"],
    # twelve warps per CTA at three or more tokens (384-thread instantiations)
    "warps=12,G=4,SP=3": ["gemv:q4_0:300:4096:8", "gemv:q8_0:200:2048:5", "gemv:q2w:150:4096:6",
                          "q81:q4_0:300:4096:8", "swiglu:q4_0:90:4096:8"],
    "warps=12,stages=3,G=2": ["gemv:q4_0:1000:2048:3", "gemv:q8_0:77:6144:4", "gemv:q2w:640:2560:8",
                              "q81:q4_0:515:2560:7", "swiglu:q4_0:300:2048:5"],
    # the fused SwiGLU keeps an even number of rows per group (G clamped to <= 16)
    "G=32": ["swiglu:q4_0:77:4096:1", "swiglu:q4_0:40:2048:8"],
    # the streaming kernel's own launch rule at the token counts the tensor cores
    # otherwise take (these tests run with that path off), including the token
    # split of eight tokens of K = 14336 into several launches
    "early=1": ["gemv:q4_0:4096:4096:8", "gemv:q8_0:2560:6144:4", "gemv:q8_0:12288:2560:8",
                "gemv:q4_0:4096:14336:8", "gemv:q4_0:515:2560:5"],
}


@pytest.mark.parametrize("tune", list(OVERRIDES))
def test_launch_overrides(orc, tmp_path, tune):
    import os
    import subprocess
    import sys
    out = tmp_path / "y.npz"
    # the streaming kernel at every token count (no tensor-core path)
    env = dict(os.environ, QMV_GEMV_TUNE=tune, QMV_TC_MIN_TOKENS="0")
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, "-m", "tests._launch_override_child", str(out)] + OVERRIDES[tune],
                       env=env, cwd=root, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    res = np.load(out)
    assert int(res["status"][0]) == 0
    for case in OVERRIDES[tune]:
        kind, fmt, n, k, m = case.split(":")
        N, K, M = int(n), int(k), int(m)
        y = res[case].astype(np.float64)
        if kind == "swiglu":
            Wg = synth.q4_0_weights(N, K, synth.seed_for(f"ovr_sg_{N}x{K}"))
            Wu = synth.q4_0_weights(N, K, synth.seed_for(f"ovr_su_{N}x{K}"))
            x = synth.activations(M, K, synth.seed_for(f"ovr_x_{K}_{M}"))
            ref = orc.swiglu(0, Wg, Wu, x, N, K, nthreads=8)
            err = H.swiglu_normalised_error(y, ref)
            assert err <= H.TOL, (tune, case, err)
            continue
        if kind == "q81":
            W = synth.q4_0_weights(N, K, synth.seed_for(f"ovr_q81_{N}x{K}"))
            x = synth.activations(M, K, synth.seed_for(f"ovr_x_{K}_{M}"))
            qo, do, _ = orc.quantize_q8_1(x)
            y_ref, S = orc.qmv_q8_1(0, W, qo, do, N, K, nthreads=8)
            err = H.normalised_error(y, y_ref, S)
            assert err <= 5e-5, (tune, case, err)
            continue
        if kind == "gemv":
            W = synth.weights(fmt, N, K, synth.seed_for(f"ovr_{fmt}_{N}x{K}"))
            x = synth.activations(M, K, synth.seed_for(f"ovr_x_{K}_{M}"))
            y_ref, S = orc.qmv(H.FMT[fmt], W, x, N, K, nthreads=8)
        else:
            E = 2 * M
            pool = synth.q4_0_weights(E * N, K, synth.seed_for(f"ovr_pool_{N}x{K}"))
            x = synth.activations(M, K, synth.seed_for(f"ovr_moe_x_{K}"))
            y_ref, S = orc.moe(0, pool, res[case + ":idx"], E, x, N, K, nthreads=8)
            assert np.array_equal(res[case], res[case + ":single"]), (tune, case, "not bit-identical")
        err = H.normalised_error(y, y_ref, S)
        assert err <= H.TOL, (tune, case, err)


@pytest.mark.parametrize("N,K,M", [(12288, 2560, 512), (8192, 2048, 512), (12288, 2560, 64), (9856, 256, 300),
                                   (8192, 2048, 64)])
def test_prefill_repeats_are_bit_identical(cuda_lib, orc, N, K, M):
    """Every slot of every ring is reused many times at these sizes; a copy that
    overtakes a read still in flight shows up as a changed output row."""
    q = cuda_lib
    W = dev(synth.q4_0_weights(N, K, synth.seed_for(f"prefill_{N}x{K}")))
    x = dev(synth.activations(M, K, synth.seed_for(f"prefill_x_{M}")))
    ys = [q.qmm_q4_0_prefill(W, x) for _ in range(5)]
    torch.cuda.synchronize()
    for y in ys[1:]:
        assert torch.equal(y, ys[0])


PREFILL_RINGS = {
    # the shallowest rings (two packed-weight slots, two operand slots)
    # one packed-weight slot, the deepest operand ring that then fits
    "1,4": ["pfrep:q4_0:12288:2560:512", "pfrep:q4_0:4096:2560:256", "pfrep:q4_0:2048:2560:64"],
    # no cluster: each CTA loads whole activation tiles itself (the rule's choice)
    "0,0,1": ["pfrep:q4_0:12288:2560:512", "pfrep:q4_0:4096:2560:256", "pfrep:q4_0:2048:2560:64",
              "pfrep:q4_0:384:512:100"],
    # CTA pairs sharing each activation tile by multicast, also with an odd tile
    # count (one CTA of the last pair lies past N)
    "0,0,2": ["pfrep:q4_0:384:512:100", "pfrep:q4_0:130:256:70", "pfrep:q4_0:8192:2048:64"],
    # 16-token tiles split along K over a cluster of 2, 3 or 8 CTAs (partials added
    # through distributed shared memory), ragged rows and a ragged chunk share
    "0,0,0,0,0,0,2": ["pfrep:q4_0:384:2560:8", "pfrep:q8_0:300:2048:16", "pfrep:q8_0:4096:6144:8"],
    "0,0,0,0,0,0,3": ["pfrep:q4_0:200:2560:5", "pfrep:q8_0:129:1792:1"],
    "0,0,0,0,0,0,8": ["pfrep:q4_0:256:2048:3", "pfrep:q8_0:130:4096:16", "pfrep:q8_0:2560:6144:8"],
    # the shallowest rings (two packed-weight slots, two operand slots), Q4_0 and Q8_0
    "2,2": ["pfrep:q4_0:12288:2560:512", "pfrep:q4_0:4096:2560:256", "pfrep:q4_0:2048:2560:64",
            "pfrep:q8_0:12288:2560:512", "pfrep:q8_0:2048:2560:64"],
}


@pytest.mark.parametrize("ring", list(PREFILL_RINGS))
def test_prefill_shallow_rings(orc, tmp_path, ring):
    import os
    import subprocess
    import sys
    out = tmp_path / "y.npz"
    env = dict(os.environ, QMV_PREFILL_RING=ring)
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, "-m", "tests._launch_override_child", str(out)] + PREFILL_RINGS[ring],
                       env=env, cwd=root, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    res = np.load(out)
    assert int(res["status"][0]) == 0
    for case in PREFILL_RINGS[ring]:
        _, fmt, n, k, m = case.split(":")
        N, K, M = int(n), int(k), int(m)
        assert bool(res[case + ":identical"][0]), (ring, case, "repeats differ")
        W = synth.weights(fmt, N, K, synth.seed_for(f"ovr_pf_{N}x{K}"))
        x = synth.activations(M, K, synth.seed_for(f"ovr_pf_x_{K}_{M}"))
        rows = _sample_rows(N, k=32)
        y_ref, S = orc.qmv_rows(H.FMT[fmt], W, x, N, K, rows, nthreads=8)
        assert H.normalised_error(res[case].astype(np.float64)[:, rows], y_ref, S) <= H.TOL, (ring, case)


def test_prefill_in_graph_on_a_new_stream(cuda_lib, orc):
    """A prefill call captured into a CUDA graph on a fresh stream (tensor maps
    are built on the host at capture time) replays correctly, twice."""
    q = cuda_lib
    N, K, M = 512, 2048, 64
    W = synth.q4_0_weights(N, K, 61)
    x = synth.activations(M, K, 62)
    Wd, xd = dev(W), dev(x)
    y = torch.empty((M, N), dtype=torch.float32, device="cuda")
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            q.qmm_q4_0_prefill(Wd, xd, y, stream=s)
    for _ in range(2):
        y.zero_()
        g.replay()
        torch.cuda.synchronize()
        y_ref, S = orc.qmv(0, W, x, N, K, nthreads=8)
        assert H.normalised_error(y.cpu().numpy(), y_ref, S) <= H.TOL


# -- sabotage: corrupted packed bytes must fail every check ----------------------------

@pytest.mark.parametrize("fmt", ["q4_0", "q8_0", "q2w"])
def test_sabotage_fails(orc, fmt):
    N, K = 512, 2048
    W = synth.weights(fmt, N, K, 60)
    x = synth.activations(2, K, 61)
    y_bad = gpu_call(fmt, H.sabotage(W, fmt), x)
    y_ref, S = orc.qmv(H.FMT[fmt], W, x, N, K, nthreads=8)
    assert H.normalised_error(y_bad, y_ref, S) > 20 * H.TOL
    # control: the kernel is consistent with the oracle on the corrupted bytes
    y_ref_bad, S_bad = orc.qmv(H.FMT[fmt], H.sabotage(W, fmt), x, N, K, nthreads=8)
    assert H.normalised_error(y_bad, y_ref_bad, S_bad) <= H.TOL


# -- prefill ---------------------------------------------------------------------------

# (9856, 256, 300) and (12000, 512, 512): on a 152-SM GPU 256-token tiles would
# need two waves, so one CTA takes 512 tokens in two accumulators (ragged
# second half, ragged last row tile).
@pytest.mark.parametrize("N,K,M", [(256, 512, 64), (384, 1024, 100), (128, 256, 1), (1024, 2560, 512),
                                   (200, 512, 70), (128, 2048, 257), (9856, 256, 300), (12000, 512, 512)])
def test_prefill(cuda_lib, orc, N, K, M):
    q = cuda_lib
    W = synth.q4_0_weights(N, K, N + K + M)
    x = synth.activations(M, K, M)
    y = q.qmm_q4_0_prefill(dev(W), dev(x))
    torch.cuda.synchronize()
    y_ref, S = orc.qmv(0, W, x, N, K, nthreads=8)
    assert H.normalised_error(y.cpu().numpy(), y_ref, S) <= H.TOL


# Q8_0 weights: 16-token tiles (M <= 16), 64-token tiles, wide tiles with one and
# two weight tiles per CTA, ragged rows and tokens.
@pytest.mark.parametrize("N,K,M", [(256, 512, 64), (384, 1024, 100), (128, 256, 1), (1024, 2560, 512),
                                   (200, 512, 70), (130, 2048, 16), (300, 4096, 9), (12000, 512, 512)])
def test_prefill_q8_0(cuda_lib, orc, N, K, M):
    q = cuda_lib
    W = synth.q8_0_weights(N, K, N + K + M)
    x = synth.activations(M, K, M)
    y = q.qmm_q8_0_prefill(dev(W), dev(x))
    torch.cuda.synchronize()
    y_ref, S = orc.qmv(1, W, x, N, K, nthreads=8)
    assert H.normalised_error(y.cpu().numpy(), y_ref, S) <= H.TOL


@pytest.mark.parametrize("N,K,M", [(12288, 2560, 512), (12288, 2560, 8), (2560, 6144, 16)])
def test_prefill_q8_0_repeats_are_bit_identical(cuda_lib, orc, N, K, M):
    q = cuda_lib
    W = dev(synth.q8_0_weights(N, K, synth.seed_for(f"prefill8_{N}x{K}")))
    x = dev(synth.activations(M, K, synth.seed_for(f"prefill8_x_{M}")))
    ys = [q.qmm_q8_0_prefill(W, x) for _ in range(5)]
    torch.cuda.synchronize()
    for y in ys[1:]:
        assert torch.equal(y, ys[0])
    rows = _sample_rows(N, k=32)
    y_ref, S = orc.qmv_rows(1, synth.q8_0_weights(N, K, synth.seed_for(f"prefill8_{N}x{K}")),
                            synth.activations(M, K, synth.seed_for(f"prefill8_x_{M}")), N, K, rows, nthreads=8)
    assert H.normalised_error(ys[0].cpu().numpy()[:, rows], y_ref, S) <= H.TOL


@pytest.mark.parametrize("N,K,M", [(12288, 2560, 64), (12288, 2560, 512), (8192, 2048, 64), (8192, 2048, 512)])
def test_prefill_full_size_sampled(cuda_lib, orc, N, K, M):
    q = cuda_lib
    W = synth.q4_0_weights(N, K, synth.seed_for(f"prefill_{N}x{K}"))
    x = synth.activations(M, K, synth.seed_for(f"prefill_x_{M}"))
    y = q.qmm_q4_0_prefill(dev(W), dev(x)).cpu().numpy()
    rows = _sample_rows(N, k=48)
    y_ref, S = orc.qmv_rows(0, W, x, N, K, rows, nthreads=8)
    assert H.normalised_error(y[:, rows], y_ref, S) <= H.TOL


# -- concurrent use from several host threads, each on its own stream ------------------

def test_concurrent_host_threads_and_streams(cuda_lib, orc):
    """The library's process-wide state (device information, shared-memory
    opt-in, the launch-shape table, the PDL switch) is shared by threads that
    call it at once, each on its own stream; every result must still match."""
    import threading
    q = cuda_lib
    cases = [("q4_0", 700, 2048, 1), ("q8_0", 300, 4096, 3), ("q2w", 515, 2560, 8), ("q4_0", 4096, 14336, 8),
             ("q8_0", 33, 768, 2), ("q4_0", 1000, 640, 4)]
    inputs = []
    for i, (fmt, N, K, M) in enumerate(cases):
        W = synth.weights(fmt, N, K, 900 + i)
        x = synth.activations(M, K, 950 + i)
        inputs.append((fmt, N, K, M, W, x, dev(W), dev(x)))
    results, errors = {}, []

    def worker(t):
        try:
            s = torch.cuda.Stream()
            fns = {"q4_0": q.qmv_q4_0, "q8_0": q.qmv_q8_0, "q2w": q.qmv_q2w}
            with torch.cuda.stream(s):
                for rep in range(3):
                    for j, (fmt, N, K, M, _, _, Wd, xd) in enumerate(inputs):
                        if (j + t) % 2 == 0:
                            y = fns[fmt](Wd, xd, stream=s)
                            results[(t, rep, j)] = y
            s.synchronize()
        except Exception as e:    # surfaced below
            errors.append(repr(e))

    torch.cuda.synchronize()           # the inputs are on the device before any side stream reads them
    threads = [threading.Thread(target=worker, args=(t,)) for t in range(4)]
    for th in threads:
        th.start()
    for th in threads:
        th.join()
    torch.cuda.synchronize()
    assert not errors, errors
    refs = {}
    for (t, rep, j), y in results.items():
        fmt, N, K, M, W, x, _, _ = inputs[j]
        if j not in refs:
            refs[j] = orc.qmv(H.FMT[fmt], W, x, N, K, nthreads=8)
        err = H.normalised_error(y.cpu().numpy().astype(np.float64), *refs[j])
        assert err <= H.TOL, (t, rep, j, err)
    assert q.qmv_device_status() == 0
