"""Pins for the CPU oracle (no GPU).

Each pin ties the oracle to something other than itself: hand-computed closed
forms (tests/golden), an exhaustive comparison of its fp16 decoder with numpy,
integer special cases that reduce to a plain numpy matmul, exact invariants,
and the sabotage check of volta-kernel-bakeoff ("Making it fair").
"""
import math

import numpy as np
import pytest

from tests import helpers as H
from weight_quantized_decode_gb300 import synth


# -- fp16 decoding -------------------------------------------------------------

def test_half_decode_exhaustive(orc):
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = np.array([orc.half_to_double(int(b)) for b in bits])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(ref[~nan]))


# -- hand-computed cases -----------------------------------------------------

@pytest.mark.parametrize("case", H.load_cases("oracle_cases.txt") + H.load_cases("q2w_cases.txt"),
                         ids=lambda c: c["name"])
def test_golden_cases(orc, case):
    y, S = orc.qmv(H.FMT[case["fmt"]], case["W"], case["xarr"], case["N"], case["K"])
    for (m, n), v in case["y"].items():
        assert y[m, n] == v, (case["name"], m, n, y[m, n], v)
    for (m, n), v in case["S"].items():
        assert S[m, n] == v, (case["name"], m, n, S[m, n], v)


def test_golden_moe(orc):
    (case,) = H.load_cases("moe_cases.txt")
    E, idx = case["moe"]
    y, S = orc.moe(H.FMT[case["fmt"]], case["W"], idx, E, case["xarr"], case["N"], case["K"])
    for (s, n), v in case["y"].items():
        assert y[s, n] == v


def test_moe_rejects_bad_index(orc):
    (case,) = H.load_cases("moe_cases.txt")
    E, _ = case["moe"]
    with pytest.raises(ValueError):
        orc.moe(0, case["W"], [0, 3, 1], E, case["xarr"], case["N"], case["K"])
    with pytest.raises(ValueError):
        orc.moe(0, case["W"], [0, -1, 1], E, case["xarr"], case["N"], case["K"])


# -- integer special cases: the product reduces to an integer matmul ----------

@pytest.mark.parametrize("K", [32, 96, 256])
def test_q4_0_integer_case_matches_numpy(orc, K):
    rng = np.random.default_rng(7 + K)
    N, M = 5, 3
    codes = rng.integers(0, 16, size=(N, K))
    d_bits = np.full((N, K // 32), 0x3C00, dtype=np.uint16)          # d = 1
    W = H.encode_q4_0(codes, d_bits)
    x = rng.integers(-50, 51, size=(M, K)).astype(np.float16)         # exact small ints
    y, S = orc.qmv(0, W, x, N, K)
    Wi = (codes - 8).astype(np.float64)
    xf = x.astype(np.float64)
    assert np.array_equal(y, xf @ Wi.T)
    assert np.array_equal(S, np.abs(xf) @ np.abs(Wi).T)


@pytest.mark.parametrize("K", [32, 128])
def test_q8_0_integer_case_matches_numpy(orc, K):
    rng = np.random.default_rng(11 + K)
    N, M = 4, 2
    codes = rng.integers(-128, 128, size=(N, K))
    d_bits = np.full((N, K // 32), 0x3C00, dtype=np.uint16)
    W = H.encode_q8_0(codes, d_bits)
    x = rng.integers(-50, 51, size=(M, K)).astype(np.float16)
    y, _ = orc.qmv(1, W, x, N, K)
    assert np.array_equal(y, x.astype(np.float64) @ codes.astype(np.float64).T)


def test_power_of_two_scales_per_block(orc):
    """d = 2^e per block (exact): y equals the integer matmul with the scale
    folded into the integer matrix column-block by column-block."""
    rng = np.random.default_rng(3)
    N, K, M = 3, 128, 2
    codes = rng.integers(0, 16, size=(N, K))
    e = rng.integers(-3, 4, size=(N, K // 32))
    d_bits = (0x3C00 + (e << 10)).astype(np.uint16)                    # 2^e
    W = H.encode_q4_0(codes, d_bits)
    x = rng.integers(-20, 21, size=(M, K)).astype(np.float16)
    y, _ = orc.qmv(0, W, x, N, K)
    scale = np.repeat(2.0 ** e, 32, axis=1)
    assert np.array_equal(y, x.astype(np.float64) @ ((codes - 8) * scale).T)


# -- invariants ------------------------------------------------------------------

def _rand(fmt, N, K, M, seed):
    W = synth.weights(fmt, N, K, seed)
    x = synth.activations(M, K, seed)
    return W, x


def test_all_code8_gives_zero(orc):
    W, x = _rand("q4_0", 7, 512, 2, 1)
    v = W.reshape(7, -1, 18)
    v[:, :, 2:] = 0x88
    y, _ = orc.qmv(0, W, x, 7, 512)
    assert np.all(y == 0.0)


def test_doubling_scales_doubles_y(orc):
    for fmt in ("q4_0", "q8_0"):
        bb = H.BLOCK_BYTES[fmt]
        W, x = _rand(fmt, 6, 256, 2, 2)
        W2 = W.copy().reshape(6, -1, bb)
        d = W2[:, :, 0:2].copy().view(np.uint16)
        W2[:, :, 0:2] = (d + 0x0400).view(np.uint8)                      # exponent + 1
        y, _ = orc.qmv(H.FMT[fmt], W, x, 6, 256)
        y2, _ = orc.qmv(H.FMT[fmt], W2.reshape(6, -1), x, 6, 256)
        assert np.array_equal(y2, 2.0 * y)


def test_linear_in_x(orc):
    rng = np.random.default_rng(5)
    W, _ = _rand("q4_0", 9, 512, 1, 3)
    x1 = rng.integers(-100, 100, size=(1, 512)).astype(np.float16)
    x2 = rng.integers(-100, 100, size=(1, 512)).astype(np.float16)
    y1, _ = orc.qmv(0, W, x1, 9, 512)
    y2, _ = orc.qmv(0, W, x2, 9, 512)
    y12, S = orc.qmv(0, W, (x1.astype(np.float32) + x2).astype(np.float16), 9, 512)
    assert np.max(np.abs(y12 - (y1 + y2)) / (S + 1e-30)) < 1e-12


def test_q2w_integer_case_matches_numpy(orc):
    rng = np.random.default_rng(71)
    N, K, M = 6, 256, 3
    codes = rng.integers(0, 4, size=(N, K))
    d_bits = np.full((N, K // 32), 0x3C00, dtype=np.uint16)          # d = 1
    W = H.encode_q2w(codes, d_bits)
    x = rng.integers(-50, 51, size=(M, K)).astype(np.float16)
    y, S = orc.qmv(2, W, x, N, K)
    Wi = (codes - 2).astype(np.float64)
    xf = x.astype(np.float64)
    assert np.array_equal(y, xf @ Wi.T)
    assert np.array_equal(S, np.abs(xf) @ np.abs(Wi).T)


def test_q2w_to_q4_reencoding_identical(orc):
    # a 2-bit code c2 is the Q4_0 code c2 + 6: same weight (c2 - 2) d, same scale
    N, K = 5, 512
    W2 = synth.q2w_weights(N, K, 72)
    x = synth.activations(3, K, 73)
    v = W2.reshape(N, K // 32, 10)
    planes = [(v[:, :, 2:10] >> (2 * p)) & 3 for p in range(4)]          # [N, nb, 8] each
    codes = np.concatenate(planes, axis=2).reshape(N, K).astype(np.int64)  # element j = plane j//8, byte j%8
    d_bits = v[:, :, 0:2].copy().view(np.uint16).reshape(N, K // 32)
    W4 = H.encode_q4_0(codes + 6, d_bits)
    y2, S2 = orc.qmv(2, W2, x, N, K)
    y4, S4 = orc.qmv(0, W4, x, N, K)
    assert np.array_equal(y2, y4) and np.array_equal(S2, S4)
    assert np.array_equal(H.encode_q2w(codes, d_bits), W2)         # the encoder is the format's inverse


def test_q2w_all_code2_gives_zero(orc):
    N, K = 4, 256
    W = H.encode_q2w(np.full((N, K), 2), np.full((N, K // 32), 0x3C00, dtype=np.uint16))
    y, S = orc.qmv(2, W, synth.activations(2, K, 74), N, K)
    assert np.all(y == 0) and np.all(S == 0)


def test_q4_to_q8_reencoding_identical(orc):
    N, K = 5, 256
    W4, x = _rand("q4_0", N, K, 2, 4)
    v = W4.reshape(N, K // 32, 18)
    lo = (v[:, :, 2:] & 0x0F).astype(np.int16) - 8
    hi = (v[:, :, 2:] >> 4).astype(np.int16) - 8
    codes = np.concatenate([lo, hi], axis=2).reshape(N, K)
    d_bits = v[:, :, 0:2].copy().view(np.uint16).reshape(N, K // 32)
    W8 = H.encode_q8_0(codes, d_bits)
    y4, S4 = orc.qmv(0, W4, x, N, K)
    y8, S8 = orc.qmv(1, W8, x, N, K)
    assert np.array_equal(y4, y8) and np.array_equal(S4, S8)


def test_block_permutation_invariance(orc):
    N, K, M = 4, 512, 2
    for fmt in ("q4_0", "q8_0"):
        bb = H.BLOCK_BYTES[fmt]
        W, x = _rand(fmt, N, K, M, 6)
        perm = np.random.default_rng(8).permutation(K // 32)
        Wp = W.reshape(N, K // 32, bb)[:, perm].reshape(N, -1)
        xp = x.reshape(M, K // 32, 32)[:, perm].reshape(M, K)
        y, S = orc.qmv(H.FMT[fmt], W, x, N, K)
        yp, _ = orc.qmv(H.FMT[fmt], Wp, xp, N, K)
        assert np.max(np.abs(y - yp) / S) < 1e-13


def test_tokens_and_rows_are_independent(orc):
    N, K, M = 11, 256, 4
    W, x = _rand("q8_0", N, K, M, 9)
    y, S = orc.qmv(1, W, x, N, K)
    for m in range(M):
        ym, Sm = orc.qmv(1, W, x[m:m + 1], N, K)
        assert np.array_equal(ym[0], y[m]) and np.array_equal(Sm[0], S[m])
    rows = [10, 0, 3, 3]
    yr, Sr = orc.qmv_rows(1, W, x, N, K, rows)
    assert np.array_equal(yr, y[:, rows]) and np.array_equal(Sr, S[:, rows])


def test_moe_identity_routing_equals_separate_gemvs(orc):
    E, N, K = 4, 6, 256
    pool = synth.q4_0_weights(E * N, K, 12)
    x = synth.activations(E, K, 12)
    y, _ = orc.moe(0, pool, np.arange(E), E, x, N, K)
    for e in range(E):
        ye, _ = orc.qmv(0, pool[e * N:(e + 1) * N], x[e:e + 1], N, K)
        assert np.array_equal(ye[0], y[e])


def test_empty_shapes(orc):
    y, S = orc.qmv(0, np.zeros(0, np.uint8), np.zeros((2, 0), np.float16), 3, 0)
    assert y.shape == (2, 3) and np.all(y == 0) and np.all(S == 0)
    y, S = orc.qmv(0, np.zeros(0, np.uint8), np.zeros((1, 64), np.float16), 0, 64)
    assert y.shape == (1, 0)


# -- sabotage: corrupting the packed bytes must fail every check ----------------

@pytest.mark.parametrize("fmt", ["q4_0", "q8_0", "q2w"])
def test_sabotage_fails_the_check(orc, fmt):
    """A check is the max error over a product's outputs.  Sabotage moves each
    weight by +-8d (Q4_0) or more (Q8_0): the expected normalised error is
    ~2.5/sqrt(K) = 0.055 at K=2048, so the check fails by a wide margin and
    almost every single output fails on its own too."""
    N, K, M = 64, 2048, 2
    W, x = _rand(fmt, N, K, M, 13)
    y, S = orc.qmv(H.FMT[fmt], W, x, N, K)
    ys, _ = orc.qmv(H.FMT[fmt], H.sabotage(W, fmt), x, N, K)
    err = np.abs(ys - y) / (S + 1e-6)
    assert err.max() > 20 * H.TOL
    assert (err > H.TOL).mean() > 0.9


def test_sabotage_fails_golden(orc):
    for case in H.load_cases("oracle_cases.txt"):
        y, _ = orc.qmv(H.FMT[case["fmt"]], H.sabotage(case["W"], case["fmt"]),
                       case["xarr"], case["N"], case["K"])
        assert any(y[m, n] != v for (m, n), v in case["y"].items()), case["name"]


def test_tolerance_helper():
    assert H.normalised_error([1.0], [1.0], [1.0]) == 0.0
    assert H.normalised_error([1.003], [1.0], [1.0]) > H.TOL
    assert H.normalised_error([np.nan], [1.0], [1.0]) == np.inf


# -- gate + up + SwiGLU (closed forms) --------------------------------------------------

def _uniform_table(code, d_bits, N=1, K=32):
    return H.encode_q4_0(np.full((N, K), code, dtype=np.int64), np.full((N, K // 32), d_bits, dtype=np.uint16))


def _silu(z):
    return z / (1.0 + math.exp(-z))


@pytest.mark.parametrize("gate_code,up_code,g,u", [
    (9, 10, 1.0, 2.0),      # w = 1/32 and 2/32 against 32 ones
    (7, 10, -1.0, 2.0),     # negative gate
    (6, 9, -2.0, 1.0),
    (12, 5, 4.0, -3.0),     # negative up
])
def test_swiglu_closed_form(orc, gate_code, up_code, g, u):
    Wg = _uniform_table(gate_code, 0x2800)      # d = 2^-5
    Wu = _uniform_table(up_code, 0x2800)
    x = np.ones((1, 32), dtype=np.float16)
    r = orc.swiglu(0, Wg, Wu, x, 1, 32)
    assert r["g"][0, 0] == g and r["u"][0, 0] == u
    assert r["Sg"][0, 0] == abs(g) and r["Su"][0, 0] == abs(u)
    assert r["y"][0, 0] == pytest.approx(_silu(g) * u, rel=1e-15)


def test_swiglu_zero_gate_or_up_gives_zero(orc):
    x = np.ones((1, 32), dtype=np.float16)
    assert orc.swiglu(0, _uniform_table(8, 0x3C00), _uniform_table(13, 0x3C00), x, 1, 32)["y"][0, 0] == 0.0
    assert orc.swiglu(0, _uniform_table(13, 0x3C00), _uniform_table(8, 0x3C00), x, 1, 32)["y"][0, 0] == 0.0


def test_swiglu_large_gate_is_linear(orc):
    # g = 7 * 32 = 224 (d = 1): silu(g) = g to double precision; u = 32
    x = np.ones((1, 32), dtype=np.float16)
    r = orc.swiglu(0, _uniform_table(15, 0x3C00), _uniform_table(9, 0x3C00), x, 1, 32)
    assert r["y"][0, 0] == 224.0 * 32.0


def test_swiglu_rows_tokens_and_subset(orc):
    # row 0: gate w = 1/32, up w = 2/32; row 1: gate w = -2/32, up w = 1/32;
    # token 0: x = 1, token 1: x = 0.5
    gc = np.array([[9] * 32, [6] * 32]); uc = np.array([[10] * 32, [9] * 32])
    d = np.full((2, 1), 0x2800, dtype=np.uint16)
    Wg, Wu = H.encode_q4_0(gc, d), H.encode_q4_0(uc, d)
    x = np.stack([np.ones(32), np.full(32, 0.5)]).astype(np.float16)
    r = orc.swiglu(0, Wg, Wu, x, 2, 32)
    want = np.array([[_silu(1.0) * 2.0, _silu(-2.0) * 1.0], [_silu(0.5) * 1.0, _silu(-1.0) * 0.5]])
    np.testing.assert_allclose(r["y"], want, rtol=1e-15, atol=0)
    sub = orc.swiglu(0, Wg, Wu, x, 2, 32, rows=[1])
    np.testing.assert_allclose(sub["y"][:, 0], want[:, 1], rtol=1e-15, atol=0)


def test_silu_slope_bound():
    # the constant of the fused tolerance: sup of silu'(z) = s(z) (1 + z (1 - s(z)))
    z = np.linspace(-40, 40, 400001)
    s = 1.0 / (1.0 + np.exp(-z))
    slope = s * (1.0 + z * (1.0 - s))
    assert np.abs(slope).max() < H.SILU_SLOPE_MAX
    assert np.abs(slope).max() > 1.09


def test_swiglu_tolerance_helper(orc):
    x = np.ones((1, 32), dtype=np.float16)
    ref = orc.swiglu(0, _uniform_table(9, 0x2800), _uniform_table(10, 0x2800), x, 1, 32)
    assert H.swiglu_normalised_error(ref["y"], ref) == 0.0
    # a gate product off by its whole allowance (TOL * Sg) stays inside
    g2 = ref["g"] + H.TOL * ref["Sg"]
    y2 = g2 / (1 + np.exp(-g2)) * ref["u"]
    assert H.swiglu_normalised_error(y2, ref) <= H.TOL
    # ten times that does not
    g3 = ref["g"] + 10 * H.TOL * ref["Sg"]
    y3 = g3 / (1 + np.exp(-g3)) * ref["u"]
    assert H.swiglu_normalised_error(y3, ref) > H.TOL


# -- fp32 activations (values enter exactly; no narrowing to fp16) ---------------------

def test_f32_equals_f16_on_half_values(orc):
    # every fp16 value is an fp32 value: both entry points must give the same doubles
    for fmt, name in ((0, "q4_0"), (1, "q8_0")):
        W, x = _rand(name, 9, 768, 3, 11 + fmt)
        y16, S16 = orc.qmv(fmt, W, x, 9, 768)
        y32, S32 = orc.qmv(fmt, W, x.astype(np.float32), 9, 768)
        assert np.array_equal(y16, y32) and np.array_equal(S16, S32)
        r16, S16r = orc.qmv_rows(fmt, W, x, 9, 768, [8, 0, 3])
        r32, S32r = orc.qmv_rows(fmt, W, x.astype(np.float32), 9, 768, [8, 0, 3])
        assert np.array_equal(r16, r32) and np.array_equal(S16r, S32r)
    Wg, x = _rand("q4_0", 5, 512, 2, 21)
    Wu = synth.q4_0_weights(5, 512, 22)
    a, b = orc.swiglu(0, Wg, Wu, x, 5, 512), orc.swiglu(0, Wg, Wu, x.astype(np.float32), 5, 512)
    assert all(np.array_equal(a[k], b[k]) for k in a)


@pytest.mark.parametrize("xv,scale", [
    (1.0 + 2.0 ** -20, 1.0),            # fp32-exact, rounds to 1.0 in fp16
    (11184811 / 2.0 ** 25, 1.0),        # the fp32 nearest to 1/3 (fp16's is 0.333251953125)
    (1.0e6, 2.0 ** -10),                # far outside fp16's range
    (2.0 ** -130, 1.0),                 # an fp32 subnormal (zero in fp16)
])
def test_f32_activations_enter_exactly(orc, xv, scale):
    # Q8_0 row of K weights all equal to q * d = 3 * scale: y = 3 * scale * K * xv exactly
    K = 64
    d_bits = np.float16(scale).view(np.uint16)
    W = H.encode_q8_0(np.full((1, K), 3, dtype=np.int64), np.full((1, K // 32), d_bits, dtype=np.uint16))
    x = np.full((1, K), xv, dtype=np.float32)
    assert float(x[0, 0]) == xv
    y, S = orc.qmv(1, W, x, 1, K)
    assert y[0, 0] == 3.0 * scale * K * xv and S[0, 0] == abs(y[0, 0])


def test_f32_swiglu_closed_form(orc):
    # gate w = 1/32 and up w = 2/32 against 32 activations of 1 + 2^-20 (fp32-exact)
    e = 1.0 + 2.0 ** -20
    x = np.full((1, 32), e, dtype=np.float32)
    r = orc.swiglu(0, _uniform_table(9, 0x2800), _uniform_table(10, 0x2800), x, 1, 32)
    assert r["g"][0, 0] == e and r["u"][0, 0] == 2.0 * e
    assert r["y"][0, 0] == pytest.approx(_silu(e) * 2.0 * e, rel=1e-15)


# -- fp16 encoder and Q8_1 activations ---------------------------------------------------

def test_float_to_half_matches_numpy(orc):
    """Round to nearest even, against numpy's float32 -> float16 cast: every finite
    half, every midpoint between neighbours (the ties), a hair either side of
    each midpoint, and log-uniform random values of both signs."""
    bits = np.arange(0x0000, 0x7c00, dtype=np.uint16)           # finite non-negative halves
    h = bits.view(np.float16).astype(np.float32)
    mids = ((h[:-1].astype(np.float64) + h[1:].astype(np.float64)) / 2).astype(np.float32)
    hair = np.float32(1 + 2.0 ** -20)
    rng = np.random.default_rng(5)
    rnd = (2.0 ** rng.uniform(-30, 17, 20000)).astype(np.float32)
    vals = np.concatenate([h, mids, mids * hair, mids / hair, rnd, [65504, 65519.99, 65520, 65536, 1e9]]).astype(np.float32)
    vals = np.concatenate([vals, -vals])
    got = np.array([orc.float_to_half(v) for v in vals], dtype=np.uint16)
    with np.errstate(over="ignore"):                          # the values above 65520 are meant to overflow
        want = vals.astype(np.float16).view(np.uint16)
    bad = np.nonzero(got != want)[0]
    assert bad.size == 0, [(float(vals[i]), hex(got[i]), hex(want[i])) for i in bad[:5]]


def _q81(orc, x):
    return orc.quantize_q8_1(np.asarray(x, dtype=np.float16).reshape(1, -1))


def test_q8_1_closed_forms(orc):
    # amax = 127: d = 1, q = x exactly
    x = np.array(list(range(-127, 128, 8))[:31] + [127], dtype=np.float64)
    q, d, s = _q81(orc, x)
    assert np.array_equal(q[0], x.astype(np.int8)) and d[0, 0] == 0x3C00 and s[0, 0] == int(x.sum())
    # all zeros: d = 0, q = 0
    q, d, s = _q81(orc, np.zeros(32))
    assert not q.any() and d[0, 0] == 0 and s[0, 0] == 0
    # amax = 254: d = 2, id = 0.5; ties go away from zero (2.5 -> 3, -1.5 -> -2, 0.5 -> 1)
    x = np.zeros(32); x[:8] = [254, 5, -3, 1, -1, 2, 7, -254]
    q, d, s = _q81(orc, x)
    assert list(q[0, :8]) == [127, 3, -2, 1, -1, 1, 4, -127] and d[0, 0] == 0x4000
    assert s[0, 0] == 127 + 3 - 2 + 1 - 1 + 1 + 4 - 127
    # amax = 1: d = 1/127 stored as the nearest fp16 (0x2008: 0.0078735...)
    x = np.zeros(32); x[0] = 1.0; x[1] = -0.5
    q, d, s = _q81(orc, x)
    assert q[0, 0] == 127 and q[0, 1] == -64 and d[0, 0] == 0x2008   # -63.5 rounds away to -64


def test_q8_1_blocks_tokens_and_symmetry(orc):
    x = synth.activations(3, 256, 81)
    q, d, s = orc.quantize_q8_1(x)
    for m in range(3):
        for b in range(8):
            qb, db, sb = _q81(orc, x[m, 32 * b:32 * b + 32])
            assert np.array_equal(qb[0], q[m, 32 * b:32 * b + 32]) and db[0, 0] == d[m, b] and sb[0, 0] == s[m, b]
    qn, dn, sn = orc.quantize_q8_1(-x)
    assert np.array_equal(qn, -q) and np.array_equal(dn, d) and np.array_equal(sn, -s)
    assert np.array_equal(s, q.reshape(3, 8, 32).astype(np.int32).sum(axis=2))
    # every code within half a step of x (d in fp32 before its fp16 rounding)
    xf = x.astype(np.float64).reshape(3, 8, 32)
    dd = np.abs(xf).max(axis=2, keepdims=True) / 127
    assert np.all(np.abs(xf - q.reshape(3, 8, 32) * dd) <= dd * (0.5 + 1e-6))
    assert np.abs(q).max() == 127


def test_q8_1_product_integer_case_matches_numpy(orc):
    # Q4_0 with d = 1 against activations whose every block has max |x| = 127:
    # d_x = 1 and q = x, so y is the integer matmul
    rng = np.random.default_rng(82)
    N, K, M = 6, 256, 2
    codes = rng.integers(0, 16, size=(N, K))
    W = H.encode_q4_0(codes, np.full((N, K // 32), 0x3C00, dtype=np.uint16))
    x = rng.integers(-127, 128, size=(M, K))
    x.reshape(M, K // 32, 32)[:, :, 0] = 127
    q, d, s = orc.quantize_q8_1(x.astype(np.float16))
    assert np.array_equal(q, x) and np.all(d == 0x3C00)
    y, S = orc.qmv_q8_1(0, W, q, d, N, K)
    Wi = (codes - 8).astype(np.float64)
    assert np.array_equal(y, x.astype(np.float64) @ Wi.T)
    assert np.array_equal(S, np.abs(x).astype(np.float64) @ np.abs(Wi).T)


def test_q8_1_product_integer_case_q8_0(orc):
    # Q8_0 with d = 1 and codes over the whole signed range, against activations
    # whose every block has max |x| = 127: y is the integer matmul of the codes
    rng = np.random.default_rng(84)
    N, K, M = 5, 512, 3
    codes = rng.integers(-128, 128, size=(N, K))
    W = H.encode_q8_0(codes, np.full((N, K // 32), 0x3C00, dtype=np.uint16))
    x = rng.integers(-127, 128, size=(M, K))
    x.reshape(M, K // 32, 32)[:, :, 31] = -127
    q, d, s = orc.quantize_q8_1(x.astype(np.float16))
    assert np.array_equal(q, x) and np.all(d == 0x3C00)
    y, S = orc.qmv_q8_1(1, W, q, d, N, K)
    Wi = codes.astype(np.float64)
    assert np.array_equal(y, x.astype(np.float64) @ Wi.T)
    assert np.array_equal(S, np.abs(x).astype(np.float64) @ np.abs(Wi).T)


def test_q8_1_product_integer_case_q2w(orc):
    # plain 2-bit with d = 1 (codes 0..3, weights c - 2) against activations
    # whose every block has max |x| = 127: y is the integer matmul
    rng = np.random.default_rng(85)
    N, K, M = 4, 768, 2
    codes = rng.integers(0, 4, size=(N, K))
    W = H.encode_q2w(codes, np.full((N, K // 32), 0x3C00, dtype=np.uint16))
    x = rng.integers(-127, 128, size=(M, K))
    x.reshape(M, K // 32, 32)[:, :, 13] = 127
    q, d, s = orc.quantize_q8_1(x.astype(np.float16))
    assert np.array_equal(q, x) and np.all(d == 0x3C00)
    y, S = orc.qmv_q8_1(2, W, q, d, N, K)
    Wi = (codes - 2).astype(np.float64)
    assert np.array_equal(y, x.astype(np.float64) @ Wi.T)
    assert np.array_equal(S, np.abs(x).astype(np.float64) @ np.abs(Wi).T)


def test_q8_1_product_is_the_product_on_dequantised_x(orc):
    N, K, M = 9, 768, 3
    W, x = _rand("q4_0", N, K, M, 83)
    q, d, _ = orc.quantize_q8_1(x)
    xhat = (q.reshape(M, K // 32, 32).astype(np.float32)
            * d.view(np.float16).astype(np.float32)[:, :, None]).reshape(M, K)   # exact in fp32
    y1, S1 = orc.qmv_q8_1(0, W, q, d, N, K)
    y2, S2 = orc.qmv(0, W, xhat, N, K)
    assert np.array_equal(y1, y2) and np.array_equal(S1, S2)
    yr, Sr = orc.qmv_q8_1(0, W, q, d, N, K, rows=[8, 0, 4])
    assert np.array_equal(yr, y1[:, [8, 0, 4]]) and np.array_equal(Sr, S1[:, [8, 0, 4]])
    # against the exact product: the quantisation error stays within its bound
    # sum |w| * (d_fp32 / 2 + |q| * |fp16(d) - d|) per output (w from the oracle's dequantisation)
    ye, _ = orc.qmv(0, W, x, N, K)
    wabs = np.abs(np.stack([orc.dequant_row(0, W, n, K) for n in range(N)]))
    xf = x.astype(np.float64).reshape(M, K // 32, 32)
    dd = np.abs(xf).max(axis=2) / 127
    dq = d.view(np.float16).astype(np.float64)
    per_x = (dd[:, :, None] / 2 + np.abs(q.reshape(M, K // 32, 32)) * np.abs(dq - dd)[:, :, None]).reshape(M, K)
    bound = per_x @ wabs.T
    assert np.all(np.abs(y1 - ye) <= bound * (1 + 1e-9))
