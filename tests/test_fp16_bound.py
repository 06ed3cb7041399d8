"""The decode kernels' fp16 partial sums cannot overflow (CPU check).

Each half of a half2 chain in the streaming kernel sums eight products
w' * x, w' the pre-scaled weight and x a finite fp16 activation, before the
chain is converted to fp32.  Round-to-nearest is monotone, so the magnitude of
the i-th partial sum is at most B_i, where B_1 = fp16(max|w'| * 65504) and
B_i = fp16(B_{i-1} + B_1).  This test reads the pre-scales the kernels are
compiled with and replays that sequence in exact fp16 rounding: every B_i must
be finite.  The page's rule is /64 for a lane that sums two words of Q4_0
codes (volta-kernel-bakeoff, "A few tokens at once"); /32 with eight products
is the overflow this guards against, and the check must catch it.
"""
import os
import re
from fractions import Fraction

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
COMMON = os.path.join(ROOT, "weight_quantized_decode_gb300", "csrc", "qmv_common.cuh")

FP16_MAX = 65504.0
CHAIN = 8                      # products per half of a chain (two 32-bit code words)
MAX_CODE = {"Q4": 8, "Q8": 128, "Q2": 2}    # largest |centred code|: c - 8, int8 q, c - 2


def prescales():
    src = open(COMMON).read()
    out = {}
    for name in MAX_CODE:
        m = re.search(rf"constexpr float k{name}Prescale = ([0-9.]+)f;", src)
        assert m, f"k{name}Prescale not found"
        out[name] = float(m.group(1))
    return out


def fp16(v):
    """Round a double to the nearest fp16 (ties to even), as the HFMA2 does."""
    with np.errstate(over="ignore"):
        return float(np.float16(v))


def bound_sequence(max_w):
    p = fp16(max_w * FP16_MAX)
    seq = [p]
    for _ in range(CHAIN - 1):
        seq.append(fp16(seq[-1] + p))
    return seq


@pytest.mark.parametrize("name", list(MAX_CODE))
def test_chain_partial_sums_stay_finite(name):
    pre = prescales()[name]
    assert pre > 0 and Fraction(pre).denominator == 1 and (int(pre) & (int(pre) - 1)) == 0, \
        "the pre-scale must be a power of two (exact in fp16 and undone exactly in fp32)"
    seq = bound_sequence(MAX_CODE[name] / pre)
    assert all(np.isfinite(v) and v <= FP16_MAX for v in seq), (name, pre, seq)


def test_the_check_catches_the_old_prescale():
    # Q4_0 at /32 (|w'| <= 1/4): the sixth partial sum already overflows.
    seq = bound_sequence(8 / 32.0)
    assert not all(np.isfinite(seq))
    # Q8_0 at /512 likewise.
    assert not all(np.isfinite(bound_sequence(128 / 512.0)))


def test_fp16_rounding_helper():
    # 65519 rounds down to the largest finite half, 65520 (the midpoint) to inf.
    assert fp16(65519.0) == FP16_MAX
    assert np.isinf(fp16(65520.0))
    # ties to even: 2049 lies between 2048 and 2050
    assert fp16(2049.0) == 2048.0 and fp16(2051.0) == 2052.0
