"""Planted mistakes in the oracle must be caught by its pins.

Each mutant is a one-line edit of oracle/qmv_oracle.c of the kind a careless
rewrite could make (a dropped term, a wrong sign, index or stride, a transposed
operand, a swapped nibble or byte order).  The mutant is compiled into a
temporary directory and the whole oracle pin suite (tests/test_oracle.py) is run
against it in a subprocess; the suite must fail.  The planted mistakes live
only in the temporary copy, on the CPU.
"""
import os
import subprocess
import sys

import pytest

from oracle import oracle as O

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "qmv_oracle.c")

# (name, original snippet, mutated snippet, occurrence index)
MUTANTS = [
    ("nibbles_swapped", "int lo = qs[j] & 0x0f;\n        int hi = qs[j] >> 4;",
     "int hi = qs[j] & 0x0f;\n        int lo = qs[j] >> 4;", 0),
    ("nibbles_interleaved", "w[j] = (double)(lo - 8) * d;\n        w[j + 16] = (double)(hi - 8) * d;",
     "w[2 * j] = (double)(lo - 8) * d;\n        w[2 * j + 1] = (double)(hi - 8) * d;", 0),
    ("low_bias_dropped", "(double)(lo - 8) * d", "(double)(lo) * d", 0),
    ("high_bias_dropped", "(double)(hi - 8) * d", "(double)(hi) * d", 0),
    ("high_index_shifted", "w[j + 16] =", "w[(j + 17) % 32] =", 0),
    ("q4_scale_big_endian", "(uint16_t)(blk[0] | (blk[1] << 8))", "(uint16_t)(blk[1] | (blk[0] << 8))", 0),
    ("q8_scale_big_endian", "(uint16_t)(blk[0] | (blk[1] << 8))", "(uint16_t)(blk[1] | (blk[0] << 8))", 1),
    ("half_exponent_bias", "expo - 25", "expo - 24", 0),
    ("half_subnormal_scale", "ldexp((double)mant, -24)", "ldexp((double)mant, -25)", 0),
    ("half_sign_ignored", "return sign ? -v : v;", "return v;", 0),
    ("half_implicit_bit", "(double)(1024 + mant)", "(double)(mant)", 0),
    ("q8_codes_unsigned", "const int8_t *q = (const int8_t *)(blk + 2);",
     "const uint8_t *q = (const uint8_t *)(blk + 2);", 0),
    ("q8_codes_offset", "const int8_t *q = (const int8_t *)(blk + 2);",
     "const int8_t *q = (const int8_t *)(blk + 1);", 0),
    ("q8_scale_dropped", "w[j] = (double)q[j] * d;", "w[j] = (double)q[j];", 0),
    ("x_transposed", "xd[m * K + k]", "xd[k * M + m]", 0),
    ("row_stride", "W + n * nblk * bb", "W + n * (nblk - 1) * bb", 0),
    ("q4_block_stride", "dequant_block_q4_0(row + b * bb, w + 32 * b)",
     "dequant_block_q4_0(row + b * 16, w + 32 * b)", 0),
    ("q4_block_order", "dequant_block_q4_0(row + b * bb, w + 32 * b)",
     "dequant_block_q4_0(row + b * bb, w + 32 * (nblk - 1 - b))", 0),
    ("q8_block_stride", "dequant_block_q8_0(row + b * bb, w + 32 * b)",
     "dequant_block_q8_0(row + b * 32, w + 32 * b)", 0),
    ("S_without_abs", "sabs += fabs(p);", "sabs += p;", 0),
    ("y_with_abs", "acc += p;", "acc += fabs(p);", 0),
    ("y_layout_transposed", "y[m * nrows + r] = acc;", "y[r * M + m] = acc;", 0),
    ("moe_slot_as_expert", "int32_t e = idx[s];", "int32_t e = (int32_t)s;", 0),
    ("moe_shared_token", "x + s * K,", "x,", 0),
    ("moe_expert_stride", "int64_t expert_bytes = N * (K / 32) * bb;",
     "int64_t expert_bytes = (N - 1) * (K / 32) * bb;", 0),
    ("moe_output_offset", "y + s * N, S + s * N", "y, S", 0),
    ("silu_sign", "gate / (1.0 + exp(-gate)) * u[i]", "gate / (1.0 + exp(gate)) * u[i]", 0),
    ("silu_dropped", "y[i] = gate / (1.0 + exp(-gate)) * u[i];", "y[i] = gate * u[i];", 0),
    ("sigmoid_without_gate", "y[i] = gate / (1.0 + exp(-gate)) * u[i];", "y[i] = 1.0 / (1.0 + exp(-gate)) * u[i];", 0),
    ("gate_and_up_swapped", "const double gate = g[i];\n        y[i] = gate / (1.0 + exp(-gate)) * u[i];",
     "const double gate = u[i];\n        y[i] = gate / (1.0 + exp(-gate)) * g[i];", 0),
    ("up_table_is_gate", "rc = qmv_rows_xd(fmt, Wu, xd,", "rc = qmv_rows_xd(fmt, Wg, xd,", 0),
    ("q2w_sequential_order", "int c = (qs[j % 8] >> (2 * (j / 8))) & 3;",
     "int c = (qs[j / 4] >> (2 * (j % 4))) & 3;", 0),
    ("q2w_planes_reversed", "int c = (qs[j % 8] >> (2 * (j / 8))) & 3;",
     "int c = (qs[j % 8] >> (6 - 2 * (j / 8))) & 3;", 0),
    ("q2w_bias_dropped", "w[j] = (double)(c - 2) * d;", "w[j] = (double)(c) * d;", 0),
    ("q2w_bias_off_by_one", "w[j] = (double)(c - 2) * d;", "w[j] = (double)(c - 1) * d;", 0),
    ("q2w_scale_dropped", "w[j] = (double)(c - 2) * d;", "w[j] = (double)(c - 2);", 0),
    ("q2w_block_bytes", "if (fmt == ORACLE_FMT_Q2W) return 10;", "if (fmt == ORACLE_FMT_Q2W) return 8;", 0),
    ("f2h_ties_away", "double mant = rint((2.0 * m - 1.0) * 1024.0);",
     "double mant = round((2.0 * m - 1.0) * 1024.0);", 0),
    ("f2h_truncates", "double mant = rint((2.0 * m - 1.0) * 1024.0);",
     "double mant = floor((2.0 * m - 1.0) * 1024.0);", 0),
    ("f2h_overflow_at_max", "if (v >= 65520.0) return", "if (v > 65504.0) return", 0),
    ("f2h_subnormal_scale", "rint(v * ldexp(1.0, 24))", "rint(v * ldexp(1.0, 23))", 0),
    ("q8_1_ties_to_even", "const int c = (int)roundf(t);", "const int c = (int)rintf(t);", 0),
    ("q8_1_scale_128", "const float d = amax / 127.0f;", "const float d = amax / 128.0f;", 0),
    ("q8_1_amax_signed", "const float a = fabsf(xf[i]);", "const float a = xf[i];", 0),
    ("q8_1_sum_first_only", "s += c;", "s = c;", 0),
    ("q8_1_scale_per_token", "xd[m * K + k] = (double)q[m * K + k] * oracle_half_to_double(d_bits[m * (K / 32) + k / 32]);",
     "xd[m * K + k] = (double)q[m * K + k] * oracle_half_to_double(d_bits[m * (K / 32)]);", 0),
    ("f32_narrowed_to_half", "xd[i] = (double)x[i];", "xd[i] = (double)(_Float16)x[i];", 0),
    ("f32_read_as_half", "double *xd = widen_float(x, M * K);",
     "double *xd = widen_half((const uint16_t *)x, M * K);", 0),
    ("f32_swiglu_read_as_half", "double *xd = widen_float(x, M * K);",
     "double *xd = widen_half((const uint16_t *)x, M * K);", 1),
]


def _mutate(src, old, new, occ):
    pos = -1
    for _ in range(occ + 1):
        pos = src.find(old, pos + 1)
        assert pos >= 0, f"snippet not found: {old!r}"
    return src[:pos] + new + src[pos + len(old):]


@pytest.mark.parametrize("name,old,new,occ", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(tmp_path, name, old, new, occ):
    src = open(SRC).read()
    mutated = _mutate(src, old, new, occ)
    assert mutated != src
    msrc = tmp_path / "mutant.c"
    msrc.write_text(mutated)
    lib = O.build(str(msrc), str(tmp_path / "libmutant.so"), force=True)
    env = dict(os.environ, QMV_ORACLE_LIB=lib)
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_oracle.py")],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode != 0, f"mutant {name} survived the oracle pins:\n{r.stdout[-2000:]}"


def test_unmutated_oracle_passes_through_same_route(tmp_path):
    lib = O.build(SRC, str(tmp_path / "libclean.so"), force=True)
    env = dict(os.environ, QMV_ORACLE_LIB=lib)
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_oracle.py")],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stdout[-2000:]
