"""Test-side helpers: fixture parser, tolerance, and a GGUF encoder for
integer special cases.  None of this is used by the product path."""
from __future__ import annotations

import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
FMT = {"q4_0": 0, "q8_0": 1, "q2w": 2}
BLOCK_BYTES = {"q4_0": 18, "q8_0": 34, "q2w": 10}
TOL = 2e-3  # max |y - y_ref| / (S + 1e-6) per output


def normalised_error(y, y_ref, S):
    y = np.asarray(y, dtype=np.float64)
    y_ref = np.asarray(y_ref, dtype=np.float64)
    S = np.asarray(S, dtype=np.float64)
    if y.size == 0:
        return 0.0
    err = np.abs(y - y_ref) / (S + 1e-6)
    err = np.where(np.isnan(err), np.inf, err)
    return float(err.max())


SILU_SLOPE_MAX = 1.1   # sup |d silu / dz| = 1.0998 (at z = 2.40)


def swiglu_normalised_error(y, ref):
    """Fused gate + up + SwiGLU against the oracle (dict with y, g, u, Sg, Su).

    Each of the two products carries the GEMV bound |dg| <= TOL * Sg,
    |du| <= TOL * Su; through y = silu(g) * u (mean value theorem on silu):
        |dy| <= TOL * (1.1 * Sg * (|u| + TOL * Su) + |silu(g)| * Su).
    Returns max |y - y_ref| / (that bound / TOL + 1e-6), to compare with TOL."""
    y = np.asarray(y, dtype=np.float64)
    g, u = ref["g"], ref["u"]
    if y.size == 0:
        return 0.0
    silu = g / (1.0 + np.exp(-g))
    scale = SILU_SLOPE_MAX * ref["Sg"] * (np.abs(u) + TOL * ref["Su"]) + np.abs(silu) * ref["Su"]
    err = np.abs(y - ref["y"]) / (scale + 1e-6)
    err = np.where(np.isnan(err), np.inf, err)
    return float(err.max())


def _x_spec(spec, K):
    kind = spec[0]
    j = np.arange(K, dtype=np.float64)
    if kind == "seq":
        v = j + 1
    elif kind == "square":
        v = (j + 1) ** 2
    elif kind == "fill":
        v = np.full(K, float(spec[1]))
    elif kind == "onehot":
        k, val, base = int(spec[1]), float(spec[2]), float(spec[3])
        v = np.full(K, base)
        v[k] = val
    elif kind == "split":
        k, a, b = int(spec[1]), float(spec[2]), float(spec[3])
        v = np.where(j < k, a, b)
    else:
        raise ValueError(kind)
    x = v.astype(np.float16)
    assert np.array_equal(x.astype(np.float64), v), "fixture x must be exact in fp16"
    return x


def load_cases(name):
    """Parse a golden fixture file into a list of dicts."""
    cases, cur = [], None
    with open(os.path.join(GOLDEN, name)) as f:
        for raw in f:
            line = raw.split("#", 1)[0].strip() if not raw.lstrip().startswith("cite") else raw.strip()
            if not line:
                continue
            tok = line.split()
            key = tok[0]
            if key == "case":
                cur = {"name": tok[1], "blocks": [], "x": {}, "y": {}, "S": {}, "moe": None}
            elif key == "cite":
                pass
            elif key == "fmt":
                cur["fmt"] = tok[1]
            elif key == "shape":
                kv = dict(t.split("=") for t in tok[1:])
                cur["N"], cur["K"], cur["M"] = int(kv["N"]), int(kv["K"]), int(kv["M"])
            elif key == "moe":
                kv = dict(t.split("=") for t in tok[1:])
                cur["moe"] = (int(kv["n_experts"]), [int(v) for v in kv["idx"].split(",")])
            elif key == "block":
                cur["blocks"].append((int(tok[1]), int(tok[2]), bytes.fromhex(tok[3])))
            elif key == "x":
                cur["x"][int(tok[1])] = tok[2:]
            elif key in ("y", "S"):
                cur[key][(int(tok[1]), int(tok[2]))] = float(tok[3])
            elif key == "end":
                cases.append(_finish(cur))
                cur = None
            else:
                raise ValueError(f"bad fixture line: {line}")
    return cases


def _finish(c):
    fmt, N, K, M = c["fmt"], c["N"], c["K"], c["M"]
    bb = BLOCK_BYTES[fmt]
    rows = N if c["moe"] is None else N * c["moe"][0]
    W = np.zeros((rows, (K // 32) * bb), dtype=np.uint8)
    seen = set()
    for r, b, data in c["blocks"]:
        assert len(data) == bb, (c["name"], len(data))
        W[r, b * bb:(b + 1) * bb] = np.frombuffer(data, dtype=np.uint8)
        seen.add((r, b))
    assert len(seen) == rows * (K // 32), f"{c['name']}: every block must be listed"
    x = np.stack([_x_spec(c["x"][m], K) for m in range(M)])
    c["W"], c["xarr"] = W, x
    return c


# -- a GGUF encoder for integer special cases (the inverse of the format) -----

def encode_q4_0(codes, d_bits):
    """codes: int array [N, K] in 0..15; d_bits: uint16 [N, K/32] -> bytes."""
    N, K = codes.shape
    nb = K // 32
    c = codes.reshape(N, nb, 32).astype(np.uint8)
    out = np.empty((N, nb, 18), dtype=np.uint8)
    out[:, :, 0] = d_bits & 0xFF
    out[:, :, 1] = d_bits >> 8
    out[:, :, 2:18] = c[:, :, :16] | (c[:, :, 16:] << 4)
    return out.reshape(N, nb * 18)


def encode_q8_0(codes, d_bits):
    """codes: int array [N, K] in -128..127; d_bits: uint16 [N, K/32] -> bytes."""
    N, K = codes.shape
    nb = K // 32
    out = np.empty((N, nb, 34), dtype=np.uint8)
    out[:, :, 0] = d_bits & 0xFF
    out[:, :, 1] = d_bits >> 8
    out[:, :, 2:34] = codes.reshape(N, nb, 32).astype(np.int8).view(np.uint8)
    return out.reshape(N, nb * 34)


def encode_q2w(codes, d_bits):
    """codes: int array [N, K] in 0..3 (w = (c - 2) d); d_bits: uint16 [N, K/32]
    -> bytes (element j in bits 2*(j//8) of byte j % 8 of its block)."""
    N, K = codes.shape
    nb = K // 32
    c = codes.reshape(N, nb, 4, 8).astype(np.uint8)      # [.., plane, byte]
    out = np.empty((N, nb, 10), dtype=np.uint8)
    out[:, :, 0] = d_bits & 0xFF
    out[:, :, 1] = d_bits >> 8
    out[:, :, 2:10] = c[:, :, 0] | (c[:, :, 1] << 2) | (c[:, :, 2] << 4) | (c[:, :, 3] << 6)
    return out.reshape(N, nb * 10)


def sabotage(W, fmt):
    """Flip code bits in every code byte (scales untouched), after
    volta-kernel-bakeoff, 'Making it fair' (its sabotage switch breaks the
    packed weights): XOR 0x88 moves each Q4_0 code by 8 in its top bit (every
    weight by +-8d); for the 2-bit format XOR 0xAA moves every code by 2."""
    bb = BLOCK_BYTES[fmt]
    W = np.array(W, dtype=np.uint8, copy=True)
    v = W.reshape(W.shape[0], -1, bb)
    v[:, :, 2:] ^= 0xAA if fmt == "q2w" else 0x88
    return W
