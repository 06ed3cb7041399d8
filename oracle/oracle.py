"""ctypes wrapper around ``qmv_oracle.c`` (test infrastructure only).

The C file is compiled with gcc into ``oracle/_build/`` on first use.  All
arithmetic lives in the C file; this module only moves numpy buffers in and
out.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

FMT_Q4_0 = 0
FMT_Q8_0 = 1
FMT_Q2W = 2

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "qmv_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LOCK = threading.Lock()

_i64 = ctypes.c_int64
_ptr = ctypes.c_void_p


def build(src: str = _SRC, out: str | None = None, force: bool = False) -> str:
    """Compile ``src`` into a shared library and return its path."""
    if out is None:
        os.makedirs(_BUILD, exist_ok=True)
        out = os.path.join(_BUILD, "liboracle.so")
    if force or not os.path.exists(out) or os.path.getmtime(out) < os.path.getmtime(src):
        tmp = out + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-shared", "-fPIC", src, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, out)
    return out


class Oracle:
    """One loaded copy of the oracle library (the default one, or a test's)."""

    def __init__(self, path: str):
        lib = ctypes.CDLL(path)
        lib.oracle_half_to_double.restype = ctypes.c_double
        lib.oracle_half_to_double.argtypes = [ctypes.c_uint16]
        lib.oracle_block_bytes.restype = _i64
        lib.oracle_block_bytes.argtypes = [ctypes.c_int]
        lib.oracle_dequant_row.restype = ctypes.c_int
        lib.oracle_dequant_row.argtypes = [ctypes.c_int, _ptr, _i64, _i64, _ptr]
        lib.oracle_qmv_rows.restype = ctypes.c_int
        lib.oracle_qmv_rows.argtypes = [ctypes.c_int, _ptr, _ptr, _i64, _i64, _i64,
                                        _ptr, _i64, _ptr, _ptr, ctypes.c_int]
        lib.oracle_qmv.restype = ctypes.c_int
        lib.oracle_qmv.argtypes = [ctypes.c_int, _ptr, _ptr, _i64, _i64, _i64,
                                   _ptr, _ptr, ctypes.c_int]
        lib.oracle_moe.restype = ctypes.c_int
        lib.oracle_moe.argtypes = [ctypes.c_int, _ptr, _ptr, _i64, _ptr, _i64, _i64, _i64,
                                   _ptr, _ptr, ctypes.c_int]
        lib.oracle_swiglu_rows.restype = ctypes.c_int
        lib.oracle_swiglu_rows.argtypes = [ctypes.c_int, _ptr, _ptr, _ptr, _i64, _i64, _i64, _ptr, _i64,
                                           _ptr, _ptr, _ptr, _ptr, _ptr, ctypes.c_int]
        lib.oracle_qmv_rows_f32.restype = ctypes.c_int
        lib.oracle_qmv_rows_f32.argtypes = lib.oracle_qmv_rows.argtypes
        lib.oracle_swiglu_rows_f32.restype = ctypes.c_int
        lib.oracle_swiglu_rows_f32.argtypes = lib.oracle_swiglu_rows.argtypes
        lib.oracle_float_to_half.restype = ctypes.c_uint16
        lib.oracle_float_to_half.argtypes = [ctypes.c_float]
        lib.oracle_quantize_q8_1.restype = ctypes.c_int
        lib.oracle_quantize_q8_1.argtypes = [_ptr, _i64, _i64, _ptr, _ptr, _ptr]
        lib.oracle_qmv_q8_1_rows.restype = ctypes.c_int
        lib.oracle_qmv_q8_1_rows.argtypes = [ctypes.c_int, _ptr, _ptr, _ptr, _i64, _i64, _i64, _ptr, _i64,
                                             _ptr, _ptr, ctypes.c_int]
        lib.oracle_max_threads.restype = ctypes.c_int
        lib.oracle_max_threads.argtypes = []
        self.lib = lib
        self.path = path

    # -- helpers -----------------------------------------------------------
    @staticmethod
    def _u8(a) -> np.ndarray:
        a = np.ascontiguousarray(a)
        return a.view(np.uint8).reshape(-1)

    @staticmethod
    def _x_bits(x) -> np.ndarray:
        x = np.ascontiguousarray(x)
        if x.dtype == np.float16:
            x = x.view(np.uint16)
        if x.dtype != np.uint16:
            raise TypeError("x must be float16 (or its uint16 bit patterns)")
        return x

    @classmethod
    def _x_arg(cls, x):
        """(activations as passed to C, True for fp32): float32 arrays go to the
        fp32 entry points, float16 / uint16 ones to the fp16 entry points."""
        x = np.ascontiguousarray(x)
        if x.dtype == np.float32:
            return x, True
        return cls._x_bits(x), False

    def half_to_double(self, bits: int) -> float:
        return self.lib.oracle_half_to_double(int(bits) & 0xFFFF)

    def block_bytes(self, fmt: int) -> int:
        return int(self.lib.oracle_block_bytes(fmt))

    def dequant_row(self, fmt: int, W, n: int, K: int) -> np.ndarray:
        Wb = self._u8(W)
        w = np.empty(K, dtype=np.float64)
        rc = self.lib.oracle_dequant_row(fmt, Wb.ctypes.data, n, K, w.ctypes.data)
        if rc != 0:
            raise ValueError(f"oracle_dequant_row failed ({rc})")
        return w

    def qmv(self, fmt: int, W, x, N: int, K: int, nthreads: int = 1):
        """Return (y, S), both float64 [M][N].  x is float16 (or its uint16 bit
        patterns) or float32; either way its values enter the fp64 sums exactly."""
        Wb = self._u8(W)
        xb, f32 = self._x_arg(x)
        xb = xb.reshape(xb.shape[0], K) if xb.ndim == 2 else xb.reshape(-1, K)
        M = xb.shape[0]
        if Wb.size < N * (K // 32) * self.block_bytes(fmt):
            raise ValueError("W buffer too small")
        y = np.empty((M, N), dtype=np.float64)
        S = np.empty((M, N), dtype=np.float64)
        if f32:
            rc = self.lib.oracle_qmv_rows_f32(fmt, Wb.ctypes.data, xb.ctypes.data, N, K, M, None, N,
                                              y.ctypes.data, S.ctypes.data, nthreads)
        else:
            rc = self.lib.oracle_qmv(fmt, Wb.ctypes.data, xb.ctypes.data, N, K, M,
                                     y.ctypes.data, S.ctypes.data, nthreads)
        if rc != 0:
            raise ValueError(f"oracle_qmv failed ({rc})")
        return y, S

    def qmv_rows(self, fmt: int, W, x, N: int, K: int, rows, nthreads: int = 1):
        """(y, S) for the listed rows only: float64 [M][len(rows)]."""
        Wb = self._u8(W)
        xb, f32 = self._x_arg(x)
        xb = xb.reshape(-1, K)
        M = xb.shape[0]
        rows = np.ascontiguousarray(rows, dtype=np.int64)
        y = np.empty((M, rows.size), dtype=np.float64)
        S = np.empty((M, rows.size), dtype=np.float64)
        fn = self.lib.oracle_qmv_rows_f32 if f32 else self.lib.oracle_qmv_rows
        rc = fn(fmt, Wb.ctypes.data, xb.ctypes.data, N, K, M,
                rows.ctypes.data, rows.size, y.ctypes.data, S.ctypes.data, nthreads)
        if rc != 0:
            raise ValueError(f"oracle_qmv_rows failed ({rc})")
        return y, S

    def moe(self, fmt: int, W_pool, idx, n_experts: int, x, N: int, K: int, nthreads: int = 1):
        """(y, S), float64 [n_slots][N]; raises on an out-of-range index."""
        Wb = self._u8(W_pool)
        idx = np.ascontiguousarray(idx, dtype=np.int32)
        xb = self._x_bits(x).reshape(-1, K)
        n_slots = idx.size
        if xb.shape[0] != n_slots:
            raise ValueError("one token per slot")
        y = np.full((n_slots, N), np.nan)
        S = np.full((n_slots, N), np.nan)
        rc = self.lib.oracle_moe(fmt, Wb.ctypes.data, idx.ctypes.data, n_experts, xb.ctypes.data,
                                 N, K, n_slots, y.ctypes.data, S.ctypes.data, nthreads)
        if rc != 0:
            raise ValueError(f"oracle_moe failed ({rc})")
        return y, S

    def swiglu(self, fmt: int, Wg, Wu, x, N: int, K: int, rows=None, nthreads: int = 1):
        """Gate + up + SwiGLU: dict of float64 [M][n] arrays y, g, u, Sg, Su
        (n = N, or len(rows) for the listed rows)."""
        Wgb, Wub = self._u8(Wg), self._u8(Wu)
        xb, f32 = self._x_arg(x)
        xb = xb.reshape(-1, K)
        M = xb.shape[0]
        need = N * (K // 32) * self.block_bytes(fmt)
        if Wgb.size < need or Wub.size < need:
            raise ValueError("W buffer too small")
        if rows is None:
            rp, nr = None, N
        else:
            rows = np.ascontiguousarray(rows, dtype=np.int64)
            rp, nr = rows.ctypes.data, rows.size
        out = {k: np.empty((M, nr), dtype=np.float64) for k in ("y", "g", "u", "Sg", "Su")}
        fn = self.lib.oracle_swiglu_rows_f32 if f32 else self.lib.oracle_swiglu_rows
        rc = fn(fmt, Wgb.ctypes.data, Wub.ctypes.data, xb.ctypes.data, N, K, M, rp, nr,
                                         out["y"].ctypes.data, out["g"].ctypes.data, out["u"].ctypes.data,
                                         out["Sg"].ctypes.data, out["Su"].ctypes.data, nthreads)
        if rc != 0:
            raise ValueError(f"oracle_swiglu_rows failed ({rc})")
        return out

    def float_to_half(self, f: float) -> int:
        return int(self.lib.oracle_float_to_half(float(f)))

    def quantize_q8_1(self, x):
        """Q8_1 blocks of fp16 activations [M][K]: (q int8 [M][K], d_bits uint16
        [M][K/32] (the fp16 scales), sumq int32 [M][K/32])."""
        xb = self._x_bits(x)
        xb = xb.reshape(xb.shape[0], -1) if xb.ndim == 2 else xb.reshape(1, -1)
        M, K = xb.shape
        q = np.empty((M, K), dtype=np.int8)
        d = np.empty((M, K // 32), dtype=np.uint16)
        s = np.empty((M, K // 32), dtype=np.int32)
        rc = self.lib.oracle_quantize_q8_1(xb.ctypes.data, M, K, q.ctypes.data, d.ctypes.data, s.ctypes.data)
        if rc != 0:
            raise ValueError(f"oracle_quantize_q8_1 failed ({rc})")
        return q, d, s

    def qmv_q8_1(self, fmt: int, W, q, d_bits, N: int, K: int, rows=None, nthreads: int = 1):
        """(y, S) of the weights against Q8_1 activations (q, d_bits): float64 [M][n]."""
        Wb = self._u8(W)
        q = np.ascontiguousarray(q, dtype=np.int8).reshape(-1, K)
        d_bits = np.ascontiguousarray(d_bits, dtype=np.uint16).reshape(q.shape[0], K // 32)
        M = q.shape[0]
        if rows is None:
            rp, nr = None, N
        else:
            rows = np.ascontiguousarray(rows, dtype=np.int64)
            rp, nr = rows.ctypes.data, rows.size
        y = np.empty((M, nr), dtype=np.float64)
        S = np.empty((M, nr), dtype=np.float64)
        rc = self.lib.oracle_qmv_q8_1_rows(fmt, Wb.ctypes.data, q.ctypes.data, d_bits.ctypes.data, N, K, M,
                                           rp, nr, y.ctypes.data, S.ctypes.data, nthreads)
        if rc != 0:
            raise ValueError(f"oracle_qmv_q8_1_rows failed ({rc})")
        return y, S

    def max_threads(self) -> int:
        return int(self.lib.oracle_max_threads())


_DEFAULT: Oracle | None = None


def default() -> Oracle:
    global _DEFAULT
    with _LOCK:
        if _DEFAULT is None:
            _DEFAULT = Oracle(build())
        return _DEFAULT


def half_to_double(bits: int) -> float:
    return default().half_to_double(bits)


def block_bytes(fmt: int) -> int:
    return default().block_bytes(fmt)


def dequant_row(fmt, W, n, K):
    return default().dequant_row(fmt, W, n, K)


def qmv(fmt, W, x, N, K, nthreads=1):
    return default().qmv(fmt, W, x, N, K, nthreads)


def swiglu(fmt, Wg, Wu, x, N, K, rows=None, nthreads=1):
    return default().swiglu(fmt, Wg, Wu, x, N, K, rows, nthreads)


def qmv_rows(fmt, W, x, N, K, rows, nthreads=1):
    return default().qmv_rows(fmt, W, x, N, K, rows, nthreads)


def moe(fmt, W_pool, idx, n_experts, x, N, K, nthreads=1):
    return default().moe(fmt, W_pool, idx, n_experts, x, N, K, nthreads)


def max_threads() -> int:
    return default().max_threads()
