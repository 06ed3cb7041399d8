"""weight_quantized_decode_gb300 -- block-quantised (GGUF Q4_0 / Q8_0) weight x
activation products for single-stream decode on one GB300 (sm_103a).

A thin ctypes binding over the C ABI in ``include/qmv.h`` (``libqmv.so``,
built in-tree by ``build.py``).  It only marshals arguments: every step of the
computation runs in the library's CUDA kernels.  There is no CPU path; calls
raise if the library is missing or a tensor is not on a CUDA device.

Functions (same names as the C ABI):
    qmv_q4_0(W, x, y=None, stream=None)          -> y fp32 [M, N]
    qmv_q8_0(W, x, y=None, stream=None)          -> y fp32 [M, N]
    qmv_q4_0_swiglu(W_gate, W_up, x, y=None, stream=None) -> silu(gate) * up, fp32 [M, N]
    qmv_q4_0_f32, qmv_q4_0_swiglu_f32            -> the same two with fp32 x
    qmv_q2w(W, x, y=None, stream=None)           -> plain 2-bit weights, y fp32 [M, N]
    qmv_q4_0_q8_1(W, x, y=None, stream=None)     -> Q4_0 against Q8_1-quantised x (integer dots)
    qmv_quantize_q8_1(x, stream=None)            -> (q, d_bits, sumq) of the Q8_1 activations
    qmv_q4_0_q8_1_pre(W, q, d_bits, sumq, ...)   -> the Q8_1 product on activations already quantised
    qmv_moe(W_pool, expert_idx, n_experts, x, N, y=None, stream=None)
    qmm_q4_0_prefill(W, x, y=None, stream=None)  -> y fp32 [M, N]
    qmm_q8_0_prefill(W, x, y=None, stream=None)  -> y fp32 [M, N]
    qmv_device_status(stream=None)               -> int (QMV_DEV_* bits, cleared)
    qmv_read_probe(buf, out=None, stream=None)   -> checksum tensor (read-only bandwidth probe)
    qmv_set_pdl(enable), qmv_status_str(code), qmv_version()
Raw-pointer forms (``*_ptr``) take integers and are what the benchmark times.
"""
from __future__ import annotations

import ctypes
import os
import threading

_HERE = os.path.dirname(os.path.abspath(__file__))
# QMV_LIB selects another build of the same library (the phase-timeline
# variant of phase_timeline.py); there is no CPU path either way.
LIB_PATH = os.environ.get("QMV_LIB") or os.path.join(_HERE, "libqmv.so")

QMV_OK = 0
QMV_DEV_BAD_EXPERT = 0x1
QMV_DEV_TIMEOUT = 0x2
Q4_0_BLOCK_BYTES = 18
Q8_0_BLOCK_BYTES = 34
Q2W_BLOCK_BYTES = 10

_lock = threading.Lock()
_lib = None


class QmvError(RuntimeError):
    def __init__(self, fn, code):
        super().__init__(f"{fn} failed: {qmv_status_str(code)} ({code})")
        self.code = code


def lib():
    """Load ``libqmv.so`` (raises loudly if it has not been built)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: run weight_quantized_decode_gb300/build.py "
                               "(there is no CPU fallback)")
        L = ctypes.CDLL(LIB_PATH)
        vp, i64 = ctypes.c_void_p, ctypes.c_int64
        for name in ("qmv_q4_0", "qmv_q8_0", "qmm_q4_0_prefill", "qmm_q8_0_prefill", "qmv_q4_0_f32", "qmv_q2w", "qmv_q4_0_q8_1",
                     "qmv_q8_0_q8_1"):
            f = getattr(L, name)
            f.restype = ctypes.c_int
            f.argtypes = [vp, vp, vp, i64, i64, i64, vp]
        L.qmv_moe.restype = ctypes.c_int
        L.qmv_moe.argtypes = [vp, vp, i64, vp, vp, i64, i64, i64, vp]
        L.qmv_q4_0_swiglu.restype = ctypes.c_int
        L.qmv_q4_0_swiglu.argtypes = [vp, vp, vp, vp, i64, i64, i64, vp]
        L.qmv_q4_0_q8_1_pre.restype = ctypes.c_int
        L.qmv_q4_0_q8_1_pre.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, vp]
        L.qmv_q8_0_q8_1_pre.restype = ctypes.c_int
        L.qmv_q8_0_q8_1_pre.argtypes = [vp, vp, vp, vp, i64, i64, i64, vp]
        L.qmv_quantize_q8_1.restype = ctypes.c_int
        L.qmv_quantize_q8_1.argtypes = [vp, vp, vp, vp, i64, i64, vp]
        L.qmv_q4_0_swiglu_f32.restype = ctypes.c_int
        L.qmv_q4_0_swiglu_f32.argtypes = [vp, vp, vp, vp, i64, i64, i64, vp]
        L.qmv_device_status.restype = ctypes.c_int
        L.qmv_device_status.argtypes = [vp, ctypes.POINTER(ctypes.c_int32)]
        L.qmv_read_probe.restype = ctypes.c_int
        L.qmv_read_probe.argtypes = [vp, i64, vp, vp]
        L.qmv_set_pdl.restype = None
        L.qmv_set_pdl.argtypes = [ctypes.c_int]
        L.qmv_status_str.restype = ctypes.c_char_p
        L.qmv_status_str.argtypes = [ctypes.c_int]
        L.qmv_version.restype = ctypes.c_char_p
        L.qmv_version.argtypes = []
        _lib = L
        return L


def qmv_status_str(code: int) -> str:
    return lib().qmv_status_str(int(code)).decode()


def qmv_version() -> str:
    return lib().qmv_version().decode()


def qmv_set_pdl(enable: bool) -> None:
    lib().qmv_set_pdl(1 if enable else 0)


# -- raw-pointer entry points ------------------------------------------------------

def _check(fn, code):
    if code != QMV_OK:
        raise QmvError(fn, code)


def qmv_q4_0_swiglu_ptr(W_gate: int, W_up: int, x: int, y: int, N: int, K: int, M: int,
                        stream: int = 0) -> None:
    _check("qmv_q4_0_swiglu", lib().qmv_q4_0_swiglu(W_gate, W_up, x, y, N, K, M, stream))


def qmv_q4_0_ptr(W: int, x: int, y: int, N: int, K: int, M: int, stream: int = 0) -> None:
    _check("qmv_q4_0", lib().qmv_q4_0(W, x, y, N, K, M, stream))


def qmv_q4_0_f32_ptr(W: int, x: int, y: int, N: int, K: int, M: int, stream: int = 0) -> None:
    _check("qmv_q4_0_f32", lib().qmv_q4_0_f32(W, x, y, N, K, M, stream))


def qmv_q4_0_swiglu_f32_ptr(W_gate: int, W_up: int, x: int, y: int, N: int, K: int, M: int,
                            stream: int = 0) -> None:
    _check("qmv_q4_0_swiglu_f32", lib().qmv_q4_0_swiglu_f32(W_gate, W_up, x, y, N, K, M, stream))


def qmv_q8_0_ptr(W: int, x: int, y: int, N: int, K: int, M: int, stream: int = 0) -> None:
    _check("qmv_q8_0", lib().qmv_q8_0(W, x, y, N, K, M, stream))


def qmv_q4_0_q8_1_ptr(W: int, x: int, y: int, N: int, K: int, M: int, stream: int = 0) -> None:
    _check("qmv_q4_0_q8_1", lib().qmv_q4_0_q8_1(W, x, y, N, K, M, stream))


def qmv_q4_0_q8_1_pre_ptr(W: int, q: int, d_bits: int, sumq: int, y: int, N: int, K: int, M: int,
                          stream: int = 0) -> None:
    _check("qmv_q4_0_q8_1_pre", lib().qmv_q4_0_q8_1_pre(W, q, d_bits, sumq, y, N, K, M, stream))


def qmv_q8_0_q8_1_ptr(W: int, x: int, y: int, N: int, K: int, M: int, stream: int = 0) -> None:
    _check("qmv_q8_0_q8_1", lib().qmv_q8_0_q8_1(W, x, y, N, K, M, stream))


def qmv_q8_0_q8_1_pre_ptr(W: int, q: int, d_bits: int, y: int, N: int, K: int, M: int, stream: int = 0) -> None:
    _check("qmv_q8_0_q8_1_pre", lib().qmv_q8_0_q8_1_pre(W, q, d_bits, y, N, K, M, stream))


def qmv_quantize_q8_1_ptr(x: int, q: int, d_bits: int, sumq: int, M: int, K: int, stream: int = 0) -> None:
    _check("qmv_quantize_q8_1", lib().qmv_quantize_q8_1(x, q, d_bits, sumq, M, K, stream))


def qmv_q2w_ptr(W: int, x: int, y: int, N: int, K: int, M: int, stream: int = 0) -> None:
    _check("qmv_q2w", lib().qmv_q2w(W, x, y, N, K, M, stream))


def qmv_moe_ptr(W_pool: int, idx: int, n_experts: int, x: int, y: int, N: int, K: int, M: int,
                stream: int = 0) -> None:
    _check("qmv_moe", lib().qmv_moe(W_pool, idx, n_experts, x, y, N, K, M, stream))


def qmm_q4_0_prefill_ptr(W: int, x: int, y: int, N: int, K: int, M: int, stream: int = 0) -> None:
    _check("qmm_q4_0_prefill", lib().qmm_q4_0_prefill(W, x, y, N, K, M, stream))


def qmm_q8_0_prefill_ptr(W: int, x: int, y: int, N: int, K: int, M: int, stream: int = 0) -> None:
    _check("qmm_q8_0_prefill", lib().qmm_q8_0_prefill(W, x, y, N, K, M, stream))


def qmv_read_probe_ptr(buf: int, nbytes: int, out: int, stream: int = 0) -> None:
    _check("qmv_read_probe", lib().qmv_read_probe(buf, nbytes, out, stream))


# -- torch-tensor entry points ---------------------------------------------------------

def _torch():
    import torch
    return torch


def _stream_handle(stream):
    torch = _torch()
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream) if hasattr(stream, "cuda_stream") else int(stream)


def _on_device(fn, *tensors):
    """All tensors on one CUDA device; returns a context that makes it current.
    The library launches on the current device and takes its status word and
    SM count from it, so a call on another device's tensors must switch first."""
    torch = _torch()
    dev = tensors[0].device
    for t in tensors[1:]:
        if t.device != dev:
            raise ValueError(f"{fn}: all tensors must be on one device ({dev} and {t.device})")
    return torch.cuda.device(dev)


def _check_y(y, M, N, fn):
    torch = _torch()
    if not (y.is_cuda and y.dtype == torch.float32 and y.is_contiguous() and y.numel() == M * N):
        raise ValueError(f"{fn}: y must be a contiguous CUDA float32 tensor of {M}x{N}")


def _prep(W, x, y, block_bytes, fn, x_dtype=None):
    torch = _torch()
    x_dtype = torch.float16 if x_dtype is None else x_dtype
    if not (W.is_cuda and x.is_cuda):
        raise TypeError(f"{fn}: W and x must be CUDA tensors (no CPU path)")
    if W.dtype != torch.uint8:
        raise TypeError(f"{fn}: W must be uint8 GGUF bytes")
    if x.dtype != x_dtype:
        raise TypeError(f"{fn}: x must be {str(x_dtype).replace('torch.', '')}")
    if x.dim() == 1:
        x = x.unsqueeze(0)
    if not (W.is_contiguous() and x.is_contiguous()):
        raise ValueError(f"{fn}: W and x must be contiguous")
    M, K = x.shape
    if K % 32:
        raise ValueError(f"{fn}: K={K} is not a multiple of 32")
    row_bytes = (K // 32) * block_bytes
    if row_bytes == 0:
        N = W.shape[0] if W.dim() >= 1 else 0
    else:
        if W.numel() % row_bytes:
            raise ValueError(f"{fn}: W size {W.numel()} is not a whole number of rows of {row_bytes} bytes")
        N = W.numel() // row_bytes
    if y is None:
        y = torch.empty((M, N), dtype=torch.float32, device=x.device)
    else:
        _check_y(y, M, N, fn)
    return W, x, y, N, K, M


def qmv_q4_0(W, x, y=None, stream=None):
    """y[M, N] = x[M, K] @ dequant(W)^T for Q4_0 weights ``W`` (uint8, N rows)."""
    W, x, y, N, K, M = _prep(W, x, y, Q4_0_BLOCK_BYTES, "qmv_q4_0")
    with _on_device("qmv_q4_0", W, x, y):
        qmv_q4_0_ptr(W.data_ptr(), x.data_ptr(), y.data_ptr(), N, K, M, _stream_handle(stream))
    return y


def qmv_q4_0_f32(W, x, y=None, stream=None):
    """qmv_q4_0 with float32 activations, rounded to fp16 inside the kernel."""
    W, x, y, N, K, M = _prep(W, x, y, Q4_0_BLOCK_BYTES, "qmv_q4_0_f32", _torch().float32)
    with _on_device("qmv_q4_0_f32", W, x, y):
        qmv_q4_0_f32_ptr(W.data_ptr(), x.data_ptr(), y.data_ptr(), N, K, M, _stream_handle(stream))
    return y


def _check_up(W_gate, W_up, fn):
    torch = _torch()
    if not (W_up.is_cuda and W_up.dtype == torch.uint8 and W_up.is_contiguous()
            and W_up.numel() == W_gate.numel()):
        raise ValueError(f"{fn}: W_up must be a contiguous CUDA uint8 table shaped like W_gate")


def qmv_q4_0_swiglu(W_gate, W_up, x, y=None, stream=None):
    """y[M, N] = silu(x @ dequant(W_gate)^T) * (x @ dequant(W_up)^T) for two
    Q4_0 tables of N rows each (the MLP's gate + up + SwiGLU in one call)."""
    W_gate, x, y, N, K, M = _prep(W_gate, x, y, Q4_0_BLOCK_BYTES, "qmv_q4_0_swiglu")
    _check_up(W_gate, W_up, "qmv_q4_0_swiglu")
    with _on_device("qmv_q4_0_swiglu", W_gate, W_up, x, y):
        qmv_q4_0_swiglu_ptr(W_gate.data_ptr(), W_up.data_ptr(), x.data_ptr(), y.data_ptr(), N, K, M,
                            _stream_handle(stream))
    return y


def qmv_q4_0_swiglu_f32(W_gate, W_up, x, y=None, stream=None):
    """qmv_q4_0_swiglu with float32 activations, rounded to fp16 inside the kernel."""
    W_gate, x, y, N, K, M = _prep(W_gate, x, y, Q4_0_BLOCK_BYTES, "qmv_q4_0_swiglu_f32", _torch().float32)
    _check_up(W_gate, W_up, "qmv_q4_0_swiglu_f32")
    with _on_device("qmv_q4_0_swiglu_f32", W_gate, W_up, x, y):
        qmv_q4_0_swiglu_f32_ptr(W_gate.data_ptr(), W_up.data_ptr(), x.data_ptr(), y.data_ptr(), N, K, M,
                                _stream_handle(stream))
    return y


def qmv_q8_0(W, x, y=None, stream=None):
    """y[M, N] = x[M, K] @ dequant(W)^T for Q8_0 weights."""
    W, x, y, N, K, M = _prep(W, x, y, Q8_0_BLOCK_BYTES, "qmv_q8_0")
    with _on_device("qmv_q8_0", W, x, y):
        qmv_q8_0_ptr(W.data_ptr(), x.data_ptr(), y.data_ptr(), N, K, M, _stream_handle(stream))
    return y


def qmv_q4_0_q8_1(W, x, y=None, stream=None):
    """qmv_q4_0 with the activations quantised to Q8_1 in the kernel (integer dots)."""
    W, x, y, N, K, M = _prep(W, x, y, Q4_0_BLOCK_BYTES, "qmv_q4_0_q8_1")
    with _on_device("qmv_q4_0_q8_1", W, x, y):
        qmv_q4_0_q8_1_ptr(W.data_ptr(), x.data_ptr(), y.data_ptr(), N, K, M, _stream_handle(stream))
    return y


def _prep_pre(W, q, d_bits, sumq, y, block_bytes, fn):
    """Checks shared by the calls on activations already in Q8_1 (sumq may be None)."""
    torch = _torch()
    tensors = [W, q, d_bits] + ([sumq] if sumq is not None else [])
    if not all(t.is_cuda for t in tensors):
        raise TypeError(f"{fn}: all tensors must be on a CUDA device (no CPU path)")
    if W.dtype != torch.uint8 or q.dtype != torch.int8 or d_bits.dtype != torch.int16 or \
            (sumq is not None and sumq.dtype != torch.int32):
        raise TypeError(f"{fn}: W uint8, q int8, d_bits int16" + (", sumq int32" if sumq is not None else ""))
    if q.dim() == 1:
        q = q.unsqueeze(0)
    M, K = q.shape
    if K % 32 or d_bits.numel() != M * (K // 32) or (sumq is not None and sumq.numel() != M * (K // 32)):
        raise ValueError(f"{fn}: q [M, K] with K % 32 == 0, d_bits" + (" and sumq" if sumq is not None else "")
                         + " [M, K/32]")
    if not all(t.is_contiguous() for t in tensors):
        raise ValueError(f"{fn}: tensors must be contiguous")
    row_bytes = (K // 32) * block_bytes
    if row_bytes and W.numel() % row_bytes:
        raise ValueError(f"{fn}: W size {W.numel()} is not a whole number of rows of {row_bytes} bytes")
    N = W.numel() // row_bytes if row_bytes else (W.shape[0] if W.dim() >= 1 else 0)
    if y is None:
        y = torch.empty((M, N), dtype=torch.float32, device=q.device)
    else:
        _check_y(y, M, N, fn)
    return q, y, N, K, M


def qmv_q4_0_q8_1_pre(W, q, d_bits, sumq, y=None, stream=None):
    """qmv_q4_0_q8_1 on activations already in Q8_1 (q int8 [M, K], d_bits int16
    [M, K/32], sumq int32 [M, K/32], as qmv_quantize_q8_1 returns them)."""
    q, y, N, K, M = _prep_pre(W, q, d_bits, sumq, y, Q4_0_BLOCK_BYTES, "qmv_q4_0_q8_1_pre")
    with _on_device("qmv_q4_0_q8_1_pre", W, q, d_bits, sumq, y):
        qmv_q4_0_q8_1_pre_ptr(W.data_ptr(), q.data_ptr(), d_bits.data_ptr(), sumq.data_ptr(), y.data_ptr(), N, K,
                              M, _stream_handle(stream))
    return y


def qmv_q8_0_q8_1(W, x, y=None, stream=None):
    """qmv_q8_0 with the activations quantised to Q8_1 in the kernel (signed integer dots)."""
    W, x, y, N, K, M = _prep(W, x, y, Q8_0_BLOCK_BYTES, "qmv_q8_0_q8_1")
    with _on_device("qmv_q8_0_q8_1", W, x, y):
        qmv_q8_0_q8_1_ptr(W.data_ptr(), x.data_ptr(), y.data_ptr(), N, K, M, _stream_handle(stream))
    return y


def qmv_q8_0_q8_1_pre(W, q, d_bits, y=None, stream=None):
    """qmv_q8_0_q8_1 on activations already in Q8_1 (q int8 [M, K], d_bits int16
    [M, K/32]; the code sums qmv_quantize_q8_1 also returns are not needed)."""
    q, y, N, K, M = _prep_pre(W, q, d_bits, None, y, Q8_0_BLOCK_BYTES, "qmv_q8_0_q8_1_pre")
    with _on_device("qmv_q8_0_q8_1_pre", W, q, d_bits, y):
        qmv_q8_0_q8_1_pre_ptr(W.data_ptr(), q.data_ptr(), d_bits.data_ptr(), y.data_ptr(), N, K, M,
                              _stream_handle(stream))
    return y


def qmv_quantize_q8_1(x, stream=None):
    """Q8_1 blocks of fp16 activations [M, K] on the GPU: (q int8 [M, K],
    d_bits int16 [M, K/32] holding the fp16 scales' bits, sumq int32 [M, K/32])."""
    torch = _torch()
    if not x.is_cuda or x.dtype != torch.float16:
        raise TypeError("qmv_quantize_q8_1: x must be a float16 CUDA tensor (no CPU path)")
    if x.dim() == 1:
        x = x.unsqueeze(0)
    x = x.contiguous()
    M, K = x.shape
    q = torch.empty((M, K), dtype=torch.int8, device=x.device)
    d = torch.empty((M, K // 32), dtype=torch.int16, device=x.device)
    s = torch.empty((M, K // 32), dtype=torch.int32, device=x.device)
    with _on_device("qmv_quantize_q8_1", x):
        qmv_quantize_q8_1_ptr(x.data_ptr(), q.data_ptr(), d.data_ptr(), s.data_ptr(), M, K, _stream_handle(stream))
    return q, d, s


def qmv_q2w(W, x, y=None, stream=None):
    """y[M, N] = x[M, K] @ dequant(W)^T for plain 2-bit weights (10-byte blocks)."""
    W, x, y, N, K, M = _prep(W, x, y, Q2W_BLOCK_BYTES, "qmv_q2w")
    with _on_device("qmv_q2w", W, x, y):
        qmv_q2w_ptr(W.data_ptr(), x.data_ptr(), y.data_ptr(), N, K, M, _stream_handle(stream))
    return y


def qmm_q4_0_prefill(W, x, y=None, stream=None):
    """Many-token (prefill) form of qmv_q4_0 on the tensor cores."""
    W, x, y, N, K, M = _prep(W, x, y, Q4_0_BLOCK_BYTES, "qmm_q4_0_prefill")
    with _on_device("qmm_q4_0_prefill", W, x, y):
        qmm_q4_0_prefill_ptr(W.data_ptr(), x.data_ptr(), y.data_ptr(), N, K, M, _stream_handle(stream))
    return y


def qmm_q8_0_prefill(W, x, y=None, stream=None):
    """Many-token (prefill) form of qmv_q8_0 on the tensor cores."""
    W, x, y, N, K, M = _prep(W, x, y, Q8_0_BLOCK_BYTES, "qmm_q8_0_prefill")
    with _on_device("qmm_q8_0_prefill", W, x, y):
        qmm_q8_0_prefill_ptr(W.data_ptr(), x.data_ptr(), y.data_ptr(), N, K, M, _stream_handle(stream))
    return y


def qmv_moe(W_pool, expert_idx, n_experts, x, N, y=None, stream=None):
    """Slot s: y[s] = x[s] @ dequant(expert expert_idx[s])^T, all slots in one launch."""
    torch = _torch()
    if not (W_pool.is_cuda and x.is_cuda and expert_idx.is_cuda):
        raise TypeError("qmv_moe: W_pool, expert_idx and x must be CUDA tensors (no CPU path)")
    if expert_idx.dtype != torch.int32 or not expert_idx.is_contiguous():
        raise TypeError("qmv_moe: expert_idx must be a contiguous int32 CUDA tensor")
    if W_pool.dtype != torch.uint8 or x.dtype != torch.float16:
        raise TypeError("qmv_moe: W_pool must be uint8, x float16")
    if x.dim() == 1:
        x = x.unsqueeze(0)
    if not (W_pool.is_contiguous() and x.is_contiguous()):
        raise ValueError("qmv_moe: W_pool and x must be contiguous")
    M, K = x.shape
    if expert_idx.numel() != M:
        raise ValueError("qmv_moe: one expert index per token")
    need = n_experts * N * (K // 32) * Q4_0_BLOCK_BYTES
    if W_pool.numel() < need:
        raise ValueError(f"qmv_moe: W_pool holds {W_pool.numel()} bytes, needs {need}")
    if y is None:
        y = torch.empty((M, N), dtype=torch.float32, device=x.device)
    else:
        _check_y(y, M, N, "qmv_moe")
    with _on_device("qmv_moe", W_pool, expert_idx, x, y):
        qmv_moe_ptr(W_pool.data_ptr(), expert_idx.data_ptr(), int(n_experts), x.data_ptr(), y.data_ptr(),
                    int(N), int(K), int(M), _stream_handle(stream))
    return y


def qmv_read_probe(buf, out=None, stream=None):
    """Stream the bytes of the CUDA tensor ``buf`` (a multiple of 256 bytes) through
    the read-only bandwidth probe; returns the device uint32 checksum tensor ``out``
    (an int32 view: the XOR of the 16 bytes at every 256-byte offset, as 32-bit words)."""
    torch = _torch()
    if not (buf.is_cuda and buf.is_contiguous()):
        raise ValueError("qmv_read_probe: buf must be a contiguous CUDA tensor (no CPU path)")
    if out is None:
        out = torch.empty(1, dtype=torch.int32, device=buf.device)
    with _on_device("qmv_read_probe", buf, out):
        qmv_read_probe_ptr(buf.data_ptr(), buf.numel() * buf.element_size(), out.data_ptr(), _stream_handle(stream))
    return out


def qmv_device_status(stream=None) -> int:
    """Read and clear the device status word (synchronises the stream)."""
    out = ctypes.c_int32(0)
    _check("qmv_device_status", lib().qmv_device_status(_stream_handle(stream), ctypes.byref(out)))
    return int(out.value)
