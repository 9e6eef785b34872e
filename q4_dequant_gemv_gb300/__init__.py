"""Python binding of the GB300 Q4_K decode library (libq4k.so, C ABI in include/q4k.h).

Argument marshalling only: every step of the computation runs in the library's
CUDA kernels.  torch supplies device memory and the current CUDA stream.  There
is no CPU fallback: if the library is not built or cannot load, every call
raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libq4k.so")

Q4K_OK = 0
Q4K_FLAG_PDL = 1
Q4K_FLAG_TENSOR_CORE = 2
Q4K_FLAG_Q8K_X = 4
Q4K_FLAG_TEST_STALL = 8
Q4K_FLAG_ROWS16 = 16
QK = 256
QBYTES = 144
MAX_BATCH = 16

_lock = threading.Lock()
_lib = None


class Q4KError(RuntimeError):
    def __init__(self, fn: str, status: int, text: str):
        super().__init__(f"{fn} failed: status {status} ({text})")
        self.status = status


class LaunchOpts(ctypes.Structure):
    _fields_ = [("split_k", ctypes.c_int), ("flags", ctypes.c_uint), ("wait_limit_us", ctypes.c_uint),
                ("reserved", ctypes.c_int * 5)]


class GemvGroup(ctypes.Structure):
    _fields_ = [("W", ctypes.c_void_p), ("y", ctypes.c_void_p), ("N", ctypes.c_int64)]


# Every symbol the header declares (checked by the CPU tests).
EXPORTS = ("q4k_status_string", "q4k_abi_version", "q4k_gemv", "q4k_gemv_argmax", "q4k_gemv_argmax_debug",
           "q4k_gemv_argmax_noalloc", "q4k_gemm_prefill", "q4k_gemm_prefill_exact", "q4k_gemv_ex",
           "q4k_gemv_grouped", "q4k_gemv_plan",
           "q4k_device_error_flags", "q4k_device_error_clear", "q4k_stream_read", "q6k_gemv",
           "q6k_planar_bytes", "q6k_repack_planar", "q6k_gemv_planar")


def lib():
    """Load libq4k.so (raises if missing -- there is no fallback path)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"libq4k.so is not built ({LIB_PATH}); run __graft_entry__.build()")
        L = ctypes.CDLL(LIB_PATH)
        P, I64, I = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
        L.q4k_status_string.argtypes = [I]
        L.q4k_status_string.restype = ctypes.c_char_p
        L.q4k_abi_version.restype = I
        L.q4k_gemv.argtypes = [P, P, P, I64, I64, I, P]
        L.q4k_gemv.restype = I
        L.q4k_gemv_ex.argtypes = [P, P, P, I64, I64, I, P, ctypes.POINTER(LaunchOpts)]
        L.q4k_gemv_ex.restype = I
        L.q4k_gemv_grouped.argtypes = [ctypes.POINTER(GemvGroup), I, P, I64, I, P, ctypes.POINTER(LaunchOpts)]
        L.q4k_gemv_grouped.restype = I
        L.q4k_gemv_argmax.argtypes = [P, P, P, I64, I64, I, P]
        L.q4k_gemv_argmax.restype = I
        L.q4k_gemv_argmax_debug.argtypes = [P, P, P, P, I64, I64, I, P]
        L.q4k_gemv_argmax_debug.restype = I
        L.q4k_gemv_argmax_noalloc.argtypes = [P, P, P, I64, I64, I, P]
        L.q4k_gemv_argmax_noalloc.restype = I
        L.q4k_gemm_prefill.argtypes = [P, P, P, I64, I64, I64, P]
        L.q4k_gemm_prefill_exact.argtypes = [P, P, P, I64, I64, I64, P]
        L.q4k_gemm_prefill_exact.restype = I
        L.q6k_gemv.argtypes = [P, P, P, I64, I64, I, P]
        L.q6k_gemv.restype = I
        L.q6k_planar_bytes.argtypes = [I64, I64]
        L.q6k_planar_bytes.restype = I64
        L.q6k_repack_planar.argtypes = [P, P, I64, I64, P]
        L.q6k_repack_planar.restype = I
        L.q6k_gemv_planar.argtypes = [P, P, P, I64, I64, I, P]
        L.q6k_gemv_planar.restype = I
        L.q4k_gemm_prefill.restype = I
        L.q4k_gemv_plan.argtypes = [I64, I64, I, ctypes.POINTER(ctypes.c_int * 4)]
        L.q4k_gemv_plan.restype = I
        L.q4k_device_error_flags.restype = ctypes.c_uint
        L.q4k_device_error_clear.restype = I
        L.q4k_stream_read.argtypes = [P, I64, ctypes.POINTER(ctypes.c_int64), P]
        L.q4k_stream_read.restype = I
        _lib = L
        return L


def status_string(s: int) -> str:
    return lib().q4k_status_string(int(s)).decode()


def _check(fn: str, st: int):
    if st != Q4K_OK:
        raise Q4KError(fn, st, status_string(st))


def _stream_ptr(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _dev(t, name, dtype, cuda=True):
    import torch
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must have dtype {dtype}, got {t.dtype}")
    if cuda and not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t


def _shape_wk(W, K):
    N = W.shape[0]
    if W.dim() != 2 or W.shape[1] != (K // QK) * QBYTES:
        raise ValueError(f"W must be uint8 [N, K/256*144] for K={K}, got {tuple(W.shape)}")
    return N


def _flags(pdl: bool, tensor_core: bool, q8k: bool = False, rows16: bool = False) -> int:
    return ((Q4K_FLAG_PDL if pdl else 0) | (Q4K_FLAG_TENSOR_CORE if tensor_core else 0)
            | (Q4K_FLAG_Q8K_X if q8k else 0) | (Q4K_FLAG_ROWS16 if rows16 else 0))


def gemv(W, x, y=None, *, stream=None, split_k: int = 0, pdl: bool = False, tensor_core: bool = False,
         q8k: bool = False, wait_limit_us: int = 0, test_stall: bool = False, rows16: bool = False):
    """y [B, N] (fp32) = W_q4k [N, K] . x [B, K] (fp32); x may also be [K].
    tensor_core: batch 1 on the tensor-core inner product instead of the integer one.
    q8k: batch 1 with x quantized Q8_K style (int8 codes per 256-block), its own error bound.
    rows16: batch 1 on the 16-row-tile kernel (chosen automatically where it applies).
    wait_limit_us, test_stall: bound of the kernel's waits, and a wait made to run out (failure tests)."""
    import torch
    _dev(W, "W", torch.uint8)
    _dev(x, "x", torch.float32)
    squeeze = x.dim() == 1
    x2 = x.view(1, -1) if squeeze else x
    B, K = x2.shape
    N = _shape_wk(W, K)
    if y is None:
        y = torch.empty((B, N), dtype=torch.float32, device=x.device)
    _dev(y, "y", torch.float32)
    if y.numel() != B * N:
        raise ValueError("y has the wrong size")
    L = lib()
    if split_k or pdl or tensor_core or q8k or wait_limit_us or test_stall or rows16:
        o = LaunchOpts(split_k, _flags(pdl, tensor_core, q8k, rows16) | (Q4K_FLAG_TEST_STALL if test_stall else 0),
                       int(wait_limit_us))
        st = L.q4k_gemv_ex(W.data_ptr(), x2.data_ptr(), y.data_ptr(), N, K, B, _stream_ptr(stream), ctypes.byref(o))
        _check("q4k_gemv_ex", st)
    else:
        st = L.q4k_gemv(W.data_ptr(), x2.data_ptr(), y.data_ptr(), N, K, B, _stream_ptr(stream))
        _check("q4k_gemv", st)
    return y.view(N) if squeeze and y.dim() == 2 else y


def q6k_gemv(W, x, y=None, *, stream=None):
    """y [B, N] (fp32) = W_q6k [N, K] . x [B, K] (fp32); x may also be [K]."""
    import torch
    _dev(W, "W", torch.uint8)
    _dev(x, "x", torch.float32)
    squeeze = x.dim() == 1
    x2 = x.view(1, -1) if squeeze else x
    B, K = x2.shape
    if K % 256 or W.dim() != 2 or W.shape[1] != (K // 256) * 210:
        raise ValueError(f"W must be [N, {(K // 256) * 210}] uint8 for K={K}")
    N = W.shape[0]
    if y is None:
        y = torch.empty((B, N), dtype=torch.float32, device=x.device)
    _dev(y, "y", torch.float32)
    if y.numel() != B * N:
        raise ValueError("y has the wrong size")
    st = lib().q6k_gemv(W.data_ptr(), x2.data_ptr(), y.data_ptr(), N, K, B, _stream_ptr(stream))
    _check("q6k_gemv", st)
    return y.view(N) if squeeze and y.dim() == 2 else y


def q6k_planar_bytes(N: int, K: int) -> int:
    """Size in bytes of the planar form of an N x K Q6_K matrix."""
    n = lib().q6k_planar_bytes(N, K)
    if n < 0:
        raise ValueError(f"bad Q6_K shape {N} x {K}")
    return n


def q6k_repack_planar(W, K: int, Wp=None, *, stream=None):
    """The planar form (flat uint8 tensor) of the Q6_K matrix W [N, K/256*210]."""
    import torch
    _dev(W, "W", torch.uint8)
    if K % 256 or W.dim() != 2 or W.shape[1] != (K // 256) * 210:
        raise ValueError(f"W must be [N, {(K // 256) * 210}] uint8 for K={K}")
    N = W.shape[0]
    nbytes = q6k_planar_bytes(N, K)
    if Wp is None:
        Wp = torch.empty(nbytes, dtype=torch.uint8, device=W.device)
    _dev(Wp, "Wp", torch.uint8)
    if Wp.numel() != nbytes:
        raise ValueError(f"Wp must hold {nbytes} bytes")
    _check("q6k_repack_planar", lib().q6k_repack_planar(W.data_ptr(), Wp.data_ptr(), N, K, _stream_ptr(stream)))
    return Wp


def q6k_gemv_planar(Wp, x, N: int, y=None, *, stream=None):
    """y [B, N] (fp32) = W x from the planar form Wp of W; x [B, K] (fp32) or [K]."""
    import torch
    _dev(Wp, "Wp", torch.uint8)
    _dev(x, "x", torch.float32)
    squeeze = x.dim() == 1
    x2 = x.view(1, -1) if squeeze else x
    B, K = x2.shape
    if Wp.numel() != q6k_planar_bytes(N, K):
        raise ValueError("Wp does not hold a planar N x K matrix")
    if y is None:
        y = torch.empty((B, N), dtype=torch.float32, device=x.device)
    _dev(y, "y", torch.float32)
    if y.numel() != B * N:
        raise ValueError("y has the wrong size")
    _check("q6k_gemv_planar", lib().q6k_gemv_planar(Wp.data_ptr(), x2.data_ptr(), y.data_ptr(), N, K, B,
                                                    _stream_ptr(stream)))
    return y.view(N) if squeeze and y.dim() == 2 else y


def gemv_grouped(Ws, x, ys=None, *, stream=None, split_k: int = 0, pdl: bool = False, tensor_core: bool = False,
                 q8k: bool = False, rows16: bool = False):
    """Several Q4_K matrices times the same x in one launch: returns [y_g [B, N_g]]."""
    import torch
    if not 1 <= len(Ws) <= 4:
        raise ValueError("1 to 4 matrices")
    _dev(x, "x", torch.float32)
    x2 = x.view(1, -1) if x.dim() == 1 else x
    B, K = x2.shape
    if ys is None:
        ys = [torch.empty((B, W.shape[0]), dtype=torch.float32, device=x.device) for W in Ws]
    arr = (GemvGroup * len(Ws))()
    for i, (W, y) in enumerate(zip(Ws, ys)):
        _dev(W, "W", torch.uint8)
        _dev(y, "y", torch.float32)
        N = _shape_wk(W, K)
        if y.numel() != B * N:
            raise ValueError("y has the wrong size")
        arr[i] = GemvGroup(W.data_ptr(), y.data_ptr(), N)
    o = LaunchOpts(split_k, _flags(pdl, tensor_core, q8k, rows16))
    st = lib().q4k_gemv_grouped(arr, len(Ws), x2.data_ptr(), K, B, _stream_ptr(stream), ctypes.byref(o))
    _check("q4k_gemv_grouped", st)
    return ys


def gemv_argmax(W, x, idx=None, *, logits=None, stream=None):
    """int32 idx [B] = argmax_n (W . x[b])[n] (lowest index on ties)."""
    import torch
    _dev(W, "W", torch.uint8)
    _dev(x, "x", torch.float32)
    x2 = x.view(1, -1) if x.dim() == 1 else x
    B, K = x2.shape
    N = _shape_wk(W, K)
    if idx is None:
        idx = torch.empty(B, dtype=torch.int32, device=x.device)
    _dev(idx, "idx", torch.int32)
    L = lib()
    if logits is not None:
        _dev(logits, "logits", torch.float32)
        st = L.q4k_gemv_argmax_debug(W.data_ptr(), x2.data_ptr(), idx.data_ptr(), logits.data_ptr(), N, K, B,
                                     _stream_ptr(stream))
        _check("q4k_gemv_argmax_debug", st)
    else:
        st = L.q4k_gemv_argmax(W.data_ptr(), x2.data_ptr(), idx.data_ptr(), N, K, B, _stream_ptr(stream))
        _check("q4k_gemv_argmax", st)
    return idx


def gemm_prefill(W, X, Y=None, *, stream=None, exact=False):
    """Y [T, N] (fp32) = X [T, K] (bf16) . W_q4k^T; exact=True: q4k_gemm_prefill_exact (no weight rounding)."""
    import torch
    _dev(W, "W", torch.uint8)
    _dev(X, "X", torch.bfloat16)
    T, K = X.shape
    N = _shape_wk(W, K)
    if Y is None:
        Y = torch.empty((T, N), dtype=torch.float32, device=X.device)
    _dev(Y, "Y", torch.float32)
    fn = "q4k_gemm_prefill_exact" if exact else "q4k_gemm_prefill"
    st = getattr(lib(), fn)(W.data_ptr(), X.data_ptr(), Y.data_ptr(), N, K, T, _stream_ptr(stream))
    _check(fn, st)
    return Y


def gemv_plan(N: int, K: int, batch: int):
    out = (ctypes.c_int * 4)()
    _check("q4k_gemv_plan", lib().q4k_gemv_plan(N, K, batch, ctypes.byref(out)))
    return {"split_k": out[0], "ctas": out[1], "rows_per_tile": out[2], "x_chunk_blocks": out[3]}


def stream_read(buf, *, stream=None) -> int:
    """Read-only streaming probe over a device buffer (any dtype, contiguous):
    launches the probe kernel and returns the number of bytes it streams."""
    import torch
    if not isinstance(buf, torch.Tensor) or not buf.is_cuda or not buf.is_contiguous():
        raise ValueError("buf must be a contiguous CUDA tensor")
    n = ctypes.c_int64(0)
    _check("q4k_stream_read", lib().q4k_stream_read(buf.data_ptr(), buf.numel() * buf.element_size(), ctypes.byref(n),
                                                    _stream_ptr(stream)))
    return int(n.value)


def device_error_flags() -> int:
    return int(lib().q4k_device_error_flags())


def device_error_clear():
    _check("q4k_device_error_clear", lib().q4k_device_error_clear())


def raw_call(name: str, *args):
    """Call an exported entry point with raw integer/pointer arguments (tests)."""
    return getattr(lib(), name)(*args)
