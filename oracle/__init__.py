"""CPU oracle for the Q4_K decode hot path -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg may import this package.  The product library (``q4_dequant_gemv_gb300``)
never imports, links or executes anything here, and this package never imports
the product.  The arithmetic lives in ``q4k_oracle.c`` (plain C, fp64
accumulation); this module only compiles it with gcc and marshals numpy arrays
through ctypes.

Parity status of each function (what pins it is in ``tests/test_oracle.py``):
  fp16 / bf16 decode ........ pinned (all 65536 patterns vs numpy's decoders)
  scale / quant unpack ...... pinned (single-bit fixtures in tests/golden)
  block dequant ............. pinned (closed-form blocks, golden fixtures)
  gemv ...................... pinned (brute force vs library matmul, one-hot,
                              all-ones closed form, batch invariance)
  argmax .................... pinned (ties, planted maximum, NaN, signed zero)
  prefill ................... pinned (brute force vs library matmul)
The byte packing of the 6-bit scales and 4-bit quants is a reading (the GGUF
Q4_K packing): the pages name the format but never print its bytes, so it is
pinned only against that written reading, not against real model files.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "q4k_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

QK = 256
QBYTES = 144


def build(force: bool = False) -> str:
    """Compile q4k_oracle.c into liboracle.so (gcc, -O2, OpenMP)."""
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared", "-fno-fast-math",
           "-ffp-contract=off", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        build()
        lib = ctypes.CDLL(_LIB)
        P = ctypes.c_void_p
        I64 = ctypes.c_int64
        I = ctypes.c_int
        lib.oracle_fp16_to_double.argtypes = [ctypes.c_uint16]
        lib.oracle_fp16_to_double.restype = ctypes.c_double
        lib.oracle_bf16_to_double.argtypes = [ctypes.c_uint16]
        lib.oracle_bf16_to_double.restype = ctypes.c_double
        lib.oracle_round_bf16.argtypes = [ctypes.c_double]
        lib.oracle_round_bf16.restype = ctypes.c_double
        lib.oracle_unpack_scales.argtypes = [P, P, P]
        lib.oracle_unpack_quants.argtypes = [P, P]
        lib.oracle_dequant_block.argtypes = [P, P]
        lib.oracle_pack_block.argtypes = [ctypes.c_uint16, ctypes.c_uint16, P, P, P, P]
        lib.oracle_dequant_matrix.argtypes = [P, I64, I64, P, I]
        lib.oracle_gemv.argtypes = [P, P, P, I64, I64, I, I]
        lib.oracle_gemv_rows.argtypes = [P, P, P, I64, I64, I, P, I64, I]
        lib.oracle_argmax_f64.argtypes = [P, I64]
        lib.oracle_argmax_f64.restype = I64
        lib.oracle_argmax_f32.argtypes = [P, I64]
        lib.oracle_argmax_f32.restype = I64
        lib.oracle_prefill.argtypes = [P, P, P, I64, I64, I64, I, I]
        lib.oracle_q8k_quantize.argtypes = [P, I64, P, P]
        lib.oracle_gemv_q8k.argtypes = [P, P, P, P, I64, I64, I]
        lib.oracle_q6k_dequant_block.argtypes = [P, P]
        lib.oracle_q6k_gemv.argtypes = [P, P, P, I64, I64, I, I]
        lib.oracle_q6k_gemv_rows.argtypes = [P, P, P, I64, I, P, I64, I]
        lib.oracle_max_threads.restype = I
        _lib = lib
        return lib


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def max_threads() -> int:
    return int(_load().oracle_max_threads())


def fp16_to_double(bits: int) -> float:
    return float(_load().oracle_fp16_to_double(int(bits) & 0xFFFF))


def bf16_to_double(bits: int) -> float:
    return float(_load().oracle_bf16_to_double(int(bits) & 0xFFFF))


def round_bf16(v: float) -> float:
    return float(_load().oracle_round_bf16(float(v)))


def unpack_scales(s12) -> tuple[np.ndarray, np.ndarray]:
    s = _c(s12, np.uint8)
    assert s.size == 12
    sc = np.zeros(8, np.int32)
    m = np.zeros(8, np.int32)
    _load().oracle_unpack_scales(_ptr(s), _ptr(sc), _ptr(m))
    return sc, m


def unpack_quants(qs128) -> np.ndarray:
    qs = _c(qs128, np.uint8)
    assert qs.size == 128
    q = np.zeros(256, np.int32)
    _load().oracle_unpack_quants(_ptr(qs), _ptr(q))
    return q


def dequant_block(blk) -> np.ndarray:
    b = _c(blk, np.uint8)
    assert b.size == QBYTES
    w = np.zeros(QK, np.float64)
    _load().oracle_dequant_block(_ptr(b), _ptr(w))
    return w


def pack_block(d_bits: int, dmin_bits: int, sc, m, q) -> np.ndarray:
    """Encode one block from its fields (test helper; inverse of the unpack)."""
    sc = _c(sc, np.int32)
    m = _c(m, np.int32)
    q = _c(q, np.int32)
    assert sc.size == 8 and m.size == 8 and q.size == 256
    assert sc.min() >= 0 and sc.max() < 64 and m.min() >= 0 and m.max() < 64
    assert q.min() >= 0 and q.max() < 16
    out = np.zeros(QBYTES, np.uint8)
    _load().oracle_pack_block(int(d_bits) & 0xFFFF, int(dmin_bits) & 0xFFFF, _ptr(sc), _ptr(m), _ptr(q), _ptr(out))
    return out


def dequant_matrix(W: np.ndarray, N: int, K: int, threads: int = 0) -> np.ndarray:
    W = _c(W, np.uint8)
    assert W.size == N * (K // QK) * QBYTES
    out = np.zeros((N, K), np.float64)
    _load().oracle_dequant_matrix(_ptr(W), N, K, _ptr(out), threads)
    return out


def gemv(W: np.ndarray, x: np.ndarray, N: int, K: int, threads: int = 0) -> np.ndarray:
    """fp64 y [B][N] = W_deq [N][K] . x[b] for x fp32 [B][K] (or [K])."""
    W = _c(W, np.uint8)
    x2 = _c(x, np.float32).reshape(-1, K)
    B = x2.shape[0]
    assert W.size == N * (K // QK) * QBYTES
    y = np.zeros((B, N), np.float64)
    _load().oracle_gemv(_ptr(W), _ptr(x2), _ptr(y), N, K, B, threads)
    return y


def gemv_rows(W: np.ndarray, x: np.ndarray, N: int, K: int, rows, threads: int = 0) -> np.ndarray:
    """fp64 y [B][len(rows)] for a subset of rows of W_deq . x."""
    W = _c(W, np.uint8)
    x2 = _c(x, np.float32).reshape(-1, K)
    B = x2.shape[0]
    r = _c(rows, np.int64)
    assert r.size == 0 or (r.min() >= 0 and r.max() < N)
    y = np.zeros((B, r.size), np.float64)
    _load().oracle_gemv_rows(_ptr(W), _ptr(x2), _ptr(y), N, K, B, _ptr(r), r.size, threads)
    return y


def argmax(v: np.ndarray) -> int:
    """First index of the maximum (NaN never wins; all-NaN -> 0)."""
    if v.dtype == np.float32:
        a = _c(v, np.float32)
        return int(_load().oracle_argmax_f32(_ptr(a), a.size))
    a = _c(v, np.float64)
    return int(_load().oracle_argmax_f64(_ptr(a), a.size))


def prefill(W: np.ndarray, X_bf16_bits: np.ndarray, N: int, K: int, round_w: bool = False,
            threads: int = 0) -> np.ndarray:
    """fp64 Y [T][N] = X [T][K] . W_deq^T with X given as bf16 bit patterns."""
    W = _c(W, np.uint8)
    X = _c(X_bf16_bits, np.uint16).reshape(-1, K)
    T = X.shape[0]
    Y = np.zeros((T, N), np.float64)
    _load().oracle_prefill(_ptr(W), _ptr(X), _ptr(Y), N, K, T, 1 if round_w else 0, threads)
    return Y


def q8k_quantize(x: np.ndarray, K: int):
    """Q8_K activation quantization of one row x fp32 [K]: int8 codes q [K] and
    float32 block scales d [K/256] (rule: oracle_q8k_quantize in q4k_oracle.c)."""
    x1 = _c(x, np.float32).reshape(K)
    q = np.zeros(K, np.int8)
    d = np.zeros(K // QK, np.float32)
    _load().oracle_q8k_quantize(_ptr(x1), K, _ptr(q), _ptr(d))
    return q, d


def gemv_q8k(W: np.ndarray, q: np.ndarray, d: np.ndarray, N: int, K: int, threads: int = 0) -> np.ndarray:
    """fp64 y [N] = W_deq . (d_block * q): the Q4_K x Q8_K product, batch 1."""
    W = _c(W, np.uint8)
    q = _c(q, np.int8)
    d = _c(d, np.float32)
    assert W.size == N * (K // QK) * QBYTES and q.size == K and d.size == K // QK
    y = np.zeros(N, np.float64)
    _load().oracle_gemv_q8k(_ptr(W), _ptr(q), _ptr(d), _ptr(y), N, K, threads)
    return y


Q6BYTES = 210


def q6k_dequant_block(blk) -> np.ndarray:
    """The 256 weights (fp64) of one 210-byte Q6_K block."""
    b = _c(np.frombuffer(bytes(blk), np.uint8) if isinstance(blk, (bytes, bytearray)) else blk, np.uint8)
    assert b.size == Q6BYTES
    w = np.zeros(QK, np.float64)
    _load().oracle_q6k_dequant_block(_ptr(b), _ptr(w))
    return w


def q6k_dequant_matrix(W: np.ndarray, N: int, K: int) -> np.ndarray:
    W = _c(W, np.uint8).reshape(N * (K // QK), Q6BYTES)
    return np.stack([q6k_dequant_block(W[i]) for i in range(W.shape[0])]).reshape(N, K) if N else np.zeros((0, K))


def q6k_gemv(W: np.ndarray, x: np.ndarray, N: int, K: int, threads: int = 0) -> np.ndarray:
    """fp64 y [B][N] = W_q6k_deq [N][K] . x[b] for x fp32 [B][K] (or [K])."""
    W = _c(W, np.uint8)
    x2 = _c(x, np.float32).reshape(-1, K)
    B = x2.shape[0]
    assert W.size == N * (K // QK) * Q6BYTES
    y = np.zeros((B, N), np.float64)
    _load().oracle_q6k_gemv(_ptr(W), _ptr(x2), _ptr(y), N, K, B, threads)
    return y


def q6k_gemv_rows(W: np.ndarray, x: np.ndarray, N: int, K: int, rows, threads: int = 0) -> np.ndarray:
    """fp64 y [B][len(rows)] for a subset of rows of a Q6_K matrix times x."""
    W = _c(W, np.uint8)
    x2 = _c(x, np.float32).reshape(-1, K)
    B = x2.shape[0]
    r = _c(rows, np.int64)
    assert W.size == N * (K // QK) * Q6BYTES and (r.size == 0 or (r.min() >= 0 and r.max() < N))
    y = np.zeros((B, r.size), np.float64)
    _load().oracle_q6k_gemv_rows(_ptr(W), _ptr(x2), _ptr(y), K, B, _ptr(r), r.size, threads)
    return y
