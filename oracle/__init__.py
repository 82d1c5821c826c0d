"""CPU oracle for the TN GEMM ``C = A @ B.T`` -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product path (the CUDA library and
its Python binding) never imports, links or executes anything here, and this
package imports nothing from the product.

The arithmetic lives in ``gemm_oracle.c`` (fp64 accumulation for fp16/bf16,
int64 for int8, operands decoded from their bit patterns by the IEEE 754
definitions).  This module only compiles it with gcc and marshals numpy
arrays.  Which page passage each function follows is stated in the C file:
"RL驱动CUDA L2 GEMM内核自动调优：A100/H100 tile size与融合优化" (tile/data-layout,
multi-precision and correctness paragraphs).

Parity status: pinned (brute force on tiny inputs, identity, permutation,
rank-1 closed forms, exact small integers, int8 extremes, exhaustive decoder
checks -- ``tests/test_oracle_pins.py``).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gemm_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

FMT_F16 = 0
FMT_BF16 = 1


def build(force: bool = False) -> str:
    """Compile gemm_oracle.c into liboracle.so next to it (OpenMP if available)."""
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    base = ["gcc", "-O2", "-ffp-contract=off", "-shared", "-fPIC", "-std=c11"]
    tmp = _LIB + ".tmp.%d" % os.getpid()
    try:
        subprocess.run(base + ["-fopenmp", _SRC, "-o", tmp, "-lm"], check=True,
                       capture_output=True, text=True)
    except subprocess.CalledProcessError:
        subprocess.run(base + [_SRC, "-o", tmp, "-lm"], check=True, capture_output=True, text=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            i64, p = ctypes.c_int64, ctypes.c_void_p
            lib.oracle_f16_to_f64.argtypes = [ctypes.c_uint16]
            lib.oracle_f16_to_f64.restype = ctypes.c_double
            lib.oracle_bf16_to_f64.argtypes = [ctypes.c_uint16]
            lib.oracle_bf16_to_f64.restype = ctypes.c_double
            lib.oracle_decode.argtypes = [p, p, i64, ctypes.c_int]
            lib.oracle_decode.restype = None
            lib.oracle_max_threads.argtypes = []
            lib.oracle_max_threads.restype = ctypes.c_int
            lib.oracle_gemm_tn_half.argtypes = [p, p, p, i64, i64, i64, ctypes.c_int, ctypes.c_int]
            lib.oracle_gemm_tn_half.restype = ctypes.c_int
            lib.oracle_gemm_tn_half_sampled.argtypes = [p, p, i64, i64, i64, ctypes.c_int,
                                                        p, p, i64, p, ctypes.c_int]
            lib.oracle_gemm_tn_half_sampled.restype = ctypes.c_int
            lib.oracle_gemm_tn_i8.argtypes = [p, p, p, p, i64, i64, i64, ctypes.c_int]
            lib.oracle_gemm_tn_i8.restype = ctypes.c_int
            lib.oracle_gemm_tn_i8_sampled.argtypes = [p, p, i64, i64, i64, p, p, i64, p, p,
                                                      ctypes.c_int]
            lib.oracle_gemm_tn_i8_sampled.restype = ctypes.c_int
            lib.oracle_epilogue.argtypes = [p, i64, i64, p, ctypes.c_int]
            lib.oracle_epilogue.restype = ctypes.c_int
            lib.oracle_epilogue_sampled.argtypes = [p, p, i64, p, ctypes.c_int]
            lib.oracle_epilogue_sampled.restype = ctypes.c_int
            lib.oracle_fma_chain.argtypes = [p, p, i64, ctypes.c_int, ctypes.c_float,
                                             ctypes.c_float]
            lib.oracle_fma_chain.restype = ctypes.c_int
            _lib = lib
    return _lib


def _ptr(a: np.ndarray):
    return ctypes.c_void_p(a.ctypes.data)


def _bits16(x: np.ndarray) -> np.ndarray:
    x = np.ascontiguousarray(x)
    if x.dtype == np.float16:
        x = x.view(np.uint16)
    if x.dtype not in (np.uint16, np.int16):
        raise TypeError("half-precision operands are passed as 16-bit patterns, got %s" % x.dtype)
    return x.view(np.uint16)


def max_threads() -> int:
    return int(_load().oracle_max_threads())


def decode(bits: np.ndarray, fmt: int) -> np.ndarray:
    """Decode fp16 (fmt 0) or bf16 (fmt 1) bit patterns to float64."""
    b = _bits16(bits).ravel()
    out = np.empty(b.shape, dtype=np.float64)
    _load().oracle_decode(_ptr(b), _ptr(out), b.size, fmt)
    return out.reshape(np.shape(bits))


def gemm_tn_half(A: np.ndarray, B: np.ndarray, fmt: int, threads: int = 0) -> np.ndarray:
    """fp64 C = A @ B.T for half-precision bit patterns A[M,K], B[N,K]."""
    A, B = _bits16(A), _bits16(B)
    M, K = A.shape
    N, K2 = B.shape
    if K != K2:
        raise ValueError("K mismatch")
    C = np.empty((M, N), dtype=np.float64)
    rc = _load().oracle_gemm_tn_half(_ptr(A), _ptr(B), _ptr(C), M, N, K, fmt, threads)
    if rc != 0:
        raise RuntimeError("oracle_gemm_tn_half failed")
    return C


def gemm_tn_half_sampled(A, B, fmt: int, rows, cols, threads: int = 0) -> np.ndarray:
    A, B = _bits16(A), _bits16(B)
    M, K = A.shape
    N, _ = B.shape
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    cols = np.ascontiguousarray(cols, dtype=np.int64)
    out = np.empty(rows.shape, dtype=np.float64)
    rc = _load().oracle_gemm_tn_half_sampled(_ptr(A), _ptr(B), M, N, K, fmt, _ptr(rows),
                                             _ptr(cols), rows.size, _ptr(out), threads)
    if rc != 0:
        raise RuntimeError("oracle_gemm_tn_half_sampled failed")
    return out


def gemm_tn_i8(A: np.ndarray, B: np.ndarray, threads: int = 0):
    """Exact int8 GEMM; returns (C64 int64, C32 int32 wrapped modulo 2^32)."""
    A = np.ascontiguousarray(A, dtype=np.int8)
    B = np.ascontiguousarray(B, dtype=np.int8)
    M, K = A.shape
    N, K2 = B.shape
    if K != K2:
        raise ValueError("K mismatch")
    C64 = np.empty((M, N), dtype=np.int64)
    C32 = np.empty((M, N), dtype=np.int32)
    rc = _load().oracle_gemm_tn_i8(_ptr(A), _ptr(B), _ptr(C64), _ptr(C32), M, N, K, threads)
    if rc != 0:
        raise RuntimeError("oracle_gemm_tn_i8 failed")
    return C64, C32


def gemm_tn_i8_sampled(A, B, rows, cols, threads: int = 0):
    A = np.ascontiguousarray(A, dtype=np.int8)
    B = np.ascontiguousarray(B, dtype=np.int8)
    M, K = A.shape
    N, _ = B.shape
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    cols = np.ascontiguousarray(cols, dtype=np.int64)
    o64 = np.empty(rows.shape, dtype=np.int64)
    o32 = np.empty(rows.shape, dtype=np.int32)
    rc = _load().oracle_gemm_tn_i8_sampled(_ptr(A), _ptr(B), M, N, K, _ptr(rows), _ptr(cols),
                                           rows.size, _ptr(o64), _ptr(o32), threads)
    if rc != 0:
        raise RuntimeError("oracle_gemm_tn_i8_sampled failed")
    return o64, o32


ACT_NONE, ACT_RELU, ACT_GELU, ACT_SILU = 0, 1, 2, 3


def epilogue(C: np.ndarray, bias, act: int) -> np.ndarray:
    """act(C + bias[None, :]) in fp64 on a copy of the fp64 GEMM result C[M,N]."""
    out = np.array(C, dtype=np.float64, copy=True, order="C")
    b = None if bias is None else np.ascontiguousarray(bias, dtype=np.float32)
    rc = _load().oracle_epilogue(_ptr(out), out.shape[0], out.shape[1],
                                 None if b is None else _ptr(b), act)
    if rc != 0:
        raise RuntimeError("oracle_epilogue failed")
    return out


def epilogue_sampled(vals: np.ndarray, cols, bias, act: int) -> np.ndarray:
    out = np.array(vals, dtype=np.float64, copy=True)
    cols = np.ascontiguousarray(cols, dtype=np.int64)
    b = None if bias is None else np.ascontiguousarray(bias, dtype=np.float32)
    rc = _load().oracle_epilogue_sampled(_ptr(out), _ptr(cols), out.size,
                                         None if b is None else _ptr(b), act)
    if rc != 0:
        raise RuntimeError("oracle_epilogue_sampled failed")
    return out


def fma_chain(x: np.ndarray, iters: int, a: float, b: float) -> np.ndarray:
    """y = x, then iters times y = fma(y, a, b) in fp32 (single rounding), elementwise."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty_like(x)
    rc = _load().oracle_fma_chain(_ptr(x), _ptr(out), x.size, iters, a, b)
    if rc != 0:
        raise RuntimeError("oracle_fma_chain failed")
    return out
