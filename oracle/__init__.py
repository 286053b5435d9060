"""CPU oracle for C = alpha*A*B + beta*C (FP16 A and B, FP32 C, double sums).

TEST INFRASTRUCTURE ONLY. Only the test suite, ``__graft_entry__.smoke()``
and the benchmark's CPU-baseline leg may import this package. The CUDA
library never calls it, and the two share no code.

The arithmetic lives in ``oracle.c`` (plain C, double accumulation, its own
binary16 decoder); this module compiles it with gcc and wraps it with ctypes.
Definitions and sources are in the header of ``oracle.c``:

* "Day 80, Capstone 4: a tensor-core GEMM", "Capability" / "Minimal model"
  (FP16 inputs, FP32 accumulation) and "Compare like with like" /
  "Independent gate" (double CPU reference, Kahan float64 in the gate).
* "Day 72: Tensor cores with WMMA", "Why this program calls cuBLAS twice"
  (every element checked against a double CPU reference).

Operands are passed as flat arrays with a leading dimension, exactly as a
BLAS caller would: ``A`` holds binary16 bit patterns (``numpy.uint16``) with
element (i, k) at ``A[i*lda + k]``; ``B`` likewise with (k, j) at
``B[k*ldb + j]`` (row-major, the default) or ``B[j*ldb + k]`` with
``b_col_major=True`` (the gate's layout on "Day 80", "Independent gate");
``C`` is ``numpy.float32`` with (i, j) at ``C[i*ldc + j]``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle.so")

_lib = None
_lock = threading.Lock()


def compile_source(src: str, out: str) -> str:
    """gcc -O2 without FMA contraction or fast-math, so the double arithmetic
    is the same IEEE sequence on x86-64 and aarch64."""
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-D_DEFAULT_SOURCE", "-ffp-contract=off", "-fno-fast-math",
           "-fPIC", "-shared", "-pthread", "-o", tmp, src, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def build(force: bool = False) -> str:
    """Compile oracle.c into oracle/_build/liboracle.so."""
    os.makedirs(_BUILD, exist_ok=True)
    fresh = os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)
    if fresh and not force:
        return _LIB_PATH
    return compile_source(_SRC, _LIB_PATH)


def bind(path: str):
    """Load a compiled oracle.c from ``path`` and declare its signatures."""
    lib = ctypes.CDLL(path)
    i64, f64, p = ctypes.c_int64, ctypes.c_double, ctypes.c_void_p
    lib.oracle_half_to_double.restype = f64
    lib.oracle_half_to_double.argtypes = [ctypes.c_uint16]
    lib.oracle_gemm.restype = ctypes.c_int
    lib.oracle_gemm.argtypes = [i64, i64, i64, f64, p, i64, p, i64, f64, p, i64,
                                p, p, ctypes.c_int, ctypes.c_int]
    lib.oracle_elements.restype = ctypes.c_int
    lib.oracle_elements.argtypes = [i64, i64, i64, f64, p, i64, p, i64, f64, p, i64,
                                    i64, p, p, p, p, ctypes.c_int, ctypes.c_int]
    lib.oracle_gemm_ex.restype = ctypes.c_int
    lib.oracle_gemm_ex.argtypes = lib.oracle_gemm.argtypes + [ctypes.c_int]
    lib.oracle_elements_ex.restype = ctypes.c_int
    lib.oracle_elements_ex.argtypes = lib.oracle_elements.argtypes + [ctypes.c_int]
    return lib


def _load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = bind(build())
        return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _as_bits(x, name):
    if x is None:
        return None
    a = np.ascontiguousarray(x)
    if a.dtype == np.float16:
        a = a.view(np.uint16)
    if a.dtype != np.uint16:
        raise TypeError(f"{name} must hold binary16 bit patterns (uint16 or float16), got {a.dtype}")
    return a.reshape(-1)


def _as_f32(x):
    if x is None:
        return None
    a = np.ascontiguousarray(x)
    if a.dtype != np.float32:
        raise TypeError(f"C must be float32, got {a.dtype}")
    return a.reshape(-1)


def _check_extent(a, rows, ld, cols, name):
    if a is None or rows == 0 or cols == 0:
        return
    need = (rows - 1) * ld + cols
    if a.size < need:
        raise ValueError(f"{name} holds {a.size} elements, needs {need}")


def half_to_double(bits: int, lib=None) -> float:
    """The oracle's own binary16 decoder applied to one bit pattern."""
    return (lib or _load()).oracle_half_to_double(int(bits) & 0xFFFF)


def gemm(M, N, K, alpha, A, lda, B, ldb, beta, C=None, ldc=None, *, kahan=False, threads=0,
         lib=None, b_col_major=False):
    """Every element of alpha*A*B + beta*C.

    Returns ``(out, S)``, both float64 arrays of shape (M, N), where
    ``S[i, j] = sum_k |A[i,k]*B[k,j]|`` (the scale the tolerance is stated in).
    """
    ldc = N if ldc is None else ldc
    A, B, C = _as_bits(A, "A"), _as_bits(B, "B"), _as_f32(C)
    need_ab = alpha != 0 and K > 0
    if need_ab:
        _check_extent(A, M, lda, K, "A")
        _check_extent(B, N, ldb, K, "B") if b_col_major else _check_extent(B, K, ldb, N, "B")
    if beta != 0:
        _check_extent(C, M, ldc, N, "C")
    out = np.empty((M, N), dtype=np.float64)
    S = np.empty((M, N), dtype=np.float64)
    rc = (lib or _load()).oracle_gemm_ex(M, N, K, float(alpha), _ptr(A), lda, _ptr(B), ldb,
                                         float(beta), _ptr(C), ldc, _ptr(out), _ptr(S),
                                         int(bool(kahan)), int(threads), int(bool(b_col_major)))
    if rc != 0:
        raise ValueError(f"oracle_gemm rejected the arguments (status {rc})")
    return out, S


def elements(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, I, J, *, kahan=False, threads=0,
             lib=None, b_col_major=False):
    """The listed elements (I[e], J[e]) of alpha*A*B + beta*C; returns ``(out, S)``."""
    A, B, C = _as_bits(A, "A"), _as_bits(B, "B"), _as_f32(C)
    I = np.ascontiguousarray(I, dtype=np.int64).reshape(-1)
    J = np.ascontiguousarray(J, dtype=np.int64).reshape(-1)
    if I.shape != J.shape:
        raise ValueError("I and J differ in length")
    if alpha != 0 and K > 0:
        _check_extent(A, M, lda, K, "A")
        _check_extent(B, N, ldb, K, "B") if b_col_major else _check_extent(B, K, ldb, N, "B")
    if beta != 0:
        _check_extent(C, M, ldc, N, "C")
    out = np.empty(I.shape, dtype=np.float64)
    S = np.empty(I.shape, dtype=np.float64)
    rc = (lib or _load()).oracle_elements_ex(M, N, K, float(alpha), _ptr(A), lda, _ptr(B), ldb,
                                             float(beta), _ptr(C), ldc, I.size, _ptr(I), _ptr(J),
                                             _ptr(out), _ptr(S), int(bool(kahan)), int(threads),
                                             int(bool(b_col_major)))
    if rc != 0:
        raise ValueError(f"oracle_elements rejected the arguments (status {rc})")
    return out, S


def tolerance(S):
    """Per-element bound |C_gpu - C_ref| <= 1e-3 * S + 1e-5, S = sum_k |A_ik * B_kj|."""
    return 1e-3 * np.asarray(S) + 1e-5
