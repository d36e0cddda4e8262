"""CPU oracle for dense GEMM, C = A @ B, accumulated in float64.

TEST INFRASTRUCTURE, NOT PART OF THE PRODUCT. Only ``tests/``,
``__graft_entry__.smoke()`` and ``bench.py`` (its ``cpu_baseline`` leg and its
``--impl reference`` arm) may import this package. The product path
(``dense_gemm_14_gb300``) never imports it, and it imports nothing from the
product.

The arithmetic lives in ``oracle_gemm.c`` (a plain i-k-j triple loop, see its
header for the definition it follows and the pages it cites). This module only
compiles that file with gcc and marshals numpy arrays to it through ctypes.

Inputs are numpy arrays: ``float32`` for ``dtype="f32"``; for ``"bf16"`` and
``"f16"`` the raw 16-bit patterns as ``uint16`` (the oracle decodes them
itself, so it sees exactly the rounded values the GPU sees).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle_gemm.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle_gemm.so")

DTYPE_CODES = {"f32": 0, "bf16": 1, "f16": 2}

_lib = None
_lock = threading.Lock()


def build(force: bool = False) -> str:
    """Compiles oracle_gemm.c into oracle/_build/liboracle_gemm.so (gcc, OpenMP).

    ``-ffp-contract=off`` keeps gcc from fusing the sum's multiply and add (the
    products are exact in double either way, so this only keeps the code
    literal) and no fast-math flag reorders the sum.
    """
    os.makedirs(_BUILD, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-fopenmp", "-ffp-contract=off", "-fPIC", "-shared",
           "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            i64, vp, dp = ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p
            lib.oracle_gemm.argtypes = [i64, i64, i64, ctypes.c_int, vp, i64, vp, i64,
                                        dp, dp, i64, ctypes.c_int]
            lib.oracle_gemm.restype = ctypes.c_int
            lib.oracle_gemm_entries.argtypes = [i64, i64, i64, ctypes.c_int, vp, i64, vp, i64,
                                                i64, vp, vp, dp, dp, ctypes.c_int]
            lib.oracle_gemm_entries.restype = ctypes.c_int
            lib.oracle_decode_matrix.argtypes = [ctypes.c_int, vp, i64, i64, i64, dp]
            lib.oracle_decode_matrix.restype = ctypes.c_int
            lib.oracle_gemm_ex.argtypes = [i64, i64, i64, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                           ctypes.c_double, vp, i64, vp, i64, ctypes.c_double,
                                           vp, i64, dp, dp, i64, ctypes.c_int]
            lib.oracle_gemm_ex.restype = ctypes.c_int
            lib.oracle_truncate_tf32.argtypes = [vp, i64]
            lib.oracle_truncate_tf32.restype = ctypes.c_int
            lib.oracle_max_threads.argtypes = []
            lib.oracle_max_threads.restype = ctypes.c_int
            _lib = lib
    return _lib


def _check(x: np.ndarray, dtype: str, name: str) -> np.ndarray:
    want = np.float32 if dtype == "f32" else np.uint16
    if x.dtype != want:
        raise TypeError(f"{name}: expected {np.dtype(want)} for dtype={dtype}, got {x.dtype}")
    if x.ndim != 2:
        raise ValueError(f"{name}: expected a 2-D array")
    if x.size and (x.strides[1] != x.itemsize or x.strides[0] % x.itemsize):
        x = np.ascontiguousarray(x)
    return x


def _ptr(x: np.ndarray) -> int:
    return x.ctypes.data if x.size else 0


def _ld(x: np.ndarray) -> int:
    """Row pitch in elements (empty or single-row arrays: the row length)."""
    if x.size == 0 or x.shape[0] <= 1:
        return x.shape[1]
    return x.strides[0] // x.itemsize


def max_threads() -> int:
    """Threads the oracle's OpenMP loops use by default."""
    return int(_load().oracle_max_threads())


def gemm(A: np.ndarray, B: np.ndarray, dtype: str = "f32", threads: int = 0,
         with_abs: bool = True):
    """Returns (C, Cabs) as float64 arrays; Cabs = |A| @ |B| (None if not asked).

    C[i, j] = sum_k A[i, k] * B[k, j], summed in float64 over k in order.
    """
    code = DTYPE_CODES[dtype]
    A = _check(A, dtype, "A")
    B = _check(B, dtype, "B")
    M, K = A.shape
    K2, N = B.shape
    if K != K2:
        raise ValueError(f"inner dimensions differ: {A.shape} @ {B.shape}")
    C = np.empty((M, N), dtype=np.float64)
    Cabs = np.empty((M, N), dtype=np.float64) if with_abs else None
    rc = _load().oracle_gemm(M, N, K, code, _ptr(A), _ld(A),
                             _ptr(B), _ld(B),
                             _ptr(C), _ptr(Cabs) if Cabs is not None else 0, N, threads)
    if rc != 0:
        raise RuntimeError(f"oracle_gemm failed with code {rc}")
    return C, Cabs


def gemm_ex(A: np.ndarray, B: np.ndarray, dtype: str = "f32", transa: bool = False,
            transb: bool = False, alpha: float = 1.0, beta: float = 0.0,
            C0: np.ndarray | None = None, threads: int = 0):
    """Returns (C, Cabs) for C = alpha * op(A) @ op(B) + beta * C0 in float64.

    A and B are the STORED arrays: op(A) = A (M x K) or A.T when transa (A is
    then K x M); likewise for B. C0 is float32 M x N, read only if beta != 0.
    """
    code = DTYPE_CODES[dtype]
    A = _check(A, dtype, "A")
    B = _check(B, dtype, "B")
    M, K = (A.shape[1], A.shape[0]) if transa else A.shape
    K2, N = (B.shape[1], B.shape[0]) if transb else B.shape
    if K != K2:
        raise ValueError(f"inner dimensions differ: op(A) {M}x{K}, op(B) {K2}x{N}")
    if beta != 0.0:
        if C0 is None or C0.shape != (M, N):
            raise ValueError("C0 of shape (M, N) is needed when beta != 0")
        C0 = np.ascontiguousarray(C0, dtype=np.float32)
    C = np.empty((M, N), dtype=np.float64)
    Cabs = np.empty((M, N), dtype=np.float64)
    rc = _load().oracle_gemm_ex(M, N, K, code, int(bool(transa)), int(bool(transb)),
                                float(alpha), _ptr(A), _ld(A), _ptr(B), _ld(B), float(beta),
                                _ptr(C0) if beta != 0.0 else 0, N, _ptr(C), _ptr(Cabs), N,
                                threads)
    if rc != 0:
        raise RuntimeError(f"oracle_gemm_ex failed with code {rc}")
    return C, Cabs


def gemm_entries(A: np.ndarray, B: np.ndarray, rows, cols, dtype: str = "f32",
                 threads: int = 0):
    """Returns (C[rows[t], cols[t]], Cabs[...]) for each t, one dot product each."""
    code = DTYPE_CODES[dtype]
    A = _check(A, dtype, "A")
    B = _check(B, dtype, "B")
    M, K = A.shape
    K2, N = B.shape
    if K != K2:
        raise ValueError(f"inner dimensions differ: {A.shape} @ {B.shape}")
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    cols = np.ascontiguousarray(cols, dtype=np.int64)
    if rows.shape != cols.shape or rows.ndim != 1:
        raise ValueError("rows and cols must be 1-D and of equal length")
    out = np.empty(rows.shape[0], dtype=np.float64)
    outabs = np.empty(rows.shape[0], dtype=np.float64)
    rc = _load().oracle_gemm_entries(M, N, K, code, _ptr(A), _ld(A),
                                     _ptr(B), _ld(B), rows.shape[0],
                                     _ptr(rows), _ptr(cols), _ptr(out), _ptr(outabs), threads)
    if rc != 0:
        raise RuntimeError(f"oracle_gemm_entries failed with code {rc}")
    return out, outabs


def truncate_tf32(X: np.ndarray) -> np.ndarray:
    """A float32 copy of X with every value truncated to tf32 (the 13 low
    fraction bits cleared: what the tensor cores take from an fp32 input)."""
    out = np.array(X, dtype=np.float32, copy=True, order="C")
    rc = _load().oracle_truncate_tf32(_ptr(out) if out.size else 0, out.size)
    if rc != 0:
        raise RuntimeError(f"oracle_truncate_tf32 failed with code {rc}")
    return out


def decode(X: np.ndarray, dtype: str) -> np.ndarray:
    """Decodes a 2-D array of fp32 values or 16-bit patterns to float64."""
    X = _check(X, dtype, "X")
    out = np.empty(X.shape, dtype=np.float64)
    rc = _load().oracle_decode_matrix(DTYPE_CODES[dtype], _ptr(X), X.shape[0], X.shape[1],
                                      _ld(X), _ptr(out))
    if rc != 0:
        raise RuntimeError(f"oracle_decode_matrix failed with code {rc}")
    return out


def within_bound(C_gpu: np.ndarray, C_ref: np.ndarray, Cabs: np.ndarray, rel: float):
    """Element-wise acceptance: |C_gpu - C_ref| <= rel * Cabs, and no NaN.

    Returns (ok, worst) where worst = max |C_gpu - C_ref| / Cabs over elements
    with Cabs > 0 (elements with Cabs == 0 must match exactly: an empty or
    all-zero dot product is exactly zero).
    """
    C_gpu = np.asarray(C_gpu, dtype=np.float64)
    diff = np.abs(C_gpu - C_ref)
    if np.isnan(C_gpu).any() and not np.isnan(C_ref).any():
        return False, float("inf")
    ok = bool(np.all(diff <= rel * Cabs))
    pos = Cabs > 0
    worst = float(np.max(diff[pos] / Cabs[pos])) if pos.any() else 0.0
    return ok, worst
