"""CPU oracle for dense row-major C = A x B (FP64 accumulation).

TEST INFRASTRUCTURE ONLY.  Only the test suite, the package smoke check
and the benchmark's CPU-baseline leg may import this package.  The
library's product path never touches it, and it imports nothing from the
library: callers hand it numpy arrays.

Definition followed: "第八课：GPU 如何完成矩阵乘法" (Lesson 8: how a GPU does
matrix multiplication), section 一: C[i][j] = sum_{k<K} A[i][k] * B[k][j]
for A in R^{M x K}, B in R^{K x N}.  The arithmetic lives in oracle.c; this
module only marshals arguments.  Pins are in tests/test_oracle.py.
"""
import ctypes
import os

import numpy as np

from . import build as _build

_lib = None


def _load():
    global _lib
    if _lib is None:
        path = _build.build()
        lib = ctypes.CDLL(path)
        i32, f32p, f64p = ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p
        lib.oracle_gemm_f64.argtypes = [i32, i32, i32, f32p, i32, f32p, i32, f64p, i32]
        lib.oracle_gemm_f64.restype = None
        lib.oracle_abs_gemm_f64.argtypes = [i32, i32, i32, f32p, i32, f32p, i32, f64p, i32]
        lib.oracle_abs_gemm_f64.restype = None
        lib.oracle_gemm_rows_f64.argtypes = [i32, ctypes.c_void_p, i32, i32, f32p, i32,
                                             f32p, i32, f64p, f64p]
        lib.oracle_gemm_rows_f64.restype = None
        lib.oracle_max_threads.argtypes = []
        lib.oracle_max_threads.restype = i32
        lib.oracle_set_threads.argtypes = [i32]
        lib.oracle_set_threads.restype = None
        _lib = lib
    return _lib


def _as_rowmajor_f32(X, name):
    """Return (array, leading dimension) for a 2-D float32 matrix whose rows
    may be strided (a row-major view into a wider buffer) but whose columns
    are contiguous."""
    X = np.asarray(X)
    if X.dtype != np.float32:
        raise TypeError(f"{name}: oracle inputs are float32 (bf16 inputs are widened "
                        f"exactly to float32 by the caller), got {X.dtype}")
    if X.ndim != 2:
        raise ValueError(f"{name}: expected a 2-D matrix")
    rows, cols = X.shape
    if cols > 1 and X.strides[1] != 4:
        X = np.ascontiguousarray(X)
    if rows > 1 and (X.strides[0] % 4 != 0 or X.strides[0] < 4 * cols):
        X = np.ascontiguousarray(X)
    ld = X.strides[0] // 4 if rows > 1 else max(cols, 1)
    return X, max(ld, 1)


def _ptr(X):
    return X.ctypes.data if X.size else 0


def max_threads():
    return _load().oracle_max_threads()


def set_threads(n):
    _load().oracle_set_threads(int(n))


def gemm(A, B):
    """C = A x B in float64 (plain definition, k ascending)."""
    lib = _load()
    A, lda = _as_rowmajor_f32(A, "A")
    B, ldb = _as_rowmajor_f32(B, "B")
    M, K = A.shape
    K2, N = B.shape
    if K != K2:
        raise ValueError(f"inner dimensions differ: A is {A.shape}, B is {B.shape}")
    C = np.empty((M, N), dtype=np.float64)
    if M and N:
        lib.oracle_gemm_f64(M, N, K, _ptr(A), lda, _ptr(B), ldb, _ptr(C), max(N, 1))
    return C


def abs_gemm(A, B):
    """S = |A| x |B| in float64: the scale of every error bound."""
    lib = _load()
    A, lda = _as_rowmajor_f32(A, "A")
    B, ldb = _as_rowmajor_f32(B, "B")
    M, K = A.shape
    K2, N = B.shape
    if K != K2:
        raise ValueError(f"inner dimensions differ: A is {A.shape}, B is {B.shape}")
    S = np.empty((M, N), dtype=np.float64)
    if M and N:
        lib.oracle_abs_gemm_f64(M, N, K, _ptr(A), lda, _ptr(B), ldb, _ptr(S), max(N, 1))
    return S


def gemm_rows(A, B, rows, with_abs=True):
    """Rows `rows` of C (and of S when with_abs): arrays of shape (len(rows), N)."""
    lib = _load()
    A, lda = _as_rowmajor_f32(A, "A")
    B, ldb = _as_rowmajor_f32(B, "B")
    M, K = A.shape
    K2, N = B.shape
    if K != K2:
        raise ValueError(f"inner dimensions differ: A is {A.shape}, B is {B.shape}")
    rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    if rows.size and (rows.min() < 0 or rows.max() >= M):
        raise IndexError("row index out of range")
    C = np.empty((rows.size, N), dtype=np.float64)
    S = np.empty((rows.size, N), dtype=np.float64) if with_abs else None
    if rows.size and N:
        lib.oracle_gemm_rows_f64(rows.size, _ptr(rows), N, K, _ptr(A), lda, _ptr(B), ldb,
                                 _ptr(C), _ptr(S) if S is not None else None)
    return (C, S) if with_abs else C


__all__ = ["gemm", "abs_gemm", "gemm_rows", "max_threads", "set_threads"]
