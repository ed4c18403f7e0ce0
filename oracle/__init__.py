"""CPU oracle for the GEMM library (fp64 accumulation, plain loops, in ``oracle.c``).

TEST INFRASTRUCTURE ONLY.  Only the test suite, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg may import this package.  The product library never
imports, links or executes anything here, and this package imports nothing from it.

Every function takes numpy arrays (float32 inputs, float64 outputs) and calls the C
routine of the same name.  bf16 inputs are passed as float32: every bf16 value is
exactly representable in float32, so the conversion loses nothing.

Citations for what each routine computes are in the header of ``oracle.c``:
"Learning to develop for GPU with GEMM as the example" (section "Matrix product") for
the GEMM, and "Three X: large convolutions in PyTorch for training" (sections "Why we
need high-dimensional convolution" and "CuBLAS") for the convolution and its im2col
lowering.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

# -O2 keeps the code plain; -ffp-contract=off keeps each multiply and add separately
# rounded; no -ffast-math, so nothing is reassociated.
CFLAGS = ["-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared", "-pthread"]


def build(force: bool = False) -> str:
    """Compile ``oracle.c`` into ``liboracle.so`` beside it (gcc, a second or two)."""
    with _lock:
        if (not force and os.path.exists(_LIB)
                and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
            return _LIB
        tmp = _LIB + ".tmp.%d" % os.getpid()
        subprocess.run(["gcc", *CFLAGS, _SRC, "-o", tmp, "-lm"], check=True)
        os.replace(tmp, _LIB)
        return _LIB


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        i64, p = ctypes.c_int64, ctypes.c_void_p
        lib.oracle_gemm.argtypes = [i64, i64, i64, p, i64, p, i64, p, i64, ctypes.c_int]
        lib.oracle_gemm_entries.argtypes = [i64, i64, i64, p, i64, p, i64, i64, i64, p, p, p, ctypes.c_int]
        d = ctypes.c_double
        lib.oracle_gemm_general.argtypes = [i64, i64, i64, d, p, i64, p, i64, d, p, i64, p, i64, ctypes.c_int]
        lib.oracle_conv4d_direct.argtypes = [i64, p, i64, p, p, p, p, ctypes.c_int]
        lib.oracle_im2col4d.argtypes = [i64, p, p, p, p]
        for f in (lib.oracle_gemm, lib.oracle_gemm_entries, lib.oracle_gemm_general, lib.oracle_conv4d_direct,
                  lib.oracle_im2col4d):
            f.restype = ctypes.c_int
        _lib = lib
    return _lib


def default_threads() -> int:
    return max(1, len(os.sched_getaffinity(0)))


def _f32(a) -> np.ndarray:
    a = np.asarray(a)
    if a.dtype != np.float32:
        raise TypeError("oracle inputs are float32 arrays (bf16 values convert exactly), got %s" % a.dtype)
    return a


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


def _check_2d(a: np.ndarray, rows: int, cols: int, name: str) -> int:
    """Return the row stride (in elements) of a 2-D row-major view."""
    if a.ndim != 2 or a.shape[0] < rows or a.shape[1] < cols:
        raise ValueError("%s must be at least %dx%d, got %s" % (name, rows, cols, a.shape))
    if a.strides[1] != a.itemsize:
        raise ValueError("%s must have unit stride along rows" % name)
    return a.strides[0] // a.itemsize


def gemm(A: np.ndarray, B: np.ndarray, nthreads: int | None = None) -> np.ndarray:
    """C = A @ B in fp64 (k ascending, separate multiply and add).

    A is M x K and B is K x N, float32, row-major; row strides (lda, ldb) may exceed
    the column counts (a 2-D slice of a wider array).
    """
    A, B = _f32(A), _f32(B)
    M, K = A.shape
    K2, N = B.shape
    if K2 != K:
        raise ValueError("inner dimensions differ: %d vs %d" % (K, K2))
    lda = _check_2d(A, M, K, "A") if M and K else max(K, 1)
    ldb = _check_2d(B, K, N, "B") if K and N else max(N, 1)
    C = np.empty((M, N), dtype=np.float64)
    if M == 0 or N == 0:
        return C
    rc = _load().oracle_gemm(M, N, K, _ptr(A), lda, _ptr(B), ldb, _ptr(C), N,
                             nthreads or default_threads())
    if rc != 0:
        raise RuntimeError("oracle_gemm rejected its arguments (rc=%d)" % rc)
    return C


def gemm_general(alpha: float, A: np.ndarray, B: np.ndarray, beta: float = 0.0, C: np.ndarray | None = None,
                 nthreads: int | None = None) -> np.ndarray:
    """D = alpha * (A @ B) + beta * C in fp64 ("generalised" GEMM; C unread when beta == 0).

    C, when given, is converted to float64 (exact for fp32 and bf16 values)."""
    A, B = _f32(A), _f32(B)
    M, K = A.shape
    N = B.shape[1]
    if B.shape[0] != K:
        raise ValueError("inner dimensions differ")
    lda = _check_2d(A, M, K, "A") if M and K else max(K, 1)
    ldb = _check_2d(B, K, N, "B") if K and N else max(N, 1)
    D = np.empty((M, N), dtype=np.float64)
    if M == 0 or N == 0:
        return D
    Cp = None
    if beta != 0.0:
        if C is None or C.shape != (M, N):
            raise ValueError("beta != 0 needs C of shape (M, N)")
        Cp = np.ascontiguousarray(C, dtype=np.float64)
    rc = _load().oracle_gemm_general(M, N, K, float(alpha), _ptr(A), lda, _ptr(B), ldb, float(beta),
                                     _ptr(Cp) if Cp is not None else None, N, _ptr(D), N,
                                     nthreads or default_threads())
    if rc != 0:
        raise RuntimeError("oracle_gemm_general rejected its arguments (rc=%d)" % rc)
    return D


def gemm_entries(A: np.ndarray, B: np.ndarray, rows, cols, nthreads: int | None = None,
                 B_transposed_copy: np.ndarray | None = None) -> np.ndarray:
    """C[rows[t], cols[t]] of A @ B, each entry by the definition's k loop, in fp64.

    ``B_transposed_copy`` (N x K, contiguous) may be given to stream columns of B
    from contiguous memory; it must hold the same values as ``B.T``.
    """
    A = _f32(A)
    M, K = A.shape
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    cols = np.ascontiguousarray(cols, dtype=np.int64)
    if rows.shape != cols.shape or rows.ndim != 1:
        raise ValueError("rows and cols must be 1-D of equal length")
    lda = _check_2d(A, M, K, "A") if M and K else max(K, 1)
    if B_transposed_copy is not None:
        Bt = _f32(B_transposed_copy)
        N = Bt.shape[0]
        b_sj = _check_2d(Bt, N, K, "B_transposed_copy")
        b_sk = 1
        base = Bt
    else:
        B = _f32(B)
        N = B.shape[1]
        b_sk = _check_2d(B, K, N, "B")
        b_sj = 1
        base = B
    out = np.empty(rows.shape[0], dtype=np.float64)
    rc = _load().oracle_gemm_entries(M, N, K, _ptr(A), lda, _ptr(base), b_sk, b_sj, rows.shape[0],
                                     _ptr(rows), _ptr(cols), _ptr(out), nthreads or default_threads())
    if rc != 0:
        raise RuntimeError("oracle_gemm_entries rejected its arguments (rc=%d)" % rc)
    return out


def conv4d_direct(x: np.ndarray, w: np.ndarray, nthreads: int | None = None) -> np.ndarray:
    """Valid 4-D cross-correlation: x[Cin, I0..I3], w[Cout, Cin, R0..R3] -> y[Cout, P0..P3], fp64."""
    x = np.ascontiguousarray(_f32(x))
    w = np.ascontiguousarray(_f32(w))
    if x.ndim != 5 or w.ndim != 6 or w.shape[1] != x.shape[0]:
        raise ValueError("x must be [Cin, I0, I1, I2, I3] and w [Cout, Cin, R0, R1, R2, R3]")
    cin, cout = x.shape[0], w.shape[0]
    ins = np.array(x.shape[1:], dtype=np.int64)
    ks = np.array(w.shape[2:], dtype=np.int64)
    outs = tuple(int(i - k + 1) for i, k in zip(ins, ks))
    if min(outs) <= 0:
        raise ValueError("kernel larger than input")
    y = np.empty((cout,) + outs, dtype=np.float64)
    rc = _load().oracle_conv4d_direct(cin, _ptr(ins), cout, _ptr(ks), _ptr(x), _ptr(w), _ptr(y),
                                      nthreads or default_threads())
    if rc != 0:
        raise RuntimeError("oracle_conv4d_direct rejected its arguments (rc=%d)" % rc)
    return y


def im2col4d(x: np.ndarray, ks) -> np.ndarray:
    """Column matrix of a valid 4-D cross-correlation: [Cin*prod(ks), prod(out)] float32."""
    x = np.ascontiguousarray(_f32(x))
    if x.ndim != 5:
        raise ValueError("x must be [Cin, I0, I1, I2, I3]")
    cin = x.shape[0]
    ins = np.array(x.shape[1:], dtype=np.int64)
    ks = np.array(ks, dtype=np.int64)
    outs = [int(i - k + 1) for i, k in zip(ins, ks)]
    if len(ks) != 4 or min(outs) <= 0:
        raise ValueError("need four kernel extents no larger than the input")
    col = np.empty((cin * int(np.prod(ks)), int(np.prod(outs))), dtype=np.float32)
    rc = _load().oracle_im2col4d(cin, _ptr(ins), _ptr(ks), _ptr(x), _ptr(col))
    if rc != 0:
        raise RuntimeError("oracle_im2col4d rejected its arguments (rc=%d)" % rc)
    return col


__all__ = ["build", "gemm", "gemm_general", "gemm_entries", "conv4d_direct", "im2col4d", "default_threads"]
