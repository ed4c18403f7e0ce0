"""Python binding of the GB300 GEMM library (``include/gemm.h``).

Argument marshalling only: every function forwards to the C entry point of the same
name in ``lib/libgemm_gb300.so``; all arithmetic runs in the library's CUDA kernels.
PyTorch is used for device memory and streams (``matmul`` and ``conv4d`` take tensors).
There is no fallback: if the library is missing, importing this package raises.
"""
from __future__ import annotations

import ctypes
import os

_PKG = os.path.dirname(os.path.abspath(__file__))
# GEMM_GB300_DEBUG=1 loads the debug build (every computed global index checked in the
# kernels; a failed check is reported by gemm_get_device_status as GEMM_ERR_DEVICE_BOUNDS).
DEBUG = os.environ.get("GEMM_GB300_DEBUG") == "1"
LIB_PATH = os.path.join(_PKG, "lib", "libgemm_gb300_debug.so" if DEBUG else "libgemm_gb300.so")

GEMM_F32, GEMM_BF16, GEMM_F16 = 0, 1, 2
GEMM_OK = 0
GEMM_ERR_INVALID_ARG = -1
GEMM_ERR_ALIGNMENT = -2
GEMM_ERR_UNSUPPORTED = -3
GEMM_ERR_CUDA = -4
GEMM_ERR_DEVICE_TIMEOUT = -5
GEMM_ERR_DEVICE_BOUNDS = -6
GEMM_OPT_F32_KERNEL, GEMM_OPT_SPLIT_K, GEMM_OPT_WAIT_LIMIT_US, GEMM_OPT_TC_CHUNK, GEMM_OPT_TC_PAIR = 1, 2, 3, 4, 5
GEMM_OPT_TEST_STALL = 6
GEMM_OPT_CONV_STACK = 7
GEMM_OPT_CONV_SPLIT = 8

# Every symbol include/gemm.h declares (the ABI test checks the library exports them).
EXPORTS = ["gemm_create", "gemm_destroy", "gemm_run", "gemm_run_ex", "gemm_run_host", "gemm_run_host_batch",
           "conv4d_im2col",
           "conv4d_forward", "conv4d_forward_cl", "conv4d_forward_tc",
           "gemm_get_device_status", "gemm_set_option", "gemm_launch_count", "gemm_status_string",
           "gemm_run_f32_skinny_noalloc"]


class HostProblem(ctypes.Structure):
    """gemm_host_problem: one product of gemm_run_host_batch."""
    _fields_ = [("M", ctypes.c_int64), ("N", ctypes.c_int64), ("K", ctypes.c_int64), ("A", ctypes.c_void_p),
                ("lda", ctypes.c_int64), ("B", ctypes.c_void_p), ("ldb", ctypes.c_int64), ("C", ctypes.c_void_p),
                ("ldc", ctypes.c_int64), ("dtype", ctypes.c_int)]


class GemmError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        super().__init__("%s%s (status %d)" % (what + ": " if what else "", status_string(status), status))


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError("%s is not built; run __graft_entry__.build() first" % LIB_PATH)
    lib = ctypes.CDLL(LIB_PATH)
    i64, p, i32 = ctypes.c_int64, ctypes.c_void_p, ctypes.c_int
    lib.gemm_create.argtypes = [ctypes.POINTER(p), i32]
    lib.gemm_destroy.argtypes = [p]
    lib.gemm_run.argtypes = [p, i64, i64, i64, p, i64, p, i64, p, i64, i32, p]
    lib.gemm_run_host.argtypes = [p, i64, i64, i64, p, i64, p, i64, p, i64, i32, p]
    lib.gemm_run_host_batch.argtypes = [p, i32, ctypes.POINTER(HostProblem), p]
    f32 = ctypes.c_float
    lib.gemm_run_ex.argtypes = [p, i64, i64, i64, f32, p, i64, p, i64, f32, p, i64, i32, i32, p]
    lib.conv4d_im2col.argtypes = [p, p, i64, ctypes.POINTER(i64), ctypes.POINTER(i64), p, p]
    lib.conv4d_forward.argtypes = [p, p, i64, ctypes.POINTER(i64), p, i64, ctypes.POINTER(i64), p, i64, p]
    lib.conv4d_forward_cl.argtypes = [p, p, i64, ctypes.POINTER(i64), p, i64, ctypes.POINTER(i64), p, i32, p]
    lib.conv4d_forward_tc.argtypes = [p, p, i64, ctypes.POINTER(i64), p, i64, ctypes.POINTER(i64), p, i64, i32, p]
    lib.gemm_get_device_status.argtypes = [p, p]
    lib.gemm_set_option.argtypes = [p, i32, i64]
    lib.gemm_launch_count.argtypes = [p]
    lib.gemm_run_f32_skinny_noalloc.argtypes = [i64, i64, i64, p, i64, p, i64, p, i64, i32, p]
    lib.gemm_status_string.argtypes = [i32]
    lib.gemm_status_string.restype = ctypes.c_char_p
    for name in EXPORTS:
        if name != "gemm_status_string":
            getattr(lib, name).restype = i32
    lib.gemm_launch_count.restype = i64
    return lib


_lib = _load()


def library():
    """The loaded ctypes library (for callers that want the raw C ABI)."""
    return _lib


# ----------------------------------------------------------------- C ABI, same names

def gemm_create(device: int = 0) -> int:
    h = ctypes.c_void_p()
    rc = _lib.gemm_create(ctypes.byref(h), int(device))
    if rc != GEMM_OK:
        raise GemmError(rc, "gemm_create")
    return h.value


def gemm_destroy(h: int) -> int:
    return _lib.gemm_destroy(h)


def gemm_run(h, M, N, K, A, lda, B, ldb, C, ldc, dtype, stream=0) -> int:
    return _lib.gemm_run(h, M, N, K, A, lda, B, ldb, C, ldc, dtype, stream)


def gemm_run_ex(h, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, ab_dtype, c_dtype, stream=0) -> int:
    return _lib.gemm_run_ex(h, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, ab_dtype, c_dtype, stream)


def gemm_run_host(h, M, N, K, A, lda, B, ldb, C, ldc, dtype, stream=0) -> int:
    return _lib.gemm_run_host(h, M, N, K, A, lda, B, ldb, C, ldc, dtype, stream)


def gemm_run_host_batch(h, problems, stream=0) -> int:
    """problems: a sequence of HostProblem (or tuples of its fields)."""
    arr = (HostProblem * len(problems))(*[q if isinstance(q, HostProblem) else HostProblem(*q) for q in problems])
    return _lib.gemm_run_host_batch(h, len(problems), arr, stream)


def conv4d_im2col(h, x, C_in, in_dims, k_dims, col, stream=0) -> int:
    ins = (ctypes.c_int64 * 4)(*[int(v) for v in in_dims])
    ks = (ctypes.c_int64 * 4)(*[int(v) for v in k_dims])
    return _lib.conv4d_im2col(h, x, C_in, ins, ks, col, stream)


def conv4d_forward(h, x, C_in, in_dims, w, C_out, k_dims, y, ldy, stream=0) -> int:
    ins = (ctypes.c_int64 * 4)(*[int(v) for v in in_dims])
    ks = (ctypes.c_int64 * 4)(*[int(v) for v in k_dims])
    return _lib.conv4d_forward(h, x, C_in, ins, w, C_out, ks, y, ldy, stream)


def conv4d_forward_cl(h, x, C_in, in_dims, w, C_out, k_dims, y, dtype, stream=0) -> int:
    ins = (ctypes.c_int64 * 4)(*[int(v) for v in in_dims])
    ks = (ctypes.c_int64 * 4)(*[int(v) for v in k_dims])
    return _lib.conv4d_forward_cl(h, x, C_in, ins, w, C_out, ks, y, dtype, stream)


def conv4d_forward_tc(h, x, C_in, in_dims, w, C_out, k_dims, y, ldy, dtype, stream=0) -> int:
    ins = (ctypes.c_int64 * 4)(*[int(v) for v in in_dims])
    ks = (ctypes.c_int64 * 4)(*[int(v) for v in k_dims])
    return _lib.conv4d_forward_tc(h, x, C_in, ins, w, C_out, ks, y, ldy, dtype, stream)


def gemm_get_device_status(h, stream=0) -> int:
    return _lib.gemm_get_device_status(h, stream)


def gemm_set_option(h, option: int, value: int) -> int:
    return _lib.gemm_set_option(h, int(option), int(value))


def gemm_launch_count(h) -> int:
    return _lib.gemm_launch_count(h)


def status_string(status: int) -> str:
    return _lib.gemm_status_string(int(status)).decode()


gemm_status_string = status_string


# ------------------------------------------------------- tensor conveniences (torch)

_DTYPES = None


def _dtype_code(t):
    global _DTYPES
    import torch
    if _DTYPES is None:
        _DTYPES = {torch.float32: GEMM_F32, torch.bfloat16: GEMM_BF16, torch.float16: GEMM_F16}
    try:
        return _DTYPES[t.dtype]
    except KeyError:
        raise TypeError("unsupported input dtype %s" % t.dtype) from None


def _row_major_2d(t, name):
    if t.dim() != 2 or (t.shape[1] > 1 and t.stride(1) != 1) or (t.shape[0] > 1 and t.stride(0) < t.shape[1]):
        raise ValueError("%s must be a 2-D row-major tensor (unit column stride), got strides %s"
                         % (name, tuple(t.stride())))
    return max(t.stride(0), t.shape[1], 1)


class Gemm:
    """A library handle bound to one CUDA device."""

    def __init__(self, device: int = 0):
        self.device = int(device)
        self.handle = gemm_create(self.device)

    def close(self):
        if self.handle:
            gemm_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def set_option(self, option: int, value: int):
        rc = gemm_set_option(self.handle, option, value)
        if rc != GEMM_OK:
            raise GemmError(rc, "gemm_set_option")

    def matmul(self, A, B, out=None, stream=None, alpha=1.0, beta=0.0, out_dtype=None):
        """out[M, N] = alpha * A[M, K] @ B[K, N] + beta * out; A, B fp32 / bf16 / fp16 CUDA
        tensors; out fp32 (default) or bf16 / fp16; out is read only when beta != 0."""
        import torch
        if A.dtype != B.dtype:
            raise TypeError("A and B must have the same dtype")
        M, K = A.shape
        K2, N = B.shape
        if K2 != K:
            raise ValueError("inner dimensions differ")
        if out is None:
            if beta != 0.0:
                raise ValueError("beta != 0 needs an existing out")
            out = torch.empty((M, N), dtype=out_dtype or torch.float32, device=A.device)
        lda, ldb, ldc = _row_major_2d(A, "A"), _row_major_2d(B, "B"), _row_major_2d(out, "out")
        s = torch.cuda.current_stream(A.device).cuda_stream if stream is None else int(stream)
        if alpha == 1.0 and beta == 0.0 and out.dtype == torch.float32:
            rc = gemm_run(self.handle, M, N, K, A.data_ptr(), lda, B.data_ptr(), ldb, out.data_ptr(), ldc,
                          _dtype_code(A), s)
        else:
            rc = gemm_run_ex(self.handle, M, N, K, float(alpha), A.data_ptr(), lda, B.data_ptr(), ldb, float(beta),
                             out.data_ptr(), ldc, _dtype_code(A), _dtype_code(out), s)
        if rc != GEMM_OK:
            raise GemmError(rc, "gemm_run")
        return out

    def matmul_host(self, A, B, out=None, stream=None):
        """The same product with CPU tensors in and out (copies inside the library)."""
        import torch
        M, K = A.shape
        N = B.shape[1]
        if out is None:
            out = torch.empty((M, N), dtype=torch.float32)
        lda, ldb, ldc = _row_major_2d(A, "A"), _row_major_2d(B, "B"), _row_major_2d(out, "out")
        s = 0 if stream is None else int(stream)
        rc = gemm_run_host(self.handle, M, N, K, A.data_ptr(), lda, B.data_ptr(), ldb, out.data_ptr(), ldc,
                           _dtype_code(A), s)
        if rc != GEMM_OK:
            raise GemmError(rc, "gemm_run_host")
        return out

    def matmul_host_batch(self, pairs, outs=None, stream=None):
        """Several products of CPU tensors as one pipeline: pairs = [(A, B), ...]."""
        import torch
        if outs is None:
            outs = [torch.empty((A.shape[0], B.shape[1]), dtype=torch.float32) for A, B in pairs]
        probs = []
        for (A, B), out in zip(pairs, outs):
            if A.shape[1] != B.shape[0] or tuple(out.shape) != (A.shape[0], B.shape[1]) or A.dtype != B.dtype:
                raise ValueError("shapes or dtypes do not match")
            probs.append(HostProblem(A.shape[0], B.shape[1], A.shape[1], A.data_ptr(), _row_major_2d(A, "A"),
                                     B.data_ptr(), _row_major_2d(B, "B"), out.data_ptr(), _row_major_2d(out, "out"),
                                     _dtype_code(A)))
        s = 0 if stream is None else int(stream)
        rc = gemm_run_host_batch(self.handle, probs, s)
        if rc != GEMM_OK:
            raise GemmError(rc, "gemm_run_host_batch")
        return outs

    def im2col4d(self, x, ks, col=None, stream=None):
        """Column matrix [C_in*prod(ks), prod(in-ks+1)] of a valid 4-D cross-correlation."""
        import torch
        if x.dim() != 5 or x.dtype != torch.float32 or not x.is_contiguous():
            raise ValueError("x must be a contiguous fp32 [C_in, I0, I1, I2, I3] tensor")
        cin = x.shape[0]
        ins = list(x.shape[1:])
        outs = [i - k + 1 for i, k in zip(ins, ks)]
        rows = cin * ks[0] * ks[1] * ks[2] * ks[3]
        cols = outs[0] * outs[1] * outs[2] * outs[3]
        if col is None:
            col = torch.empty((rows, cols), dtype=torch.float32, device=x.device)
        s = torch.cuda.current_stream(x.device).cuda_stream if stream is None else int(stream)
        rc = conv4d_im2col(self.handle, x.data_ptr(), cin, ins, ks, col.data_ptr(), s)
        if rc != GEMM_OK:
            raise GemmError(rc, "conv4d_im2col")
        return col

    def conv4d_implicit(self, x, w, out=None, stream=None):
        """Valid 4-D cross-correlation as an implicit GEMM: y[C_out, P0, P1, P2, P3]."""
        import torch
        if x.dim() != 5 or w.dim() != 6 or x.dtype != torch.float32 or w.dtype != torch.float32:
            raise ValueError("x must be fp32 [C_in, I0..I3] and w fp32 [C_out, C_in, R0..R3]")
        if not (x.is_contiguous() and w.is_contiguous()):
            raise ValueError("x and w must be contiguous")
        cin, cout = x.shape[0], w.shape[0]
        ks = list(w.shape[2:])
        outs = [i - k + 1 for i, k in zip(x.shape[1:], ks)]
        npos = outs[0] * outs[1] * outs[2] * outs[3]
        if out is None:
            out = torch.empty((cout, npos), dtype=torch.float32, device=x.device)
        ldy = _row_major_2d(out, "out")
        s = torch.cuda.current_stream(x.device).cuda_stream if stream is None else int(stream)
        rc = conv4d_forward(self.handle, x.data_ptr(), cin, list(x.shape[1:]), w.data_ptr(), cout, ks,
                            out.data_ptr(), ldy, s)
        if rc != GEMM_OK:
            raise GemmError(rc, "conv4d_forward")
        return out.view(cout, *outs) if out.is_contiguous() else out

    def conv4d_cl(self, x, w, out=None, stream=None):
        """Valid 4-D cross-correlation on the tensor cores, channel-last 16-bit operands.

        x: [I0, I1, I2, I3, C_in] and w: [C_out, R0, R1, R2, R3, C_in], both bf16 or both
        fp16, contiguous; returns y: fp32 [P0, P1, P2, P3, C_out]."""
        import torch
        dt = {torch.bfloat16: GEMM_BF16, torch.float16: GEMM_F16}.get(x.dtype)
        if x.dim() != 5 or w.dim() != 6 or dt is None or w.dtype != x.dtype:
            raise ValueError("x must be [I0..I3, C_in] and w [C_out, R0..R3, C_in], both bf16 or both fp16")
        if not (x.is_contiguous() and w.is_contiguous()) or w.shape[5] != x.shape[4]:
            raise ValueError("x and w must be contiguous with the same C_in")
        cin, cout = x.shape[4], w.shape[0]
        ins, ks = list(x.shape[:4]), list(w.shape[1:5])
        outs = [i - k + 1 for i, k in zip(ins, ks)]
        if out is None:
            out = torch.empty(outs + [cout], dtype=torch.float32, device=x.device)
        elif list(out.shape) != outs + [cout] or out.dtype != torch.float32 or not out.is_contiguous():
            raise ValueError("out must be contiguous fp32 %s" % (outs + [cout],))
        s = torch.cuda.current_stream(x.device).cuda_stream if stream is None else int(stream)
        rc = conv4d_forward_cl(self.handle, x.data_ptr(), cin, ins, w.data_ptr(), cout, ks, out.data_ptr(), dt, s)
        if rc != GEMM_OK:
            raise GemmError(rc, "conv4d_forward_cl")
        return out

    def conv4d_tc(self, x, w, out=None, stream=None):
        """Valid 4-D cross-correlation on the tensor cores, channel-first 16-bit operands.

        x: [C_in, I0, I1, I2, I3] and w: [C_out, C_in, R0, R1, R2, R3], both bf16 or both
        fp16, contiguous; returns y: fp32 [C_out, P0, P1, P2, P3] (or writes `out`, whose
        rows over the output positions may be strided: out[o] at out.data_ptr() + o
        out.stride(0))."""
        import torch
        dt = {torch.bfloat16: GEMM_BF16, torch.float16: GEMM_F16}.get(x.dtype)
        if x.dim() != 5 or w.dim() != 6 or dt is None or w.dtype != x.dtype:
            raise ValueError("x must be [C_in, I0..I3] and w [C_out, C_in, R0..R3], both bf16 or both fp16")
        if not (x.is_contiguous() and w.is_contiguous()) or w.shape[1] != x.shape[0]:
            raise ValueError("x and w must be contiguous with the same C_in")
        cin, cout = x.shape[0], w.shape[0]
        ins, ks = list(x.shape[1:]), list(w.shape[2:])
        outs = [i - k + 1 for i, k in zip(ins, ks)]
        npos = 1
        for v in outs:
            npos *= v
        if out is None:
            out = torch.empty([cout] + outs, dtype=torch.float32, device=x.device)
        if out.dtype != torch.float32 or out.shape[0] != cout or out[0].numel() != npos or \
                not out[0].is_contiguous():
            raise ValueError("out must be fp32 [%d, %s] with contiguous rows" % (cout, outs))
        s = torch.cuda.current_stream(x.device).cuda_stream if stream is None else int(stream)
        rc = conv4d_forward_tc(self.handle, x.data_ptr(), cin, ins, w.data_ptr(), cout, ks, out.data_ptr(),
                               out.stride(0), dt, s)
        if rc != GEMM_OK:
            raise GemmError(rc, "conv4d_forward_tc")
        return out

    def conv4d(self, x, w, col=None, out=None, stream=None):
        """Valid 4-D cross-correlation as im2col + GEMM: y[C_out, P0, P1, P2, P3]."""
        ks = list(w.shape[2:])
        col = self.im2col4d(x, ks, col=col, stream=stream)
        cout = w.shape[0]
        y = self.matmul(w.reshape(cout, -1), col, out=out, stream=stream)
        outs = [i - k + 1 for i, k in zip(x.shape[1:], ks)]
        return y.view(cout, *outs)

    def launch_count(self) -> int:
        return gemm_launch_count(self.handle)

    def device_status(self, stream=None) -> int:
        import torch
        s = torch.cuda.current_stream(self.device).cuda_stream if stream is None else int(stream)
        return gemm_get_device_status(self.handle, s)


__all__ = ["Gemm", "GemmError", "HostProblem", "gemm_create", "gemm_destroy", "gemm_run", "gemm_run_ex",
           "gemm_run_host", "gemm_run_host_batch",
           "conv4d_im2col", "conv4d_forward", "conv4d_forward_cl", "conv4d_forward_tc", "gemm_get_device_status", "gemm_set_option", "gemm_launch_count",
           "gemm_status_string",
           "status_string", "library", "LIB_PATH", "EXPORTS"]
