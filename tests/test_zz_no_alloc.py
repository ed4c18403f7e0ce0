"""The allocation-free skinny fp32 entry point, gemm_run_f32_skinny_noalloc.

It is meant for callers that may not allocate device memory (code running inside
another framework's memory manager, or on a path where cudaMalloc's device-wide
synchronisation is not acceptable): it takes no handle and keeps its split-K partial
sums in a fixed 32 MiB array inside the library instead of an allocated workspace.

These tests call it through the C ABI (ctypes, no binding helper) twice in a row and
compare each result with the existing entry point, gemm_run, on the same inputs, within
the fp32 tolerance the other tests use (1e-5 * sqrt(K)).  With gemm_run told to use the
same kernel (the register-streaming skinny kernel) and the default split, both run the
same code with the same split, so those results are also expected to be identical.
The file sorts last so that a run that stops at the first failure has run every other
test first; it also passes on its own in a fresh process.
"""
import ctypes
import math

import numpy as np
import pytest
import torch

import seeded_inputs as si

pytestmark = pytest.mark.gpu

SCRATCH_FLOATS = 8 << 20


@pytest.fixture(scope="module")
def g():
    import __graft_entry__
    __graft_entry__.build()
    import programming_tiled_gemm_gb300 as g
    return g


def noalloc(g, A, B, C, split_k=0, stream=None):
    M, K = A.shape
    N = B.shape[1]
    s = torch.cuda.current_stream().cuda_stream if stream is None else stream
    return g.library().gemm_run_f32_skinny_noalloc(
        ctypes.c_int64(M), ctypes.c_int64(N), ctypes.c_int64(K), ctypes.c_void_p(A.data_ptr()),
        ctypes.c_int64(A.stride(0)), ctypes.c_void_p(B.data_ptr()), ctypes.c_int64(B.stride(0)),
        ctypes.c_void_p(C.data_ptr()), ctypes.c_int64(C.stride(0)), ctypes.c_int(split_k), ctypes.c_void_p(s))


@pytest.mark.parametrize("M,N,K,split_k", [
    (16, 16384, 16384, 0),   # the skinny workload, default split
    (13, 3001, 4097, 0),     # ragged columns, K not a multiple of the A step
    (32, 20736, 10000, 0),   # the convolution GEMM shape
    (5, 777, 2000, 9),       # a forced split
    (1, 64, 64, 1),          # no split: the scratch array is not used
])
def test_matches_gemm_run_on_two_calls_in_a_row(g, M, N, K, split_k):
    dev = torch.device("cuda")
    A, B = si.gemm_operands(M, N, K, seed=M + N + K)
    Ad, Bd = A.to(dev), B.to(dev)
    ref_lib = g.Gemm(0)
    if split_k:
        ref_lib.set_option(g.GEMM_OPT_SPLIT_K, split_k)
    ref_default = ref_lib.matmul(Ad, Bd)  # gemm_run's default kernel choice
    ref_lib.set_option(g.GEMM_OPT_F32_KERNEL, 3)
    ref = ref_lib.matmul(Ad, Bd)  # the kernel this entry point runs
    torch.cuda.synchronize()
    tol = 1e-5 * math.sqrt(K)
    outs = []
    for _ in range(2):
        C = torch.full((M, N), float("nan"), device=dev)
        assert noalloc(g, Ad, Bd, C, split_k) == g.GEMM_OK
        torch.cuda.synchronize()
        assert torch.isfinite(C).all()
        assert (C - ref).abs().max().item() <= tol
        assert (C - ref_default).abs().max().item() <= tol
        outs.append(C)
    assert torch.equal(outs[0], outs[1])
    assert torch.equal(outs[0], ref)  # same kernel, same split: identical sums
    ref_lib.close()


def test_integer_inputs_exact(g):
    import oracle
    dev = torch.device("cuda")
    A, B = si.integer_copy(24, 5000, 3000, seed=17)
    C = torch.empty((24, 5000), device=dev)
    for _ in range(2):
        assert noalloc(g, A.to(dev), B.to(dev), C) == g.GEMM_OK
        torch.cuda.synchronize()
        assert np.array_equal(C.cpu().double().numpy(), oracle.gemm(A.numpy(), B.numpy()))


def test_size_limit_and_argument_errors(g):
    dev = torch.device("cuda")
    A = torch.ones((32, 64), device=dev)
    B = torch.ones((64, 16384), device=dev)
    C = torch.empty((32, 16384), device=dev)
    # 64 slices x 32 x 16384 floats = 32 Mi floats > the 8 Mi-float scratch array
    assert 64 * 32 * 16384 > SCRATCH_FLOATS
    assert noalloc(g, A, B, C, split_k=64) == g.GEMM_ERR_UNSUPPORTED
    A33 = torch.ones((33, 64), device=dev)
    C33 = torch.empty((33, 16384), device=dev)
    assert noalloc(g, A33, B, C33) == g.GEMM_ERR_UNSUPPORTED
    assert noalloc(g, A, B, C, split_k=5000) == g.GEMM_ERR_INVALID_ARG
    lib = g.library()
    assert lib.gemm_run_f32_skinny_noalloc(4, 4, 4, None, 4, None, 4, None, 4, 0, None) == g.GEMM_ERR_INVALID_ARG
    assert lib.gemm_run_f32_skinny_noalloc(4, 4, 4, A.data_ptr(), 3, B.data_ptr(), 16384, C.data_ptr(), 16384,
                                           0, None) == g.GEMM_ERR_INVALID_ARG


def test_leftover_scratch_from_a_larger_split_never_reaches_the_sum(g):
    """A call with a large split x M x N layout fills the shared scratch array with NaN
    partial sums (its inputs hold NaNs); the next call, on the same stream, uses a smaller
    layout over the same array and must still equal gemm_run: every partial sum it adds
    was written by itself."""
    dev = torch.device("cuda")
    # shape X: split 9, 24 x 8000 -> 1.73 Mi floats of partials, all NaN
    Ax = torch.full((24, 900), float("nan"), device=dev)
    Bx = torch.ones((900, 8000), device=dev)
    Cx = torch.empty((24, 8000), device=dev)
    assert noalloc(g, Ax, Bx, Cx, split_k=9) == g.GEMM_OK
    # shape Y: split 3, 7 x 3001 -> a different slice stride over the same array
    A, B = si.gemm_operands(7, 3001, 1500, seed=23)
    Ad, Bd = A.to(dev), B.to(dev)
    ref_lib = g.Gemm(0)
    ref_lib.set_option(g.GEMM_OPT_SPLIT_K, 3)
    ref_lib.set_option(g.GEMM_OPT_F32_KERNEL, 3)
    ref = ref_lib.matmul(Ad, Bd)
    for _ in range(2):
        Cy = torch.full((7, 3001), float("nan"), device=dev)
        assert noalloc(g, Ad, Bd, Cy, split_k=3) == g.GEMM_OK
        torch.cuda.synchronize()
        assert torch.isnan(Cx).all()  # the first call really left NaNs behind
        assert torch.isfinite(Cy).all()
        assert torch.equal(Cy, ref)
        assert (Cy - ref).abs().max().item() <= 1e-5 * math.sqrt(1500)
        assert noalloc(g, Ax, Bx, Cx, split_k=9) == g.GEMM_OK  # NaNs again before the repeat
    ref_lib.close()


def test_sizes_beyond_the_kernels_limits_are_refused_before_any_launch(g):
    """The entry point applies gemm_run's checks: 32-bit kernel limits (unsupported) and
    the element-offset range (invalid), and compares the scratch need without
    overflowing."""
    dev = torch.device("cuda")
    A = torch.ones((16, 64), device=dev)
    B = torch.ones((64, 256), device=dev)
    C = torch.empty((16, 256), device=dev)
    lib = g.library()
    big = 1 << 40  # N far beyond 32-bit indexing; split * M * N would not overflow int64 here
    assert lib.gemm_run_f32_skinny_noalloc(16, big, 64, A.data_ptr(), 64, B.data_ptr(), big, C.data_ptr(), big,
                                           0, None) == g.GEMM_ERR_UNSUPPORTED
    huge = 1 << 62  # leading dimensions whose offsets leave the int64 range
    assert lib.gemm_run_f32_skinny_noalloc(16, 256, 64, A.data_ptr(), 64, B.data_ptr(), huge, C.data_ptr(), 256,
                                           0, None) == g.GEMM_ERR_INVALID_ARG
    assert noalloc(g, A, B, C) == g.GEMM_OK  # a valid call still runs after the refusals
    torch.cuda.synchronize()
    assert torch.equal(C, torch.full_like(C, 64.0))
