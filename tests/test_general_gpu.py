"""The generalised product C = alpha * A.B + beta * C (gemm_run_ex) against the oracle.

The oracle's gemm_general follows the GEMM page's "Generalised matrix multiplication GEMM"
section in fp64.  Exact cases use integer-valued inputs with dyadic alpha and beta, whose
results are representable in the output type (fp32 always; bf16 / fp16 for small
magnitudes); general cases allow the fp32 GEMM tolerance scaled by |alpha| plus one
rounding of the output type.  Every kernel family is covered: tensor-core CTA pairs and
single CTAs (bf16 and fp16 inputs, fused epilogue) and the fp32 tiled and skinny kernels
(separate epilogue pass).
"""
import math

import numpy as np
import pytest
import torch

import oracle
import seeded_inputs as si

pytestmark = pytest.mark.gpu
GUARD = 2

PATHS = [  # (name, input dtype, M, N, K, tc pair option)
    ("tc_pair", "bf16", 520, 264, 136, 2),
    ("tc_single", "f16", 300, 264, 72, 1),
    ("tc_split_k", "bf16", 100, 1000, 1100, 0),  # M <= 128, 4 tiles: K in 2 slices
    ("tc_pair_last_wave", "bf16", 520, 264, 4160, 2),  # 6 pair tiles, each in 2 K slices
    ("f32_tiled", "f32", 200, 250, 130, 0),
    ("f32_skinny", "f32", 20, 1030, 300, 0),
]
OUT = {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16}


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__
    __graft_entry__.build()
    import programming_tiled_gemm_gb300 as g
    h = g.Gemm(0)
    yield h
    h.close()


def padded_operands(A, B, dev):
    M, K = A.shape
    N = B.shape[1]
    Ad = torch.zeros((M, (K + 7) // 8 * 8 + 8), dtype=A.dtype, device=dev)
    Ad[:, :K] = A.to(dev)
    Bd = torch.zeros((K, (N + 7) // 8 * 8 + 8), dtype=B.dtype, device=dev)
    Bd[:, :N] = B.to(dev)
    return Ad[:, :K], Bd[:, :N]


def run_general(lib, A, B, C0, alpha, beta, out_dtype, pair):
    """C (guard-banded, padded rows) = alpha A B + beta C0; returns C as float64 numpy."""
    import programming_tiled_gemm_gb300 as g
    dev = torch.device("cuda")
    lib.set_option(g.GEMM_OPT_TC_PAIR, pair)
    M, N = C0.shape
    Ad, Bd = padded_operands(A, B, dev)
    big = torch.full((M + 2 * GUARD, N + 8 + 2 * GUARD), -7.0, dtype=OUT[out_dtype], device=dev)
    C = big[GUARD:GUARD + M, GUARD:GUARD + N]
    C.copy_(C0.to(dev))
    lib.matmul(Ad, Bd, out=C, alpha=alpha, beta=beta)
    torch.cuda.synchronize()
    lib.set_option(g.GEMM_OPT_TC_PAIR, 0)
    assert lib.device_status() == 0
    host = big.float().cpu()
    mask = torch.ones_like(host, dtype=torch.bool)
    mask[GUARD:GUARD + M, GUARD:GUARD + N] = False
    assert torch.all(host[mask] == -7.0), "kernel wrote outside C"
    return host[GUARD:GUARD + M, GUARD:GUARD + N].double().numpy()


@pytest.mark.parametrize("out_dtype", ["f32", "bf16", "f16"])
@pytest.mark.parametrize("name,dt,M,N,K,pair", PATHS)
def test_integer_inputs_dyadic_weights_exact(lib, name, dt, M, N, K, pair, out_dtype):
    # |A B| <= 16 K; with bf16 / fp16 outputs keep the results small enough to be exact
    Kx = K if out_dtype == "f32" else 8
    A, B = si.integer_copy(M, N, Kx, seed=M + N, dtype=dt)
    C0 = si.ints((M, N), si.generator(M * N)).float()
    alpha, beta = (0.5, -2.0) if out_dtype == "f32" else (0.5, 1.0)
    got = run_general(lib, A, B, C0.to(OUT[out_dtype]), alpha, beta, out_dtype, pair)
    ref = oracle.gemm_general(alpha, A.float().numpy(), B.float().numpy(), beta, C0.double().numpy())
    assert np.array_equal(got, ref)


@pytest.mark.parametrize("out_dtype", ["f32", "bf16"])
@pytest.mark.parametrize("name,dt,M,N,K,pair", PATHS)
def test_uniform_inputs_within_tolerance(lib, name, dt, M, N, K, pair, out_dtype):
    A, B = si.gemm_operands(M, N, K, seed=7, dist="uniform", dtype=dt)
    C0 = si.uniform((M, N), si.generator(9)).to(OUT[out_dtype])
    alpha, beta = 1.5, -0.75
    got = run_general(lib, A, B, C0, alpha, beta, out_dtype, pair)
    ref = oracle.gemm_general(alpha, A.float().numpy(), B.float().numpy(), beta, C0.double().numpy())
    gemm_tol = (2e-5 if dt != "f32" else 1e-5) * math.sqrt(K) * abs(alpha)
    out_ulp = 2.0 ** -8 if out_dtype == "bf16" else 2.0 ** -23  # one rounding of the output
    assert np.all(np.abs(got - ref) <= gemm_tol + out_ulp * np.abs(ref) + 1e-6)


@pytest.mark.parametrize("name,dt,M,N,K,pair", PATHS)
def test_beta_zero_does_not_read_C(lib, name, dt, M, N, K, pair):
    A, B = si.integer_copy(M, N, K, seed=3, dtype=dt)
    C0 = torch.full((M, N), float("nan"))
    got = run_general(lib, A, B, C0, 2.0, 0.0, "f32", pair)
    assert np.array_equal(got, 2.0 * oracle.gemm(A.float().numpy(), B.float().numpy()))


@pytest.mark.parametrize("out_dtype", ["f32", "bf16"])
def test_empty_inner_dimension_scales_C(lib, out_dtype):
    import programming_tiled_gemm_gb300 as g
    dev = torch.device("cuda")
    C = torch.full((5, 9), 3.0, dtype=OUT[out_dtype], device=dev)
    A = torch.empty((5, 0), dtype=torch.bfloat16, device=dev)
    B = torch.empty((0, 9), dtype=torch.bfloat16, device=dev)
    lib.matmul(A, B, out=C, alpha=4.0, beta=-0.5)
    torch.cuda.synchronize()
    assert torch.all(C.float() == -1.5)
    lib.matmul(A, B, out=C, alpha=4.0, beta=0.0)
    torch.cuda.synchronize()
    assert torch.all(C.float() == 0.0)
    assert g.GEMM_OK == lib.device_status()


def test_output_alignment_and_type_errors(lib):
    import programming_tiled_gemm_gb300 as g
    dev = torch.device("cuda")
    A = torch.ones((8, 8), dtype=torch.bfloat16, device=dev)
    buf = torch.zeros(100, dtype=torch.bfloat16, device=dev)
    h = lib.handle
    # fp32 output at a 2-byte offset
    assert g.gemm_run_ex(h, 8, 8, 8, 1.0, A.data_ptr(), 8, A.data_ptr(), 8, 0.0, buf.data_ptr() + 2, 8,
                         g.GEMM_BF16, g.GEMM_F32) == g.GEMM_ERR_ALIGNMENT
    # unknown output type
    assert g.gemm_run_ex(h, 8, 8, 8, 1.0, A.data_ptr(), 8, A.data_ptr(), 8, 0.0, buf.data_ptr(), 8,
                         g.GEMM_BF16, 7) == g.GEMM_ERR_INVALID_ARG
