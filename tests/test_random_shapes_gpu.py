"""Seeded random shapes through every default path, exact against the oracle.

The other GPU tests pick their shapes by hand (tails, waves, slices, splits).  These draw
them: sizes from 1 up to a few tiles in every dimension, so that edge tiles, partial waves,
K tails and the automatic kernel, split and stack choices meet in combinations nobody
chose.  Inputs are integers in [-4, 4], so every partial sum is an integer below 2^24 and
the results must equal the fp64 oracle exactly, whatever the summation order.
"""
import random

import numpy as np
import pytest
import torch

import oracle
import seeded_inputs as si

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__
    __graft_entry__.build()
    import programming_tiled_gemm_gb300 as g
    h = g.Gemm(0)
    yield h
    h.close()


def _shapes(seed, count, lo, hi, k_hi, multiple=1):
    rng = random.Random(seed)
    out = []
    for _ in range(count):
        M = rng.randint(lo, hi)
        N = rng.randint(lo, hi) // multiple * multiple or multiple
        K = rng.randint(lo, k_hi) // multiple * multiple or multiple
        out.append((M, N, K))
    return out


F32_SHAPES = _shapes(101, 16, 1, 900, 1500)
BF16_SHAPES = _shapes(202, 16, 1, 1100, 1800, multiple=8)  # 16-byte rows for the TMA


@pytest.mark.parametrize("M,N,K", F32_SHAPES)
def test_fp32_default_path_exact(lib, M, N, K):
    import programming_tiled_gemm_gb300 as g
    A, B = si.integer_copy(M, N, K, seed=M * 7 + N * 3 + K)
    C = lib.matmul(A.cuda(), B.cuda())
    torch.cuda.synchronize()
    assert lib.device_status() == g.GEMM_OK
    assert np.array_equal(C.cpu().double().numpy(), oracle.gemm(A.numpy(), B.numpy()))


@pytest.mark.parametrize("M,N,K", BF16_SHAPES)
def test_bf16_default_path_exact(lib, M, N, K):
    import programming_tiled_gemm_gb300 as g
    A, B = si.integer_copy(M, N, K, seed=M * 5 + N + K * 11, dtype="bf16")
    C = lib.matmul(A.cuda(), B.cuda())
    torch.cuda.synchronize()
    assert lib.device_status() == g.GEMM_OK
    assert np.array_equal(C.cpu().double().numpy(), oracle.gemm(A.float().numpy(), B.float().numpy()))


def _conv_shapes(seed, count):
    rng = random.Random(seed)
    out = []
    for _ in range(count):
        ks = [rng.randint(1, 5) for _ in range(4)]
        ins = [k + rng.randint(0, 9) for k in ks]
        out.append((rng.randint(1, 24), rng.choice([16, 32, 48]), tuple(ins), tuple(ks)))
    return out


@pytest.mark.parametrize("cin,cout,ins,ks", _conv_shapes(303, 10))
def test_implicit_convolution_exact(lib, cin, cout, ins, ks):
    import programming_tiled_gemm_gb300 as g
    gen = si.generator(cin + cout + sum(ins))
    x = si.ints((cin,) + ins, gen).float()
    w = si.ints((cout, cin) + ks, gen).float()
    y = lib.conv4d_implicit(x.cuda(), w.cuda())
    torch.cuda.synchronize()
    assert lib.device_status() == g.GEMM_OK
    assert np.array_equal(y.cpu().double().numpy(), oracle.conv4d_direct(x.numpy(), w.numpy()))


@pytest.mark.parametrize("cin,cout,ins,ks", _conv_shapes(404, 10))
def test_tensor_core_convolution_channel_first_exact(lib, cin, cout, ins, ks):
    """Channel counts padded to 16 by the re-layout; stack and K split chosen by the plan."""
    import programming_tiled_gemm_gb300 as g
    gen = si.generator(2 * cin + cout + sum(ks))
    x = si.ints((cin,) + ins, gen).float()
    w = si.ints((cout, cin) + ks, gen).float()
    try:
        y = lib.conv4d_tc(x.to(torch.bfloat16).cuda(), w.to(torch.bfloat16).cuda())
    except g.GemmError as e:  # shapes the kernel does not take (a stage that does not fit)
        assert e.status == g.GEMM_ERR_UNSUPPORTED
        pytest.skip("shape outside the tensor-core convolution's plan")
    torch.cuda.synchronize()
    assert lib.device_status() == g.GEMM_OK
    assert np.array_equal(y.cpu().double().numpy(), oracle.conv4d_direct(x.numpy(), w.numpy()))
