"""Failure detection on the GPU without a fault.

Every mbarrier wait in the tensor-core kernels and the TMA-fed fp32 kernels is bounded
by a wall-clock limit.  GEMM_OPT_TEST_STALL makes the kernel wait once on a barrier that
nothing ever arrives on, so that wait runs out: the kernel records a timeout in the
handle's status word, lets its other roles give up, waits (bounded) for the copies and
MMAs it already issued, frees its tensor memory and returns.  The host then reads
GEMM_ERR_DEVICE_TIMEOUT, and the same context keeps computing correct products.
No trap, assert, bad address or unbounded loop is involved.
"""
import numpy as np
import pytest
import torch

import oracle
import seeded_inputs as si

pytestmark = pytest.mark.gpu


@pytest.fixture()
def lib():
    import __graft_entry__
    __graft_entry__.build()
    import programming_tiled_gemm_gb300 as g
    h = g.Gemm(0)
    h.set_option(g.GEMM_OPT_WAIT_LIMIT_US, 20000)  # 20 ms
    yield h
    h.set_option(g.GEMM_OPT_TEST_STALL, 0)
    h.close()


@pytest.mark.parametrize("pair", [1, 2])
def test_tensor_core_wait_runs_out_and_is_reported(lib, pair):
    import programming_tiled_gemm_gb300 as g
    dev = torch.device("cuda")
    A, B = si.integer_copy(512, 512, 1024, seed=31, dtype="bf16")
    Ad, Bd = A.to(dev), B.to(dev)
    lib.set_option(g.GEMM_OPT_TC_PAIR, pair)
    lib.set_option(g.GEMM_OPT_TEST_STALL, 1)
    C = torch.zeros((512, 512), device=dev)
    lib.matmul(Ad, Bd, out=C)  # the launch itself succeeds
    assert lib.device_status() == g.GEMM_ERR_DEVICE_TIMEOUT
    assert lib.device_status() == g.GEMM_OK  # reading the status clears it
    # the context is intact: the next product is correct
    lib.set_option(g.GEMM_OPT_TEST_STALL, 0)
    C = lib.matmul(Ad, Bd)
    torch.cuda.synchronize()
    assert lib.device_status() == g.GEMM_OK
    assert np.array_equal(C.cpu().double().numpy(), oracle.gemm(A.float().numpy(), B.float().numpy()))


def test_skinny_wait_runs_out_and_is_reported(lib):
    import programming_tiled_gemm_gb300 as g
    dev = torch.device("cuda")
    A, B = si.integer_copy(16, 4096, 2048, seed=32)
    Ad, Bd = A.to(dev), B.to(dev)
    lib.set_option(g.GEMM_OPT_F32_KERNEL, 4)
    lib.set_option(g.GEMM_OPT_TEST_STALL, 1)
    lib.matmul(Ad, Bd)
    assert lib.device_status() == g.GEMM_ERR_DEVICE_TIMEOUT
    lib.set_option(g.GEMM_OPT_TEST_STALL, 0)
    C = lib.matmul(Ad, Bd)
    torch.cuda.synchronize()
    assert lib.device_status() == g.GEMM_OK
    assert np.array_equal(C.cpu().double().numpy(), oracle.gemm(A.numpy(), B.numpy()))


def test_persistent_fp32_wait_runs_out_and_is_reported(lib):
    import programming_tiled_gemm_gb300 as g
    dev = torch.device("cuda")
    A, B = si.integer_copy(700, 900, 1000, seed=33)
    Ad, Bd = A.to(dev), B.to(dev)
    lib.set_option(g.GEMM_OPT_F32_KERNEL, 5)
    lib.set_option(g.GEMM_OPT_TEST_STALL, 1)
    lib.matmul(Ad, Bd)
    assert lib.device_status() == g.GEMM_ERR_DEVICE_TIMEOUT
    lib.set_option(g.GEMM_OPT_TEST_STALL, 0)
    C = lib.matmul(Ad, Bd)
    torch.cuda.synchronize()
    assert lib.device_status() == g.GEMM_OK
    assert np.array_equal(C.cpu().double().numpy(), oracle.gemm(A.numpy(), B.numpy()))
    lib.set_option(g.GEMM_OPT_F32_KERNEL, 0)


def test_test_hook_rejects_other_values(lib):
    import programming_tiled_gemm_gb300 as g
    assert g.gemm_set_option(lib.handle, g.GEMM_OPT_TEST_STALL, 2) == g.GEMM_ERR_INVALID_ARG
