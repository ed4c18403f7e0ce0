"""Tensor-core 4-D convolution with channel-last 16-bit operands (conv4d_forward_cl)
against the oracle's direct convolution.

The oracle computes y[o][p] = sum_{c, r} x[c][p + r] w[o][c][r] in fp64; the operands are
the same bf16 / fp16 values (exact in float32) moved to channel-first order for it, and
its output is moved to channel-last order for the comparison.
  * integer-valued inputs in [-4, 4]: exact (every partial sum is an integer below 2^24);
  * uniform[-1, 1] inputs rounded to bf16: max |y - y_ref| <= 2e-5 * sqrt(K), K = C_in x taps.
Shapes cover the 16^4 x 16 -> 32 channel, 5^4 workload, ragged extents, planes that need
one to several tiles and CTAs, and more than one 16-channel step per tap.  A guard band
around y checks that nothing is written outside it.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import seeded_inputs as si

pytestmark = pytest.mark.gpu
GUARD = 16  # floats on each side of y (keeps y 16-byte aligned)
SENTINEL = -777.0


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__
    __graft_entry__.build()
    import programming_tiled_gemm_gb300 as g
    h = g.Gemm(0)
    yield h
    h.close()


def conv_ref(x_cl: torch.Tensor, w_cl: torch.Tensor) -> np.ndarray:
    """Oracle direct convolution of channel-last operands, returned channel-last."""
    x = x_cl.float().permute(4, 0, 1, 2, 3).contiguous().numpy()
    w = w_cl.float().permute(0, 5, 1, 2, 3, 4).contiguous().numpy()
    return np.ascontiguousarray(np.moveaxis(oracle.conv4d_direct(x, w), 0, -1))


def run_guarded(lib, x_cl, w_cl):
    dev = torch.device("cuda")
    ins, ks = list(x_cl.shape[:4]), list(w_cl.shape[1:5])
    outs = [i - k + 1 for i, k in zip(ins, ks)] + [w_cl.shape[0]]
    n = int(np.prod(outs))
    big = torch.full((n + 2 * GUARD,), SENTINEL, device=dev)
    y = big[GUARD:GUARD + n].view(outs)
    lib.conv4d_cl(x_cl.to(dev), w_cl.to(dev), out=y)
    torch.cuda.synchronize()
    assert lib.device_status() == 0
    host = big.cpu()
    assert torch.all(host[:GUARD] == SENTINEL) and torch.all(host[GUARD + n:] == SENTINEL), "wrote outside y"
    return host[GUARD:GUARD + n].view(outs).double().numpy()


def int_operands(cin, cout, ins, ks, seed, dtype="bf16"):
    g = si.generator(seed)
    x = si.ints((cin,) + tuple(ins), g).float()
    w = si.ints((cout, cin) + tuple(ks), g).float()
    return si.channel_last(x, w, dtype)


SHAPES = [  # (C_in, C_out, input extents, kernel extents); odd in[3] or 2 C_out > 256 run unstacked
    (16, 32, (6, 5, 16, 16), (3, 2, 5, 5)),     # two tiles per plane, one CTA
    (32, 48, (5, 6, 7, 9), (2, 3, 2, 4)),       # two 16-channel steps per tap, one tile
    (16, 16, (3, 3, 20, 30), (1, 2, 3, 3)),     # five tiles per plane over three CTAs
    (64, 32, (3, 4, 9, 10), (2, 2, 3, 3)),      # four steps per tap
    (16, 256, (2, 2, 4, 4), (1, 1, 2, 2)),      # widest N, one accumulation chunk
    (16, 32, (2, 2, 2, 130), (1, 1, 1, 3)),     # long rows, planes of three tiles
    (48, 16, (1, 1, 1, 1), (1, 1, 1, 1)),       # a single output position
    (16, 32, (7, 7, 7, 7), (7, 7, 7, 7)),       # kernel as large as the input
]


@pytest.mark.parametrize("cin,cout,ins,ks", SHAPES)
def test_integer_inputs_are_exact(lib, cin, cout, ins, ks):
    x, w = int_operands(cin, cout, ins, ks, seed=cin + cout + sum(ins))
    assert np.array_equal(run_guarded(lib, x, w), conv_ref(x, w))


STACKED = [  # (stack S, C_in, C_out, input extents, kernel extents): S | in[3], S C_out <= 256
    (1, 16, 32, (6, 5, 16, 16), (3, 2, 5, 5)),
    (2, 16, 32, (6, 5, 16, 16), (3, 2, 5, 5)),
    (4, 16, 32, (6, 5, 16, 16), (3, 2, 5, 5)),
    (2, 32, 48, (5, 6, 7, 10), (2, 3, 2, 4)),
    (2, 16, 16, (3, 3, 20, 30), (1, 2, 3, 3)),
    (4, 16, 64, (3, 3, 9, 12), (2, 1, 4, 5)),
    (2, 16, 128, (2, 2, 4, 4), (1, 1, 2, 2)),
    (4, 16, 32, (7, 7, 7, 8), (7, 7, 7, 7)),
]


@pytest.mark.parametrize("stack,cin,cout,ins,ks", STACKED)
def test_stacked_positions_are_exact(lib, stack, cin, cout, ins, ks):
    """S output positions per tile row, stacked along the MMA's N (GEMM_OPT_CONV_STACK)."""
    import programming_tiled_gemm_gb300 as g
    x, w = int_operands(cin, cout, ins, ks, seed=7 * stack + cin + sum(ks))
    lib.set_option(g.GEMM_OPT_CONV_STACK, stack)
    try:
        got = run_guarded(lib, x, w)
    finally:
        lib.set_option(g.GEMM_OPT_CONV_STACK, 0)
    assert np.array_equal(got, conv_ref(x, w))


SPLIT = [  # (stack S, C_in, C_out, input extents, kernel extents) run with and without the K split
    (4, 16, 32, (16, 16, 16, 16), (5, 5, 5, 5)),   # the workload: 36 tiles, 144 CTAs split
    (2, 16, 32, (6, 5, 16, 16), (3, 2, 5, 5)),     # a few tiles
    (4, 32, 32, (3, 4, 9, 12), (2, 2, 3, 3)),      # two 16-channel steps per tap
    (2, 16, 64, (2, 3, 5, 6), (1, 2, 2, 3)),       # two stages, a ring shorter than the partial parts
]


@pytest.mark.parametrize("stack,cin,cout,ins,ks", SPLIT)
def test_k_split_over_two_pairs_is_exact_and_matches_one_pair(lib, stack, cin, cout, ins, ks):
    """GEMM_OPT_CONV_SPLIT 1 (one CTA pair per tile) and 2 (two pairs per tile in a cluster
    of four, partial tiles added through distributed shared memory): both exact on integer
    inputs, so both equal the oracle and each other."""
    import programming_tiled_gemm_gb300 as g
    x, w = int_operands(cin, cout, ins, ks, seed=3 * stack + cout + sum(ins))
    ref = conv_ref(x, w)
    lib.set_option(g.GEMM_OPT_CONV_STACK, stack)
    try:
        outs = []
        for split in (1, 2):
            lib.set_option(g.GEMM_OPT_CONV_SPLIT, split)
            outs.append(run_guarded(lib, x, w))
    finally:
        lib.set_option(g.GEMM_OPT_CONV_STACK, 0)
        lib.set_option(g.GEMM_OPT_CONV_SPLIT, 0)
    assert np.array_equal(outs[0], ref)
    assert np.array_equal(outs[1], ref)


def test_k_split_refusals(lib):
    """Two pairs per tile need S C_out a multiple of 32 and at least two stages."""
    import programming_tiled_gemm_gb300 as g
    dev = torch.device("cuda")
    h = lib.handle
    x = torch.zeros((2, 2, 4, 4, 16), dtype=torch.bfloat16, device=dev)
    w = torch.zeros((16, 1, 1, 2, 2, 16), dtype=torch.bfloat16, device=dev)
    y = torch.zeros((2, 2, 3, 3, 16), device=dev)
    s = torch.cuda.current_stream().cuda_stream
    lib.set_option(g.GEMM_OPT_CONV_SPLIT, 2)
    try:
        # N = 2 x 16 = 32 but a single stage (one tap triple, one channel step)
        assert g.conv4d_forward_cl(h, x.data_ptr(), 16, [2, 2, 4, 4], w.data_ptr(), 16, [1, 1, 2, 2], y.data_ptr(),
                                   g.GEMM_BF16, s) == g.GEMM_ERR_UNSUPPORTED
        lib.set_option(g.GEMM_OPT_CONV_STACK, 1)  # N = 16: not a multiple of 32
        w2 = torch.zeros((16, 2, 1, 2, 2, 16), dtype=torch.bfloat16, device=dev)
        y2 = torch.zeros((1, 2, 3, 3, 16), device=dev)
        assert g.conv4d_forward_cl(h, x.data_ptr(), 16, [2, 2, 4, 4], w2.data_ptr(), 16, [2, 1, 2, 2], y2.data_ptr(),
                                   g.GEMM_BF16, s) == g.GEMM_ERR_UNSUPPORTED
    finally:
        lib.set_option(g.GEMM_OPT_CONV_SPLIT, 0)
        lib.set_option(g.GEMM_OPT_CONV_STACK, 0)
    assert g.gemm_set_option(h, g.GEMM_OPT_CONV_SPLIT, 3) == g.GEMM_ERR_INVALID_ARG
    assert g.gemm_set_option(h, g.GEMM_OPT_CONV_SPLIT, -1) == g.GEMM_ERR_INVALID_ARG
    torch.cuda.synchronize()
    assert lib.device_status() == g.GEMM_OK


def test_integer_inputs_fp16_are_exact(lib):
    x, w = int_operands(32, 32, (4, 4, 9, 11), (2, 3, 3, 4), seed=5, dtype="f16")
    assert np.array_equal(run_guarded(lib, x, w), conv_ref(x, w))


@pytest.mark.parametrize("cin,cout,ins,ks", SHAPES[:4])
def test_uniform_bf16_within_tolerance(lib, cin, cout, ins, ks):
    g = si.generator(11)
    x, w = si.channel_last(si.uniform((cin,) + tuple(ins), g), si.uniform((cout, cin) + tuple(ks), g))
    K = cin * int(np.prod(ks))
    assert np.abs(run_guarded(lib, x, w) - conv_ref(x, w)).max() <= 2e-5 * math.sqrt(K)


def test_workload_shape_exact_and_within_tolerance(lib):
    wl = si.WORKLOADS["conv4d"]
    c = wl.conv
    x, w = si.channel_last(*si.workload_operands(wl))
    got = run_guarded(lib, x, w)
    assert np.abs(got - conv_ref(x, w)).max() <= 2e-5 * math.sqrt(wl.K)
    xi, wi = int_operands(c["cin"], c["cout"], c["ins"], c["ks"], seed=wl.seed)
    assert np.array_equal(run_guarded(lib, xi, wi), conv_ref(xi, wi))


def test_results_are_deterministic(lib):
    g = si.generator(3)
    x, w = si.channel_last(si.uniform((16, 8, 8, 12, 12), g), si.uniform((32, 16, 3, 3, 3, 3), g))
    xd, wd = x.cuda(), w.cuda()
    y1 = lib.conv4d_cl(xd, wd).clone()
    y2 = lib.conv4d_cl(xd, wd)
    assert torch.equal(y1, y2)


def test_argument_errors_are_reported(lib):
    import programming_tiled_gemm_gb300 as g
    dev = torch.device("cuda")
    h = lib.handle
    x = torch.zeros(4096, dtype=torch.bfloat16, device=dev)
    y = torch.zeros(4096, device=dev)
    ins, ks = [2, 2, 4, 4], [1, 1, 2, 2]
    run = g.conv4d_forward_cl
    assert run(h, x.data_ptr(), 8, ins, x.data_ptr(), 16, ks, y.data_ptr(), g.GEMM_BF16) == g.GEMM_ERR_UNSUPPORTED
    assert run(h, x.data_ptr(), 16, ins, x.data_ptr(), 24, ks, y.data_ptr(), g.GEMM_BF16) == g.GEMM_ERR_UNSUPPORTED
    assert run(h, x.data_ptr(), 16, ins, x.data_ptr(), 272, ks, y.data_ptr(), g.GEMM_BF16) == g.GEMM_ERR_UNSUPPORTED
    assert run(h, x.data_ptr() + 2, 16, ins, x.data_ptr(), 16, ks, y.data_ptr(), g.GEMM_BF16) == g.GEMM_ERR_ALIGNMENT
    assert run(h, x.data_ptr(), 16, ins, x.data_ptr(), 16, ks, y.data_ptr() + 4, g.GEMM_BF16) == g.GEMM_ERR_ALIGNMENT
    assert run(h, x.data_ptr(), 16, ins, x.data_ptr(), 16, ks, y.data_ptr(), g.GEMM_F32) == g.GEMM_ERR_INVALID_ARG
    assert run(h, x.data_ptr(), 16, ins, x.data_ptr(), 16, [1, 1, 5, 2], y.data_ptr(),
               g.GEMM_BF16) == g.GEMM_ERR_INVALID_ARG
    # (every call below is refused before anything is launched: the buffers are far smaller
    # than the shapes they stand for)
    # one filter triple's weights for one 16-channel step (2 boxes of 20 slices x 128
    # channels x 16 bytes) do not fit three pipeline stages; N = 2 C_out > 256 rules out S = 2
    assert run(h, x.data_ptr(), 16, [1, 1, 2, 24], x.data_ptr(), 256, [1, 1, 1, 20], y.data_ptr(),
               g.GEMM_BF16) == g.GEMM_ERR_UNSUPPORTED
    # a filter row longer than one input box reaches (more than 256 rows of S positions)
    assert run(h, x.data_ptr(), 16, [1, 1, 1, 258], x.data_ptr(), 16, [1, 1, 1, 258], y.data_ptr(),
               g.GEMM_BF16) == g.GEMM_ERR_UNSUPPORTED
    # a stack that does not divide in[3], or makes N = S C_out wider than 256
    lib.set_option(g.GEMM_OPT_CONV_STACK, 4)
    try:
        assert run(h, x.data_ptr(), 16, [2, 2, 4, 6], x.data_ptr(), 16, ks, y.data_ptr(),
                   g.GEMM_BF16) == g.GEMM_ERR_UNSUPPORTED
        assert run(h, x.data_ptr(), 16, ins, x.data_ptr(), 128, ks, y.data_ptr(),
                   g.GEMM_BF16) == g.GEMM_ERR_UNSUPPORTED
    finally:
        lib.set_option(g.GEMM_OPT_CONV_STACK, 0)
    assert g.gemm_set_option(h, g.GEMM_OPT_CONV_STACK, 3) == g.GEMM_ERR_INVALID_ARG
    torch.cuda.synchronize()
    assert lib.device_status() == g.GEMM_OK


def test_wait_runs_out_and_is_reported(lib):
    """The failure-detection hook: the epilogue's wait on a barrier nothing arrives on runs
    out; the kernel drains its copies and MMAs, frees TMEM and returns an error status."""
    import programming_tiled_gemm_gb300 as g
    x, w = int_operands(16, 32, (6, 5, 16, 16), (3, 2, 5, 5), seed=9)
    xd, wd = x.cuda(), w.cuda()
    lib.set_option(g.GEMM_OPT_WAIT_LIMIT_US, 20000)
    lib.set_option(g.GEMM_OPT_TEST_STALL, 1)
    try:
        lib.conv4d_cl(xd, wd)
        assert lib.device_status() == g.GEMM_ERR_DEVICE_TIMEOUT
    finally:
        lib.set_option(g.GEMM_OPT_TEST_STALL, 0)
        lib.set_option(g.GEMM_OPT_WAIT_LIMIT_US, 0)
    y = lib.conv4d_cl(xd, wd)
    torch.cuda.synchronize()
    assert lib.device_status() == g.GEMM_OK
    assert np.array_equal(y.cpu().double().numpy(), conv_ref(x, w))
