"""4-D convolution lowered to a GEMM (im2col on the GPU + the fp32 GEMM) against the oracle.

* im2col is a pure copy: compared bit for bit with the oracle's im2col.
* the convolution output: integer-valued inputs exactly, uniform[-1, 1] inputs within
  1e-5 * sqrt(K) with K = C_in * prod(kernel), against the oracle's direct nested-loop
  cross-correlation (and, at full size, against the oracle GEMM of the oracle im2col).
"""
import math

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


SHAPES = [
    (1, (1, 1, 1, 1), 1, (1, 1, 1, 1)),
    (2, (5, 5, 1, 1), 3, (3, 3, 1, 1)),
    (3, (6, 7, 5, 9), 4, (2, 3, 1, 4)),   # column count 5*5*5*6 = 750: not a multiple of 4
    (4, (8, 8, 8, 8), 32, (3, 3, 3, 3)),
    (16, (9, 9, 9, 9), 32, (5, 5, 5, 5)),
    (3, (6, 5, 7, 12), 4, (2, 1, 3, 5)),  # five-tap rows, p3 = 8: the tap-group im2col path
    (2, (4, 5, 6, 16), 3, (2, 3, 2, 5)),  # the same with p3 = 12, as in the 16^4 workload
]


def draw(cin, ins, cout, ks, seed, ints=False):
    g = si.generator(seed)
    if ints:
        x = si.ints((cin,) + ins, g).float()
        w = si.ints((cout, cin) + ks, g).float()
    else:
        x = si.uniform((cin,) + ins, g)
        w = si.uniform((cout, cin) + ks, g)
    return x, w


@pytest.mark.parametrize("cin,ins,cout,ks", SHAPES)
def test_im2col_is_bit_exact(lib, cin, ins, cout, ks):
    x, _ = draw(cin, ins, cout, ks, seed=1)
    col = lib.im2col4d(x.cuda(), list(ks))
    torch.cuda.synchronize()
    assert np.array_equal(col.cpu().numpy(), oracle.im2col4d(x.numpy(), ks))


@pytest.mark.parametrize("cin,ins,cout,ks", SHAPES)
def test_conv_integer_inputs_exact(lib, cin, ins, cout, ks):
    x, w = draw(cin, ins, cout, ks, seed=2, ints=True)
    y = lib.conv4d(x.cuda(), w.cuda())
    assert np.array_equal(y.cpu().double().numpy(), oracle.conv4d_direct(x.numpy(), w.numpy()))


@pytest.mark.parametrize("cin,ins,cout,ks", SHAPES)
def test_conv_uniform_within_tolerance(lib, cin, ins, cout, ks):
    x, w = draw(cin, ins, cout, ks, seed=3)
    y = lib.conv4d(x.cuda(), w.cuda())
    K = cin * int(np.prod(ks))
    err = np.abs(y.cpu().double().numpy() - oracle.conv4d_direct(x.numpy(), w.numpy())).max()
    assert err <= 1e-5 * math.sqrt(K)


def oracle_conv(x, w):
    """The oracle's convolution; large cases take its im2col + GEMM route, which the oracle
    pins show to be bit-identical to the direct nested loops and is much faster."""
    if x[0].numel() * w.numel() <= 2e8:
        return oracle.conv4d_direct(x.numpy(), w.numpy())
    col = oracle.im2col4d(x.numpy(), tuple(w.shape[2:]))
    y = oracle.gemm(np.ascontiguousarray(w.reshape(w.shape[0], -1).numpy()), col)
    outs = tuple(i - k + 1 for i, k in zip(x.shape[1:], w.shape[2:]))
    return y.reshape((w.shape[0],) + outs)


IMPLICIT_SHAPES = SHAPES + [
    (16, (16, 16, 16, 16), 32, (5, 5, 5, 5)),   # the workload's geometry (float4 gather path)
    (3, (9, 8, 10, 12), 7, (2, 3, 4, 5)),       # float4 path with C_out < 32
    (2, (7, 6, 9, 10), 40, (3, 2, 2, 5)),       # C_out > 32: two output-channel blocks
]


@pytest.mark.parametrize("split", [0, 1, 3])
@pytest.mark.parametrize("cin,ins,cout,ks", IMPLICIT_SHAPES)
def test_implicit_conv_integer_inputs_exact(lib, split, cin, ins, cout, ks):
    import programming_tiled_gemm_gb300 as g
    lib.set_option(g.GEMM_OPT_SPLIT_K, split)
    try:
        x, w = draw(cin, ins, cout, ks, seed=4, ints=True)
        y = lib.conv4d_implicit(x.cuda(), w.cuda())
        torch.cuda.synchronize()
        assert np.array_equal(y.cpu().double().numpy(), oracle_conv(x, w))
    finally:
        lib.set_option(g.GEMM_OPT_SPLIT_K, 0)


@pytest.mark.parametrize("cin,ins,cout,ks", IMPLICIT_SHAPES)
def test_implicit_conv_uniform_within_tolerance(lib, cin, ins, cout, ks):
    x, w = draw(cin, ins, cout, ks, seed=6)
    y = lib.conv4d_implicit(x.cuda(), w.cuda())
    K = cin * int(np.prod(ks))
    err = np.abs(y.cpu().double().numpy() - oracle_conv(x, w)).max()
    assert err <= 1e-5 * math.sqrt(K)


def test_implicit_conv_guard_band_and_padded_output(lib):
    x, w = draw(3, (6, 7, 5, 9), 5, (2, 3, 1, 4), seed=8, ints=True)
    npos = 5 * 5 * 5 * 6
    big = torch.full((5 + 2, npos + 9), -5.5, device="cuda")
    out = big[1:6, 2:2 + npos]
    lib.conv4d_implicit(x.cuda(), w.cuda(), out=out)
    torch.cuda.synchronize()
    host = big.cpu()
    mask = torch.ones_like(host, dtype=torch.bool)
    mask[1:6, 2:2 + npos] = False
    assert torch.all(host[mask] == -5.5)
    ref = oracle.conv4d_direct(x.numpy(), w.numpy()).reshape(5, -1)
    assert np.array_equal(host[1:6, 2:2 + npos].double().numpy(), ref)


def test_im2col_rejects_bad_geometry(lib):
    import programming_tiled_gemm_gb300 as g
    x = torch.zeros(2 * 4 * 4 * 4 * 4, device="cuda")
    col = torch.zeros(10, device="cuda")
    assert g.conv4d_im2col(lib.handle, x.data_ptr(), 2, [4, 4, 4, 4], [5, 1, 1, 1], col.data_ptr()) \
        == g.GEMM_ERR_INVALID_ARG
    assert g.conv4d_im2col(lib.handle, x.data_ptr(), 0, [4, 4, 4, 4], [1, 1, 1, 1], col.data_ptr()) \
        == g.GEMM_ERR_INVALID_ARG


@pytest.mark.slow
def test_full_config(lib):
    w_ = si.WORKLOADS["conv4d"]
    c = w_.conv
    x, w = si.workload_operands(w_)
    xd, wd = x.cuda(), w.cuda()
    col = lib.im2col4d(xd, list(c["ks"]))
    y = lib.matmul(wd.reshape(c["cout"], -1), col)
    torch.cuda.synchronize()
    col_ref = oracle.im2col4d(x.numpy(), c["ks"])
    assert np.array_equal(col.cpu().numpy(), col_ref)
    del col
    ref = oracle.gemm(w.reshape(c["cout"], -1).numpy(), col_ref)
    assert np.abs(y.cpu().double().numpy() - ref).max() <= 1e-5 * math.sqrt(w_.K)
    # the direct nested-loop route on one output channel (a thin, independent check)
    direct = oracle.conv4d_direct(x.numpy(), w[:1].numpy())
    assert np.abs(y[:1].cpu().double().numpy() - direct.reshape(1, -1)).max() <= 1e-5 * math.sqrt(w_.K)
    # the implicit GEMM on the same inputs, against the oracle GEMM of the oracle im2col
    yi = lib.conv4d_implicit(xd, wd).reshape(c["cout"], -1)
    torch.cuda.synchronize()
    assert np.abs(yi.cpu().double().numpy() - ref).max() <= 1e-5 * math.sqrt(w_.K)
