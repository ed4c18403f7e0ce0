"""Tensor-core 4-D convolution with channel-first 16-bit operands (conv4d_forward_tc)
against the oracle's direct convolution.

The entry point takes x [C_in][I0..I3] and w [C_out][C_in][R0..R3] in PyTorch's order,
re-lays both channel-last (channels padded with zeros to a multiple of 16) and runs the
channel-last tensor-core kernel, which stores y channel-first.  Checks:
  * integer-valued inputs in [-4, 4]: exact against the fp64 oracle;
  * uniform[-1, 1] inputs rounded to bf16: max |y - y_ref| <= 2e-5 * sqrt(K), K = C_in x taps;
  * bit-identical to conv4d_forward_cl on operands laid out channel-last (and zero-padded)
    by the test itself;
  * a strided y (ldy > positions) with sentinels in the gaps and around it: nothing written
    outside the output rows.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import seeded_inputs as si

pytestmark = pytest.mark.gpu
SENTINEL = -777.0


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__
    __graft_entry__.build()
    import programming_tiled_gemm_gb300 as g
    h = g.Gemm(0)
    yield h
    h.close()


def int_operands(cin, cout, ins, ks, seed, dtype=torch.bfloat16):
    g = si.generator(seed)
    x = si.ints((cin,) + tuple(ins), g).float()
    w = si.ints((cout, cin) + tuple(ks), g).float()
    return x.to(dtype), w.to(dtype)


def run_strided(lib, x, w, pad=8):
    """y in rows of npos + pad floats, sentinels in the gaps and on both sides."""
    dev = torch.device("cuda")
    cout = w.shape[0]
    outs = [i - k + 1 for i, k in zip(x.shape[1:], w.shape[2:])]
    npos = int(np.prod(outs))
    ldy = npos + pad
    big = torch.full((16 + cout * ldy + 16,), SENTINEL, device=dev)
    rows = big[16:16 + cout * ldy].view(cout, ldy)
    out = rows[:, :npos]
    lib.conv4d_tc(x.to(dev), w.to(dev), out=out)
    torch.cuda.synchronize()
    assert lib.device_status() == 0
    host = big.cpu()
    assert torch.all(host[:16] == SENTINEL) and torch.all(host[16 + cout * ldy:] == SENTINEL), "wrote outside y"
    hrows = host[16:16 + cout * ldy].view(cout, ldy)
    assert torch.all(hrows[:, npos:] == SENTINEL), "wrote into the gaps between rows"
    return hrows[:, :npos].double().numpy().reshape([cout] + outs)


SHAPES = [  # (C_in, C_out, input extents, kernel extents)
    (16, 32, (6, 5, 16, 16), (3, 2, 5, 5)),     # the workload's channel counts, two tiles per plane
    (3, 16, (4, 5, 6, 8), (2, 2, 3, 3)),        # three channels padded to 16
    (20, 48, (5, 6, 7, 9), (2, 3, 2, 4)),       # 20 channels padded to 32: two steps per tap
    (32, 32, (3, 3, 20, 30), (1, 2, 3, 3)),     # five tiles per plane
    (1, 16, (1, 1, 1, 1), (1, 1, 1, 1)),        # a single output position, one channel
]


@pytest.mark.parametrize("cin,cout,ins,ks", SHAPES)
def test_integer_inputs_are_exact(lib, cin, cout, ins, ks):
    x, w = int_operands(cin, cout, ins, ks, seed=cin + 3 * cout + sum(ins))
    y = run_strided(lib, x, w)
    ref = oracle.conv4d_direct(x.float().numpy(), w.float().numpy())
    assert np.array_equal(y, ref)


def test_fp16_integer_inputs_are_exact(lib):
    x, w = int_operands(16, 32, (4, 4, 9, 9), (2, 2, 3, 3), seed=5, dtype=torch.float16)
    y = run_strided(lib, x, w, pad=0)
    assert np.array_equal(y, oracle.conv4d_direct(x.float().numpy(), w.float().numpy()))


def test_workload_shape_is_exact(lib):
    x, w = int_operands(16, 32, (16, 16, 16, 16), (5, 5, 5, 5), seed=11)
    y = lib.conv4d_tc(x.cuda(), w.cuda())
    torch.cuda.synchronize()
    assert lib.device_status() == 0
    assert np.array_equal(y.cpu().double().numpy(), oracle.conv4d_direct(x.float().numpy(), w.float().numpy()))


@pytest.mark.parametrize("cin,cout,ins,ks", SHAPES[:3])
def test_uniform_bf16_within_tolerance(lib, cin, cout, ins, ks):
    g = si.generator(cin + cout)
    x = si.uniform((cin,) + tuple(ins), g).to(torch.bfloat16)
    w = si.uniform((cout, cin) + tuple(ks), g).to(torch.bfloat16)
    y = run_strided(lib, x, w)
    ref = oracle.conv4d_direct(x.float().numpy(), w.float().numpy())
    K = cin * int(np.prod(ks))
    assert np.abs(y - ref).max() <= 2e-5 * math.sqrt(K)


@pytest.mark.parametrize("cin", [16, 20])
def test_bit_identical_to_the_channel_last_entry_point(lib, cin):
    g = si.generator(cin)
    x = si.uniform((cin, 5, 6, 7, 12), g).to(torch.bfloat16)
    w = si.uniform((32, cin, 2, 3, 2, 5), g).to(torch.bfloat16)
    cp = (cin + 15) // 16 * 16
    xp = torch.zeros((cp,) + tuple(x.shape[1:]), dtype=x.dtype)
    xp[:cin] = x
    wp = torch.zeros((32, cp) + tuple(w.shape[2:]), dtype=w.dtype)
    wp[:, :cin] = w
    x_cl = xp.permute(1, 2, 3, 4, 0).contiguous()
    w_cl = wp.permute(0, 2, 3, 4, 5, 1).contiguous()
    y_cf = lib.conv4d_tc(x.cuda(), w.cuda())
    y_cl = lib.conv4d_cl(x_cl.cuda(), w_cl.cuda())
    torch.cuda.synchronize()
    assert lib.device_status() == 0
    assert torch.equal(y_cf, y_cl.permute(4, 0, 1, 2, 3))


def test_argument_errors_are_reported(lib):
    import programming_tiled_gemm_gb300 as g
    dev = torch.device("cuda")
    x = torch.zeros((16, 4, 4, 4, 4), dtype=torch.bfloat16, device=dev)
    w = torch.zeros((32, 16, 2, 2, 2, 2), dtype=torch.bfloat16, device=dev)
    y = torch.zeros((32, 81), device=dev)
    ins, ks = [4, 4, 4, 4], [2, 2, 2, 2]

    def call(xp, wp, cin, cout, yp, ldy, dt=g.GEMM_BF16, ins=ins, ks=ks):
        return g.conv4d_forward_tc(lib.handle, xp, cin, ins, wp, cout, ks, yp, ldy, dt,
                                   torch.cuda.current_stream().cuda_stream)

    assert call(x.data_ptr(), w.data_ptr(), 16, 32, y.data_ptr(), 81) == g.GEMM_OK
    torch.cuda.synchronize()
    assert call(x.data_ptr(), w.data_ptr(), 16, 32, y.data_ptr(), 80) == g.GEMM_ERR_INVALID_ARG  # ldy < positions
    assert call(x.data_ptr(), w.data_ptr(), 16, 32, y.data_ptr(), 81, dt=g.GEMM_F32) == g.GEMM_ERR_INVALID_ARG
    assert call(x.data_ptr() + 1, w.data_ptr(), 16, 32, y.data_ptr(), 81) == g.GEMM_ERR_ALIGNMENT
    assert call(x.data_ptr(), w.data_ptr(), 16, 32, y.data_ptr() + 2, 81) == g.GEMM_ERR_ALIGNMENT
    assert call(x.data_ptr(), w.data_ptr(), 16, 24, y.data_ptr(), 81) == g.GEMM_ERR_UNSUPPORTED  # C_out % 16
    assert call(x.data_ptr(), w.data_ptr(), 16, 32, y.data_ptr(), 81, ks=[5, 2, 2, 2]) == g.GEMM_ERR_INVALID_ARG
    assert call(0, w.data_ptr(), 16, 32, y.data_ptr(), 81) == g.GEMM_ERR_INVALID_ARG
    assert lib.device_status() == 0
