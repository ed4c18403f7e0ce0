"""Pins of the CPU oracle to facts that do not come from the oracle itself.

Each check is a closed form, an exact special case, a library routine (numpy / scipy)
or a worked example from the pages.  Together they are chosen so that a plausible slip
in the oracle -- a dropped term, a transposed operand, a wrong stride or index, a
reversed summation -- fails at least one of them; ``test_oracle_mutants.py`` plants
such slips in a copy of the oracle and checks exactly that.

GEMM definition: "Learning to develop for GPU with GEMM as the example", section
"Matrix product".  Convolution and im2col: "Three X: large convolutions in PyTorch for
training", sections "Why we need high-dimensional convolution" and "CuBLAS".
"""
import os

import numpy as np
import pytest

import oracle

RNG = np.random.default_rng(12345)
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def f32(a):
    return np.ascontiguousarray(a, dtype=np.float32)


# ----------------------------------------------------------------------- GEMM pins

@pytest.mark.parametrize("M,K,N", [(1, 1, 1), (4, 4, 4), (37, 37, 53), (64, 64, 3)])
def test_left_identity_gives_B(M, K, N):
    A = f32(np.eye(M, K))
    B = f32(RNG.uniform(-1, 1, (K, N)))
    C = oracle.gemm(A, B)
    assert np.array_equal(C, B.astype(np.float64))


@pytest.mark.parametrize("M,K,N", [(4, 4, 4), (29, 41, 41), (3, 64, 64)])
def test_right_identity_gives_A(M, K, N):
    A = f32(RNG.uniform(-1, 1, (M, K)))
    B = f32(np.eye(K, N))
    C = oracle.gemm(A, B)
    assert np.array_equal(C, A.astype(np.float64))


def test_permutation_permutes_rows_of_B():
    K, N = 50, 23
    perm = RNG.permutation(K)
    P = np.zeros((K, K), dtype=np.float32)
    P[np.arange(K), perm] = 1.0
    B = f32(RNG.uniform(-1, 1, (K, N)))
    C = oracle.gemm(P, B)
    assert np.array_equal(C, B[perm].astype(np.float64))


def test_permutation_on_the_right_permutes_columns_of_A():
    M, K = 19, 31
    perm = RNG.permutation(K)
    P = np.zeros((K, K), dtype=np.float32)
    P[perm, np.arange(K)] = 1.0          # (A P)[:, j] = A[:, perm[j]]
    A = f32(RNG.uniform(-1, 1, (M, K)))
    C = oracle.gemm(A, P)
    assert np.array_equal(C, A[:, perm].astype(np.float64))


@pytest.mark.parametrize("M,K,N", [(1, 1, 1), (7, 300, 5), (16, 4097, 9)])
def test_all_ones_gives_K(M, K, N):
    C = oracle.gemm(f32(np.ones((M, K))), f32(np.ones((K, N))))
    assert np.array_equal(C, np.full((M, N), float(K)))


def test_zero_inner_dimension_gives_zeros():
    C = oracle.gemm(np.zeros((5, 0), np.float32), np.zeros((0, 7), np.float32))
    assert C.shape == (5, 7) and np.array_equal(C, np.zeros((5, 7)))


def test_empty_outputs():
    assert oracle.gemm(np.zeros((0, 4), np.float32), np.zeros((4, 3), np.float32)).shape == (0, 3)
    assert oracle.gemm(np.zeros((2, 4), np.float32), np.zeros((4, 0), np.float32)).shape == (2, 0)


@pytest.mark.parametrize("K", [1, 3, 64, 1000])
def test_rank_one(K):
    # A = u 1^T, B = 1 w^T  =>  C[i][j] = K u_i w_j.  Dyadic values keep every sum exact.
    M, N = 13, 11
    u = RNG.integers(-32, 33, M) / 8.0
    w = RNG.integers(-32, 33, N) / 8.0
    A = f32(np.repeat(u[:, None], K, axis=1))
    B = f32(np.repeat(w[None, :], K, axis=0))
    C = oracle.gemm(A, B)
    assert np.array_equal(C, K * np.outer(u, w))


def test_outer_product_when_K_is_one():
    u = f32(RNG.uniform(-1, 1, (9, 1)))
    w = f32(RNG.uniform(-1, 1, (1, 6)))
    C = oracle.gemm(u, w)
    assert np.array_equal(C, u.astype(np.float64) @ w.astype(np.float64))


def test_triangular_closed_forms_fix_operand_orientation():
    # U upper-triangular ones (U[i][k] = 1 for k >= i) times ones: C[i][j] = K - i.
    # A transposed A would give i + 1 instead.
    K, N = 17, 5
    U = f32(np.triu(np.ones((K, K))))
    C = oracle.gemm(U, f32(np.ones((K, N))))
    assert np.array_equal(C, np.repeat((K - np.arange(K, dtype=np.float64))[:, None], N, axis=1))
    # ones times L (L[k][j] = 1 for k >= j): C[i][j] = K - j; a transposed B gives j + 1.
    L = f32(np.tril(np.ones((K, K))))
    C = oracle.gemm(f32(np.ones((3, K))), L)
    assert np.array_equal(C, np.repeat((K - np.arange(K, dtype=np.float64))[None, :], 3, axis=0))


@pytest.mark.parametrize("K", [1, 2, 5, 4096])
def test_arithmetic_series_counts_every_term(K):
    # A[i][k] = k + 1, B = ones  =>  C = K (K + 1) / 2; dropping any term changes it.
    A = f32(np.tile(np.arange(1, K + 1), (3, 1)))
    C = oracle.gemm(A, f32(np.ones((K, 4))))
    assert np.array_equal(C, np.full((3, 4), K * (K + 1) / 2.0))


def test_brute_force_4x4_small_integers_match_numpy_exactly():
    # All 4x4 products of small integers are exact in fp64, so any summation order
    # agrees bit for bit with numpy's matmul.
    for _ in range(200):
        A = RNG.integers(-4, 5, (4, 4)).astype(np.float32)
        B = RNG.integers(-4, 5, (4, 4)).astype(np.float32)
        assert np.array_equal(oracle.gemm(A, B), A.astype(np.float64) @ B.astype(np.float64))


@pytest.mark.parametrize("M,K,N", [(33, 65, 17), (128, 256, 96), (5, 1000, 300)])
def test_random_floats_match_numpy_float64(M, K, N):
    A = f32(RNG.uniform(-1, 1, (M, K)))
    B = f32(RNG.uniform(-1, 1, (K, N)))
    C = oracle.gemm(A, B)
    ref = A.astype(np.float64) @ B.astype(np.float64)
    scale = np.abs(A).astype(np.float64) @ np.abs(B).astype(np.float64)
    assert np.all(np.abs(C - ref) <= 1e-13 * K * scale + 1e-300)


def test_leading_dimensions_skip_padding():
    M, K, N = 9, 14, 11
    A_full = f32(np.full((M, K + 5), np.nan))
    B_full = f32(np.full((K, N + 3), np.nan))
    A_full[:, :K] = RNG.uniform(-1, 1, (M, K))
    B_full[:, :N] = RNG.uniform(-1, 1, (K, N))
    C = oracle.gemm(A_full[:, :K], B_full[:, :N])
    assert np.all(np.isfinite(C))
    assert np.array_equal(C, oracle.gemm(f32(A_full[:, :K]), f32(B_full[:, :N])))


def test_sum_runs_over_k_ascending():
    # fp64 sum of [2^60, -2^60, 1] is 1 in ascending order and 0 in descending order.
    A = f32([[2.0 ** 60, -(2.0 ** 60), 1.0]])
    B = f32(np.ones((3, 1)))
    assert oracle.gemm(A, B)[0, 0] == 1.0
    A = f32([[1.0, 2.0 ** 60, -(2.0 ** 60)]])
    assert oracle.gemm(A, B)[0, 0] == 0.0


def test_thread_count_does_not_change_results():
    A = f32(RNG.uniform(-1, 1, (61, 333)))
    B = f32(RNG.uniform(-1, 1, (333, 47)))
    C1 = oracle.gemm(A, B, nthreads=1)
    for t in (2, 3, 7, 64):
        assert np.array_equal(C1, oracle.gemm(A, B, nthreads=t))


def test_entries_equal_full_product_bit_for_bit():
    M, K, N = 40, 123, 57
    A = f32(RNG.uniform(-1, 1, (M, K)))
    B = f32(RNG.uniform(-1, 1, (K, N)))
    C = oracle.gemm(A, B)
    ri = RNG.integers(0, M, 500)
    rj = RNG.integers(0, N, 500)
    e1 = oracle.gemm_entries(A, B, ri, rj)
    e2 = oracle.gemm_entries(A, None, ri, rj, B_transposed_copy=f32(B.T))
    assert np.array_equal(e1, C[ri, rj])
    assert np.array_equal(e2, C[ri, rj])


def test_rejects_mismatched_shapes():
    with pytest.raises(ValueError):
        oracle.gemm(np.zeros((3, 4), np.float32), np.zeros((5, 2), np.float32))
    with pytest.raises(TypeError):
        oracle.gemm(np.zeros((3, 4)), np.zeros((4, 2)))


# ----------------------------------------------------------- generalised GEMM pins

def test_general_with_alpha_one_beta_zero_is_the_product():
    A = f32(RNG.uniform(-1, 1, (13, 21)))
    B = f32(RNG.uniform(-1, 1, (21, 8)))
    assert np.array_equal(oracle.gemm_general(1.0, A, B), oracle.gemm(A, B))


def test_general_beta_zero_never_reads_C():
    A = f32(np.ones((3, 4)))
    B = f32(np.ones((4, 5)))
    C = np.full((3, 5), np.nan)
    assert np.array_equal(oracle.gemm_general(2.0, A, B, 0.0, C), np.full((3, 5), 8.0))


def test_general_zero_product_scales_the_accumulator():
    # A = 0: D = beta * C exactly
    C = RNG.uniform(-1, 1, (6, 7))
    D = oracle.gemm_general(3.0, f32(np.zeros((6, 5))), f32(RNG.uniform(-1, 1, (5, 7))), -0.25, C)
    assert np.array_equal(D, -0.25 * C)


def test_general_closed_form_with_dyadic_weights():
    # A = all ones (M x K), B = all ones (K x N), C = i - j: D = alpha*K + beta*(i - j)
    M, K, N = 9, 12, 7
    alpha, beta = 0.5, -2.0
    C = np.subtract.outer(np.arange(M), np.arange(N)).astype(np.float64)
    D = oracle.gemm_general(alpha, f32(np.ones((M, K))), f32(np.ones((K, N))), beta, C)
    assert np.array_equal(D, alpha * K + beta * C)


def test_general_matches_numpy_float64():
    A = f32(RNG.uniform(-1, 1, (17, 33)))
    B = f32(RNG.uniform(-1, 1, (33, 11)))
    C = RNG.uniform(-1, 1, (17, 11))
    D = oracle.gemm_general(1.75, A, B, 0.5, C)
    ref = 1.75 * (A.astype(np.float64) @ B.astype(np.float64)) + 0.5 * C
    assert np.allclose(D, ref, rtol=0, atol=1e-12)


# ------------------------------------------------------------------ convolution pins

def conv_case(cin, ins, cout, ks, seed=7):
    g = np.random.default_rng(seed)
    x = f32(g.uniform(-1, 1, (cin,) + tuple(ins)))
    w = f32(g.uniform(-1, 1, (cout, cin) + tuple(ks)))
    return x, w


def test_conv_all_ones_counts_taps():
    cin, ins, cout, ks = 3, (7, 6, 5, 8), 2, (2, 3, 1, 4)
    y = oracle.conv4d_direct(f32(np.ones((cin,) + ins)), f32(np.ones((cout, cin) + ks)))
    assert y.shape == (cout, 6, 4, 5, 5)
    assert np.array_equal(y, np.full(y.shape, float(cin * 2 * 3 * 1 * 4)))


def test_conv_all_ones_full_config_gives_10000():
    # The 4-D workload: 16 channels, 16^4 input, 5^4 kernel -> every output is 16 * 625.
    # A thin output-channel slice keeps the CPU time small; the sum per output is the same.
    y = oracle.conv4d_direct(f32(np.ones((16, 16, 16, 16, 16))), f32(np.ones((1, 16, 5, 5, 5, 5))))
    assert y.shape == (1, 12, 12, 12, 12)
    assert np.array_equal(y, np.full(y.shape, 10000.0))


def test_conv_delta_filter_is_a_shifted_crop():
    cin, ins, cout, ks = 4, (6, 7, 5, 6), 3, (3, 2, 2, 3)
    x, _ = conv_case(cin, ins, cout, ks)
    P = tuple(i - k + 1 for i, k in zip(ins, ks))
    for (o, c, a, b, d, e) in [(0, 0, 0, 0, 0, 0), (1, 2, 2, 1, 0, 2), (2, 3, 1, 0, 1, 1)]:
        w = np.zeros((cout, cin) + ks, np.float32)
        w[o, c, a, b, d, e] = 1.0
        y = oracle.conv4d_direct(x, w)
        expect = np.zeros((cout,) + P)
        expect[o] = x[c, a:a + P[0], b:b + P[1], d:d + P[2], e:e + P[3]]
        assert np.array_equal(y, expect)


def test_conv_matches_scipy_correlate():
    scipy_signal = pytest.importorskip("scipy.signal")
    cin, ins, cout, ks = 3, (6, 5, 7, 6), 2, (3, 2, 4, 2)
    x, w = conv_case(cin, ins, cout, ks)
    y = oracle.conv4d_direct(x, w)
    for o in range(cout):
        ref = sum(scipy_signal.correlate(x[c].astype(np.float64), w[o, c].astype(np.float64),
                                         mode="valid", method="direct") for c in range(cin))
        assert np.allclose(y[o], ref, rtol=0, atol=1e-12)


def test_im2col_matches_numpy_sliding_windows():
    cin, ins, ks = 3, (6, 5, 7, 4), (2, 3, 4, 2)
    x, _ = conv_case(cin, ins, 1, ks)
    col = oracle.im2col4d(x, ks)
    win = np.lib.stride_tricks.sliding_window_view(x, ks, axis=(1, 2, 3, 4))
    # win: [cin, P0, P1, P2, P3, R0, R1, R2, R3] -> rows (c, r...), columns (p...)
    P = win.shape[1:5]
    ref = win.transpose(0, 5, 6, 7, 8, 1, 2, 3, 4).reshape(cin * int(np.prod(ks)), int(np.prod(P)))
    assert np.array_equal(col, ref)


def test_two_routes_to_the_convolution_agree_exactly():
    # Direct nested loops and im2col followed by the oracle GEMM sum the same products
    # in the same (c, r0, r1, r2, r3) order, so they agree bit for bit.
    cin, ins, cout, ks = 4, (7, 6, 6, 5), 5, (3, 3, 2, 2)
    x, w = conv_case(cin, ins, cout, ks)
    y = oracle.conv4d_direct(x, w)
    col = oracle.im2col4d(x, ks)
    y2 = oracle.gemm(f32(w.reshape(cout, -1)), col)
    assert np.array_equal(y.reshape(cout, -1), y2)


def test_im2col_worked_example_from_the_pages():
    """The 3x3 image / 3x3 filter / nine-output example of the convolution page.

    Fixture: tests/golden/im2col_toy_3x3.txt.  The page numbers the GEMM outputs
    o1..o9 and maps o7 to the 2-D output position [2, 0] of the 3x3 result: the
    columns are ordered row-major over output positions.  A 3x3 output from a 3x3
    image and a 3x3 filter needs a one-pixel zero border, so the image is padded to
    5x5 here and the two trailing dimensions are given extent 1.
    """
    fixture = {}
    with open(os.path.join(GOLDEN, "im2col_toy_3x3.txt")) as fh:
        for line in fh:
            line = line.split("#", 1)[0].strip()
            if line:
                key, val = line.split("=")
                fixture[key.strip()] = [int(v) for v in val.split(",")]
    img = np.arange(1, 10, dtype=np.float32).reshape(3, 3)
    padded = np.zeros((5, 5), np.float32)
    padded[1:4, 1:4] = img
    x = padded.reshape(1, 5, 5, 1, 1)
    col = oracle.im2col4d(x, (3, 3, 1, 1))
    assert col.shape == (9, fixture["n_outputs"][0])
    n = fixture["gemm_output_index_1based"][0] - 1
    p, q = fixture["output_position"]
    assert divmod(n, 3) == (p, q)
    assert np.array_equal(col[:, n], padded[p:p + 3, q:q + 3].reshape(-1))
