"""bf16 / fp16 tensor-core path (tcgen05) on the GPU against the CPU oracle, via the C ABI.

Tolerances (max |C - C_ref|):
  * integer-valued inputs in [-4, 4] (exact in bf16 and fp16; every partial sum is an
    integer below 2^24): exact;
  * normal(0, 1) inputs rounded to bf16, compared with the oracle on the same rounded
    values: 2e-5 * sqrt(K).
At 8192^3 the oracle cannot do all 6.7e7 entries one by one in seconds, so the full-size
test compares 128 full rows, 128 full columns and 65536 random entries exactly against
the oracle, and checks the whole matrix with Freivalds' test: for random x,
|C x - A (B x)| per row is bounded by sqrt(N) times the per-entry tolerance (the
per-entry errors are independent across columns) plus the fp64 rounding of A (B x).
"""
import math

import numpy as np
import pytest
import torch

import oracle
import seeded_inputs as si

pytestmark = pytest.mark.gpu
SENTINEL = -777.25


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__
    __graft_entry__.build()
    import programming_tiled_gemm_gb300 as g
    h = g.Gemm(0)
    yield h
    h.close()


@pytest.fixture(autouse=True)
def _reset(lib):
    import programming_tiled_gemm_gb300 as g
    yield
    lib.set_option(g.GEMM_OPT_TC_CHUNK, 0)
    lib.set_option(g.GEMM_OPT_TC_PAIR, 0)


def padded(t, ld, dev):
    buf = torch.zeros((t.shape[0], ld), dtype=t.dtype, device=dev)
    buf[:, : t.shape[1]] = t.to(dev)
    return buf[:, : t.shape[1]]


def run_guarded(lib, A, B, guard=3, pad_c=5):
    dev = torch.device("cuda")
    M, K = A.shape
    N = B.shape[1]
    Ad = padded(A, (K + 7) // 8 * 8 + 8, dev)
    Bd = padded(B, (N + 7) // 8 * 8 + 16, dev)
    Cbig = torch.full((M + 2 * guard, N + pad_c + 2 * guard), SENTINEL, device=dev)
    Cv = Cbig[guard:guard + M, guard:guard + N]
    lib.matmul(Ad, Bd, out=Cv)
    torch.cuda.synchronize()
    assert lib.device_status() == 0
    host = Cbig.cpu()
    mask = torch.ones_like(host, dtype=torch.bool)
    mask[guard:guard + M, guard:guard + N] = False
    assert torch.all(host[mask] == SENTINEL), "kernel wrote outside C"
    return host[guard:guard + M, guard:guard + N].double().numpy()


SHAPES = [(1, 1, 1), (128, 256, 64), (128, 256, 16), (129, 257, 65), (200, 300, 100), (64, 1000, 8),
          (256, 512, 1024), (1000, 24, 520), (1024, 2048, 512), (2048, 4096, 384)]


@pytest.mark.parametrize("pair", [1, 2])
@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("M,N,K", SHAPES)
def test_integer_inputs_exact(lib, pair, dtype, M, N, K):
    """pair 1: one CTA per 128 x 256 tile; pair 2: CTA pairs (cta_group::2) per 256 x 256 tile."""
    import programming_tiled_gemm_gb300 as g
    lib.set_option(g.GEMM_OPT_TC_PAIR, pair)
    A, B = si.integer_copy(M, N, K, seed=M + 3 * N + 7 * K, dtype=dtype)
    got = run_guarded(lib, A, B)
    assert np.array_equal(got, oracle.gemm(A.float().numpy(), B.float().numpy()))


@pytest.mark.parametrize("pair", [1, 2])
@pytest.mark.parametrize("chunk", [1, 3, 16, 4096])
def test_accumulation_chunks_exact(lib, pair, chunk):
    import programming_tiled_gemm_gb300 as g
    lib.set_option(g.GEMM_OPT_TC_CHUNK, chunk)
    lib.set_option(g.GEMM_OPT_TC_PAIR, pair)
    A, B = si.integer_copy(300, 520, 1100, seed=chunk)
    got = run_guarded(lib, A, B)
    assert np.array_equal(got, oracle.gemm(A.float().numpy(), B.float().numpy()))


@pytest.mark.parametrize("pair", [1, 2])
@pytest.mark.parametrize("M,N,K", [(256, 512, 1024), (384, 256, 4096), (200, 300, 8192)])
def test_normal_bf16_within_tolerance(lib, pair, M, N, K):
    import programming_tiled_gemm_gb300 as g
    lib.set_option(g.GEMM_OPT_TC_PAIR, pair)
    A, B = si.gemm_operands(M, N, K, seed=21, dist="normal", dtype="bf16")
    got = run_guarded(lib, A, B)
    err = np.abs(got - oracle.gemm(A.float().numpy(), B.float().numpy())).max()
    assert err <= 2e-5 * math.sqrt(K), err


def test_tile_option_accepts_single_and_pair_only(lib):
    """GEMM_OPT_TC_PAIR takes 0 (choose), 1 (single CTA) or 2 (CTA pair); nothing else."""
    import programming_tiled_gemm_gb300 as g
    for bad in (3, 4, -1):
        with pytest.raises(g.GemmError) as e:
            lib.set_option(g.GEMM_OPT_TC_PAIR, bad)
        assert e.value.status == g.GEMM_ERR_INVALID_ARG


@pytest.mark.parametrize("M,N,K", [(1024, 2048, 2048), (4096, 4096, 4096)])
def test_results_are_deterministic(lib, M, N, K):
    """Every kernel family repeats its result bit for bit.  The families agree within the
    tolerance: the CTA-pair kernel may cut a last wave's tiles along K, which regroups the
    chunk sums of those tiles."""
    import programming_tiled_gemm_gb300 as g
    A, B = si.gemm_operands(M, N, K, seed=5, dist="normal", dtype="bf16")
    Ad, Bd = A.cuda(), B.cuda()
    ref = None
    for pair in (0, 1, 2):
        lib.set_option(g.GEMM_OPT_TC_PAIR, pair)
        c1 = lib.matmul(Ad, Bd).clone()
        for _ in range(2):
            assert torch.equal(c1, lib.matmul(Ad, Bd)), pair
        if ref is None:
            ref = c1
        assert (c1 - ref).abs().max().item() <= 2 * 2e-5 * math.sqrt(K)


LAST_WAVE_SHAPES = [  # CTA-pair tiles (256 x 256) whose last wave is cut along K (76 pairs)
    (4096, 4096, 4096),   # 256 tiles: 228 whole, the last 28 in 2 slices
    (3072, 2048, 6144),   # 96 tiles: the last 20 in 3 slices of 32 k-blocks
    (1024, 1024, 8192),   # 16 tiles, all in 4 slices
    (1000, 1000, 8400),   # ragged M, N and K: slices of 32 and 33 k-blocks, a partial k-block
    (1024, 2048, 4096),   # 32 tiles, all in 2 slices
]


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("M,N,K", LAST_WAVE_SHAPES)
def test_last_wave_split_integer_inputs_exact(lib, dtype, M, N, K):
    """The CTA-pair kernel's last-wave tiles run as K slices; the warp finishing a tile
    part's last slice adds the slices' partials in slice order and stores C."""
    A, B = si.integer_copy(M, N, K, seed=M + 7 * N + K, dtype=dtype)
    got = run_guarded(lib, A, B)
    assert np.array_equal(got, oracle.gemm(A.float().numpy(), B.float().numpy()))


@pytest.mark.parametrize("M,N,K", [(4096, 4096, 4096), (1024, 2048, 4096), (1500, 1504, 4200)])
def test_last_wave_two_slices_into_aligned_C_exact(lib, M, N, K):
    """Two K slices and a plain fp32 C with 16-byte aligned rows: the part's first slice
    to finish stores C (TMA), the second adds itself to C (TMA reduce-add).  The rows
    around C and the padding past column N stay untouched."""
    dev = torch.device("cuda")
    A, B = si.integer_copy(M, N, K, seed=M + N + 3 * K, dtype="bf16")
    ldc = (N + 4 + 3) // 4 * 4
    big = torch.full((M + 2, ldc), SENTINEL, device=dev)
    C = big[1:M + 1, :N]
    lib.matmul(A.to(dev), B.to(dev), out=C)
    torch.cuda.synchronize()
    assert lib.device_status() == 0
    host = big.cpu()
    assert torch.all(host[0] == SENTINEL) and torch.all(host[M + 1] == SENTINEL)
    assert torch.all(host[1:M + 1, N:] == SENTINEL)
    assert np.array_equal(host[1:M + 1, :N].double().numpy(), oracle.gemm(A.float().numpy(), B.float().numpy()))


def test_last_wave_split_within_tolerance(lib):
    A, B = si.gemm_operands(4096, 4096, 4096, seed=41, dist="normal", dtype="bf16")
    got = run_guarded(lib, A, B)
    err = np.abs(got - oracle.gemm(A.float().numpy(), B.float().numpy())).max()
    assert err <= 2e-5 * math.sqrt(4096), err


SPLIT_SHAPES = [  # M <= 128 with 128 x 256 tiles filling under half the SMs: K is split
    (128, 2048, 4096),   # 8 tiles, up to 16 slices of 4 k-blocks (clusters above 8 CTAs)
    (100, 1000, 4296),   # ragged M and K: slices of 4 and 5 k-blocks, a partial k-block
    (1, 256, 1024),      # one row, one tile, 4 slices
    (37, 4104, 8192),    # 17 tiles, a partial last tile column
    (50, 1001, 2000),    # odd N: C stored element by element
    (128, 8, 2048),      # one narrow tile, 8 slices
]


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("M,N,K", SPLIT_SHAPES)
def test_split_k_integer_inputs_exact(lib, dtype, M, N, K):
    """The default tile choice splits K for small M: the CTAs of a cluster each take one K
    slice of a tile and add the fp32 partial tiles, read from each other's shared memory,
    in slice order."""
    A, B = si.integer_copy(M, N, K, seed=M + 5 * N + K, dtype=dtype)
    got = run_guarded(lib, A, B)
    assert np.array_equal(got, oracle.gemm(A.float().numpy(), B.float().numpy()))


def test_split_k_within_tolerance_deterministic_and_close_to_unsplit(lib):
    import programming_tiled_gemm_gb300 as g
    M, N, K = 128, 2048, 8192
    A, B = si.gemm_operands(M, N, K, seed=31, dist="normal", dtype="bf16")
    got = run_guarded(lib, A, B)
    ref = oracle.gemm(A.float().numpy(), B.float().numpy())
    tol = 2e-5 * math.sqrt(K)
    assert np.abs(got - ref).max() <= tol
    Ad, Bd = A.cuda(), B.cuda()
    launches = lib.launch_count()
    c1 = lib.matmul(Ad, Bd).clone()
    assert lib.launch_count() - launches == 1  # the slices are added inside the one kernel
    for _ in range(3):
        assert torch.equal(c1, lib.matmul(Ad, Bd))
    lib.set_option(g.GEMM_OPT_TC_PAIR, 1)  # explicit single-CTA tiles: no split
    c2 = lib.matmul(Ad, Bd)
    assert (c1 - c2).abs().max().item() <= 2 * tol


def test_split_k_general_epilogue(lib):
    """alpha / beta and a bf16 C through the split path, alternating shapes."""
    dev = torch.device("cuda")
    for M, N, K in [(96, 1024, 4096), (128, 2048, 2048), (96, 1024, 4096)]:
        A, B = si.integer_copy(M, N, K, seed=M + N + K, dtype="bf16")
        C0 = si.ints((M, N), si.generator(3)).to(torch.bfloat16)  # integer-valued, exact in bf16
        C = C0.to(dev)
        lib.matmul(A.to(dev), B.to(dev), out=C, alpha=0.5, beta=-2.0)
        torch.cuda.synchronize()
        assert lib.device_status() == 0
        # the exact result (integers and halves below 2^24) rounded once to bf16
        ref = oracle.gemm_general(0.5, A.float().numpy(), B.float().numpy(), -2.0, C0.double().numpy())
        want = torch.from_numpy(ref).float().to(torch.bfloat16)
        assert torch.equal(C.cpu(), want)


def test_alignment_rules(lib):
    import programming_tiled_gemm_gb300 as g
    dev = torch.device("cuda")
    buf = torch.zeros(64 * 72 + 8, dtype=torch.bfloat16, device=dev)
    C = torch.empty((64, 64), device=dev)
    B = torch.zeros((72, 64), dtype=torch.bfloat16, device=dev)
    h = lib.handle
    # A base 2 bytes off a 16-byte boundary
    assert g.gemm_run(h, 64, 64, 72, buf.data_ptr() + 2, 72, B.data_ptr(), 64, C.data_ptr(), 64,
                      g.GEMM_BF16) == g.GEMM_ERR_ALIGNMENT
    # lda not a multiple of 8 elements
    assert g.gemm_run(h, 64, 64, 70, buf.data_ptr(), 70, B.data_ptr(), 64, C.data_ptr(), 64,
                      g.GEMM_BF16) == g.GEMM_ERR_ALIGNMENT
    # the aligned call succeeds
    assert g.gemm_run(h, 64, 64, 72, buf.data_ptr(), 72, B.data_ptr(), 64, C.data_ptr(), 64,
                      g.GEMM_BF16) == g.GEMM_OK
    torch.cuda.synchronize()


def test_zero_K_and_empty(lib):
    dev = torch.device("cuda")
    C = torch.full((4, 8), 5.0, device=dev)
    lib.matmul(torch.empty((4, 0), dtype=torch.bfloat16, device=dev),
               torch.empty((0, 8), dtype=torch.bfloat16, device=dev), out=C)
    assert torch.all(C == 0)


def test_host_buffer_entry_point_bf16(lib):
    A, B = si.integer_copy(130, 250, 190, seed=8, dtype="bf16")
    C = lib.matmul_host(A, B)
    assert np.array_equal(C.double().numpy(), oracle.gemm(A.float().numpy(), B.float().numpy()))


@pytest.mark.slow
def test_config_8192_sampled_and_freivalds(lib):
    w = si.WORKLOADS["bf16_8192"]
    A, B = si.workload_operands(w)
    C = lib.matmul(A.cuda(), B.cuda())
    torch.cuda.synchronize()
    assert lib.device_status() == 0
    tol = 2e-5 * math.sqrt(w.K)
    Af, Bf = A.float().numpy(), B.float().numpy()
    Cd = C.cpu().double().numpy()
    rows, cols, ri, rj = si.sample_indices(w.M, w.N, w.seed)
    rows, cols, ri, rj = rows.numpy(), cols.numpy(), ri.numpy(), rj.numpy()
    err_rows = np.abs(Cd[rows] - oracle.gemm(Af[rows], Bf)).max()
    err_cols = np.abs(Cd[:, cols] - oracle.gemm(Af, np.ascontiguousarray(Bf[:, cols]))).max()
    err_rand = np.abs(Cd[ri, rj] - oracle.gemm_entries(Af, None, ri, rj,
                                                       B_transposed_copy=np.ascontiguousarray(Bf.T))).max()
    assert max(err_rows, err_cols, err_rand) <= tol, (err_rows, err_cols, err_rand)
    # Freivalds: every row of C x against A (B x), x with entries +-1
    g = np.random.default_rng(2)
    A64, B64 = Af.astype(np.float64), Bf.astype(np.float64)
    for _ in range(2):
        x = g.choice([-1.0, 1.0], size=w.N)
        lhs = Cd @ x
        rhs = A64 @ (B64 @ x)
        bound = tol * math.sqrt(w.N) * 6 + 1e-9 * np.abs(A64) @ np.abs(B64 @ x)
        assert np.all(np.abs(lhs - rhs) <= bound)


@pytest.mark.parametrize("pinned", [True, False])
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_host_entry_point_pipelined_chunks(lib, pinned, dtype):
    """M >= 4096 takes the chunked copy/compute pipeline; rows not a multiple of the chunk,
    a padded host leading dimension for A and C, integer inputs: exact."""
    M, N, K = 4352 + 3, 264, 72
    A, B = si.integer_copy(M, N, K, seed=44, dtype=dtype)
    tdt = A.dtype
    Abig = torch.zeros((M, K + 8), dtype=tdt)
    Abig[:, :K] = A
    Cbig = torch.full((M, N + 5), -3.0)
    if pinned:
        Abig, Cbig, B = Abig.pin_memory(), Cbig.pin_memory(), B.pin_memory()
    lib.matmul_host(Abig[:, :K], B, out=Cbig[:, :N])
    ref = oracle.gemm(A.float().numpy(), B.float().numpy())
    assert np.array_equal(Cbig[:, :N].double().numpy(), ref)
    assert torch.all(Cbig[:, N:] == -3.0)


def test_host_batch_pipelines_several_products(lib):
    """gemm_run_host_batch: a chunked bf16 product, an fp32 product, an fp16 product with
    padded host leading dimensions and an empty one, in one pipeline; integer inputs: exact,
    and each result equals the single-product entry point's."""
    import programming_tiled_gemm_gb300 as g
    shapes = [(4352 + 3, 264, 72, "bf16"), (4100, 136, 40, "f32"), (300, 72, 520, "f16"), (0, 8, 8, "bf16"),
              (4863, 16, 8, "f32"), (4864, 24, 16, "f32")]  # fp32 row chunks rounded past M, or ending at M
    pairs, outs, refs = [], [], []
    for i, (M, N, K, dt) in enumerate(shapes):
        A, B = si.integer_copy(M, N, K, seed=60 + i, dtype=dt)
        Abig = torch.zeros((M, K + 8), dtype=A.dtype).pin_memory()
        Abig[:, :K] = A
        Cbig = torch.full((M, N + 4), -3.0).pin_memory()
        pairs.append((Abig[:, :K], B.pin_memory()))
        outs.append(Cbig)
        refs.append(oracle.gemm(A.float().numpy(), B.float().numpy()))
    lib.matmul_host_batch(pairs, outs=[c[:, :N] for c, (_, N, _, _) in zip(outs, shapes)])
    for (M, N, K, dt), Cbig, ref, (A, B) in zip(shapes, outs, refs, pairs):
        assert np.array_equal(Cbig[:, :N].double().numpy(), ref)
        assert torch.all(Cbig[:, N:] == -3.0)
        if M:
            assert torch.equal(lib.matmul_host(A, B), Cbig[:, :N])
    # a bad problem anywhere in the batch: nothing runs
    C0 = torch.full((4, 4), 5.0)
    bad = [g.HostProblem(4, 4, 4, pairs[0][0].data_ptr(), 80, pairs[0][1].data_ptr(), 264, C0.data_ptr(), 4,
                         g.GEMM_BF16),
           g.HostProblem(4, 4, 4, 0, 4, 0, 4, C0.data_ptr(), 4, g.GEMM_BF16)]
    assert g.gemm_run_host_batch(lib.handle, bad) == g.GEMM_ERR_INVALID_ARG
    assert torch.all(C0 == 5.0)
