"""fp32 path on the GPU against the CPU oracle (through the C ABI).

Tolerances (max |C - C_ref| over the compared entries):
  * integer-valued inputs in [-4, 4]: exact (every partial sum is an integer below 2^24);
  * uniform[-1, 1] inputs: 1e-5 * sqrt(K).
Kernels: the 128x256 and 64x128 tiled FFMA kernels (with and without split-K), the
persistent TMA-fed 128x256 kernel (one launch; K slices added by the slice that finishes
last) and the two skinny kernels (B streamed through registers, or through a TMA ring in
shared memory), each forced on shapes with ragged tails, padded leading dimensions and
guard bands around C.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import seeded_inputs as si

pytestmark = pytest.mark.gpu

SENTINEL = 1234.5


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__
    __graft_entry__.build()
    import programming_tiled_gemm_gb300 as g
    h = g.Gemm(0)
    yield h
    h.close()


@pytest.fixture(autouse=True)
def _reset_options(lib):
    import programming_tiled_gemm_gb300 as g
    yield
    lib.set_option(g.GEMM_OPT_F32_KERNEL, 0)
    lib.set_option(g.GEMM_OPT_SPLIT_K, 0)


def run_padded(lib, A, B, pad_a=0, pad_b=0, pad_c=0, guard=2):
    """Run with leading dimensions padded and a sentinel band around C; check the band."""
    dev = torch.device("cuda")
    M, K = A.shape
    N = B.shape[1]
    Ad = torch.full((M, K + pad_a), float("nan"), device=dev)
    Ad[:, :K] = A.to(dev)
    Bd = torch.full((K, N + pad_b), float("nan"), device=dev)
    Bd[:, :N] = B.to(dev)
    Cbig = torch.full((M + 2 * guard, N + pad_c + 2 * guard), SENTINEL, device=dev)
    Cv = Cbig[guard:guard + M, guard:guard + N]
    lib.matmul(Ad[:, :K], Bd[:, :N], out=Cv)
    torch.cuda.synchronize()
    assert lib.device_status() == 0
    host = Cbig.cpu()
    mask = torch.ones_like(host, dtype=torch.bool)
    mask[guard:guard + M, guard:guard + N] = False
    assert torch.all(host[mask] == SENTINEL), "kernel wrote outside C"
    return host[guard:guard + M, guard:guard + N].double().numpy()


def ref_of(A, B):
    return oracle.gemm(A.numpy(), B.numpy())


KERNELS = [(1, 0), (1, 3), (2, 0), (2, 2), (3, 0), (3, 5), (4, 0), (4, 5), (5, 0), (5, 3)]  # (kernel, split-K: 0 = auto)
TMA_FED = (4, 5)  # kernels that need 16-byte rows of B (5: and of A)


def pad_to_16_bytes(n):
    """Padding that makes a row of n floats a multiple of 16 bytes (plus 4 floats of slack)."""
    return (4 - n % 4) % 4 + 4


@pytest.mark.parametrize("kernel,split", KERNELS)
@pytest.mark.parametrize("M,N,K", [(1, 1, 1), (7, 13, 5), (31, 129, 67), (32, 1030, 300), (130, 257, 129)])
def test_integer_inputs_are_exact(lib, kernel, split, M, N, K):
    import programming_tiled_gemm_gb300 as g
    if kernel in (3, 4) and M > 32:
        pytest.skip("skinny kernels take M <= 32")
    lib.set_option(g.GEMM_OPT_F32_KERNEL, kernel)
    lib.set_option(g.GEMM_OPT_SPLIT_K, split)
    A, B = si.integer_copy(M, N, K, seed=M * 1000 + N + K)
    # the TMA-fed kernels need 16-byte rows: pad ldb (and lda) to a multiple of 4 floats
    got = run_padded(lib, A, B, pad_a=pad_to_16_bytes(K) if kernel == 5 else 3,
                     pad_b=pad_to_16_bytes(N) if kernel in TMA_FED else 5, pad_c=1)
    assert np.array_equal(got, ref_of(A, B))


@pytest.mark.parametrize("kernel,split", KERNELS)
@pytest.mark.parametrize("M,N,K", [(17, 100, 1000), (29, 515, 777), (200, 136, 520)])
def test_uniform_inputs_within_tolerance(lib, kernel, split, M, N, K):
    import programming_tiled_gemm_gb300 as g
    if kernel in (3, 4) and M > 32:
        pytest.skip("skinny kernels take M <= 32")
    lib.set_option(g.GEMM_OPT_F32_KERNEL, kernel)
    lib.set_option(g.GEMM_OPT_SPLIT_K, split)
    A, B = si.gemm_operands(M, N, K, seed=5)
    got = run_padded(lib, A, B, pad_a=pad_to_16_bytes(K) if kernel == 5 else 0, pad_b=pad_to_16_bytes(N))
    assert np.abs(got - ref_of(A, B)).max() <= 1e-5 * math.sqrt(K)


def test_misaligned_operands_take_the_scalar_path(lib):
    dev = torch.device("cuda")
    M, N, K = 45, 61, 39
    A, B = si.integer_copy(M, N, K, seed=3)
    buf_a = torch.zeros(M * K + 1, device=dev)
    buf_a[1:] = A.reshape(-1).to(dev)
    buf_b = torch.zeros(K * N + 1, device=dev)
    buf_b[1:] = B.reshape(-1).to(dev)
    Ad = buf_a[1:].view(M, K)  # 4-byte offset: no float4 loads
    Bd = buf_b[1:].view(K, N)
    C = lib.matmul(Ad, Bd)
    assert np.array_equal(C.cpu().double().numpy(), ref_of(A, B))


def test_zero_K_writes_zeros_and_empty_shapes_are_noops(lib):
    dev = torch.device("cuda")
    C = torch.full((5, 7), 3.0, device=dev)
    lib.matmul(torch.empty((5, 0), device=dev), torch.empty((0, 7), device=dev), out=C)
    assert torch.all(C == 0)
    C = torch.full((0, 7), 3.0, device=dev)
    lib.matmul(torch.empty((0, 4), device=dev), torch.empty((4, 7), device=dev), out=C)
    C = torch.full((3, 2), 3.0, device=dev)
    lib.matmul(torch.ones((3, 4), device=dev)[:, :0], torch.ones((0, 2), device=dev), out=C)
    assert torch.all(C == 0)


def test_config_256_uniform_and_integer_copy(lib):
    w = si.WORKLOADS["f32_256"]
    A, B = si.workload_operands(w)
    C = lib.matmul(A.cuda(), B.cuda())
    assert np.abs(C.cpu().double().numpy() - ref_of(A, B)).max() <= 1e-5 * math.sqrt(w.K)
    Ai, Bi = si.integer_copy(w.M, w.N, w.K, w.seed)
    C = lib.matmul(Ai.cuda(), Bi.cuda())
    assert np.array_equal(C.cpu().double().numpy(), ref_of(Ai, Bi))


@pytest.mark.slow
def test_config_4096_full_matrix(lib):
    w = si.WORKLOADS["f32_4096"]
    A, B = si.workload_operands(w)
    C = lib.matmul(A.cuda(), B.cuda()).cpu().double().numpy()
    assert np.abs(C - ref_of(A, B)).max() <= 1e-5 * math.sqrt(w.K)
    Ai, Bi = si.integer_copy(w.M, w.N, w.K, w.seed)
    C = lib.matmul(Ai.cuda(), Bi.cuda()).cpu().double().numpy()
    assert np.array_equal(C, ref_of(Ai, Bi))


@pytest.mark.slow
def test_config_skinny_full_matrix(lib):
    w = si.WORKLOADS["f32_skinny"]
    A, B = si.workload_operands(w)
    C = lib.matmul(A.cuda(), B.cuda()).cpu().double().numpy()
    assert np.abs(C - ref_of(A, B)).max() <= 1e-5 * math.sqrt(w.K)
    # |partial sums| <= 16 * 16384 < 2^24: integer inputs are exact at this K too
    Ai, Bi = si.integer_copy(w.M, w.N, w.K, w.seed)
    C = lib.matmul(Ai.cuda(), Bi.cuda()).cpu().double().numpy()
    assert np.array_equal(C, ref_of(Ai, Bi))


def last_wave_plan(interior, slots, K):
    """The launcher's rule for the tiles of a last, partial wave: (tiles, pieces along K)."""
    if interior <= slots or interior % slots == 0:
        return 0, 1
    rem = interior % slots
    best_t, best_rs = 1.0, 1
    for rs in range(2, 9):
        if K // rs < 32 * 16:
            break
        t = ((rem * rs + slots - 1) // slots) / rs
        if t < best_t - 1e-9:
            best_t, best_rs = t, rs
    return (0, 1) if best_t > 0.85 else (rem, best_rs)


@pytest.mark.parametrize("M,N", [(1664, 3328), (1701, 3341)])
def test_last_wave_tiles_split_along_K(lib, M, N):
    # 13 x 13 = 169 interior 128 x 256 tiles: on 152 SMs the 17 tiles of the last wave run
    # cut into K slices whose partial tiles are summed in a separate fixed-order pass
    import programming_tiled_gemm_gb300 as g
    lib.set_option(g.GEMM_OPT_F32_KERNEL, 1)
    K = 2048
    slots = torch.cuda.get_device_properties(0).multi_processor_count
    rem, rs = last_wave_plan((M // 128) * (N // 256), slots, K)
    Ai, Bi = si.integer_copy(M, N, K, seed=M)
    n0 = lib.launch_count()
    got = run_padded(lib, Ai, Bi, pad_b=-N % 4, pad_c=4)  # rows of B 16-byte aligned: vector loads
    edge = (M % 128 != 0) or (N % 256 != 0)
    assert lib.launch_count() - n0 == 1 + (2 if rem else 0) + (1 if edge else 0)
    assert np.array_equal(got, ref_of(Ai, Bi))
    A, B = si.gemm_operands(M, N, K, seed=M + 1)
    got = run_padded(lib, A, B)
    assert np.abs(got - ref_of(A, B)).max() <= 1e-5 * math.sqrt(K)


def test_back_to_back_split_products_share_the_workspace(lib):
    """Products whose K slices or split-K partials go through the handle's workspace,
    queued on one stream with no synchronisation in between: the later launches of one
    call start as the earlier ones drain (programmatic dependent launches), and the next
    call's partials must not overwrite a workspace that is still being read."""
    shapes = [(1664, 3328, 2048), (16, 4096, 8192), (1664, 3328, 1024), (32, 1000, 3000)]
    ops = []
    for i, (M, N, K) in enumerate(shapes):
        Ai, Bi = si.integer_copy(M, N, K, seed=100 + i)
        ops.append((Ai, Bi, Ai.cuda(), Bi.cuda(), torch.empty((M, N), device="cuda")))
    torch.cuda.synchronize()
    for _, _, Ad, Bd, C in ops:
        lib.matmul(Ad, Bd, out=C)
    torch.cuda.synchronize()
    assert lib.device_status() == 0
    for Ai, Bi, _, _, C in ops:
        assert np.array_equal(C.cpu().double().numpy(), ref_of(Ai, Bi))


def test_results_are_deterministic(lib):
    import programming_tiled_gemm_gb300 as g
    A, B = si.gemm_operands(24, 3000, 5000, seed=9)
    Ad, Bd = A.cuda(), B.cuda()
    for kernel in (1, 2, 3, 4, 5):
        lib.set_option(g.GEMM_OPT_F32_KERNEL, kernel)
        lib.set_option(g.GEMM_OPT_SPLIT_K, 7)
        c1 = lib.matmul(Ad, Bd).clone()
        c2 = lib.matmul(Ad, Bd)
        assert torch.equal(c1, c2)


def test_argument_errors_are_reported(lib):
    import programming_tiled_gemm_gb300 as g
    dev = torch.device("cuda")
    A = torch.ones((4, 4), device=dev)
    C = torch.empty((4, 4), device=dev)
    h = lib.handle
    assert g.gemm_run(h, -1, 4, 4, A.data_ptr(), 4, A.data_ptr(), 4, C.data_ptr(), 4, 0) == g.GEMM_ERR_INVALID_ARG
    assert g.gemm_run(h, 4, 4, 4, A.data_ptr(), 3, A.data_ptr(), 4, C.data_ptr(), 4, 0) == g.GEMM_ERR_INVALID_ARG
    assert g.gemm_run(h, 4, 4, 4, A.data_ptr(), 4, A.data_ptr(), 4, C.data_ptr(), 3, 0) == g.GEMM_ERR_INVALID_ARG
    assert g.gemm_run(h, 4, 4, 4, 0, 4, A.data_ptr(), 4, C.data_ptr(), 4, 0) == g.GEMM_ERR_INVALID_ARG
    assert g.gemm_run(h, 4, 4, 4, A.data_ptr(), 4, A.data_ptr(), 4, C.data_ptr(), 4, 7) == g.GEMM_ERR_INVALID_ARG
    assert g.gemm_set_option(h, g.GEMM_OPT_F32_KERNEL, 9) == g.GEMM_ERR_INVALID_ARG
    assert g.gemm_set_option(h, g.GEMM_OPT_SPLIT_K, 5000) == g.GEMM_ERR_INVALID_ARG
    lib.set_option(g.GEMM_OPT_F32_KERNEL, 3)
    assert g.gemm_run(h, 40, 4, 4, A.data_ptr(), 4, A.data_ptr(), 4, C.data_ptr(), 4, 0) == g.GEMM_ERR_UNSUPPORTED
    lib.set_option(g.GEMM_OPT_F32_KERNEL, 4)
    # the TMA-fed kernel needs 16-byte aligned B rows
    assert g.gemm_run(h, 4, 3, 4, A.data_ptr(), 4, A.data_ptr(), 3, C.data_ptr(), 4, 0) == g.GEMM_ERR_ALIGNMENT


def test_sizes_beyond_the_kernels_and_failed_allocations_leave_the_handle_usable(lib):
    """A size or leading dimension past the kernels' 32-bit indexing is refused before
    anything is allocated or launched; a workspace too large to allocate is reported as a
    CUDA error; neither leaves an error behind for the next call."""
    import programming_tiled_gemm_gb300 as g
    h = lib.handle
    A = torch.ones(64, device="cuda")
    C = torch.zeros(64, device="cuda")
    big = 2**31 - 1
    assert g.gemm_run(h, big, 4, 4, A.data_ptr(), 4, A.data_ptr(), 4, C.data_ptr(), 4, 0) == g.GEMM_ERR_UNSUPPORTED
    assert g.gemm_run(h, 4, 4, 4, A.data_ptr(), big, A.data_ptr(), 4, C.data_ptr(), 4, 0) == g.GEMM_ERR_UNSUPPORTED
    assert g.gemm_run(h, 4, 4, 4, A.data_ptr(), 8, A.data_ptr(), 8, C.data_ptr(), 4, g.GEMM_BF16) == g.GEMM_OK
    torch.cuda.synchronize()
    assert g.gemm_run(h, 4, big, 4, A.data_ptr(), 8, A.data_ptr(), big, C.data_ptr(), big,
                      g.GEMM_BF16) == g.GEMM_ERR_UNSUPPORTED
    # 1024 K slices of a 65536 x 65536 product: a ~17.6 TB workspace that cudaMalloc refuses
    lib.set_option(g.GEMM_OPT_SPLIT_K, 1024)
    try:
        n = 65536
        assert g.gemm_run(h, n, n, 1024, A.data_ptr(), 1024, A.data_ptr(), n, C.data_ptr(), n, 0) == g.GEMM_ERR_CUDA
    finally:
        lib.set_option(g.GEMM_OPT_SPLIT_K, 0)
    # the handle and the thread's CUDA state are clean: a normal product runs and is exact
    Ai, Bi = si.integer_copy(40, 72, 56, seed=77)
    got = lib.matmul(Ai.cuda(), Bi.cuda())
    torch.cuda.synchronize()
    assert lib.device_status() == 0
    assert np.array_equal(got.cpu().double().numpy(), ref_of(Ai, Bi))


def test_host_buffer_entry_point(lib):
    A, B = si.integer_copy(70, 90, 110, seed=4)
    C = lib.matmul_host(A, B)
    assert np.array_equal(C.double().numpy(), ref_of(A, B))


def persistent_plan(M, N, K, slots):
    """The persistent kernel's rule for a last, partial wave of 128 x 256 tiles:
    (first split tile, K slices)."""
    tiles = -(-M // 128) * -(-N // 256)
    k_tiles = -(-K // 32)
    r = tiles % slots
    if r == 0:
        return tiles, 1
    tile_us = 2.0 * 128 * 256 * K / 4.0e5
    best, S = float(-(-r // slots)), 1
    for s in range(2, 17):
        if k_tiles // s < 8:
            break
        t = (-(-(r * s) // slots)) / s + ((s - 1) + 2.0) / tile_us
        if t < best - 1e-9:
            best, S = t, s
    if S == 1:
        return tiles, 1
    kps = -(-k_tiles // S)
    return tiles - r, -(-k_tiles // kps)


@pytest.mark.parametrize("M,N,K", [
    (1664, 3328, 2048),  # 169 whole tiles: the last 17 in K slices
    (1701, 3341, 2050),  # ragged M, N and K (zero-filled boxes; predicated edge stores)
    (4096, 4096, 1024),  # 512 tiles: 3 rounds + 56 tiles in slices
    (520, 1030, 3000),   # fewer tiles than SMs: every tile in slices
    (256, 256, 4096),    # one tile in 16 slices
    (100, 8000, 700),    # 32 tiles, K of 22 k-tiles with a ragged last one
])
def test_persistent_kernel_one_launch_exact_and_within_tolerance(lib, M, N, K):
    """The persistent kernel is one launch whatever the split; the slice that finishes a
    tile last adds every slice's partial in slice order."""
    import programming_tiled_gemm_gb300 as g
    slots = torch.cuda.get_device_properties(0).multi_processor_count
    first, S = persistent_plan(M, N, K, slots)
    if M >= 1664:
        assert S > 1  # these shapes exercise the slices
    lib.set_option(g.GEMM_OPT_F32_KERNEL, 5)
    Ai, Bi = si.integer_copy(M, N, K, seed=M + N)
    n0 = lib.launch_count()
    got = run_padded(lib, Ai, Bi, pad_a=pad_to_16_bytes(K), pad_b=pad_to_16_bytes(N), pad_c=3)
    assert lib.launch_count() - n0 == 1
    assert np.array_equal(got, ref_of(Ai, Bi))
    A, B = si.gemm_operands(M, N, K, seed=M + N + 1)
    got = run_padded(lib, A, B, pad_a=pad_to_16_bytes(K), pad_b=pad_to_16_bytes(N))
    assert np.abs(got - ref_of(A, B)).max() <= 1e-5 * math.sqrt(K)


def test_persistent_kernel_is_the_default_for_aligned_operands(lib):
    """With 16-byte rows (M > 64) the default choice is the persistent kernel: one launch."""
    A, B = si.integer_copy(1024, 1024, 512, seed=41)
    Ad, Bd = A.cuda(), B.cuda()
    n0 = lib.launch_count()
    C = lib.matmul(Ad, Bd)
    assert lib.launch_count() - n0 == 1
    assert np.array_equal(C.cpu().double().numpy(), ref_of(A, B))


def test_persistent_kernel_refuses_unaligned_rows(lib):
    import programming_tiled_gemm_gb300 as g
    lib.set_option(g.GEMM_OPT_F32_KERNEL, 5)
    A = torch.ones((100, 66), device="cuda")
    C = torch.empty((100, 66), device="cuda")
    h = lib.handle
    # lda = 66: rows of A are not a multiple of 16 bytes
    assert g.gemm_run(h, 100, 64, 66, A.data_ptr(), 66, A.data_ptr(), 66, C.data_ptr(), 66, 0) == g.GEMM_ERR_ALIGNMENT


def test_persistent_forced_split_matches_the_split_partials_of_the_tiled_kernel(lib):
    """A forced split cuts every tile at the same k-tile boundaries as the tiled kernel's
    split-K, and both add the slices in slice order: the two agree bit for bit."""
    import programming_tiled_gemm_gb300 as g
    A, B = si.gemm_operands(384, 512, 2000, seed=43)
    Ad, Bd = A.cuda(), B.cuda()
    lib.set_option(g.GEMM_OPT_SPLIT_K, 5)
    lib.set_option(g.GEMM_OPT_F32_KERNEL, 5)
    c5 = lib.matmul(Ad, Bd).clone()
    lib.set_option(g.GEMM_OPT_F32_KERNEL, 1)
    c1 = lib.matmul(Ad, Bd)
    torch.cuda.synchronize()
    assert lib.device_status() == 0
    assert np.abs(c5.cpu().double().numpy() - ref_of(A, B)).max() <= 1e-5 * math.sqrt(2000)
    assert np.abs(c5.cpu().double().numpy() - c1.cpu().double().numpy()).max() <= 2e-5 * math.sqrt(2000)
