// bf16 / fp16 GEMM on the 5th-generation tensor cores (tcgen05) of sm_103a.
//
// The tiling idea is the one "Learning to develop for GPU with GEMM as the example"
// builds up (sections "Making the GPU implementation better", "How loading into local
// memory is organised", "Improving the solution and balancing memory work"): blocks of
// A and B are staged in on-chip memory and multiplied into a block of accumulators that
// never leaves the chip until the block is done.  On this GPU every level is done by the
// hardware unit made for it:
//   * global -> shared: the Tensor Memory Accelerator (cp.async.bulk.tensor) copies a
//     128 x 64 tile of A and a 64 x 256 tile of B per k-block, 128-byte swizzled (the
//     swizzle is what the page's padding does by hand against bank conflicts, section
//     "How to do even better");
//   * the multiply: tcgen05.mma (M=128, N=256, K=16) issued by one thread, reading both
//     operands from shared memory through matrix descriptors;
//   * the accumulators: a 128 x 256 fp32 block in tensor memory (TMEM).  The tensor
//     core's own fp32 accumulation rounds toward zero, so its error grows faster than
//     the length of the sum (measured on GB300: max error 4.5e-3 at K = 8192 for
//     normal(0,1) bf16 inputs, against 2.6e-4 .. 6.2e-4 when the sum is cut into
//     512- to 1024-long pieces).  The K loop is therefore cut into chunks of `kc`
//     k-blocks: each chunk starts a fresh TMEM accumulator, alternating between two
//     TMEM buffers, and the epilogue warps add every finished chunk into fp32
//     registers with ordinary round-to-nearest adds, in chunk order;
//   * the epilogue ("Three X: large convolutions in PyTorch for training", section
//     "CUTLASS": the step after the MMA that moves accumulators out): tcgen05.ld into
//     registers, chunk sums in registers, then, once the tile's last chunk is in, plain
//     fp32 C goes out 32 x 32 at a time through a swizzled shared-memory block and a TMA
//     store (coalesced 128-byte rows, clipped at the matrix edge); alpha / beta and 16-bit
//     C use vectorised per-thread stores.  While it works on one chunk, the MMA fills the
//     other buffer, so the epilogue is hidden behind the main loop.
//   * M <= 128 with few tiles: K is split over the CTAs of a cluster, which add their
//     partial tiles through distributed shared memory (see split_reduce_store).
// Warp roles (320 threads): warp 0 = TMA producer, warp 1 = MMA issuer (and TMEM owner),
// warps 2..9 = epilogue (two warps per 32-lane TMEM quarter, 128 columns each).  A ring
// of shared-memory stages (4 for single CTAs, 6 for CTA pairs) links producer and MMA
// through mbarriers.  The grid is persistent (one CTA, or CTA pair, per SM or SM pair)
// and walks output tiles in groups of tile-rows (16 rows of 128 for single CTAs, 2048 rows
// for pairs) so that concurrently running tiles share A rows and B columns in L2 ("CUDA
// overview: performance surprises", section "Parallelism first": enough independent work
// per SM, no idle units).  The CTA-pair kernel below (cta_group::2) is the default for
// M > 128.
//
// Every wait on an mbarrier is bounded (a wall-clock limit read from %globaltimer).  On
// expiry the thread records an error code in the caller-visible status word, the CTA
// waits (again bounded) for its own TMA copies and MMAs in flight, frees its TMEM and
// returns; the host reads the code through gemm_get_device_status.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <atomic>
#include <mutex>

#include "internal.h"
#include "ptx.h"

namespace gemm_gb300 {

GEMM_DEBUG_UNIT(tc_gemm)

namespace {

constexpr int BM = 128;              // rows of an output tile (TMEM lanes)
constexpr int BN = 256;              // columns of an output tile (fp32 TMEM columns)
constexpr int BK = 64;               // k per stage: 64 x 2 bytes = one 128-byte swizzle row
constexpr int UMMA_K = 16;           // k of one tcgen05.mma for 16-bit inputs
constexpr int STAGES = 4;
constexpr int GROUP_M = 16;          // tile rows per raster group
constexpr int EPI_WARPS = 8;        // two per TMEM lane quarter, each owning 128 columns
constexpr int THREADS = 64 + 32 * EPI_WARPS;
constexpr int EPI_COLS = BN / 2;     // columns per epilogue thread (fp32 registers)
constexpr int A_STAGE_BYTES = BM * BK * 2;   // 16 KiB
constexpr int B_BOX_N = 64;                  // TMA box width along N (128 bytes)
constexpr int B_BOX_BYTES = B_BOX_N * BK * 2;  // 8 KiB
constexpr int B_STAGE_BYTES = BN * BK * 2;   // 32 KiB
constexpr int STAGE_BYTES = A_STAGE_BYTES + B_STAGE_BYTES;
constexpr int TMEM_COLS = 2 * BN;            // two chunk accumulators
// TMA-store epilogue: one 32 x 32 fp32 staging block per epilogue warp, after the ring
constexpr int EPI_STAGE_BYTES = 32 * 32 * 4;
constexpr int EPI_STAGE_TOTAL = EPI_WARPS * EPI_STAGE_BYTES;  // 32 KiB
constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + EPI_STAGE_TOTAL + 1024 /*barriers*/ + 1024 /*alignment slack*/;
constexpr int EPI_THREADS = 32 * EPI_WARPS;
// Split-K: a slice's fp32 partial tile, kept in its CTA's shared memory (the operand ring,
// free once the tile's MMAs are done) as BM rows of BN * 4 bytes; 16-byte chunk c of row r
// sits at chunk c ^ (r & 7), so that the epilogue's row-per-thread stores and the
// reduction's row-contiguous loads are both free of bank conflicts.
constexpr int SPLIT_ROW_BYTES = BN * 4;
constexpr int MAX_SPLIT = 16;  // K slices per tile (cluster size; above 8 is non-portable)
static_assert(BM * SPLIT_ROW_BYTES <= STAGES * STAGE_BYTES, "partial tile must fit the operand ring");

// Instruction descriptor, kind::f16: fp32 accumulator, A K-major, B N-major (B is the
// row-major K x N operand), N = 256; M = 128 for one CTA, 256 for a CTA pair.
__host__ __device__ constexpr uint32_t make_idesc(bool bf16, int m = BM)
{
    return (1u << 4)                         // D format: f32
           | ((bf16 ? 1u : 0u) << 7)         // A format: bf16 = 1, f16 = 0
           | ((bf16 ? 1u : 0u) << 10)        // B format
           | (0u << 15)                      // A major: K
           | (1u << 16)                      // B major: MN
           | ((uint32_t)(BN >> 3) << 17)     // N >> 3
           | ((uint32_t)(m >> 4) << 24);     // M >> 4
}

struct TileCoord {
    int m_blk, n_blk;
};

__device__ __forceinline__ TileCoord tile_coord(int t, int m_blocks, int n_blocks, int group_m = GROUP_M)
{
    const int per_group = group_m * n_blocks;
    const int g = t / per_group;
    const int first_m = g * group_m;
    const int gm = min(m_blocks - first_m, group_m);
    const int r = t - g * per_group;
    return {first_m + r % gm, r / gm};
}

struct TcParams {
    int M, N, K;
    void* C;  // fp32, bf16 or fp16 (c_dtype)
    int64_t ldc;
    int m_blocks, n_blocks, num_tiles, k_blocks;
    int kc;       // k-blocks per accumulation chunk
    int nchunks;  // chunks per tile (per K slice with split-K)
    int nsplit;   // single-CTA kernel: K slices of a tile, one CTA each, as one cluster
                  // (work item = tile * nsplit + slice); 1 = no split.  Slice z covers
                  // k-blocks [z * k_blocks / nsplit, (z + 1) * k_blocks / nsplit)
    int group_m;  // tile rows per raster group
    // CTA-pair kernel, last-wave split: work items [0, rem_first) are whole tiles; the
    // tiles from rem_first on are cut into rem_split K slices, item rem_first + j being
    // slice j % rem_split of tile rem_first + j / rem_split.  rem_split = 1: no split.
    int num_items, rem_first, rem_split;
    float* rem_ws;                  // [tile - rem_first][slice][CTA][warp][4096] partials
    unsigned long long* rem_cnt;    // [tile - rem_first][CTA][warp] arrivals, tagged rem_seq
    uint32_t* rem_flag;             // [same] rem_seq once the first slice's part is in C
    uint32_t rem_seq;               // this launch's tag (nonzero)
    int rem_direct;                 // 2 slices, plain fp32 C by TMA: C = first, then += second
    uint32_t idesc;
    int vec_store;
    int* status;
    uint64_t limit_ns;
    int test_stall;  // test hook: the epilogue first waits on a barrier nothing arrives on
    float alpha, beta;  // C = alpha * (A . B) + beta * C; C unread when beta == 0
    int c_dtype;        // GEMM_F32, GEMM_BF16 or GEMM_F16
    int epi_plain;      // alpha == 1, beta == 0, fp32: plain stores
    int c_tma;          // plain fp32 C stored by TMA through per-warp staging (tmC valid)
};

// Four adjacent outputs of the generalised product: C = alpha * acc + beta * C, in the
// output type; one 16- or 8-byte access when `vec`, else element by element.
__device__ __forceinline__ void epi_store4(const TcParams& p, int64_t off, int ncols, float a0, float a1, float a2,
                                           float a3, bool vec)
{
    float v[4] = {p.alpha * a0, p.alpha * a1, p.alpha * a2, p.alpha * a3};
    if (p.c_dtype == GEMM_F32) {
        float* c = static_cast<float*>(p.C) + off;
        if (vec) {
            if (p.beta != 0.f) {
                const float4 o = *reinterpret_cast<const float4*>(c);
                v[0] = fmaf(p.beta, o.x, v[0]), v[1] = fmaf(p.beta, o.y, v[1]);
                v[2] = fmaf(p.beta, o.z, v[2]), v[3] = fmaf(p.beta, o.w, v[3]);
            }
            *reinterpret_cast<float4*>(c) = make_float4(v[0], v[1], v[2], v[3]);
        } else {
#pragma unroll
            for (int j = 0; j < 4; ++j)
                if (j < ncols) c[j] = (p.beta != 0.f) ? fmaf(p.beta, c[j], v[j]) : v[j];
        }
    } else if (p.c_dtype == GEMM_BF16) {
        __nv_bfloat16* c = static_cast<__nv_bfloat16*>(p.C) + off;
        if (vec) {
            uint2 raw = make_uint2(0, 0);
            if (p.beta != 0.f) raw = *reinterpret_cast<const uint2*>(c);
            __nv_bfloat162 lo = *reinterpret_cast<__nv_bfloat162*>(&raw.x), hi = *reinterpret_cast<__nv_bfloat162*>(&raw.y);
            if (p.beta != 0.f) {
                v[0] = fmaf(p.beta, __low2float(lo), v[0]), v[1] = fmaf(p.beta, __high2float(lo), v[1]);
                v[2] = fmaf(p.beta, __low2float(hi), v[2]), v[3] = fmaf(p.beta, __high2float(hi), v[3]);
            }
            lo = __floats2bfloat162_rn(v[0], v[1]);
            hi = __floats2bfloat162_rn(v[2], v[3]);
            raw.x = *reinterpret_cast<uint32_t*>(&lo);
            raw.y = *reinterpret_cast<uint32_t*>(&hi);
            *reinterpret_cast<uint2*>(c) = raw;
        } else {
#pragma unroll
            for (int j = 0; j < 4; ++j)
                if (j < ncols)
                    c[j] = __float2bfloat16_rn((p.beta != 0.f) ? fmaf(p.beta, __bfloat162float(c[j]), v[j]) : v[j]);
        }
    } else {
        __half* c = static_cast<__half*>(p.C) + off;
        if (vec) {
            uint2 raw = make_uint2(0, 0);
            if (p.beta != 0.f) raw = *reinterpret_cast<const uint2*>(c);
            __half2 lo = *reinterpret_cast<__half2*>(&raw.x), hi = *reinterpret_cast<__half2*>(&raw.y);
            if (p.beta != 0.f) {
                v[0] = fmaf(p.beta, __low2float(lo), v[0]), v[1] = fmaf(p.beta, __high2float(lo), v[1]);
                v[2] = fmaf(p.beta, __low2float(hi), v[2]), v[3] = fmaf(p.beta, __high2float(hi), v[3]);
            }
            lo = __floats2half2_rn(v[0], v[1]);
            hi = __floats2half2_rn(v[2], v[3]);
            raw.x = *reinterpret_cast<uint32_t*>(&lo);
            raw.y = *reinterpret_cast<uint32_t*>(&hi);
            *reinterpret_cast<uint2*>(c) = raw;
        } else {
#pragma unroll
            for (int j = 0; j < 4; ++j)
                if (j < ncols)
                    c[j] = __float2half_rn((p.beta != 0.f) ? fmaf(p.beta, __half2float(c[j]), v[j]) : v[j]);
        }
    }
}

// Plain fp32 C from an epilogue warp: its 32 rows (thread = row lane) x EPI_COLS columns
// of `tot`, 32 columns at a time through a 32 x 32 staging block in the 128-byte-swizzle
// layout of tmC's box (16-byte chunk c of row r at chunk c ^ (r & 7): the row-per-thread
// writes meet no bank conflicts), then one TMA store of full 128-byte row segments.  The
// TMA clips rows past M and columns past N.
template <bool ADD = false>
__device__ __forceinline__ void store_rows_tma(const CUtensorMap* tmC, const float (&tot)[EPI_COLS], uint8_t* stg,
                                               int row0, int col0, int M, int N, int lane, uint64_t cpol = 0)
{
    if (row0 >= M) return;
#pragma unroll
    for (int j = 0; j < EPI_COLS / 32; ++j) {
        if (col0 + 32 * j >= N) break;
        if (lane == 0) bulk_wait_group_read0();  // the previous block has left the staging buffer
        __syncwarp();
#pragma unroll
        for (int c = 0; c < 8; ++c)
            *reinterpret_cast<float4*>(stg + lane * 128 + ((c ^ (lane & 7)) << 4)) =
                make_float4(tot[32 * j + 4 * c], tot[32 * j + 4 * c + 1], tot[32 * j + 4 * c + 2], tot[32 * j + 4 * c + 3]);
        fence_proxy_async_shared();
        __syncwarp();
        if (lane == 0) {
            if (ADD)
                tma_reduce_add_2d(tmC, smem_u32(stg), col0 + 32 * j, row0);
            else if (cpol)
                tma_store_2d_hint(tmC, smem_u32(stg), col0 + 32 * j, row0, cpol);
            else
                tma_store_2d(tmC, smem_u32(stg), col0 + 32 * j, row0);
            bulk_commit_group();
        }
    }
}

__device__ __forceinline__ void record_error(int* status, int code, volatile int* abort_flag)
{
    atomicCAS(status, 0, code);
    *abort_flag = 1;
}

// A work item of the CTA-pair kernel: tile t, k-blocks [kb0, kb1), K slice sl (-1: whole).
struct PairItem {
    int t, sl, kb0, kb1;
};

__device__ __forceinline__ PairItem pair_item(const TcParams& p, int it)
{
    if (it < p.rem_first) return {it, -1, 0, p.k_blocks};
    const int j = it - p.rem_first, sl = j % p.rem_split;
    return {p.rem_first + j / p.rem_split, sl, (int)((int64_t)sl * p.k_blocks / p.rem_split),
            (int)((int64_t)(sl + 1) * p.k_blocks / p.rem_split)};
}

constexpr int MAX_REM_SPLIT = 4;
constexpr int REM_PART_FLOATS = 32 * EPI_COLS;  // one epilogue warp's 32 rows x 128 columns

// Last-wave split, one epilogue warp's part (32 rows x 128 columns, thread = row) of K
// slice `sl` of split tile j: publish it, count it, and if it is the part's last slice to
// finish, replace `tot` by the sum of all slices in slice order (true: store C).  Nothing
// waits for another warp or CTA.
__device__ __forceinline__ bool rem_slice_combine(const TcParams& p, float (&tot)[EPI_COLS], int j, int sl, int cta,
                                                  int w, int lane, int* status, volatile int* abort_flag)
{
    const int S = p.rem_split;
    if (!in_range(j, p.num_tiles - p.rem_first) || !in_range(sl, S) || !in_range(cta, 2) || !in_range(w, EPI_WARPS))
        return false;
    float* base = p.rem_ws + ((int64_t)(j * S) * 2 * EPI_WARPS + cta * EPI_WARPS + w) * REM_PART_FLOATS;
    const int64_t zstride = (int64_t)2 * EPI_WARPS * REM_PART_FLOATS;  // between slices
    float4* mine = reinterpret_cast<float4*>(base + sl * zstride) + lane;
#pragma unroll
    for (int q = 0; q < EPI_COLS / 4; ++q)
        __stcg(mine + q * 32, make_float4(tot[4 * q], tot[4 * q + 1], tot[4 * q + 2], tot[4 * q + 3]));
    __threadfence();
    __syncwarp();
    int n = 0;
    if (lane == 0) {
        n = tagged_arrive(p.rem_cnt + ((int64_t)j * 2 + cta) * EPI_WARPS + w, p.rem_seq);
        if (n == 0) record_error(status, kDevTimeoutEpilogue, abort_flag);
    }
    n = __shfl_sync(0xffffffffu, n, 0);
    if (n != S) return false;
    __threadfence();
    // every slice, this warp's own included, is read back, so that no partial stays live
    // in registers while the slices are added
    const float4* src = reinterpret_cast<const float4*>(base) + lane;
#pragma unroll
    for (int q = 0; q < EPI_COLS / 4; ++q) {
        float4 acc = __ldcg(src + q * 32);
#pragma unroll
        for (int z = 1; z < MAX_REM_SPLIT; ++z)
            if (z < S) {
                const float4 u = __ldcg(src + z * (zstride / 4) + q * 32);
                acc.x = __fadd_rn(acc.x, u.x), acc.y = __fadd_rn(acc.y, u.y);
                acc.z = __fadd_rn(acc.z, u.z), acc.w = __fadd_rn(acc.w, u.w);
            }
        tot[4 * q] = acc.x, tot[4 * q + 1] = acc.y, tot[4 * q + 2] = acc.z, tot[4 * q + 3] = acc.w;
    }
    return true;
}

__device__ __forceinline__ int slice_begin(const TcParams& p, int z)
{
    return (int)((int64_t)z * p.k_blocks / p.nsplit);
}

// Split-K output: this CTA (rank r of the tile's cluster of S slices) adds, for its share
// of the tile's 16-byte chunks, the S partial tiles in slice order (read from each CTA's
// shared memory) and stores C.  e = 0 .. EPI_THREADS - 1.
__device__ __forceinline__ void split_reduce_store(const TcParams& p, uint32_t part, int tile, int e)
{
    constexpr int CHUNKS = BM * BN / 4;
    const int S = p.nsplit;
    const int r = (int)cluster_ctarank();
    const TileCoord tc = tile_coord(tile, p.m_blocks, p.n_blocks);
    const int lo = (int)((int64_t)CHUNKS * r / S), hi = (int)((int64_t)CHUNKS * (r + 1) / S);
    uint32_t peer[MAX_SPLIT];
#pragma unroll
    for (int z = 0; z < MAX_SPLIT; ++z)
        if (z < S) peer[z] = mapa_shared(part, (uint32_t)z);
#pragma unroll 2
    for (int idx = lo + e; idx < hi; idx += EPI_THREADS) {
        const int rr = idx / (BN / 4), c = idx % (BN / 4);
        const uint32_t off = (uint32_t)(rr * SPLIT_ROW_BYTES + ((c ^ (rr & 7)) << 4));
        float4 v[MAX_SPLIT];
#pragma unroll
        for (int z = 0; z < MAX_SPLIT; ++z)
            if (z < S) v[z] = ld_shared_cluster_f4(peer[z] + off);
        float4 acc = v[0];
#pragma unroll
        for (int z = 1; z < MAX_SPLIT; ++z)
            if (z < S) {
                acc.x = __fadd_rn(acc.x, v[z].x), acc.y = __fadd_rn(acc.y, v[z].y);
                acc.z = __fadd_rn(acc.z, v[z].z), acc.w = __fadd_rn(acc.w, v[z].w);
            }
        const int row = tc.m_blk * BM + rr, col = tc.n_blk * BN + 4 * c;
        if (row >= p.M || col >= p.N) continue;
        const bool full = p.vec_store && col + 4 <= p.N;
        if (!p.epi_plain) {
            epi_store4(p, (int64_t)row * p.ldc + col, p.N - col, acc.x, acc.y, acc.z, acc.w, full);
        } else {
            float* cp = static_cast<float*>(p.C) + (int64_t)row * p.ldc + col;
            if (full) {
                *reinterpret_cast<float4*>(cp) = acc;
            } else {
                const float w[4] = {acc.x, acc.y, acc.z, acc.w};
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    if (col + j < p.N) cp[j] = w[j];
            }
        }
    }
}

__global__ void __launch_bounds__(THREADS, 1)
tc_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
               const __grid_constant__ CUtensorMap tmC, TcParams p)
{
    extern __shared__ uint8_t smem_raw[];
    // 1024-byte alignment for the 128-byte swizzle atoms
    const uint32_t raw = smem_u32(smem_raw);
    uint8_t* smem = smem_raw + ((1024 - (raw & 1023)) & 1023);
    uint8_t* smem_a = smem;
    uint8_t* smem_b = smem + STAGES * A_STAGE_BYTES;
    uint8_t* epi_stage = smem + STAGES * STAGE_BYTES;  // [EPI_WARPS][32 rows][128 bytes]
    uint64_t* bars = reinterpret_cast<uint64_t*>(epi_stage + EPI_STAGE_TOTAL);
    uint64_t* full_bar = bars;                    // [STAGES] TMA bytes landed
    uint64_t* empty_bar = bars + STAGES;          // [STAGES] MMAs reading the stage done
    uint64_t* tfull_bar = bars + 2 * STAGES;      // [2] chunk accumulator complete
    uint64_t* tempty_bar = bars + 2 * STAGES + 2; // [2] chunk accumulator read by the epilogue
    uint64_t* drain_bar = bars + 2 * STAGES + 4;  // MMA issuer's final completion check
    uint64_t* never_bar = bars + 2 * STAGES + 5;  // never completes (test hook)
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bars + 2 * STAGES + 6);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);

    const int warp = threadIdx.x / 32;
    const int lane = threadIdx.x % 32;

    if (warp == 0 && lane == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(smem_u32(&full_bar[s]), 1);
            mbar_init(smem_u32(&empty_bar[s]), 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(smem_u32(&tfull_bar[a]), 1);
            mbar_init(smem_u32(&tempty_bar[a]), EPI_WARPS);  // one arrival per epilogue warp
        }
        mbar_init(smem_u32(drain_bar), 1);
        mbar_init(smem_u32(never_bar), 1);
        *abort_flag = 0;
        mbar_fence_init();
        prefetch_tensormap(&tmA);
        prefetch_tensormap(&tmB);
        if (p.c_tma) prefetch_tensormap(&tmC);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_holder), TMEM_COLS);
        tc_fence_before();
    }
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_holder;

    if (warp == 0) {
        // ---------------------------------------------------------------- producer
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            uint32_t issued_mask = 0, last_parity = 0;
            bool ok = true;
            for (int it = blockIdx.x; it < p.num_tiles * p.nsplit && ok; it += gridDim.x) {
                const int t = it / p.nsplit, sl = it % p.nsplit;
                const TileCoord tc = tile_coord(t, p.m_blocks, p.n_blocks);
                const int kb_end = slice_begin(p, sl + 1);
                for (int kb = slice_begin(p, sl); kb < kb_end; ++kb) {
                    if (*abort_flag || !mbar_wait(smem_u32(&empty_bar[stage]), phase ^ 1, p.limit_ns)) {
                        record_error(p.status, kDevTimeoutProducer, abort_flag);
                        ok = false;
                        break;
                    }
                    const uint32_t fb = smem_u32(&full_bar[stage]);
                    mbar_arrive_expect_tx(fb, STAGE_BYTES);
                    tma_load_2d(smem_u32(smem_a + stage * A_STAGE_BYTES), &tmA, fb, kb * BK, tc.m_blk * BM);
                    uint8_t* b_dst = smem_b + stage * B_STAGE_BYTES;
#pragma unroll
                    for (int j = 0; j < BN / B_BOX_N; ++j)
                        tma_load_2d(smem_u32(b_dst + j * B_BOX_BYTES), &tmB, fb, tc.n_blk * BN + j * B_BOX_N, kb * BK);
                    issued_mask |= 1u << stage;
                    last_parity = (last_parity & ~(1u << stage)) | (phase << stage);
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1;
                    }
                }
            }
            // every copy this CTA issued must have landed before its shared memory goes away
            for (int s = 0; s < STAGES; ++s)
                if ((issued_mask >> s) & 1)
                    if (!mbar_wait(smem_u32(&full_bar[s]), (last_parity >> s) & 1, p.limit_ns))
                        record_error(p.status, kDevTimeoutDrain, abort_flag);
        }
        __syncwarp();
    } else if (warp == 1) {
        // ---------------------------------------------------------------- MMA issuer
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            int buf = 0;
            uint32_t buf_phase = 0;
            bool ok = true;
            const uint32_t a_base = smem_u32(smem_a), b_base = smem_u32(smem_b);
            for (int it = blockIdx.x; it < p.num_tiles * p.nsplit && ok; it += gridDim.x) {
                const int sl = it % p.nsplit;
                const int kb_beg = slice_begin(p, sl), kb_end = slice_begin(p, sl + 1);
                for (int ch = 0; ch < p.nchunks && ok; ++ch) {
                    const int kb0 = kb_beg + ch * p.kc;
                    if (kb0 >= kb_end) break;  // a short last slice has fewer chunks
                    if (*abort_flag || !mbar_wait(smem_u32(&tempty_bar[buf]), buf_phase ^ 1, p.limit_ns)) {
                        record_error(p.status, kDevTimeoutMma, abort_flag);
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t d_tmem = tmem_base + (uint32_t)(buf * BN);
                    const int kb1 = min(kb0 + p.kc, kb_end);
                    for (int kb = kb0; kb < kb1; ++kb) {
                        if (*abort_flag || !mbar_wait(smem_u32(&full_bar[stage]), phase, p.limit_ns)) {
                            record_error(p.status, kDevTimeoutMma, abort_flag);
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        const uint32_t a_st = a_base + stage * A_STAGE_BYTES;
                        const uint32_t b_st = b_base + stage * B_STAGE_BYTES;
#pragma unroll
                        for (int k = 0; k < BK / UMMA_K; ++k) {
                            // A: K-major rows of 128 bytes, 8-row atoms 1024 bytes apart; step k
                            //    moves 32 bytes along the row inside the swizzle atom.
                            const uint64_t a_desc = smem_desc_sw128(a_st + k * UMMA_K * 2, 16, 1024);
                            // B: N-major, 8 k-rows of 128 bytes per atom; atoms 1024 bytes apart
                            //    along K, 64-column boxes 8 KiB apart along N; step k = 16 rows.
                            const uint64_t b_desc = smem_desc_sw128(b_st + k * UMMA_K * 128, B_BOX_BYTES, 1024);
                            umma_f16(d_tmem, a_desc, b_desc, p.idesc, (kb > kb0 || k > 0) ? 1u : 0u);
                        }
                        umma_commit(smem_u32(&empty_bar[stage]));  // stage free once these MMAs finish
                        if (++stage == STAGES) {
                            stage = 0;
                            phase ^= 1;
                        }
                    }
                    if (!ok) break;
                    umma_commit(smem_u32(&tfull_bar[buf]));  // chunk sum ready for the epilogue
                    if (++buf == 2) {
                        buf = 0;
                        buf_phase ^= 1;
                    }
                }
            }
            // no MMA of this CTA may still be running when TMEM and shared memory are released
            umma_commit(smem_u32(drain_bar));
            if (!mbar_wait(smem_u32(drain_bar), 0, p.limit_ns)) record_error(p.status, kDevTimeoutDrain, abort_flag);
        }
        __syncwarp();
    } else {
        // ---------------------------------------------------------------- epilogue
        const int q = warp & 3;            // TMEM lane quarter this warp may access
        const int half = (warp - 2) >> 2;  // which 128 of the tile's 256 columns
        int buf = 0;
        uint32_t buf_phase = 0;
        float tot[EPI_COLS];
        int t_first = blockIdx.x;
        if (p.test_stall) {
            // test hook: a wait nothing will satisfy runs out and takes the abort path
            bool ok = mbar_wait(smem_u32(never_bar), 0, p.limit_ns);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok && lane == 0) record_error(p.status, kDevTimeoutEpilogue, abort_flag);
            t_first = p.num_tiles * p.nsplit;
        }
        for (int it = t_first; it < p.num_tiles * p.nsplit; it += gridDim.x) {
            const int t = it / p.nsplit, sl = it % p.nsplit;
            const int kb_beg = slice_begin(p, sl), kb_end = slice_begin(p, sl + 1);
            bool ok = true;
#pragma unroll
            for (int i = 0; i < EPI_COLS; ++i) tot[i] = 0.f;  // (no value lives on from the last tile)
            for (int ch = 0; ch < p.nchunks; ++ch) {
                if (kb_beg + ch * p.kc >= kb_end) break;  // as the MMA issuer
                ok = !*abort_flag && mbar_wait(smem_u32(&tfull_bar[buf]), buf_phase, p.limit_ns);
                ok = __all_sync(0xffffffffu, ok);
                if (!ok) {
                    if (lane == 0) record_error(p.status, kDevTimeoutEpilogue, abort_flag);
                    break;
                }
                tc_fence_after();
                const uint32_t t_addr =
                    tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(buf * BN + half * EPI_COLS);
#pragma unroll
                for (int j = 0; j < EPI_COLS / 32; ++j) {
                    uint32_t v[32];
                    tmem_ld_32x32b_x32(t_addr + j * 32, v);
                    tmem_ld_wait();
                    if (ch == 0) {
#pragma unroll
                        for (int i = 0; i < 32; ++i) tot[j * 32 + i] = __uint_as_float(v[i]);
                    } else {
#pragma unroll
                        for (int i = 0; i < 32; ++i) tot[j * 32 + i] = __fadd_rn(tot[j * 32 + i], __uint_as_float(v[i]));
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&tempty_bar[buf]));
                if (++buf == 2) {
                    buf = 0;
                    buf_phase ^= 1;
                }
            }
            if (!ok) break;
            const TileCoord tc = tile_coord(t, p.m_blocks, p.n_blocks);
            const int row = tc.m_blk * BM + q * 32 + lane;
            if (p.nsplit > 1) {
                // K-sliced tile (this CTA's only one): the partial product goes to this
                // CTA's shared memory; the cluster adds the slices after the loop
                const int rr = q * 32 + lane;
                uint8_t* prow = smem + rr * SPLIT_ROW_BYTES;
#pragma unroll
                for (int j = 0; j < EPI_COLS / 4; ++j) {
                    const int c = half * (EPI_COLS / 4) + j;
                    *reinterpret_cast<float4*>(prow + ((c ^ (rr & 7)) << 4)) =
                        make_float4(tot[4 * j], tot[4 * j + 1], tot[4 * j + 2], tot[4 * j + 3]);
                }
                continue;
            }
            if (p.c_tma) {
                store_rows_tma(&tmC, tot, epi_stage + (warp - 2) * EPI_STAGE_BYTES, tc.m_blk * BM + q * 32,
                               tc.n_blk * BN + half * EPI_COLS, p.M, p.N, lane);
            } else if (row < p.M && !p.epi_plain) {
                const int col0 = tc.n_blk * BN + half * EPI_COLS;
                const bool full = p.vec_store && col0 + EPI_COLS <= p.N;
#pragma unroll
                for (int j = 0; j < EPI_COLS; j += 4)
                    if (col0 + j < p.N)
                        epi_store4(p, (int64_t)row * p.ldc + col0 + j, p.N - (col0 + j), tot[j], tot[j + 1], tot[j + 2],
                                   tot[j + 3], full);
            } else if (row < p.M) {
                float* crow = static_cast<float*>(p.C) + (int64_t)row * p.ldc;
                const int col0 = tc.n_blk * BN + half * EPI_COLS;
                if (p.vec_store && col0 + EPI_COLS <= p.N) {
#pragma unroll
                    for (int j = 0; j < EPI_COLS; j += 4)
                        *reinterpret_cast<float4*>(crow + col0 + j) =
                            make_float4(tot[j], tot[j + 1], tot[j + 2], tot[j + 3]);
                } else {
#pragma unroll
                    for (int j = 0; j < EPI_COLS; ++j)
                        if (col0 + j < p.N) crow[col0 + j] = tot[j];
                }
            }
        }
        // the TMA stores of C have landed before the CTA retires
        if (p.c_tma && lane == 0) bulk_wait_group0();
        __syncwarp();
    }

    if (p.nsplit > 1) {
        // Every thread of every CTA of the cluster passes both barriers, on every path:
        // the first publishes all slices' partial tiles, the second keeps each CTA's
        // shared memory alive until the others have read it.
        __syncwarp();
        cluster_sync_all();
        if (warp >= 2) split_reduce_store(p, smem_u32(smem), (int)(blockIdx.x / p.nsplit), threadIdx.x - 64);
        __syncwarp();
        cluster_sync_all();
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, TMEM_COLS);
    }
}


// ============================================================================ CTA pair
// The same pipeline on a pair of CTAs (a cluster of two, one per SM of a TPC) with
// tcgen05's cta_group::2 MMAs: one instruction computes a 256 x 256 x 16 block, rows
// 0..127 into the even CTA's TMEM and rows 128..255 into the odd CTA's.  Each CTA stages
// only its own half of A (128 rows) and its own half of B (128 columns) in shared
// memory; the pair's tensor cores read both halves.  Per SM that is 32 KiB of operands
// per 64-deep k-block instead of 48 KiB, which is what limited the one-CTA kernel (its
// shared-memory data path was saturated by operand reads plus TMA fills).
// The even CTA's warp 1 issues every MMA; its commits arrive on barriers in both CTAs
// (multicast).  Both CTAs' TMA loads complete on the even CTA's "full" barrier.  The odd
// CTA's epilogue warps arrive remotely on the even CTA's "accumulator drained" barrier.
constexpr int P_STAGES_DEFAULT = 6;
constexpr int P_A_STAGE_BYTES = BM * BK * 2;                     // 16 KiB: this CTA's 128 rows of A
constexpr int P_B_STAGE_BYTES = (BN / 2) * BK * 2;               // 16 KiB: this CTA's 128 columns of B
constexpr int P_STAGE_BYTES = P_A_STAGE_BYTES + P_B_STAGE_BYTES; // per CTA
constexpr int p_smem_bytes(int stages) { return stages * P_STAGE_BYTES + EPI_STAGE_TOTAL + 1024 + 1024; }

// A cluster is one CTA pair computing 256 x 256 tiles; each CTA loads its own operand
// halves with plain (per-CTA) TMA loads.
template <int P_STAGES>
__global__ void __launch_bounds__(THREADS, 1)
tc_gemm_pair_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                    const __grid_constant__ CUtensorMap tmC, TcParams p)
{
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    uint8_t* smem = smem_raw + ((1024 - (raw & 1023)) & 1023);
    uint8_t* smem_a = smem;
    uint8_t* smem_b = smem + P_STAGES * P_A_STAGE_BYTES;
    uint8_t* epi_stage = smem + P_STAGES * P_STAGE_BYTES;  // [EPI_WARPS][32 rows][128 bytes]
    uint64_t* bars = reinterpret_cast<uint64_t*>(epi_stage + EPI_STAGE_TOTAL);
    uint64_t* full_bar = bars;                       // [P_STAGES] (used in the even CTA)
    uint64_t* empty_bar = bars + P_STAGES;           // [P_STAGES] (both CTAs, multicast)
    uint64_t* tfull_bar = bars + 2 * P_STAGES;       // [2] (both CTAs, multicast)
    uint64_t* tempty_bar = bars + 2 * P_STAGES + 2;  // [2] (used in the even CTA)
    uint64_t* drain_bar = bars + 2 * P_STAGES + 4;   // (both CTAs, multicast)
    uint64_t* never_bar = bars + 2 * P_STAGES + 5;   // never completes (test hook)
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bars + 2 * P_STAGES + 6);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);

    const int warp = threadIdx.x / 32;
    const int lane = threadIdx.x % 32;
    const uint32_t rank = cluster_ctarank();  // CTA within its pair
    const uint32_t leader = 0;                 // the pair's even CTA (issues its MMAs)
    const uint16_t pair_mask = 0x3;
    const int pair = blockIdx.x / 2;  // cluster index: walks pair tiles
    const int npairs = gridDim.x / 2;

    if (warp == 0 && lane == 0) {
        for (int s = 0; s < P_STAGES; ++s) {
            mbar_init(smem_u32(&full_bar[s]), 1);
            mbar_init(smem_u32(&empty_bar[s]), 1);  // the pair's commit
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(smem_u32(&tfull_bar[a]), 1);
            mbar_init(smem_u32(&tempty_bar[a]), 2 * EPI_WARPS);  // epilogue warps of both CTAs
        }
        mbar_init(smem_u32(drain_bar), 1);
        mbar_init(smem_u32(never_bar), 1);
        *abort_flag = 0;
        mbar_fence_init();
        prefetch_tensormap(&tmA);
        prefetch_tensormap(&tmB);
        if (p.c_tma) prefetch_tensormap(&tmC);
    }
    if (warp == 1) {
        tmem_alloc_pair(smem_u32(tmem_holder), TMEM_COLS);
        tc_fence_before();
    }
    __syncthreads();
    cluster_sync_all();  // the peer's barriers and TMEM exist before anything targets them
    tc_fence_after();
    const uint32_t tmem_base = *tmem_holder;
    bool aborted = false;

    if (warp == 0) {
        // ---------------------------------------------------------------- producer
        if (lane == 0) {
            const uint64_t pol_keep = l2_policy_evict_last();
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true;
            for (int it = pair; it < p.num_items && ok; it += npairs) {
                const PairItem w = pair_item(p, it);
                const TileCoord tc = tile_coord(w.t, p.m_blocks, p.n_blocks, p.group_m);
                for (int kb = w.kb0; kb < w.kb1; ++kb) {
                    if (!mbar_wait_cluster(smem_u32(&empty_bar[stage]), phase ^ 1, p.limit_ns, abort_flag)) {
                        record_error(p.status, kDevTimeoutProducer, abort_flag);
                        ok = false;
                        break;
                    }
                    const uint32_t fb_local = smem_u32(&full_bar[stage]);
                    const uint32_t fb_even = mapa_shared(fb_local, leader);
                    if (rank == 0) mbar_arrive_expect_tx(fb_local, 2 * P_STAGE_BYTES);
                    // A rows are read again by every tile of their raster group: keep them in L2
                    // (measured at 8192^3: DRAM reads 1084 -> 1018 MB with the C stores below
                    // marked evict-first; B marked evict-first instead re-read B: 1222+ MB)
                    tma_load_2d_pair_hint(smem_u32(smem_a + stage * P_A_STAGE_BYTES), &tmA, fb_even, kb * BK,
                                          tc.m_blk * (2 * BM) + (int)rank * BM, pol_keep);
                    uint8_t* b_dst = smem_b + stage * P_B_STAGE_BYTES;
#pragma unroll
                    for (int j = 0; j < (BN / 2) / B_BOX_N; ++j)
                        tma_load_2d_pair(smem_u32(b_dst + j * B_BOX_BYTES), &tmB, fb_even,
                                         tc.n_blk * BN + (int)rank * (BN / 2) + j * B_BOX_N, kb * BK);
                    if (++stage == P_STAGES) {
                        stage = 0;
                        phase ^= 1;
                    }
                }
            }
            if (!ok) aborted = true;
        }
        __syncwarp();
    } else if (warp == 1) {
        // ---------------------------------------------------------------- MMA issuer (even CTA)
        if (lane == 0 && rank == 0) {
            int stage = 0;
            uint32_t phase = 0;
            int buf = 0;
            uint32_t buf_phase = 0;
            bool ok = true;
            const uint32_t a_base = smem_u32(smem_a), b_base = smem_u32(smem_b);
            const uint32_t idesc = p.idesc;
            for (int it = pair; it < p.num_items && ok; it += npairs) {
                const PairItem w = pair_item(p, it);
                for (int ch = 0; ch < p.nchunks && ok; ++ch) {
                    const int kb0 = w.kb0 + ch * p.kc;
                    if (kb0 >= w.kb1) break;  // a K slice has fewer chunks
                    if (!mbar_wait_cluster(smem_u32(&tempty_bar[buf]), buf_phase ^ 1, p.limit_ns, abort_flag)) {
                        record_error(p.status, kDevTimeoutMma, abort_flag);
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t d_tmem = tmem_base + (uint32_t)(buf * BN);
                    const int kb1 = min(kb0 + p.kc, w.kb1);
                    for (int kb = kb0; kb < kb1; ++kb) {
                        if (!mbar_wait_cluster(smem_u32(&full_bar[stage]), phase, p.limit_ns, abort_flag)) {
                            record_error(p.status, kDevTimeoutMma, abort_flag);
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        const uint32_t a_st = a_base + stage * P_A_STAGE_BYTES;
                        const uint32_t b_st = b_base + stage * P_B_STAGE_BYTES;
#pragma unroll
                        for (int k = 0; k < BK / UMMA_K; ++k) {
                            const uint64_t a_desc = smem_desc_sw128(a_st + k * UMMA_K * 2, 16, 1024);
                            const uint64_t b_desc = smem_desc_sw128(b_st + k * UMMA_K * 128, B_BOX_BYTES, 1024);
                            umma_f16_pair(d_tmem, a_desc, b_desc, idesc, (kb > kb0 || k > 0) ? 1u : 0u);
                        }
                        umma_commit_mask(smem_u32(&empty_bar[stage]), pair_mask);  // both CTAs that filled it
                        if (++stage == P_STAGES) {
                            stage = 0;
                            phase ^= 1;
                        }
                    }
                    if (!ok) break;
                    umma_commit_mask(smem_u32(&tfull_bar[buf]), pair_mask);
                    if (++buf == 2) {
                        buf = 0;
                        buf_phase ^= 1;
                    }
                }
            }
            if (!ok) aborted = true;
            umma_commit_mask(smem_u32(drain_bar), pair_mask);  // reaches both CTAs once every MMA is done
        }
        if (lane == 0) {
            if (!mbar_wait_cluster(smem_u32(drain_bar), 0, p.limit_ns, nullptr)) {
                record_error(p.status, kDevTimeoutDrain, abort_flag);
                aborted = true;
            }
        }
        __syncwarp();
    } else {
        // ---------------------------------------------------------------- epilogue (both CTAs)
        const int q = warp & 3;
        const int half = (warp - 2) >> 2;
        int buf = 0;
        uint32_t buf_phase = 0;
        float tot[EPI_COLS];
        int t_first = pair;
        if (p.test_stall) {
            // test hook: a wait nothing will satisfy runs out and takes the abort path
            bool ok = mbar_wait_cluster(smem_u32(never_bar), 0, p.limit_ns, nullptr);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok && lane == 0) record_error(p.status, kDevTimeoutEpilogue, abort_flag);
            aborted = true;
            t_first = p.num_items;
        }
        for (int it = t_first; it < p.num_items; it += npairs) {
            const PairItem w = pair_item(p, it);
            const int t = w.t;
            bool ok = true;
#pragma unroll
            for (int i = 0; i < EPI_COLS; ++i) tot[i] = 0.f;  // (no value lives on from the last item)
            for (int ch = 0; ch < p.nchunks; ++ch) {
                if (w.kb0 + ch * p.kc >= w.kb1) break;  // as the MMA issuer
                ok = mbar_wait_cluster(smem_u32(&tfull_bar[buf]), buf_phase, p.limit_ns, abort_flag);
                ok = __all_sync(0xffffffffu, ok);
                if (!ok) {
                    if (lane == 0) record_error(p.status, kDevTimeoutEpilogue, abort_flag);
                    break;
                }
                tc_fence_after();
                const uint32_t t_addr =
                    tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(buf * BN + half * EPI_COLS);
#pragma unroll
                for (int j = 0; j < EPI_COLS / 32; ++j) {
                    uint32_t v[32];
                    tmem_ld_32x32b_x32(t_addr + j * 32, v);
                    tmem_ld_wait();
                    if (ch == 0) {
#pragma unroll
                        for (int i = 0; i < 32; ++i) tot[j * 32 + i] = __uint_as_float(v[i]);
                    } else {
#pragma unroll
                        for (int i = 0; i < 32; ++i) tot[j * 32 + i] = __fadd_rn(tot[j * 32 + i], __uint_as_float(v[i]));
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive_cluster(mapa_shared(smem_u32(&tempty_bar[buf]), leader));
                if (++buf == 2) {
                    buf = 0;
                    buf_phase ^= 1;
                }
            }
            if (!ok) {
                aborted = true;
                break;
            }
            const TileCoord tc = tile_coord(t, p.m_blocks, p.n_blocks, p.group_m);
            if (w.sl >= 0 && p.rem_direct) {
                // a last-wave tile in two K slices, plain fp32 C: the part's first slice to
                // finish stores it, the second adds itself in L2 (a + b = b + a: the same
                // bits whichever comes first)
                const int64_t part = ((int64_t)(t - p.rem_first) * 2 + rank) * EPI_WARPS + (warp - 2);
                if (!in_range(part, (int64_t)(p.num_tiles - p.rem_first) * 2 * EPI_WARPS)) continue;
                int n = 0;
                if (lane == 0) {
                    n = tagged_arrive(p.rem_cnt + part, p.rem_seq);
                    if (n == 0) record_error(p.status, kDevTimeoutEpilogue, abort_flag);
                }
                n = __shfl_sync(0xffffffffu, n, 0);
                uint8_t* stg = epi_stage + (warp - 2) * EPI_STAGE_BYTES;
                const int row0 = tc.m_blk * (2 * BM) + (int)rank * BM + q * 32;
                const int col0 = tc.n_blk * BN + half * EPI_COLS;
                if (n == 1) {
                    store_rows_tma<false>(&tmC, tot, stg, row0, col0, p.M, p.N, lane);
                    if (lane == 0) {
                        bulk_wait_group0();  // the part is in C
                        fence_proxy_async_global();
                        __threadfence();
                        st_release_gpu(p.rem_flag + part, p.rem_seq);
                    }
                    __syncwarp();
                } else if (n == 2) {
                    // the first slice's warp has counted itself, so it is running and
                    // publishes without waiting on anything; the wait is bounded all the same
                    bool ok2 = true;
                    if (lane == 0) {
                        const uint64_t t0 = global_timer();
                        while (ld_acquire_gpu(p.rem_flag + part) != p.rem_seq) {
                            if (*abort_flag || global_timer() - t0 > p.limit_ns) {
                                record_error(p.status, kDevTimeoutEpilogue, abort_flag);
                                ok2 = false;
                                break;
                            }
                            __nanosleep(64);
                        }
                        fence_proxy_async_global();
                    }
                    ok2 = __shfl_sync(0xffffffffu, ok2 ? 1 : 0, 0) != 0;
                    if (ok2) store_rows_tma<true>(&tmC, tot, stg, row0, col0, p.M, p.N, lane);
                }
                continue;
            }
            // a K slice of a last-wave tile: only the part's last slice to finish stores C
            if (w.sl >= 0 && !rem_slice_combine(p, tot, t - p.rem_first, w.sl, (int)rank, warp - 2, lane, p.status,
                                                abort_flag))
                continue;
            const int row = tc.m_blk * (2 * BM) + (int)rank * BM + q * 32 + lane;
            if (p.c_tma) {
                // C is written once and not read here: first out of L2
                store_rows_tma(&tmC, tot, epi_stage + (warp - 2) * EPI_STAGE_BYTES, tc.m_blk * (2 * BM) + (int)rank * BM + q * 32,
                               tc.n_blk * BN + half * EPI_COLS, p.M, p.N, lane, l2_policy_evict_first());
            } else if (row < p.M && !p.epi_plain) {
                const int col0 = tc.n_blk * BN + half * EPI_COLS;
                const bool full = p.vec_store && col0 + EPI_COLS <= p.N;
#pragma unroll
                for (int j = 0; j < EPI_COLS; j += 4)
                    if (col0 + j < p.N)
                        epi_store4(p, (int64_t)row * p.ldc + col0 + j, p.N - (col0 + j), tot[j], tot[j + 1], tot[j + 2],
                                   tot[j + 3], full);
            } else if (row < p.M) {
                float* crow = static_cast<float*>(p.C) + (int64_t)row * p.ldc;
                const int col0 = tc.n_blk * BN + half * EPI_COLS;
                if (p.vec_store && col0 + EPI_COLS <= p.N) {
#pragma unroll
                    for (int j = 0; j < EPI_COLS; j += 4)
                        *reinterpret_cast<float4*>(crow + col0 + j) =
                            make_float4(tot[j], tot[j + 1], tot[j + 2], tot[j + 3]);
                } else {
#pragma unroll
                    for (int j = 0; j < EPI_COLS; ++j)
                        if (col0 + j < p.N) crow[col0 + j] = tot[j];
                }
            }
        }
        // the TMA stores of C have landed before the CTA retires
        if (p.c_tma && lane == 0) bulk_wait_group0();
        __syncwarp();
    }

    // after an abort, give copies and MMAs already issued time to land before the pair's
    // shared memory and TMEM are released
    if (__syncthreads_or(aborted ? 1 : 0)) grace_period(2000000ull);
    tc_fence_before();
    __syncthreads();
    cluster_sync_all();  // no MMA, remote arrival or TMA of the pair still targets this CTA
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc_pair(tmem_base, TMEM_COLS);
    }
}

// ------------------------------------------------------------------ host side

// Row-major [rows][cols] 16-bit matrix with row stride `ld` elements; box = box_cols x box_rows.
bool encode_2d(CUtensorMap* map, const void* base, bool bf16, uint64_t rows, uint64_t cols, uint64_t ld,
               uint32_t box_cols, uint32_t box_rows)
{
    auto enc = tensor_map_encoder();
    if (!enc) return false;
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {ld * 2};
    cuuint32_t box[2] = {box_cols, box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2,
                     const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                     CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// Row-major [rows][cols] fp32 C with row stride `ld` floats, stored in 32 x 32 boxes of
// 128-byte rows in the 128-byte-swizzle layout.
bool encode_c_f32(CUtensorMap* map, void* base, uint64_t rows, uint64_t cols, uint64_t ld)
{
    auto enc = tensor_map_encoder();
    if (!enc) return false;
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {ld * 4};
    cuuint32_t box[2] = {32, 32};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, base, dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

}  // namespace

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder()
{
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    });
    return fn;
}

namespace {

// Clusters of `S` single-CTA kernels that can be resident at once (0: none), per size.
// Cached per process: every device a process drives is taken to be the same part.
int split_clusters_fit(int S)
{
    static std::atomic<int> cache[MAX_SPLIT + 1];
    static std::once_flag once;
    std::call_once(once, [] {
        for (auto& c : cache) c.store(-1);
    });
    int v = cache[S].load();
    if (v >= 0) return v;
    v = 0;
    if (cudaFuncSetAttribute(tc_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES) ==
            cudaSuccess &&
        cudaFuncSetAttribute(tc_gemm_kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) == cudaSuccess) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(S, 1, 1);
        cfg.blockDim = dim3(THREADS, 1, 1);
        cfg.dynamicSmemBytes = SMEM_BYTES;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = S;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        if (cudaOccupancyMaxActiveClusters(&v, tc_gemm_kernel, &cfg) != cudaSuccess) v = 0;
    }
    cudaGetLastError();  // a refused size leaves no sticky error behind
    cache[S].store(v);
    return v;
}

// K slices for a product whose 128 x 256 tiles fill under half the SMs: the largest
// power of two that keeps every slice at least 4 k-blocks deep, the grid within the SMs
// and every tile's cluster resident at once.  1 = no split.
int choose_split(int64_t tiles, int64_t k_blocks, int num_sms)
{
    if (2 * tiles > num_sms) return 1;
    for (int S = MAX_SPLIT; S >= 2; S /= 2)
        if (k_blocks >= 4 * S && tiles * S <= num_sms && split_clusters_fit(S) >= tiles) return S;
    return 1;
}

}  // namespace

namespace {

// Clusters of the CTA-pair kernel resident at once (0: unknown).
// Cached per process: every device a process drives is taken to be the same part.
int pair_clusters_fit()
{
    static std::atomic<int> cache{-1};
    int v = cache.load();
    if (v >= 0) return v;
    v = 0;
    auto kern = tc_gemm_pair_kernel<P_STAGES_DEFAULT>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, p_smem_bytes(P_STAGES_DEFAULT)) ==
        cudaSuccess) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(2, 1, 1);
        cfg.blockDim = dim3(THREADS, 1, 1);
        cfg.dynamicSmemBytes = p_smem_bytes(P_STAGES_DEFAULT);
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 2;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        if (cudaOccupancyMaxActiveClusters(&v, kern, &cfg) != cudaSuccess) v = 0;
    }
    cudaGetLastError();
    cache.store(v);
    return v;
}

// How a product is laid on the tensor-core kernels.
struct TcPlan {
    bool pair = false;
    int64_t tiles = 0;    // output tiles of the chosen kernel
    int clusters = 0;     // pair kernels: clusters launched
    int rem_first = 0;    // pair kernel: first split tile (tiles = none)
    int rem_split = 1;    // pair kernel: K slices of each last-wave tile
    bool c_tma = false;   // plain fp32 C with 16-byte aligned rows: TMA stores
    bool rem_direct = false;  // two slices added straight into C (no partial workspace)
    int single_split = 1;     // single-CTA kernel: K slices per tile on a cluster (1 = none)
};

TcPlan plan_tc(const TcArgs& a, int num_sms, int pair_mode)
{
    TcPlan pl;
    pl.c_tma = a.epi.plain() && (reinterpret_cast<uintptr_t>(a.C) & 15) == 0 && a.ldc % 4 == 0;
    pl.pair = (pair_mode == 2) || (pair_mode == 0 && a.M > BM && num_sms >= 2);
    const int64_t n_blocks = (a.N + BN - 1) / BN;
    const int64_t k_blocks = (a.K + BK - 1) / BK;
    const int64_t single_tiles = ((a.M + BM - 1) / BM) * n_blocks;
    if (!pl.pair) {
        pl.tiles = single_tiles;
        // M <= 128 with few tiles (chosen tiles only; the stall hook runs unsplit)
        if (pair_mode == 0 && !a.test_stall && a.M <= BM) pl.single_split = choose_split(single_tiles, k_blocks, num_sms);
        return pl;
    }
    pl.tiles = ((a.M + 2 * BM - 1) / (2 * BM)) * n_blocks;
    // a persistent grid must be co-resident: clusters are placed within one GPC each, so
    // fewer than num_sms / 2 of them may fit
    int64_t clusters = num_sms / 2;
    const int fit = pair_clusters_fit();
    if (fit > 0 && fit < clusters) clusters = fit;
    pl.rem_first = (int)pl.tiles;
    // the tiles of a last wave that leaves pairs idle are cut along K (CTA pairs only;
    // the stall hook runs unsplit).  Adding a tile's slices costs about 7 us (each part
    // published to L2, counted, the others read back), so every slice keeps at least 32
    // k-blocks (about 11 us of MMAs on a pair): shorter slices measured slower than none.
    const int64_t r = pl.tiles % clusters;  // tiles of the last wave (all of them if fewer than pairs)
    if (!a.test_stall && r != 0) {
        int64_t sp = clusters / r;
        if (sp > MAX_REM_SPLIT) sp = MAX_REM_SPLIT;
        while (sp > 1 && k_blocks / sp < 32) --sp;
        if (sp >= 2) {
            pl.rem_first = (int)(pl.tiles - r);
            pl.rem_split = (int)sp;
            pl.rem_direct = (sp == 2) && pl.c_tma;
        }
    }
    // (Small products with M > 128 stay on pairs even when the single-CTA kernel's K split
    // would keep more SMs busy: its exchange through distributed shared memory costs about
    // 10 us, more than it saves below ~10 GFLOP, e.g. 0.017 -> 0.019 ms at 1024^3.)
    const int64_t items = pl.rem_first + (pl.tiles - pl.rem_first) * pl.rem_split;
    pl.clusters = (int)(items < clusters ? items : clusters);
    return pl;
}

}  // namespace

TcWorkspace tc_workspace_need(const TcArgs& a, int num_sms, int pair_mode)
{
    TcWorkspace w;
    if (a.M <= 0 || a.N <= 0 || a.K <= 0) return w;
    const TcPlan pl = plan_tc(a, num_sms, pair_mode);
    if (pl.rem_split < 2) return w;
    const int64_t split_tiles = pl.tiles - pl.rem_first;
    w.floats = pl.rem_direct ? 0 : split_tiles * pl.rem_split * 2 * EPI_WARPS * REM_PART_FLOATS;
    w.counters = split_tiles * 2 * EPI_WARPS;
    return w;
}

int launch_tc_gemm(const TcArgs& a, int num_sms, int* dev_status, uint64_t wait_limit_ns, int kc_blocks,
                   int pair_mode, cudaStream_t stream, int* launches)
{
    // sizes must fit the kernel's 32-bit tile arithmetic and TMA's 32-bit coordinates
    if (a.M > (1ll << 31) - BM || a.N > (1ll << 31) - BN || a.K > (1ll << 31) - BK) return GEMM_ERR_UNSUPPORTED;
    CUtensorMap tmA, tmB;
    const bool bf16 = a.is_bf16 != 0;
    if (!encode_2d(&tmA, a.A, bf16, (uint64_t)a.M, (uint64_t)a.K, (uint64_t)a.lda, BK, BM) ||
        !encode_2d(&tmB, a.B, bf16, (uint64_t)a.K, (uint64_t)a.N, (uint64_t)a.ldb, B_BOX_N, BK))
        return GEMM_ERR_CUDA;
    if (cudaFuncSetAttribute(tc_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES) !=
        cudaSuccess)
        return GEMM_ERR_CUDA;
    TcParams p;
    p.M = (int)a.M;
    p.N = (int)a.N;
    p.K = (int)a.K;
    p.C = a.C;
    p.ldc = a.ldc;
    p.m_blocks = (int)((a.M + BM - 1) / BM);
    p.n_blocks = (int)((a.N + BN - 1) / BN);
    const int64_t tiles = (int64_t)p.m_blocks * p.n_blocks;
    if (tiles > 0x7fffffffLL) return GEMM_ERR_UNSUPPORTED;
    p.num_tiles = (int)tiles;
    p.k_blocks = (int)((a.K + BK - 1) / BK);
    p.kc = kc_blocks > 0 ? kc_blocks : 16;
    p.group_m = GROUP_M;
    p.nsplit = 1;
    p.nchunks = (p.k_blocks + p.kc - 1) / p.kc;
    p.idesc = make_idesc(bf16);
    // vector stores: 4 outputs per access (16 bytes fp32, 8 bytes bf16/fp16)
    const uintptr_t c_align = (a.epi.c_dtype == GEMM_F32) ? 15 : 7;
    p.vec_store = ((reinterpret_cast<uintptr_t>(a.C) & c_align) == 0) && (a.ldc % 4 == 0);
    p.alpha = a.epi.alpha;
    p.beta = a.epi.beta;
    p.c_dtype = a.epi.c_dtype;
    p.epi_plain = a.epi.plain() ? 1 : 0;
    // plain fp32 C with 16-byte aligned rows goes out through TMA stores
    CUtensorMap tmC = tmA;  // (unused unless c_tma)
    p.c_tma = p.epi_plain && (reinterpret_cast<uintptr_t>(a.C) & 15) == 0 && a.ldc % 4 == 0 &&
              encode_c_f32(&tmC, a.C, (uint64_t)a.M, (uint64_t)a.N, (uint64_t)a.ldc);
    p.status = dev_status;
    p.limit_ns = wait_limit_ns;
    p.test_stall = a.test_stall;
    // CTA pairs: 256 x 256 tiles on clusters of two; single CTAs: 128 x 256 tiles
    const TcPlan pl = plan_tc(a, num_sms, pair_mode);
    p.num_items = p.num_tiles;
    p.rem_first = p.num_tiles;
    p.rem_split = 1;
    p.rem_ws = nullptr;
    p.rem_cnt = nullptr;
    p.rem_flag = nullptr;
    p.rem_seq = 0;
    p.rem_direct = 0;
    if (pl.pair) {
        const int cl = 2;  // CTAs per cluster
        p.m_blocks = (int)((a.M + cl * BM - 1) / (cl * BM));
        const int64_t ctiles = (int64_t)p.m_blocks * p.n_blocks;
        p.num_tiles = (int)ctiles;
        p.num_items = p.num_tiles;
        p.rem_first = p.num_tiles;
        if (pl.rem_split > 1 && (pl.rem_direct || a.rem_ws) && a.rem_cnt && a.rem_flag && a.rem_seq &&
            pl.c_tma == (p.c_tma != 0)) {
            p.rem_first = pl.rem_first;
            p.rem_split = pl.rem_split;
            p.num_items = pl.rem_first + (p.num_tiles - pl.rem_first) * pl.rem_split;
            p.rem_ws = a.rem_ws;
            p.rem_cnt = a.rem_cnt;
            p.rem_flag = a.rem_flag;
            p.rem_seq = a.rem_seq;
            p.rem_direct = pl.rem_direct ? 1 : 0;
        }
        p.idesc = make_idesc(bf16, 2 * BM);
        const int clusters = pl.clusters;
        // 6 stages of 32 KiB; 7 measured no faster.  Raster groups of 2048 rows of C
        // (8 pair tiles) measured best among 512 .. 4096 rows, within run-to-run noise.
        constexpr int stages = P_STAGES_DEFAULT;
        p.group_m = 8;
        auto kern = tc_gemm_pair_kernel<stages>;
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, p_smem_bytes(stages)) !=
            cudaSuccess)
            return GEMM_ERR_CUDA;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(cl * clusters, 1, 1);
        cfg.blockDim = dim3(THREADS, 1, 1);
        cfg.dynamicSmemBytes = p_smem_bytes(stages);
        cfg.stream = stream;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = cl;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        if (cudaLaunchKernelEx(&cfg, kern, tmA, tmB, tmC, p) != cudaSuccess) return GEMM_ERR_CUDA;
        *launches += 1;
        return GEMM_OK;
    }
    // few tiles (see plan_tc): K slices of a tile on a cluster of CTAs, one slice each,
    // added through distributed shared memory in slice order
    const int S = pl.single_split;
    if (S > 1) {
        p.nsplit = S;
        const int depth = (p.k_blocks + S - 1) / S;  // the deepest slice
        p.nchunks = (depth + p.kc - 1) / p.kc;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)(tiles * S), 1, 1);
        cfg.blockDim = dim3(THREADS, 1, 1);
        cfg.dynamicSmemBytes = SMEM_BYTES;
        cfg.stream = stream;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = S;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        if (S > 8 && cudaFuncSetAttribute(tc_gemm_kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) !=
                         cudaSuccess)
            return GEMM_ERR_CUDA;
        if (cudaLaunchKernelEx(&cfg, tc_gemm_kernel, tmA, tmB, tmC, p) != cudaSuccess) return GEMM_ERR_CUDA;
        *launches += 1;
        return GEMM_OK;
    }
    const int grid = (int)(tiles < num_sms ? tiles : num_sms);
    tc_gemm_kernel<<<grid, THREADS, SMEM_BYTES, stream>>>(tmA, tmB, tmC, p);
    if (cudaGetLastError() != cudaSuccess) return GEMM_ERR_CUDA;
    *launches += 1;
    return GEMM_OK;
}

}  // namespace gemm_gb300
