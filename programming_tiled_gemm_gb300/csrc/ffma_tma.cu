// fp32 GEMM on the FP32 pipe as ONE persistent launch whose tiles arrive by TMA.
//
// The arithmetic is the register-blocked outer product of "Learning to develop for GPU with
// GEMM as the example", section "Improving the solution and balancing memory work": every
// thread owns an 8 x 16 block of accumulators and, per k, multiplies 8 values of A by 16
// values of B from shared memory (packed fp32 FMAs, fma.rn.f32x2, two independent
// round-to-nearest FMAs per instruction).  The staging through shared memory is that of
// sections "Making the GPU implementation better" and "How loading into local memory is
// organised", with the block's cooperative copy replaced by the Tensor Memory Accelerator:
//   * one lane issues, per 32-deep k-tile, a 128 x 32 box of A and a 32 x 256 box of B into
//     a ring of stages; each stage completes on an mbarrier ("full"), and the eight warps
//     release it on another ("empty") once they have read it.  No block-wide barrier sits in
//     the main loop, and TMA fills rows past M, columns past N and k past K with zeros, so
//     the main loop has no predicates;
//   * A lands as [row][k] in the 128-byte swizzle layout.  A thread's eight rows are spaced
//     eight apart, so the eight rows a warp reads at once fall into eight different bank
//     groups (section "How to do even better": conflict-free shared-memory access, here
//     without a transposing store).  Each A value is loaded into both halves of the
//     register pair the packed FMA takes, so no register moves duplicate it (measured:
//     about 3 % of the FMA pipe);
//   * the grid is persistent, one CTA per SM ("CUDA overview: performance surprises",
//     section "Parallelism first"), walking tiles in grouped raster order (GROUP_M tile
//     rows sweep the tile columns together, for L2 reuse of B).  The work is handed out
//     dynamically: after its first item a CTA takes the next one from a per-launch
//     counter, so SMs that run slower (measured: up to 7 % on some SMs) take fewer items.
//     The producer runs ahead across item boundaries, so the next item's first k-tiles
//     load during an epilogue, and passes each item's index to the consumer warps through
//     a small ring in shared memory;
//   * a last, partial wave of tiles is cut along K into `split` slices (work items of
//     their own, spread over the CTAs).  Every slice publishes its partial tile to a
//     workspace and counts itself on a per-tile counter tagged with the launch; the slice
//     that counts last adds all partials in slice order (fixed order: deterministic) and
//     stores C.  Nothing waits for another CTA.
// Every mbarrier wait is bounded (wall clock) and reports to the handle's status word.
#include "internal.h"
#include "ptx.h"

namespace gemm_gb300 {

GEMM_DEBUG_UNIT(ffma_tma)

namespace {

constexpr int PT_THREADS = 256;
constexpr int PT_WARPS = PT_THREADS / 32;
constexpr int PT_BM = 128, PT_BN = 256, PT_BK = 32;
constexpr int PT_STAGES = 4;
constexpr int PT_AHEAD = PT_STAGES - 2;  // k-tiles the producer keeps issued ahead of the consumers
constexpr int PT_A_STAGE = PT_BM * PT_BK * 4;  // 16 KiB: [128 rows][32 k], 128-byte swizzle
constexpr int PT_B_STAGE = PT_BK * PT_BN * 4;  // 32 KiB: [32 k][256 columns]
constexpr int PT_STAGE = PT_A_STAGE + PT_B_STAGE;
constexpr int PT_RING = 8;  // item indices the producer may hand out ahead of the consumers
constexpr int PT_SMEM = PT_STAGES * PT_STAGE + 1024 + 512;  // + alignment slack + barriers and ring
constexpr int PT_TILE_FLOATS = PT_BM * PT_BN;
constexpr int PT_MAX_SPLIT = 16;

struct PtParams {
    int M, N, K;  // (32-bit: the host keeps sizes and leading dimensions below 2^31)
    int m_tiles, n_tiles, group_m;
    int num_tiles;
    int split_first;  // tiles [split_first, num_tiles) run as `split` K slices each
    int split;
    int kt_per_slice;  // 32-deep k-tiles per slice
    int k_tiles;
    int num_items;  // split_first + (num_tiles - split_first) * split
    float* C;
    int ldc;
    int vec_out;              // C 16-byte aligned with ldc % 4 == 0: float4 stores
    float* ws;                // [split tile][slice][256 threads x 32 float4] partial tiles
    unsigned long long* cnt;  // one tagged arrival counter per split tile, then the item counter
    uint32_t seq;             // this launch's tag (nonzero)
    int* status;
    uint64_t limit_ns;
    int test_stall;  // test hook: every warp first waits on a barrier nothing arrives on
};

struct PtItem {
    int tile, sl, kt0, kt1;  // sl = -1: the whole tile
};

__device__ __forceinline__ PtItem pt_item(const PtParams& p, int it)
{
    PtItem w;
    if (it < p.split_first) {
        w.tile = it;
        w.sl = -1;
        w.kt0 = 0;
        w.kt1 = p.k_tiles;
    } else {
        const int j = it - p.split_first;
        w.tile = p.split_first + j / p.split;
        w.sl = j % p.split;
        w.kt0 = w.sl * p.kt_per_slice;
        w.kt1 = min(w.kt0 + p.kt_per_slice, p.k_tiles);
    }
    return w;
}

// Grouped raster: group_m consecutive tile rows sweep the tile columns together.
__device__ __forceinline__ void pt_tile_coord(const PtParams& p, int t, int& mt, int& nt)
{
    const int width = p.group_m * p.n_tiles;
    const int first_m = (t / width) * p.group_m;
    const int gsize = min(p.m_tiles - first_m, p.group_m);
    mt = first_m + (t % width) % gsize;
    nt = (t % width) / gsize;
}

__device__ __forceinline__ void pt_fail(int* status, int code, volatile int* abort_flag)
{
    atomicCAS(status, 0, code);
    *abort_flag = 1;
}

__global__ void __launch_bounds__(PT_THREADS, 1)
ffma_persistent_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB, PtParams p)
{
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    uint8_t* smem = smem_raw + ((1024 - (raw & 1023)) & 1023);
    const uint32_t sa = smem_u32(smem);                        // [STAGES][A_STAGE]
    const uint32_t sb = sa + PT_STAGES * PT_A_STAGE;           // [STAGES][B_STAGE]
    uint64_t* full_bar = reinterpret_cast<uint64_t*>(smem + PT_STAGES * PT_STAGE);
    uint64_t* empty_bar = full_bar + PT_STAGES;
    uint64_t* item_bar = empty_bar + PT_STAGES;  // [PT_RING]: the ring slot's item index is written
    uint64_t* never_bar = item_bar + PT_RING;    // never completes (test hook)
    volatile int* abort_flag = reinterpret_cast<volatile int*>(never_bar + 1);
    volatile int* bcast = abort_flag + 1;
    volatile int* item_ring = bcast + 1;  // [PT_RING]

    const int tid = threadIdx.x;
    const int warp = tid / 32, lane = tid % 32;
    if (tid == 0) {
        for (int s = 0; s < PT_STAGES; ++s) {
            mbar_init(smem_u32(&full_bar[s]), 1);
            mbar_init(smem_u32(&empty_bar[s]), PT_WARPS);
        }
        for (int r = 0; r < PT_RING; ++r) mbar_init(smem_u32(&item_bar[r]), 1);
        mbar_init(smem_u32(never_bar), 1);
        *abort_flag = 0;
        mbar_fence_init();
        prefetch_tensormap(&tmA);
        prefetch_tensormap(&tmB);
    }
    __syncthreads();

    // ---------------------------------------------------------------- producer (thread 0)
    // It takes this CTA's items (the first is blockIdx.x, every later one comes from the
    // launch's item counter), publishes each item's index in the ring for the consumers,
    // and walks the items' k-tiles in the order the consumers do.
    int p_item = 0, p_kt = 0, p_kt1 = 0, p_m0 = 0, p_n0 = 0;
    // A rows are read again by every tile of their raster group: keep them in L2
    const uint64_t pol_keep = l2_policy_evict_last();
    uint32_t p_items = 0;                       // items published so far (the sentinel included)
    uint32_t p_count = 0;                       // loads issued so far
    uint32_t issued_mask = 0, last_parity = 0;  // per stage: issued at all, parity of the last load
    bool p_done = false;
    auto p_publish = [&](int it) {  // ring slot p_items % RING <- it (it >= num_items: no more work)
        item_ring[p_items % PT_RING] = it;
        mbar_arrive(smem_u32(&item_bar[p_items % PT_RING]));  // release: the index is visible
        ++p_items;
    };
    auto p_next = [&](bool first) {
        if (first) {
            p_item = blockIdx.x;
        } else {
            const int n = tagged_arrive(p.cnt + (p.num_tiles - p.split_first), p.seq);
            p_item = n > 0 ? (int)gridDim.x + n - 1 : p.num_items;
            if (n == 0) pt_fail(p.status, kDevTimeoutProducer, abort_flag);
        }
        if (p_item >= p.num_items) {
            p_done = true;
            p_publish(p.num_items);
            return;
        }
        const PtItem w = pt_item(p, p_item);
        int mt, nt;
        pt_tile_coord(p, w.tile, mt, nt);
        p_kt = w.kt0;
        p_kt1 = w.kt1;
        p_m0 = mt * PT_BM;
        p_n0 = nt * PT_BN;
        p_publish(p_item);
    };
    // issue the next k-tile's loads, if any (false: gave up waiting for a free stage)
    auto produce = [&]() -> bool {
        if (p_done) return true;
        const int slot = (int)(p_count % PT_STAGES);
        const uint32_t use = p_count / PT_STAGES;
        if (use > 0 && !mbar_wait(smem_u32(&empty_bar[slot]), (use & 1) ^ 1, p.limit_ns, abort_flag)) {
            pt_fail(p.status, kDevTimeoutProducer, abort_flag);
            return false;
        }
        const uint32_t fb = smem_u32(&full_bar[slot]);
        mbar_arrive_expect_tx(fb, PT_STAGE);
        tma_load_2d_hint(sa + slot * PT_A_STAGE, &tmA, fb, p_kt * PT_BK, p_m0, pol_keep);
        tma_load_2d(sb + slot * PT_B_STAGE, &tmB, fb, p_n0, p_kt * PT_BK);
        issued_mask |= 1u << slot;
        last_parity = (last_parity & ~(1u << slot)) | ((use & 1) << slot);
        ++p_count;
        if (++p_kt == p_kt1) p_next(false);
        return true;
    };

    bool aborted = false;
    bool stalled = false;
    if (p.test_stall) {
        // test hook: a wait nothing will satisfy runs out and takes the abort path
        const bool got = mbar_wait(smem_u32(never_bar), 0, p.limit_ns, abort_flag);
        if (!got && lane == 0) pt_fail(p.status, kDevTimeoutMma, abort_flag);
        stalled = true;
    } else if (tid == 0) {
        p_next(true);
        for (int i = 0; i < PT_AHEAD && !aborted; ++i) aborted = !produce();
    }

    // ---------------------------------------------------------------- consumers (all warps)
    const int wm = warp / 4, wn = warp % 4;  // 2 x 4 warps of 64 x 64
    const int ty = lane / 4, tx = lane % 4;  // 8 x 4 lanes
    // rows wm*64 + ty + 8 i (i = 0..7): in the 128-byte swizzle, the 16-byte chunk c of row r
    // sits at chunk c ^ (r & 7), and r & 7 = ty for all eight rows
    const uint32_t a_row = sa + (uint32_t)(wm * 64 + ty) * (PT_BK * 4);
    const uint32_t a_sw = (uint32_t)ty;
    const uint32_t b_col = (uint32_t)(wn * 64 + tx * 4) * 4;  // columns b + 16 h + {0..3}, h = 0..3
    uint32_t c_count = 0;  // k-tiles consumed so far

    float2 acc[8][8];  // acc[i][2h + e] = columns (16 h + 2 e, + 1) of row i
    for (uint32_t j = 0; !stalled; ++j) {
        // the j-th item of this CTA, as the producer published it
        bool have = mbar_wait(smem_u32(&item_bar[j % PT_RING]), (j / PT_RING) & 1, p.limit_ns, abort_flag);
        if (!have && lane == 0) pt_fail(p.status, kDevTimeoutMma, abort_flag);
        // every warp takes the same branch (the barriers below are CTA-wide)
        if (!__syncthreads_and(have ? 1 : 0)) {
            aborted = true;
            break;
        }
        const int it = item_ring[j % PT_RING];
        if (it >= p.num_items) break;
        const PtItem w = pt_item(p, it);
#pragma unroll
        for (int i = 0; i < 8; ++i)
#pragma unroll
            for (int j = 0; j < 8; ++j) acc[i][j] = make_float2(0.f, 0.f);
        bool ok = true;
        for (int kt = w.kt0; kt < w.kt1; ++kt) {
            if (tid == 0 && !aborted) aborted = !produce();
            __syncwarp();
            const int slot = (int)(c_count % PT_STAGES);
            const uint32_t par = (c_count / PT_STAGES) & 1;
            bool got = mbar_wait(smem_u32(&full_bar[slot]), par, p.limit_ns, abort_flag);
            got = __all_sync(0xffffffffu, got);
            if (!got) {
                if (lane == 0) pt_fail(p.status, kDevTimeoutMma, abort_flag);
                ok = false;
                break;
            }
            const uint32_t as = a_row + slot * PT_A_STAGE;
            const uint8_t* bs = smem + PT_STAGES * PT_A_STAGE + slot * PT_B_STAGE + b_col;
#pragma unroll
            for (int k = 0; k < PT_BK; ++k) {
                // (a, a) for each of the eight rows, loaded into both halves of the pair
                float2 ad[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const uint32_t addr = as + i * (8 * PT_BK * 4) + ((((uint32_t)(k >> 2)) ^ a_sw) << 4) + (k & 3) * 4;
                    asm("ld.shared.f32 %0, [%1];" : "=f"(ad[i].x) : "r"(addr) : "memory");
                    asm("ld.shared.f32 %0, [%1];" : "=f"(ad[i].y) : "r"(addr) : "memory");
                }
                float2 bp[8];
#pragma unroll
                for (int h = 0; h < 4; ++h) {
                    const float4 b = *reinterpret_cast<const float4*>(bs + k * PT_BN * 4 + h * 64);
                    bp[2 * h] = make_float2(b.x, b.y);
                    bp[2 * h + 1] = make_float2(b.z, b.w);
                }
                // columns outer, rows inner: measured 2 % faster than rows outer (the compiler's
                // schedule of the 64 packed FMAs per k differs)
#pragma unroll
                for (int jj = 0; jj < 8; ++jj)
#pragma unroll
                    for (int i = 0; i < 8; ++i) acc[i][jj] = __ffma2_rn(ad[i], bp[jj], acc[i][jj]);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&empty_bar[slot]));
            ++c_count;
        }
        // every warp leaves the k-loop (done or aborted) before anyone goes on
        if (__syncthreads_or(ok ? 0 : 1) || *abort_flag) {
            aborted = true;
            break;
        }

        int mt, nt;
        pt_tile_coord(p, w.tile, mt, nt);
        const int m0 = mt * PT_BM, n0 = nt * PT_BN;
        const int row0 = m0 + wm * 64 + ty;  // rows row0 + 8 i
        const int col0 = n0 + wn * 64 + tx * 4;  // columns col0 + 16 h + {0..3}

        if (w.sl >= 0) {
            // a K slice: publish the partial tile, count it; the last slice to finish adds all
            // slices in slice order and stores C
            const int st = w.tile - p.split_first;
            const bool ws_ok = in_range(st, p.num_tiles - p.split_first) && in_range(w.sl, p.split);
            float4* base = reinterpret_cast<float4*>(p.ws + (int64_t)(ws_ok ? st : 0) * p.split * PT_TILE_FLOATS);
            float4* mine = base + (int64_t)w.sl * (PT_TILE_FLOATS / 4) + tid;
#pragma unroll
            for (int i = 0; i < 8; ++i)
#pragma unroll
                for (int h = 0; h < 4; ++h)
                    if (ws_ok)
                        __stcg(mine + (i * 4 + h) * PT_THREADS,
                               make_float4(acc[i][2 * h].x, acc[i][2 * h].y, acc[i][2 * h + 1].x, acc[i][2 * h + 1].y));
            __threadfence();
            __syncthreads();
            if (tid == 0) {
                const int n = ws_ok ? tagged_arrive(p.cnt + st, p.seq) : 0;
                if (n == 0) pt_fail(p.status, kDevTimeoutEpilogue, abort_flag);
                *bcast = n;
            }
            __syncthreads();
            const int n = *bcast;
            if (n != p.split) continue;  // another slice finishes the tile
            __threadfence();
            const float4* src = base + tid;
#pragma unroll
            for (int i = 0; i < 8; ++i)
#pragma unroll
                for (int h = 0; h < 4; ++h) {
                    const float4 v = __ldcg(src + (i * 4 + h) * PT_THREADS);
                    acc[i][2 * h] = make_float2(v.x, v.y);
                    acc[i][2 * h + 1] = make_float2(v.z, v.w);
                }
            for (int s = 1; s < p.split; ++s) {
                const float4* q = src + (int64_t)s * (PT_TILE_FLOATS / 4);
#pragma unroll
                for (int i = 0; i < 8; ++i)
#pragma unroll
                    for (int h = 0; h < 4; ++h) {
                        const float4 v = __ldcg(q + (i * 4 + h) * PT_THREADS);
                        acc[i][2 * h].x = __fadd_rn(acc[i][2 * h].x, v.x);
                        acc[i][2 * h].y = __fadd_rn(acc[i][2 * h].y, v.y);
                        acc[i][2 * h + 1].x = __fadd_rn(acc[i][2 * h + 1].x, v.z);
                        acc[i][2 * h + 1].y = __fadd_rn(acc[i][2 * h + 1].y, v.w);
                    }
            }
        }

        // store C: whole tiles unpredicated, edge tiles predicated; C is written once and not
        // read here, so its lines are the first to leave L2
        const uint64_t pol_out = l2_policy_evict_first();
        const bool whole = p.vec_out && m0 + PT_BM <= p.M && n0 + PT_BN <= p.N;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int gm = row0 + 8 * i;
            if (!whole && gm >= p.M) continue;
            if (!in_range(gm, p.M)) continue;
            float* crow = p.C + (int64_t)gm * p.ldc;
#pragma unroll
            for (int h = 0; h < 4; ++h) {
                const int gn = col0 + 16 * h;
                const float v[4] = {acc[i][2 * h].x, acc[i][2 * h].y, acc[i][2 * h + 1].x, acc[i][2 * h + 1].y};
                if (whole || (p.vec_out && gn + 3 < p.N)) {
                    if (in_range(gn, p.N) && in_range(gn + 3, p.N))
                        st_global_v4_hint(crow + gn, v[0], v[1], v[2], v[3], pol_out);
                } else {
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        if (gn + e < p.N && in_range(gn + e, p.N)) crow[gn + e] = v[e];
                }
            }
        }
    }

    // every TMA copy issued must have landed before shared memory is released
    __syncthreads();
    if (tid == 0)
        for (int s = 0; s < PT_STAGES; ++s)
            if ((issued_mask >> s) & 1)
                if (!mbar_wait(smem_u32(&full_bar[s]), (last_parity >> s) & 1, p.limit_ns, nullptr))
                    atomicCAS(p.status, 0, kDevTimeoutDrain);
    __syncthreads();
}

// fp32 [rows][cols] tensor map, row stride ld floats, box box_cols x box_rows.
bool encode_f32(CUtensorMap* map, const float* base, int64_t rows, int64_t cols, int64_t ld, uint32_t box_cols,
                uint32_t box_rows, CUtensorMapSwizzle swz)
{
    auto enc = tensor_map_encoder();
    if (!enc) return false;
    cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)ld * 4};
    cuuint32_t box[2] = {box_cols, box_rows};
    cuuint32_t estr[2] = {1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float*>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

bool ffma_persistent_supported(const F32Args& a)
{
    // TMA: 16-byte aligned bases and row strides; the kernel's 32-bit sizes
    const int64_t lim = 0x7fffffffLL - 1024;
    return ((reinterpret_cast<uintptr_t>(a.A) | reinterpret_cast<uintptr_t>(a.B)) & 15) == 0 && a.lda % 4 == 0 &&
           a.ldb % 4 == 0 && a.M <= lim && a.N <= lim && a.K <= lim && a.lda <= lim && a.ldb <= lim && a.ldc <= lim;
}

FfmaPlan ffma_persistent_plan(const F32Args& a, int split_opt, int num_sms)
{
    FfmaPlan pl;
    const int64_t m_tiles = (a.M + PT_BM - 1) / PT_BM, n_tiles = (a.N + PT_BN - 1) / PT_BN;
    const int64_t tiles = m_tiles * n_tiles;
    const int64_t k_tiles = (a.K + PT_BK - 1) / PT_BK;
    pl.tiles = tiles;
    pl.k_tiles = k_tiles;
    pl.split_first = tiles;
    pl.split = 1;
    pl.counters = 1;  // the item counter
    if (tiles <= 0 || k_tiles <= 0 || num_sms <= 0) return pl;
    int S = 1;
    int64_t first = tiles;
    if (split_opt > 0) {
        // a forced split cuts every tile
        S = split_opt;
        first = 0;
    } else {
        // The tiles of a last, partial wave are cut into S slices so that they fill the
        // CTAs.  Time model, in units of one tile's main loop: whole waves + the slices'
        // rounds + the last slice's read-back of the other partials (each ~128 KiB from L2,
        // about 1 us per slice at ~130 GB/s per SM, plus ~2 us for the count and fences).
        const int64_t r = tiles % num_sms;
        if (r != 0) {
            const double tile_us = 2.0 * PT_BM * PT_BN * (double)a.K / 4.0e5;  // ~400 GFLOP/s per SM
            double best = (double)((r + num_sms - 1) / num_sms);
            for (int s = 2; s <= PT_MAX_SPLIT; ++s) {
                if (k_tiles / s < 8) break;  // keep at least 8 k-tiles (256 of K) per slice
                const double rounds = (double)((r * s + num_sms - 1) / num_sms) / s;
                const double t = rounds + ((s - 1) * 1.0 + 2.0) / tile_us;
                if (t < best - 1e-9) {
                    best = t;
                    S = s;
                }
            }
            if (S > 1) first = tiles - r;
        }
    }
    if (S > 1) {
        int64_t kps = (k_tiles + S - 1) / S;
        S = (int)((k_tiles + kps - 1) / kps);  // every slice nonempty
        pl.kt_per_slice = kps;
    }
    // counters: one per split tile, then the launch's item counter
    if (S <= 1) {
        pl.split = 1;
        pl.split_first = tiles;
        pl.counters = 1;
        return pl;
    }
    pl.split = S;
    pl.split_first = first;
    pl.ws_floats = (tiles - first) * S * (int64_t)PT_TILE_FLOATS;
    pl.counters = tiles - first + 1;
    return pl;
}

cudaError_t launch_ffma_persistent(const F32Args& a, const FfmaPlan& pl, float* ws, unsigned long long* cnt,
                                   uint32_t seq, int num_sms, int* dev_status, uint64_t limit_ns, int test_stall,
                                   cudaStream_t stream, int* launches)
{
    CUtensorMap tmA, tmB;
    if (!encode_f32(&tmA, a.A, a.M, a.K, a.lda, PT_BK, PT_BM, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_f32(&tmB, a.B, a.K, a.N, a.ldb, PT_BN, PT_BK, CU_TENSOR_MAP_SWIZZLE_NONE))
        return cudaErrorInvalidValue;
    PtParams p;
    p.M = (int)a.M;
    p.N = (int)a.N;
    p.K = (int)a.K;
    p.m_tiles = (int)((a.M + PT_BM - 1) / PT_BM);
    p.n_tiles = (int)((a.N + PT_BN - 1) / PT_BN);
    // raster groups of 16 tile rows: at 4096^3 DRAM traffic 416 -> 374 MB against groups of 8
    // (363 MB with the L2 policies above; time unchanged), 454 MB with one group
    p.group_m = 16;
    if (pl.tiles > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    p.num_tiles = (int)pl.tiles;
    p.k_tiles = (int)pl.k_tiles;
    p.split = pl.split;
    p.split_first = (int)pl.split_first;
    p.kt_per_slice = pl.split > 1 ? (int)pl.kt_per_slice : p.k_tiles;
    const int64_t items = pl.split_first + (pl.tiles - pl.split_first) * pl.split;
    if (items > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    p.num_items = (int)items;
    p.C = a.C;
    p.ldc = (int)a.ldc;
    p.vec_out = (reinterpret_cast<uintptr_t>(a.C) & 15) == 0 && a.ldc % 4 == 0;
    p.ws = ws;
    p.cnt = cnt;
    p.seq = seq;
    if ((pl.split > 1 && !ws) || !cnt || seq == 0) return cudaErrorInvalidValue;
    p.status = dev_status;
    p.limit_ns = limit_ns;
    p.test_stall = test_stall;
    cudaError_t e = cudaFuncSetAttribute(ffma_persistent_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, PT_SMEM);
    if (e != cudaSuccess) return e;
    const int grid = (int)(items < num_sms ? items : num_sms);
    ffma_persistent_kernel<<<grid, PT_THREADS, PT_SMEM, stream>>>(tmA, tmB, p);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    *launches += 1;
    return cudaSuccess;
}

}  // namespace gemm_gb300
