// fp32 GEMM for few rows (M <= 32), B streamed through a TMA ring in shared memory.
//
// With M this small the product is bound by reading B once from HBM ("CUDA overview:
// performance surprises", sections "Coalescing memory blocks" and "Parallelism first"),
// or, at M = 32, close to the ridge where the FP32 pipe binds too.  Holding B rows in
// registers (skinny.cu) keeps only ~32 KiB per SM in flight, far less than HBM's
// latency-bandwidth product; here a producer warp keeps a ring of 32 KiB stages of B in
// flight per SM with the Tensor Memory Accelerator, and the consumers only read shared
// memory:
//   * one stage = KROWS k-rows x COLS columns of B (256-wide TMA boxes; zero fill past N
//     and past K), plus the matching KROWS x MR slice of A, which the producer warp
//     transposes into [k][m] rows;
//   * MSPLIT groups of COLW consumer warps: group g owns rows g*RT .. g*RT+RT-1, and thread
//     t of a group owns CPT/4 column quads (4t, 4t + SPAN, ...) of the work item: an outer
//     product per k-row ("Learning to develop for GPU with GEMM as the example", section
//     "Improving the solution and balancing memory work") done with packed fp32 FMAs
//     (fma.rn.f32x2) on (a_m, a_m+1) x (b_n, b_n): one 16-byte load of A feeds 4 CPT
//     packed FMAs, and each B value is paired with itself once per k-row;
//   * a persistent grid walks (column block, K slice) work items; K slices write partial
//     products that a fixed-order reduction adds, so results are deterministic.
// Every mbarrier wait is bounded (wall clock) and reports to the handle's status word.
#include <cuda.h>
#include <cudaTypedefs.h>


#include "internal.h"
#include "ptx.h"

namespace gemm_gb300 {

GEMM_DEBUG_UNIT(skinny_tma)

namespace {

constexpr int ST_BOX_COLS = 256;  // TMA box width (max 256 elements)
constexpr int ST_STAGE_BUDGET = 224 * 1024;  // shared memory for the stage ring (opt-in limit 227 KiB)

// COLW consumer warps across the columns of a work item, MSPLIT groups of them across the
// rows, KROWS k-rows per stage, CPT columns per thread.  The register file is split over
// the SM's four schedulers, so the thread count sets the register budget: 9 warps allow
// 168 registers per thread, 13 warps 128.  A rows are padded by 4 floats so that the
// producer's transposing stores spread over the banks while 16-byte loads stay aligned.
template <int MR, int COLW, int MSPLIT, int KROWS, int CPT>
struct StCfg {
    static constexpr int COLS = CPT * 32 * COLW;    // columns per work item
    static constexpr int SPAN = 4 * 32 * COLW;      // a thread's column quads are SPAN apart
    static constexpr int CONSUMER_WARPS = COLW * MSPLIT;
    static constexpr int THREADS = 32 * (1 + CONSUMER_WARPS);
    static constexpr int RT = MR / MSPLIT;          // rows per consumer thread
    static constexpr int A_LD = MR + 4;             // A row stride in the stage, floats
    static constexpr int B_STAGE_BYTES = KROWS * COLS * 4;
    static constexpr int A_STAGE_BYTES = KROWS * A_LD * 4;
    static constexpr int STAGES_FIT = ST_STAGE_BUDGET / (B_STAGE_BYTES + A_STAGE_BYTES);
    static constexpr int STAGES = STAGES_FIT > 8 ? 8 : STAGES_FIT;
    static constexpr int BYTES = STAGES * (B_STAGE_BYTES + A_STAGE_BYTES) + 256 + 1024;
    static_assert(COLS % ST_BOX_COLS == 0 && MR % MSPLIT == 0 && RT % 4 == 0, "shape");
    static_assert(CPT == 4 || CPT == 8, "columns per thread");
    static_assert(STAGES >= 3 && KROWS % 8 == 0 && KROWS <= 256 && (KROWS * MR) % 32 == 0, "stages");
};

struct StParams {
    F32Args a;
    int k_per_split;  // (sizes in 32 bits: the host keeps K and lda below 2^31)
    int K, lda;
    int nsplit;
    int col_blocks;
    int num_items;  // col_blocks * nsplit
    float* ws;      // split-K partials [nsplit][M][N] (nsplit > 1)
    int vec_out;
    int* status;
    uint64_t limit_ns;
    int test_stall;  // test hook: consumers first wait on a barrier nothing arrives on
};

template <int MR, int COLW, int MSPLIT, int KROWS, int CPT>
__global__ void __launch_bounds__(StCfg<MR, COLW, MSPLIT, KROWS, CPT>::THREADS, 1)
skinny_tma_kernel(const __grid_constant__ CUtensorMap tmB, StParams p)
{
    using SM = StCfg<MR, COLW, MSPLIT, KROWS, CPT>;
    // the split-K reduction launched next may start its blocks now; it waits for this grid
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    constexpr int NQ = CPT / 4;  // column quads per thread
    constexpr int ST_KROWS = KROWS;
    constexpr int ST_STAGES = SM::STAGES;
    constexpr int CONSUMER_WARPS = SM::CONSUMER_WARPS;
    constexpr int RT = SM::RT;
    constexpr int ST_COLS = SM::COLS;
    constexpr int ST_B_STAGE_BYTES = SM::B_STAGE_BYTES;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    uint8_t* smem = smem_raw + ((1024 - (raw & 1023)) & 1023);
    uint8_t* smem_b = smem;                                      // [ST_STAGES][ST_KROWS][ST_COLS] fp32
    uint8_t* smem_a = smem + ST_STAGES * ST_B_STAGE_BYTES;       // [ST_STAGES][ST_KROWS][A_LD] fp32
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + ST_STAGES * (ST_B_STAGE_BYTES + SM::A_STAGE_BYTES));
    uint64_t* full_bar = bars;
    uint64_t* empty_bar = bars + ST_STAGES;
    uint64_t* never_bar = bars + 2 * ST_STAGES;  // never completes (test hook)
    volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + 2 * ST_STAGES + 1);

    const int warp = threadIdx.x / 32;
    const int lane = threadIdx.x % 32;
    const F32Args& a = p.a;

    if (threadIdx.x == 0) {
        for (int s = 0; s < ST_STAGES; ++s) {
            mbar_init(smem_u32(&full_bar[s]), 1);
            mbar_init(smem_u32(&empty_bar[s]), CONSUMER_WARPS);
        }
        mbar_init(smem_u32(never_bar), 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmB)) : "memory");
    }
    __syncthreads();

    if (warp == 0) {
        // ------------------------------------------------------------ producer warp
        int stage = 0;
        uint32_t phase = 0;
        uint32_t issued_mask = 0, last_parity = 0;
        bool ok = true;
        for (int item = blockIdx.x; item < p.num_items && ok; item += gridDim.x) {
            const int cb = item % p.col_blocks, sp = item / p.col_blocks;
            const int kbeg = sp * p.k_per_split;
            const int kend = (int)min((int64_t)p.K, (int64_t)kbeg + p.k_per_split);
            const int col0 = cb * ST_COLS;
            for (int k0 = kbeg; k0 < kend; k0 += ST_KROWS) {
                // this stage's A[m][k0 .. k0+KROWS-1] into registers first: its L2 latency overlaps
                // the wait for a free stage (zero past M and past this slice's K)
                float av[ST_KROWS * MR / 32];
#pragma unroll
                for (int i = 0; i < ST_KROWS * MR / 32; ++i) {
                    const int e = lane + 32 * i;
                    const int kk = e % ST_KROWS, m = e / ST_KROWS;
                    const int gk = k0 + kk;
                    av[i] = (m < a.M && gk < kend && in_range(m, a.M) && in_range(gk, a.K))
                                ? __ldg(a.A + (int64_t)m * p.lda + gk)
                                : 0.f;
                }
                bool got = (lane == 0) ? mbar_wait(smem_u32(&empty_bar[stage]), phase ^ 1, p.limit_ns, abort_flag)
                                       : true;
                got = __shfl_sync(0xffffffffu, got ? 1 : 0, 0) != 0;
                if (!got) {
                    if (lane == 0) {
                        atomicCAS(p.status, 0, kDevTimeoutProducer);
                        *abort_flag = 1;
                    }
                    ok = false;
                    break;
                }
                const uint32_t fb = smem_u32(&full_bar[stage]);
                if (lane == 0) {
                    mbar_expect_tx(fb, ST_B_STAGE_BYTES);
                    uint8_t* dst = smem_b + stage * ST_B_STAGE_BYTES;
#pragma unroll
                    for (int j = 0; j < ST_COLS / ST_BOX_COLS; ++j)
                        tma_load_2d(smem_u32(dst + j * ST_BOX_COLS * 4 * ST_KROWS), &tmB, fb, col0 + j * ST_BOX_COLS,
                                       (int)k0);
                    issued_mask |= 1u << stage;
                    last_parity = (last_parity & ~(1u << stage)) | (phase << stage);
                }
                // A transposed to [k][m]
                float* adst = reinterpret_cast<float*>(smem_a + stage * SM::A_STAGE_BYTES);
#pragma unroll
                for (int i = 0; i < ST_KROWS * MR / 32; ++i) {
                    const int e = lane + 32 * i;
                    adst[(e % ST_KROWS) * SM::A_LD + e / ST_KROWS] = av[i];
                }
                __syncwarp();
                // the A writes of all lanes are ordered before this arrival (syncwarp);
                // the barrier completes once the B bytes have landed too
                if (lane == 0) mbar_arrive(fb);
                if (++stage == ST_STAGES) {
                    stage = 0;
                    phase ^= 1;
                }
            }
        }
        // every TMA copy issued must have landed before shared memory is released
        if (lane == 0)
            for (int s = 0; s < ST_STAGES; ++s)
                if ((issued_mask >> s) & 1)
                    if (!mbar_wait(smem_u32(&full_bar[s]), (last_parity >> s) & 1, p.limit_ns, nullptr))
                        atomicCAS(p.status, 0, kDevTimeoutDrain);
    } else {
        // ------------------------------------------------------------ consumer warps
        const int ct = (threadIdx.x - 32) % (32 * COLW);  // column slot
        const int mg = (threadIdx.x - 32) / (32 * COLW);  // row group 0 .. MSPLIT-1
        const int m_base = mg * RT;
        int stage = 0;
        uint32_t phase = 0;
        int item_first = blockIdx.x;
        if (p.test_stall) {
            // test hook: a wait nothing will satisfy runs out and takes the abort path
            bool got = mbar_wait(smem_u32(never_bar), 0, p.limit_ns, abort_flag);
            got = __all_sync(0xffffffffu, got);
            if (!got && lane == 0) {
                atomicCAS(p.status, 0, kDevTimeoutMma);
                *abort_flag = 1;
            }
            item_first = p.num_items;
        }
        for (int item = item_first; item < p.num_items; item += gridDim.x) {
            const int cb = item % p.col_blocks, sp = item / p.col_blocks;
            const int kbeg = sp * p.k_per_split;
            const int kend = (int)min((int64_t)p.K, (int64_t)kbeg + p.k_per_split);
            // column quads of this thread: q * SPAN + 4 ct (q < NQ); in the stage, box j holds
            // columns 256j .. 256j+255, stored [k][256] per box
            int b_off[NQ];
#pragma unroll
            for (int q = 0; q < NQ; ++q) {
                const int c = q * SM::SPAN + ct * 4;
                b_off[q] = (c / ST_BOX_COLS) * ST_BOX_COLS * ST_KROWS + c % ST_BOX_COLS;
            }
            // acc[i][4q + j] = (C[m_base + 2i][col_q + j], C[m_base + 2i + 1][col_q + j])
            float2 acc[RT / 2][CPT];
#pragma unroll
            for (int i = 0; i < RT / 2; ++i)
#pragma unroll
                for (int j = 0; j < CPT; ++j) acc[i][j] = make_float2(0.f, 0.f);
            bool ok = true;
            for (int k0 = kbeg; k0 < kend; k0 += ST_KROWS) {
                bool got = mbar_wait(smem_u32(&full_bar[stage]), phase, p.limit_ns, abort_flag);
                got = __all_sync(0xffffffffu, got);
                if (!got) {
                    if (lane == 0) {
                        atomicCAS(p.status, 0, kDevTimeoutMma);
                        *abort_flag = 1;
                    }
                    ok = false;
                    break;
                }
                const float* bst = reinterpret_cast<const float*>(smem_b + stage * ST_B_STAGE_BYTES);
                const float* ast = reinterpret_cast<const float*>(smem_a + stage * SM::A_STAGE_BYTES) + m_base;
#pragma unroll
                for (int kk = 0; kk < ST_KROWS; ++kk) {
                    float2 bb[CPT];  // (b, b) per column
#pragma unroll
                    for (int q = 0; q < NQ; ++q) {
                        const float4 b = *reinterpret_cast<const float4*>(bst + b_off[q] + kk * ST_BOX_COLS);
                        bb[4 * q] = make_float2(b.x, b.x);
                        bb[4 * q + 1] = make_float2(b.y, b.y);
                        bb[4 * q + 2] = make_float2(b.z, b.z);
                        bb[4 * q + 3] = make_float2(b.w, b.w);
                    }
#pragma unroll
                    for (int m = 0; m < RT; m += 4) {
                        const float4 ap = *reinterpret_cast<const float4*>(ast + kk * SM::A_LD + m);  // a_m .. a_m+3
                        const float2 a01 = make_float2(ap.x, ap.y), a23 = make_float2(ap.z, ap.w);
#pragma unroll
                        for (int j = 0; j < CPT; ++j) {
                            acc[m / 2][j] = __ffma2_rn(a01, bb[j], acc[m / 2][j]);
                            acc[m / 2 + 1][j] = __ffma2_rn(a23, bb[j], acc[m / 2 + 1][j]);
                        }
                    }
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&empty_bar[stage]));
                if (++stage == ST_STAGES) {
                    stage = 0;
                    phase ^= 1;
                }
            }
            if (!ok) break;
            // write this item's product (or K-slice partial)
            float* out;
            int64_t ldo;
            if (p.nsplit > 1) {
                out = p.ws + (int64_t)sp * a.M * a.N;
                ldo = a.N;
            } else {
                out = a.C;
                ldo = a.ldc;
            }
#pragma unroll
            for (int q = 0; q < NQ; ++q) {
                const int64_t col = (int64_t)cb * ST_COLS + q * SM::SPAN + ct * 4;
                if (col >= a.N) continue;
#pragma unroll
                for (int m = 0; m < RT; ++m) {
                    if (m_base + m >= a.M) break;
                    if (!in_range(m_base + m, a.M) || !in_range(col, a.N)) break;
                    float* dst = out + (int64_t)(m_base + m) * ldo + col;
                    float v[4];
#pragma unroll
                    for (int j = 0; j < 4; ++j) v[j] = (m & 1) ? acc[m / 2][4 * q + j].y : acc[m / 2][4 * q + j].x;
                    if (p.vec_out && col + 3 < a.N) {
                        *reinterpret_cast<float4*>(dst) = make_float4(v[0], v[1], v[2], v[3]);
                    } else {
#pragma unroll
                        for (int j = 0; j < 4; ++j)
                            if (col + j < a.N) dst[j] = v[j];
                    }
                }
            }
        }
    }
    __syncthreads();
}

template <int MR, int COLW, int MSPLIT, int KROWS, int CPT>
cudaError_t launch_mr_tma(const F32Args& a, int split, float* ws, int num_sms, int* dev_status,
                          uint64_t limit_ns, int test_stall, cudaStream_t stream, int* launches)
{
    // B as a [K][N] fp32 tensor, box 256 columns x 8 rows, no swizzle, zero fill outside
    CUtensorMap tmB;
    auto enc = tensor_map_encoder();
    if (!enc) return cudaErrorNotSupported;
    cuuint64_t dims[2] = {(cuuint64_t)a.N, (cuuint64_t)a.K};
    cuuint64_t strides[1] = {(cuuint64_t)a.ldb * 4};
    cuuint32_t box[2] = {ST_BOX_COLS, KROWS};
    cuuint32_t estr[2] = {1, 1};
    if (enc(&tmB, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float*>(a.B), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    StParams p;
    p.a = a;
    int64_t kps = (a.K + split - 1) / split;
    kps = (kps + KROWS - 1) / KROWS * KROWS;  // slices start on a stage boundary
    p.k_per_split = (int)kps;
    p.K = (int)a.K;
    p.lda = (int)a.lda;
    p.nsplit = (int)((a.K + kps - 1) / kps);
    p.col_blocks = (int)((a.N + StCfg<MR, COLW, MSPLIT, KROWS, CPT>::COLS - 1) / StCfg<MR, COLW, MSPLIT, KROWS, CPT>::COLS);
    const int64_t items = (int64_t)p.col_blocks * p.nsplit;
    if (items > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    p.num_items = (int)items;
    p.ws = ws;
    if (p.nsplit > 1)
        p.vec_out = (a.N % 4 == 0);
    else
        p.vec_out = (reinterpret_cast<uintptr_t>(a.C) & 15) == 0 && a.ldc % 4 == 0;
    p.status = dev_status;
    p.limit_ns = limit_ns;
    p.test_stall = test_stall;
    constexpr int smem = StCfg<MR, COLW, MSPLIT, KROWS, CPT>::BYTES;
    constexpr int threads = StCfg<MR, COLW, MSPLIT, KROWS, CPT>::THREADS;
    auto kern = skinny_tma_kernel<MR, COLW, MSPLIT, KROWS, CPT>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    const int grid = (int)(items < num_sms ? items : num_sms);
    kern<<<grid, threads, smem, stream>>>(tmB, p);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    *launches += 1;
    if (p.nsplit == 1) return cudaSuccess;
    *launches += 1;
    return launch_splitk_reduce(ws, p.nsplit, a.M, a.N, a.C, a.ldc, num_sms, stream);
}

}  // namespace

bool skinny_tma_supported(const F32Args& a)
{
    // TMA: 16-byte aligned base, row stride a multiple of 16 bytes
    return a.M <= 32 && (reinterpret_cast<uintptr_t>(a.B) & 15) == 0 && a.ldb % 4 == 0 && a.K < (1ll << 31) - 64 &&
           a.lda < (1ll << 31) &&
           a.N < (1ll << 31);
}

// The configurations launch_skinny_tma picks:
//   M <= 16: 8 warps x 128 columns, every row in one thread (16 x 4), 8 k-rows per stage;
//   M <= 32: 4 row groups of 2 warps x 256 columns (8 x 8 per thread), 16 k-rows per stage.
// At M = 32 the smaller register tile (134 registers, no spills) with deeper stages ran
// 1.27x faster than 16 x 4 per thread in 13 warps (GB300, 32 x 20736 x 10000).
using StSmall = StCfg<16, 8, 1, 8, 4>;
using StWide = StCfg<32, 2, 4, 16, 8>;
struct StShape { int64_t cols, krows; };
static StShape st_shape_for(int64_t M)
{
    if (M <= 16) return {StSmall::COLS, 8};
    return {StWide::COLS, 16};
}

int skinny_tma_auto_split(const F32Args& a, int num_sms)
{
    // the fewest K slices whose (column block, slice) items fill the persistent grid's
    // waves to at least 97 %; more slices only add partial-sum traffic
    const StShape sh = st_shape_for(a.M);
    const int64_t cols = sh.cols;
    const int64_t cbs = (a.N + cols - 1) / cols;
    int64_t max_s = (a.K + 16 * sh.krows - 1) / (16 * sh.krows);  // at least 16 stages per slice
    if (max_s > 1024) max_s = 1024;
    if (max_s < 1) max_s = 1;
    int64_t best = 1;
    double best_eff = 0.0;
    for (int64_t s = 1; s <= max_s; ++s) {
        const int64_t items = cbs * s;
        const int64_t waves = (items + num_sms - 1) / num_sms;
        const double eff = (double)items / (double)(waves * num_sms);
        if (eff >= 0.97) return (int)s;
        if (eff > best_eff + 1e-9) {
            best_eff = eff;
            best = s;
        }
        if (items >= 4 * num_sms) break;
    }
    return (int)best;
}

cudaError_t launch_skinny_tma(const F32Args& a, int split, float* ws, int num_sms, int* dev_status,
                              uint64_t limit_ns, int test_stall, cudaStream_t stream, int* launches)
{
    if (split < 1) split = 1;
    if (a.M <= 16)
        return launch_mr_tma<16, 8, 1, 8, 4>(a, split, ws, num_sms, dev_status, limit_ns, test_stall, stream, launches);
    if (a.M <= 32)
        return launch_mr_tma<32, 2, 4, 16, 8>(a, split, ws, num_sms, dev_status, limit_ns, test_stall, stream, launches);
    return cudaErrorInvalidValue;
}

}  // namespace gemm_gb300
