// fp32 GEMM for few rows (M <= 32), B streamed through a TMA ring in shared memory.
//
// With M this small the product is bound by reading B once from HBM ("CUDA overview:
// performance surprises", sections "Coalescing memory blocks" and "Parallelism first").
// Holding B rows in registers (skinny.cu) keeps only ~32 KiB per SM in flight, far less
// than HBM's latency-bandwidth product; here a producer warp keeps four 32 KiB stages of B
// in flight per SM with the Tensor Memory Accelerator, and the consumers only read shared
// memory:
//   * one stage = 8 k-rows x 1024 columns of B (four 256-wide TMA boxes; zero fill past
//     N and past K), plus the matching 8 x MR slice of A that the producer warp writes as
//     (a, a) pairs;
//   * 8 consumer warps per group of rows (16 rows per thread; 32-row products use two
//     groups, 16 warps); thread t of a group owns columns 4t .. 4t+3 of the block,
//     an outer product per k-row ("Learning to develop for GPU with GEMM as the example",
//     section "Improving the solution and balancing memory work") done with packed fp32
//     FMAs (fma.rn.f32x2) on the pre-paired A values;
//   * a persistent grid walks (column block, K slice) work items; K slices write partial
//     products that a fixed-order reduction adds, so results are deterministic.
// Every mbarrier wait is bounded (wall clock) and reports to the handle's status word.
#include <cuda.h>
#include <cudaTypedefs.h>


#include "internal.h"
#include "ptx.h"

namespace gemm_gb300 {
namespace {

constexpr int ST_BOX_COLS = 256;  // TMA box width (max 256 elements)
constexpr int ST_KROWS = 8;        // k-rows per stage
constexpr int ST_STAGES = 6;

// COLW consumer warps across the columns of a work item (128 columns each), MSPLIT
// groups of them across the rows.  The register file is split over the SM's four
// schedulers, so the thread count sets the register budget: 9 warps allow 168 registers
// per thread (16 rows x 4 columns), 13 warps 128 (two groups of 16 rows).
template <int MR, int COLW, int MSPLIT>
struct StCfg {
    static constexpr int COLS = 4 * 32 * COLW;                    // columns per work item
    static constexpr int CONSUMER_WARPS = COLW * MSPLIT;
    static constexpr int THREADS = 32 * (1 + CONSUMER_WARPS);
    static constexpr int RT = MR / MSPLIT;                        // rows per consumer thread
    static constexpr int B_STAGE_BYTES = ST_KROWS * COLS * 4;
    static constexpr int A_STAGE_BYTES = ST_KROWS * MR * 8;       // (a, a) pairs
    static constexpr int BYTES = ST_STAGES * (B_STAGE_BYTES + A_STAGE_BYTES) + 256 + 1024;
    static_assert(COLS % ST_BOX_COLS == 0 && MR % MSPLIT == 0 && RT % 2 == 0, "shape");
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

template <int MR, int COLW, int MSPLIT>
__global__ void __launch_bounds__(StCfg<MR, COLW, MSPLIT>::THREADS, 1)
skinny_tma_kernel(const __grid_constant__ CUtensorMap tmB, StParams p)
{
    using SM = StCfg<MR, COLW, MSPLIT>;
    constexpr int CONSUMER_WARPS = SM::CONSUMER_WARPS;
    constexpr int RT = SM::RT;
    constexpr int ST_COLS = SM::COLS;
    constexpr int ST_B_STAGE_BYTES = SM::B_STAGE_BYTES;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    uint8_t* smem = smem_raw + ((1024 - (raw & 1023)) & 1023);
    uint8_t* smem_b = smem;                                      // [ST_STAGES][ST_KROWS][ST_COLS] fp32
    float2* smem_a = reinterpret_cast<float2*>(smem + ST_STAGES * ST_B_STAGE_BYTES);  // [ST_STAGES][ST_KROWS][MR]
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
                // this stage's A[m][k0 .. k0+7] into registers first: its L2 latency overlaps
                // the wait for a free stage (zero past M and past this slice's K)
                float av[ST_KROWS * MR / 32];
#pragma unroll
                for (int i = 0; i < ST_KROWS * MR / 32; ++i) {
                    const int e = lane + 32 * i;
                    const int kk = e % ST_KROWS, m = e / ST_KROWS;
                    const int gk = k0 + kk;
                    av[i] = (m < a.M && gk < kend) ? __ldg(a.A + (int64_t)m * p.lda + gk) : 0.f;
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
                // A as (a, a) pairs, [k][m]
                float2* adst = smem_a + stage * ST_KROWS * MR;
#pragma unroll
                for (int i = 0; i < ST_KROWS * MR / 32; ++i) {
                    const int e = lane + 32 * i;
                    adst[(e % ST_KROWS) * MR + e / ST_KROWS] = make_float2(av[i], av[i]);
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
            // column offset inside the stage: box j holds columns 256j .. 256j+255, stored
            // [k][256] per box
            const int box = ct / 64, in_box = (ct % 64) * 4;
            float2 acc[RT][2];
#pragma unroll
            for (int m = 0; m < RT; ++m) acc[m][0] = acc[m][1] = make_float2(0.f, 0.f);
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
                const float* bst = reinterpret_cast<const float*>(smem_b + stage * ST_B_STAGE_BYTES) +
                                   box * ST_BOX_COLS * ST_KROWS + in_box;
                const float2* ast = smem_a + stage * ST_KROWS * MR + m_base;
#pragma unroll
                for (int kk = 0; kk < ST_KROWS; ++kk) {
                    const float4 b = *reinterpret_cast<const float4*>(bst + kk * ST_BOX_COLS);
                    const float2 b01 = make_float2(b.x, b.y), b23 = make_float2(b.z, b.w);
#pragma unroll
                    for (int m = 0; m < RT; m += 2) {
                        const float4 ap = *reinterpret_cast<const float4*>(ast + kk * MR + m);  // (a_m,a_m,a_m+1,a_m+1)
                        const float2 a0 = make_float2(ap.x, ap.y), a1 = make_float2(ap.z, ap.w);
                        acc[m][0] = __ffma2_rn(a0, b01, acc[m][0]);
                        acc[m][1] = __ffma2_rn(a0, b23, acc[m][1]);
                        acc[m + 1][0] = __ffma2_rn(a1, b01, acc[m + 1][0]);
                        acc[m + 1][1] = __ffma2_rn(a1, b23, acc[m + 1][1]);
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
            const int64_t col = (int64_t)cb * ST_COLS + ct * 4;
            if (col < a.N) {
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
                for (int m = 0; m < RT; ++m) {
                    if (m_base + m >= a.M) break;
                    float* dst = out + (int64_t)(m_base + m) * ldo + col;
                    const float v[4] = {acc[m][0].x, acc[m][0].y, acc[m][1].x, acc[m][1].y};
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

template <int MR, int COLW, int MSPLIT>
cudaError_t launch_mr_tma(const F32Args& a, int split, float* ws, int num_sms, int* dev_status,
                          uint64_t limit_ns, int test_stall, cudaStream_t stream, int* launches)
{
    // B as a [K][N] fp32 tensor, box 256 columns x 8 rows, no swizzle, zero fill outside
    CUtensorMap tmB;
    auto enc = tensor_map_encoder();
    if (!enc) return cudaErrorNotSupported;
    cuuint64_t dims[2] = {(cuuint64_t)a.N, (cuuint64_t)a.K};
    cuuint64_t strides[1] = {(cuuint64_t)a.ldb * 4};
    cuuint32_t box[2] = {ST_BOX_COLS, ST_KROWS};
    cuuint32_t estr[2] = {1, 1};
    if (enc(&tmB, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float*>(a.B), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    StParams p;
    p.a = a;
    int64_t kps = (a.K + split - 1) / split;
    kps = (kps + ST_KROWS - 1) / ST_KROWS * ST_KROWS;  // slices start on a stage boundary
    p.k_per_split = (int)kps;
    p.K = (int)a.K;
    p.lda = (int)a.lda;
    p.nsplit = (int)((a.K + kps - 1) / kps);
    p.col_blocks = (int)((a.N + StCfg<MR, COLW, MSPLIT>::COLS - 1) / StCfg<MR, COLW, MSPLIT>::COLS);
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
    constexpr int smem = StCfg<MR, COLW, MSPLIT>::BYTES;
    constexpr int threads = StCfg<MR, COLW, MSPLIT>::THREADS;
    auto kern = skinny_tma_kernel<MR, COLW, MSPLIT>;
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

// columns per work item of the configuration launch_skinny_tma picks for M
static int64_t st_cols_for(int64_t M) { return M <= 16 ? StCfg<16, 8, 1>::COLS : StCfg<32, 6, 2>::COLS; }

int skinny_tma_auto_split(const F32Args& a, int num_sms)
{
    // the fewest K slices whose (column block, slice) items fill the persistent grid's
    // waves to at least 97 %; more slices only add partial-sum traffic
    const int64_t cols = st_cols_for(a.M);
    const int64_t cbs = (a.N + cols - 1) / cols;
    int64_t max_s = (a.K + 16 * ST_KROWS - 1) / (16 * ST_KROWS);  // at least 16 stages per slice
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
        return launch_mr_tma<16, 8, 1>(a, split, ws, num_sms, dev_status, limit_ns, test_stall, stream, launches);
    if (a.M <= 32)
        return launch_mr_tma<32, 6, 2>(a, split, ws, num_sms, dev_status, limit_ns, test_stall, stream, launches);
    return cudaErrorInvalidValue;
}

}  // namespace gemm_gb300
