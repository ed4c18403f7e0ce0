// Valid 4-D cross-correlation on the tensor cores, channel-last bf16 / fp16 operands.
//
// "Three X: large convolutions in PyTorch for training", section "CUTLASS": the implicit
// GEMM runs best with 128-bit aligned tensors, channel and filter counts that are
// multiples of the MMA's K, and channel-last memory order.  With channels innermost, one
// filter tap (r0, r1, r2, r3) times C_in channels is a contiguous run of the GEMM's K, and
// the operand rows of that tap are input positions shifted by the tap:
//     y[p][o] = sum_{tap} sum_c x[p + tap][c] * w[o][tap][c]
// (p an output position, x[p + tap] the input position p0+r0, p1+r1, p2+r2, p3+r3).
//
// GEMM view: M = output positions, N = C_out, K = taps x C_in.  The A operand is never
// built, not even in shared memory: the input plane (i0, i1) = (p0 + r0, p1 + r1) is
// staged once, by the Tensor Memory Accelerator, as a no-swizzle K-major tile (channel
// group g of 8 channels: positions (i2, i3) row-major, 16 bytes each).  For output rows
// q = p2 * I3 + p3 of one output plane (p0, p1), the rows for tap (r2, r3) are the staged
// positions q + r2 * I3 + r3: 128 consecutive 16-byte rows.  So each tcgen05.mma takes
// its A operand through a descriptor whose start address is the tap's shift; the rows
// q with p3 >= P3 are computed too (I3 - P3 of every I3) and never stored.
//   * tiles: 128 rows (one TMEM lane each); a plane's Q = P2 * I3 rows are covered by
//     tiles starting at 0, 128, ..., the last one moved back to end at Q (it overlaps the
//     previous tile; the overlap is stored once).  A CTA computes up to two tiles of one
//     output plane, sharing every staged input plane between them.
//   * stages: input plane (r0, r1) and a group of g2 filter rows r2 (g2 * R3 taps), with
//     the weights of those taps: [C_out][64 k] tiles, 128-byte swizzled (TMA), the B
//     operand (K-major, N = C_out).
//   * accumulation: consecutive k-steps (16 channels of one tap) go round-robin to up
//     to 8 TMEM accumulators per tile.  With N = C_out as small as 32 one MMA is short,
//     and MMAs into the same accumulator wait for each other; independent accumulators
//     keep the tensor core fed.  It also shortens every accumulator's sum, which matters
//     because the tensor core's fp32 accumulator rounds toward zero; the epilogue adds
//     the accumulators in fp32 round-to-nearest, in order.
// Warp roles (192 threads): warp 0 = TMA producer, warp 1 = MMA issuer and TMEM owner,
// warps 2..5 = epilogue (one per 32-lane TMEM quarter).  Every mbarrier wait is bounded
// (wall clock); on expiry the CTA records an error in the status word, waits (bounded)
// for its own copies and MMAs in flight, frees its TMEM and returns.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "internal.h"
#include "ptx.h"

namespace gemm_gb300 {
namespace {

constexpr int CT_THREADS = 192;
constexpr int CT_TILE_M = 128;
constexpr int CT_MAX_TILES = 2;      // tiles of one output plane per CTA
constexpr int CT_MAX_ACC = 8;       // TMEM accumulators per tile
constexpr int CT_TMEM_COLS = 512;  // most TMEM columns a CTA allocates
constexpr int CT_SMEM_BUDGET = 200 * 1024;  // pipeline stages
constexpr int CT_MAX_STAGES = 8;

struct ConvTcParams {
    int cin, cout;
    int I[4], R[4], P[4];
    int q_rows;          // Q = P2 * I3 rows per output plane
    int tiles_per_plane;
    int ctas_per_plane;
    int g2;              // filter rows r2 per stage
    int stages_per_plane;
    int num_stages;      // R0 * R1 * stages_per_plane
    int rows_box;        // input rows (i2) staged per channel group
    int cg_stride;       // bytes between channel groups of the A region
    int a_region;        // bytes of the A region (multiple of 1024)
    int nbox_b;          // 64-wide weight boxes per stage
    int b_box_bytes;     // C_out * 128
    int stage_bytes;
    int nstages_ring;
    int tx_bytes;        // bytes one stage's copies deliver
    int nacc;            // TMEM accumulators per tile (k-steps round-robin)
    int tmem_cols;       // allocated TMEM columns: power of two >= nacc * 2 tiles * C_out
    uint32_t idesc;
    float* y;
    int* status;
    uint64_t limit_ns;
    int test_stall;
};

__host__ __device__ inline int tile_start(const ConvTcParams& p, int j)
{
    if (p.q_rows <= CT_TILE_M) return 0;
    const int s = j * CT_TILE_M;
    return s < p.q_rows - CT_TILE_M ? s : p.q_rows - CT_TILE_M;
}

// kind::f16 instruction descriptor: fp32 accumulator, A and B K-major, M = 128, N = C_out.
__host__ inline uint32_t conv_idesc(bool bf16, int n)
{
    return (1u << 4) | ((bf16 ? 1u : 0u) << 7) | ((bf16 ? 1u : 0u) << 10) | ((uint32_t)(n >> 3) << 17) |
           ((uint32_t)(CT_TILE_M >> 4) << 24);
}

__device__ __forceinline__ void ct_record_error(int* status, int code, volatile int* abort_flag)
{
    atomicCAS(status, 0, code);
    *abort_flag = 1;
}

__global__ void __launch_bounds__(CT_THREADS, 1)
conv4d_tc_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW,
                 ConvTcParams p)
{
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    uint8_t* smem = smem_raw + ((1024 - (raw & 1023)) & 1023);
    const int SA = p.nstages_ring;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + SA * p.stage_bytes);
    uint64_t* full_bar = bars;             // [SA] stage copies landed
    uint64_t* empty_bar = bars + SA;       // [SA] MMAs reading the stage done
    uint64_t* done_bar = bars + 2 * SA;    // all MMAs of the CTA done
    uint64_t* drain_bar = bars + 2 * SA + 1;
    uint64_t* never_bar = bars + 2 * SA + 2;  // never completes (test hook)
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bars + 2 * SA + 3);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);

    const int warp = threadIdx.x / 32;
    const int lane = threadIdx.x % 32;

    // this CTA: output plane (p0, p1) and its tiles [t0, t0 + ntile)
    const int plane = blockIdx.x / p.ctas_per_plane;
    const int cta_in_plane = blockIdx.x % p.ctas_per_plane;
    const int p0 = plane / p.P[1], p1 = plane % p.P[1];
    const int t0 = cta_in_plane * CT_MAX_TILES;
    const int ntile = min(CT_MAX_TILES, p.tiles_per_plane - t0);
    const int row0 = tile_start(p, t0) / p.I[3];  // first staged input row (before r2)

    if (warp == 0 && lane == 0) {
        for (int s = 0; s < SA; ++s) {
            mbar_init(smem_u32(&full_bar[s]), 1);
            mbar_init(smem_u32(&empty_bar[s]), 1);
        }
        mbar_init(smem_u32(done_bar), 1);
        mbar_init(smem_u32(drain_bar), 1);
        mbar_init(smem_u32(never_bar), 1);
        *abort_flag = 0;
        mbar_fence_init();
        prefetch_tensormap(&tmX);
        prefetch_tensormap(&tmW);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_holder), (uint32_t)p.tmem_cols);
        tc_fence_before();
    }
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_holder;
    const int cgroups = p.cin / 8;

    if (warp == 0) {
        // ---------------------------------------------------------------- producer
        if (lane == 0) {
            uint32_t issued_mask = 0, last_parity = 0;
            for (int st = 0; st < p.num_stages; ++st) {
                const int slot = st % SA;
                const uint32_t ph = (uint32_t)(st / SA) & 1;
                if (*abort_flag || !mbar_wait(smem_u32(&empty_bar[slot]), ph ^ 1, p.limit_ns, abort_flag)) {
                    ct_record_error(p.status, kDevTimeoutProducer, abort_flag);
                    break;
                }
                const int pi = st / p.stages_per_plane;
                const int r0 = pi / p.R[1], r1 = pi % p.R[1];
                const int r2s = (st % p.stages_per_plane) * p.g2;
                const uint32_t fb = smem_u32(&full_bar[slot]);
                mbar_arrive_expect_tx(fb, (uint32_t)p.tx_bytes);
                uint8_t* a_dst = smem + slot * p.stage_bytes;
                const int plane_in = (p0 + r0) * p.I[1] + (p1 + r1);
                for (int g = 0; g < cgroups; ++g)
                    tma_load_5d(smem_u32(a_dst + g * p.cg_stride), &tmX, fb, 0, g, 0, row0 + r2s, plane_in);
                uint8_t* b_dst = a_dst + p.a_region;
                const int k0 = ((pi * p.R[2] + r2s) * p.R[3]) * p.cin;
                for (int b = 0; b < p.nbox_b; ++b)
                    tma_load_2d(smem_u32(b_dst + b * p.b_box_bytes), &tmW, fb, k0 + 64 * b, 0);
                issued_mask |= 1u << slot;
                last_parity = (last_parity & ~(1u << slot)) | (ph << slot);
            }
            // every copy this CTA issued must have landed before its shared memory goes away
            for (int s = 0; s < SA; ++s)
                if ((issued_mask >> s) & 1)
                    if (!mbar_wait(smem_u32(&full_bar[s]), (last_parity >> s) & 1, p.limit_ns))
                        ct_record_error(p.status, kDevTimeoutDrain, abort_flag);
        }
        __syncwarp();
    } else if (warp == 1) {
        // ---------------------------------------------------------------- MMA issuer
        if (lane == 0) {
            bool ok = true;
            const int ksteps = p.cin / 16;
            const bool two = ntile > 1;
            // tile row offsets inside the staged rows, in 16-byte positions; descriptors
            // hold the start address in 16-byte units in their low bits, so moving an
            // operand by n positions is adding n to its descriptor (no carry: shared
            // memory addresses stay below 2^18 bytes)
            const uint32_t qoff0 = (uint32_t)(tile_start(p, t0) - row0 * p.I[3]);
            const uint32_t qoff1 = two ? (uint32_t)(tile_start(p, t0 + 1) - row0 * p.I[3]) : 0u;
            const uint32_t cg2 = (uint32_t)(2 * p.cg_stride) >> 4;  // next 16 channels of A
            const uint32_t box16 = (uint32_t)p.b_box_bytes >> 4;    // next 64-wide weight box
            const uint32_t acc_cols = (uint32_t)(CT_MAX_TILES * p.cout);  // TMEM columns per accumulator
            uint32_t kstep = 0, acc_idx = 0;
            for (int st = 0; st < p.num_stages; ++st) {
                const int slot = st % SA;
                const uint32_t ph = (uint32_t)(st / SA) & 1;
                if (*abort_flag || !mbar_wait(smem_u32(&full_bar[slot]), ph, p.limit_ns, abort_flag)) {
                    ct_record_error(p.status, kDevTimeoutMma, abort_flag);
                    ok = false;
                    break;
                }
                tc_fence_after();
                const int r2s = (st % p.stages_per_plane) * p.g2;
                const int g = min(p.g2, p.R[2] - r2s);
                const uint32_t a_st = smem_u32(smem + slot * p.stage_bytes);
                const uint64_t a_desc0 = smem_desc(a_st, (uint32_t)p.cg_stride, 128, kLayoutNoSwizzle);
                uint64_t b_box = smem_desc_sw128(a_st + p.a_region, 16, 1024);  // current weight box
                uint32_t b_step = 0;                                            // 16-k step inside it
                for (int rr = 0; rr < g; ++rr) {
                    for (int r3 = 0; r3 < p.R[3]; ++r3) {
                        // position shift of tap (r2s + rr, r3)
                        uint64_t a_desc = a_desc0 + (uint32_t)(rr * p.I[3] + r3);
                        for (int s = 0; s < ksteps; ++s) {
                            const uint64_t b_desc = b_box + 2 * b_step;  // 32 bytes per step
                            const uint32_t d0 = tmem_base + acc_idx * acc_cols;
                            const uint32_t acc = kstep >= (uint32_t)p.nacc ? 1u : 0u;  // first use overwrites
                            umma_f16(d0, a_desc + qoff0, b_desc, p.idesc, acc);
                            if (two) umma_f16(d0 + (uint32_t)p.cout, a_desc + qoff1, b_desc, p.idesc, acc);
                            ++kstep;
                            if (++acc_idx == (uint32_t)p.nacc) acc_idx = 0;
                            a_desc += cg2;
                            if (++b_step == 4) {
                                b_step = 0;
                                b_box += box16;
                            }
                        }
                    }
                }
                umma_commit(smem_u32(&empty_bar[slot]));  // stage free once these MMAs finish
            }
            if (ok) umma_commit(smem_u32(done_bar));
            // no MMA of this CTA may still be running when TMEM and shared memory are released
            umma_commit(smem_u32(drain_bar));
            if (!mbar_wait(smem_u32(drain_bar), 0, p.limit_ns))
                ct_record_error(p.status, kDevTimeoutDrain, abort_flag);
        }
        __syncwarp();
    } else {
        // ---------------------------------------------------------------- epilogue
        const int quarter = warp & 3;  // TMEM lane quarter this warp may access
        bool ok = true;
        if (p.test_stall) {
            // test hook: a wait nothing will satisfy runs out and takes the abort path
            ok = mbar_wait(smem_u32(never_bar), 0, p.limit_ns);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok && lane == 0) ct_record_error(p.status, kDevTimeoutEpilogue, abort_flag);
        }
        if (ok) {
            ok = mbar_wait(smem_u32(done_bar), 0, p.limit_ns, abort_flag);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok && lane == 0) ct_record_error(p.status, kDevTimeoutEpilogue, abort_flag);
        }
        if (ok) {
            tc_fence_after();
            const int r = quarter * 32 + lane;  // tile row of this thread
            const int P23 = p.P[2] * p.P[3];
            float* yplane = p.y + ((int64_t)plane * P23) * p.cout;
            for (int j = 0; j < ntile; ++j) {
                const int t = t0 + j;
                const int q = tile_start(p, t) + r;
                const int q_min = (t == 0) ? 0 : tile_start(p, t - 1) + CT_TILE_M;  // rows of earlier tiles
                const int p2 = q / p.I[3], p3 = q % p.I[3];
                const bool store = q < p.q_rows && q >= q_min && p3 < p.P[3];
                float* yrow = yplane + ((int64_t)p2 * p.P[3] + p3) * p.cout;
                for (int c0 = 0; c0 < p.cout; c0 += 16) {
                    float acc[16];
                    for (int a = 0; a < p.nacc; ++a) {  // accumulators in fixed order
                        uint32_t v[16];
                        tmem_ld_32x32b_x16(tmem_base + ((uint32_t)(quarter * 32) << 16) +
                                               (uint32_t)((a * CT_MAX_TILES + j) * p.cout + c0),
                                           v);
                        tmem_ld_wait();
#pragma unroll
                        for (int i = 0; i < 16; ++i)
                            acc[i] = (a == 0) ? __uint_as_float(v[i]) : __fadd_rn(acc[i], __uint_as_float(v[i]));
                    }
                    if (store) {
#pragma unroll
                        for (int i = 0; i < 16; i += 4)
                            *reinterpret_cast<float4*>(yrow + c0 + i) =
                                make_float4(acc[i], acc[i + 1], acc[i + 2], acc[i + 3]);
                    }
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, (uint32_t)p.tmem_cols);
    }
}

}  // namespace

int launch_conv4d_tc(const void* x, int64_t cin, const int64_t in[4], const void* w, int64_t cout,
                     const int64_t k[4], float* y, bool bf16, int* dev_status, uint64_t limit_ns, int test_stall,
                     cudaStream_t stream, int* launches)
{
    if (cin % 16 != 0 || cout % 16 != 0 || cout < 16 || cout > 256) return GEMM_ERR_UNSUPPORTED;
    ConvTcParams p = {};
    int64_t P[4];
    for (int d = 0; d < 4; ++d) {
        P[d] = in[d] - k[d] + 1;
        if (in[d] > (1 << 20) || k[d] > (1 << 20)) return GEMM_ERR_UNSUPPORTED;
        p.I[d] = (int)in[d];
        p.R[d] = (int)k[d];
        p.P[d] = (int)P[d];
    }
    const int64_t taps = k[0] * k[1] * k[2] * k[3];
    const int64_t K = taps * cin;
    const int64_t planes_out = P[0] * P[1];
    const int64_t Q = P[2] * in[3];
    if (in[3] > 256 || K >= (1ll << 31) || in[0] * in[1] >= (1ll << 31) || Q >= (1 << 30) || cin > 2048)
        return GEMM_ERR_UNSUPPORTED;
    p.cin = (int)cin;
    p.cout = (int)cout;
    p.q_rows = (int)Q;
    p.tiles_per_plane = (int)((Q + CT_TILE_M - 1) / CT_TILE_M);
    p.ctas_per_plane = (p.tiles_per_plane + CT_MAX_TILES - 1) / CT_MAX_TILES;
    const int64_t grid = planes_out * p.ctas_per_plane;
    if (grid >= (1ll << 31)) return GEMM_ERR_UNSUPPORTED;
    p.b_box_bytes = (int)cout * 128;

    // largest r2 group whose stage leaves room for at least three stages; the staged
    // input rows must cover every tile's rows shifted by every tap of the group
    int chosen = 0;
    for (int g2 = (int)k[2]; g2 >= 1 && !chosen; --g2) {
        int rows_box = 0;
        for (int c = 0; c < p.ctas_per_plane; ++c) {
            const int t0 = c * CT_MAX_TILES;
            const int tl = (t0 + CT_MAX_TILES < p.tiles_per_plane ? t0 + CT_MAX_TILES : p.tiles_per_plane) - 1;
            const int row0 = tile_start(p, t0) / p.I[3];
            const int64_t span = (int64_t)tile_start(p, tl) - (int64_t)row0 * in[3] + CT_TILE_M +
                                 (int64_t)(g2 - 1) * in[3] + (k[3] - 1);
            const int64_t rows = (span + in[3] - 1) / in[3];
            if (rows > rows_box) rows_box = (int)(rows > (1 << 20) ? (1 << 20) : rows);
        }
        if (rows_box > 256) continue;
        const int64_t cg_bytes = (int64_t)rows_box * in[3] * 16;
        const int64_t cg_stride = (cg_bytes + 127) / 128 * 128;
        const int64_t a_region = ((cin / 8) * cg_stride + 1023) / 1024 * 1024;
        const int64_t nbox_b = ((int64_t)g2 * k[3] * cin + 63) / 64;
        const int64_t stage = a_region + nbox_b * p.b_box_bytes;
        if (3 * stage > CT_SMEM_BUDGET) continue;
        p.g2 = g2;
        p.rows_box = rows_box;
        p.cg_stride = (int)cg_stride;
        p.a_region = (int)a_region;
        p.nbox_b = (int)nbox_b;
        p.stage_bytes = (int)stage;
        p.tx_bytes = (int)((cin / 8) * cg_bytes + nbox_b * p.b_box_bytes);
        chosen = 1;
    }
    if (!chosen) return GEMM_ERR_UNSUPPORTED;
    p.stages_per_plane = (p.R[2] + p.g2 - 1) / p.g2;
    const int64_t nst = k[0] * k[1] * p.stages_per_plane;
    if (nst >= (1ll << 30)) return GEMM_ERR_UNSUPPORTED;
    p.num_stages = (int)nst;
    int ring = CT_SMEM_BUDGET / p.stage_bytes;
    if (ring > CT_MAX_STAGES) ring = CT_MAX_STAGES;
    if (ring > p.num_stages) ring = p.num_stages;
    p.nstages_ring = ring;
    const int64_t ksteps = taps * (cin / 16);
    int nacc = CT_TMEM_COLS / (CT_MAX_TILES * p.cout);
    if (nacc > CT_MAX_ACC) nacc = CT_MAX_ACC;
    if (nacc > ksteps) nacc = (int)ksteps;
    p.nacc = nacc;
    p.tmem_cols = 32;
    while (p.tmem_cols < nacc * CT_MAX_TILES * p.cout) p.tmem_cols *= 2;
    p.idesc = conv_idesc(bf16, p.cout);
    p.y = y;
    p.status = dev_status;
    p.limit_ns = limit_ns;
    p.test_stall = test_stall;

    // x as [plane = i0*I1 + i1][i2][i3][channel group][8 channels]: one box = one
    // channel group of `rows_box` input rows (zero fill past I2)
    auto enc = tensor_map_encoder();
    if (!enc) return GEMM_ERR_CUDA;
    const CUtensorMapDataType dt = bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    CUtensorMap tmX, tmW;
    {
        cuuint64_t dims[5] = {8, (cuuint64_t)(cin / 8), (cuuint64_t)in[3], (cuuint64_t)in[2],
                              (cuuint64_t)(in[0] * in[1])};
        cuuint64_t strides[4] = {16, (cuuint64_t)cin * 2, (cuuint64_t)(in[3] * cin * 2),
                                 (cuuint64_t)(in[2] * in[3] * cin * 2)};
        cuuint32_t box[5] = {8, 1, (cuuint32_t)in[3], (cuuint32_t)p.rows_box, 1};
        cuuint32_t estr[5] = {1, 1, 1, 1, 1};
        if (enc(&tmX, dt, 5, const_cast<void*>(x), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return GEMM_ERR_CUDA;
    }
    {
        // w as the row-major [C_out][K] matrix; box = 64 k x C_out rows, 128-byte swizzle
        cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)cout};
        cuuint64_t strides[1] = {(cuuint64_t)K * 2};
        cuuint32_t box[2] = {64, (cuuint32_t)cout};
        cuuint32_t estr[2] = {1, 1};
        if (enc(&tmW, dt, 2, const_cast<void*>(w), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return GEMM_ERR_CUDA;
    }
    const int smem = p.nstages_ring * p.stage_bytes + 1024 /*barriers*/ + 1024 /*alignment slack*/;
    if (cudaFuncSetAttribute(conv4d_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
        return GEMM_ERR_CUDA;
    conv4d_tc_kernel<<<(unsigned)grid, CT_THREADS, smem, stream>>>(tmX, tmW, p);
    if (cudaGetLastError() != cudaSuccess) return GEMM_ERR_CUDA;
    *launches += 1;
    return GEMM_OK;
}

}  // namespace gemm_gb300
