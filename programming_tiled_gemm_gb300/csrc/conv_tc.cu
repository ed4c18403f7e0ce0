// Valid 4-D cross-correlation on the tensor cores, channel-last bf16 / fp16 operands.
//
// "Three X: large convolutions in PyTorch for training", section "CUTLASS": the implicit
// GEMM runs best with 128-bit aligned tensors, channel and filter counts that are
// multiples of the MMA's K, and channel-last memory order.  With channels innermost, one
// filter tap (r0, r1, r2, r3) times C_in channels is a contiguous run of the GEMM's K, and
// the operand rows of that tap are input positions shifted by the tap:
//     y[p][o] = sum_{tap} sum_c x[p + tap][c] * w[o][tap][c].
//
// GEMM view.  For one i0-slab (output p0), input positions are numbered linearly over
// (i1, i2, i3): u = (i1 * I2 + i2) * I3 + i3; output position (p1, p2, p3) is u with
// p1 < P1, p2 < P2, p3 < P3, and tap (r1, r2, r3) of input plane i0 = p0 + r0 adds the
// shift (r1 * I2 + r2) * I3 + r3.  So the A operand of a tap is a run of consecutive
// staged positions, addressed by a descriptor shifted by the tap: no column matrix is
// built anywhere.  Positions u with p1 >= P1, p2 >= P2 or p3 >= P3 are computed too and
// never stored.
//
// MMA shape.  tcgen05 needs M = 128 and N >= 128 (or the shared-memory reads of A, 4 KiB
// per MMA, bound it) to run at full rate, while N = C_out is often 32.  So S output
// positions are stacked along N: tile row g stands for positions u0 + S g + t (t < S),
// column block t of N (C_out wide) holds the output at offset t, and one MMA multiplies
// the staged window at shift s by a B whose block t holds the weights of tap r3 = s - t
// (zero outside 0..R3-1).  Windows s = r3' for r3' < R3 + S - 1 cover every tap of every
// block; R3 / (R3 + S - 1) of the products are useful.  Window rows are S positions
// apart, so the input is staged split by phase (u mod S): row g of window s is entry
// (s div S) + g of phase s mod S.  The weights of one (r0, r1, r2) are staged as
// R3 + 2S - 2 slices in reverse r3 order with zero slices at both ends, so the B of every
// window is one contiguous run of S * C_out rows.
//
// Data flow.  A preparation kernel writes the phase-split input and the padded, reversed
// weight slices into the handle's workspace (16-byte rows of 8 channels, the no-swizzle
// K-major core-matrix layout).  The conv kernel stages, per filter triple (r0, r1, r2),
// the input rows one tile needs and that triple's weights with contiguous bulk copies into
// a ring of shared-memory stages; up to four threads issue the MMAs into TMEM; 4 epilogue warps
// add the accumulators and store fp32 channel-last output.
//   * accumulation: each issuer's MMAs go round-robin to its share of up to 8 TMEM accumulators; the
//     tensor core's fp32 accumulator rounds toward zero, so shorter sums per accumulator
//     keep the error small; the epilogue adds them in fp32 round-to-nearest, in order.
// Warp roles (288 threads): warp 0 = producer, warps 1..4 = MMA issuers (lane 0 each; warp
// 1 owns TMEM), warps 5..8 = epilogue (one per 32-lane TMEM quarter).  Every mbarrier wait is bounded
// (wall clock); on expiry the CTA records an error in the status word, waits (bounded)
// for its own copies and MMAs in flight, frees its TMEM and returns.
#include <algorithm>

#include "internal.h"
#include "ptx.h"

namespace gemm_gb300 {

GEMM_DEBUG_UNIT(conv_tc)

namespace {

constexpr int CT_MAX_ISSUERS = 8;   // warps whose lane 0 issues MMAs (fewer when TMEM holds fewer accumulators)
constexpr int CT_THREADS = 32 * (1 + CT_MAX_ISSUERS + 4);
constexpr int CT_G = 128;           // tile rows (TMEM lanes); each stands for S positions
constexpr int CT_MAX_ACC = 8;       // TMEM accumulators (round-robin)
constexpr int CT_TMEM_COLS = 512;
constexpr int CT_SMEM_BUDGET = 200 * 1024;  // pipeline stages
constexpr int CT_MAX_STAGES = 12;

struct ConvTcParams {
    int cin, cout, S;
    int I[4], R[4], P[4];
    int U;              // linear positions u per i0-slab covering every valid (p1, p2, p3)
    int tiles_per_p0;
    int rows_box;       // staged input rows (i1, i2 merged) per tile, one filter row r2
    int g2;             // filter rows r2 per stage (a stage: r0, r1 and g2 consecutive r2)
    int groups;         // stages per (r0, r1): ceil(R2 / g2)
    int xp_rows;        // merged rows per (i0, channel group, phase) block of the staged input
    int a_blk;          // bytes of one (channel group, phase) block of a stage
    int a_region;       // A bytes per stage, rounded up to 1024
    int nslices;        // R3 + 2S - 2 weight slices per filter triple
    int b_trip;         // weight bytes of one filter triple (r0, r1, r2)
    int stage_bytes;
    int nstages_ring;
    int num_stages;     // R0 * R1 * groups
    int issuers;        // MMA-issuing threads (1 .. CT_MAX_ISSUERS)
    int nacc;           // TMEM accumulators (issuer i owns i, i + issuers, ...)
    uint32_t acc_used;  // bit a: accumulator a receives at least one MMA
    int s_log2;         // log2(S)
    int tmem_cols;
    uint32_t idesc;
    const uint8_t* xp;  // staged input (workspace)
    const uint8_t* wp;  // staged weights (workspace)
    int64_t xp_bytes, wp_bytes;  // their sizes (index checks of debug builds)
    float* y;
    int* status;
    uint64_t limit_ns;
    int test_stall;
};

// kind::f16 instruction descriptor: fp32 accumulator, A and B K-major, M = 128, N = n.
__host__ inline uint32_t conv_idesc(bool bf16, int n)
{
    return (1u << 4) | ((bf16 ? 1u : 0u) << 7) | ((bf16 ? 1u : 0u) << 10) | ((uint32_t)(n >> 3) << 17) |
           ((uint32_t)(CT_G >> 4) << 24);
}

__device__ __forceinline__ void ct_record_error(int* status, int code, volatile int* abort_flag)
{
    atomicCAS(status, 0, code);
    *abort_flag = 1;
}

// Staged operands, in 16-byte chunks of 8 channels:
//   xp[i0][g][phase][row][m]   = x[i0][row / I2][row % I2][phase + S m][8 g .. 8 g + 7]
//                                (zero for row >= I1 * I2; rows 0 .. xp_rows - 1)
//   wp[trip][g][j][o]          = w[o][r0][r1][r2][R3 + S - 2 - j][8 g .. 8 g + 7]
//                                (zero when that r3 is outside 0 .. R3 - 1)
// One flat index over four segments, one 16-byte chunk per thread: the input in its own
// order (coalesced reads, scattered writes), the input's zero rows, the weights in their
// own order, the zero weight slices.  The chunk counts fit 31 bits (checked by the plan).
__global__ void __launch_bounds__(256)
conv_tc_prepare_kernel(const uint4* __restrict__ x, const uint4* __restrict__ w, ConvTcParams p, uint4* xp, uint4* wp)
{
    // the conv kernel may start its set-up now; it waits for this grid before reading xp / wp
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int cg = p.cin / 8, S = p.S, mS = p.I[3] / S;
    const int plane_rows = p.I[1] * p.I[2];
    const int trips = p.R[0] * p.R[1] * p.R[2];
    const int n_x = p.I[0] * plane_rows * p.I[3] * cg;
    const int tail = p.xp_rows - plane_rows;
    const int n_xz = p.I[0] * cg * S * tail * mS;
    const int n_w = p.cout * trips * p.R[3] * cg;
    const int zs = 2 * S - 2;  // zero slices per (trip, g)
    const int n_wz = trips * cg * zs * p.cout;
    const uint4 zero = make_uint4(0, 0, 0, 0);
    for (int e = blockIdx.x * blockDim.x + threadIdx.x; e < n_x + n_xz + n_w + n_wz; e += gridDim.x * blockDim.x) {
        if (e < n_x) {
            const int g = e % cg, pos = e / cg;
            const int i3 = pos % p.I[3], rest = pos / p.I[3];
            const int row = rest % plane_rows, i0 = rest / plane_rows;
            const int ph = i3 % S, m = i3 / S;
            const int64_t d = ((int64_t)((i0 * cg + g) * S + ph) * p.xp_rows + row) * mS + m;
            if (in_range(d, p.xp_bytes / 16)) xp[d] = x[e];
        } else if (e < n_x + n_xz) {
            const int f = e - n_x;
            const int m = f % mS, r = f / mS;
            const int row = plane_rows + r % tail, blk = r / tail;  // blk = (i0 * cg + g) * S + ph
            const int64_t d = ((int64_t)blk * p.xp_rows + row) * mS + m;
            if (in_range(d, p.xp_bytes / 16)) xp[d] = zero;
        } else if (e < n_x + n_xz + n_w) {
            const int f = e - n_x - n_xz;
            const int g = f % cg, r = f / cg;
            const int r3 = r % p.R[3], r2 = r / p.R[3];
            const int trip = r2 % trips, o = r2 / trips;
            const int j = p.R[3] + S - 2 - r3;
            const int64_t d = ((int64_t)(trip * cg + g) * p.nslices + j) * p.cout + o;
            if (in_range(d, p.wp_bytes / 16)) wp[d] = w[f];
        } else {
            const int f = e - n_x - n_xz - n_w;
            const int o = f % p.cout, r = f / p.cout;
            const int z = r % zs, r2 = r / zs;  // z < S - 1: the first slices, else the last
            const int g = r2 % cg, trip = r2 / cg;
            const int j = z < S - 1 ? z : p.R[3] + S - 1 + (z - (S - 1));
            const int64_t d = ((int64_t)(trip * cg + g) * p.nslices + j) * p.cout + o;
            if (in_range(d, p.wp_bytes / 16)) wp[d] = zero;
        }
    }
}

__global__ void __launch_bounds__(CT_THREADS, 1) conv4d_tc_kernel(ConvTcParams p)
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

    // this CTA: output slab p0, positions u0 .. u0 + 128 S - 1
    const int p0 = blockIdx.x / p.tiles_per_p0;
    const int u0 = (blockIdx.x % p.tiles_per_p0) * CT_G * p.S;
    const int row0 = u0 / p.I[3];            // first staged row before the tap's row shift
    const int col0 = u0 - row0 * p.I[3];     // a multiple of S
    const int N = p.S * p.cout;

    if (warp == 0 && lane == 0) {
        for (int s = 0; s < SA; ++s) {
            mbar_init(smem_u32(&full_bar[s]), 1);
            mbar_init(smem_u32(&empty_bar[s]), (uint32_t)p.issuers);  // one commit per issuer
        }
        mbar_init(smem_u32(done_bar), (uint32_t)p.issuers);
        mbar_init(smem_u32(drain_bar), (uint32_t)p.issuers);
        mbar_init(smem_u32(never_bar), 1);
        *abort_flag = 0;
        mbar_fence_init();
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
            // launched as a programmatic dependent of the staging kernel: its writes to the
            // workspace are complete and visible once this returns
            asm volatile("griddepcontrol.wait;" ::: "memory");
            uint32_t issued_mask = 0, last_parity = 0;
            const int64_t row_bytes = (int64_t)(p.I[3] / p.S) * 16;
            const int64_t blk_stride = (int64_t)p.xp_rows * row_bytes;  // one (i0, g, phase) block
            int slot = 0, r0 = 0, r1 = 0, grp = 0;
            uint32_t ph = 0;
            for (int st = 0; st < p.num_stages; ++st) {
                if (*abort_flag || !mbar_wait_sleep(smem_u32(&empty_bar[slot]), ph ^ 1, p.limit_ns, abort_flag, 200)) {
                    ct_record_error(p.status, kDevTimeoutProducer, abort_flag);
                    break;
                }
                const int r2s = grp * p.g2;
                const int g = min(p.g2, p.R[2] - r2s);
                const int row = row0 + r1 * p.I[2] + r2s;
                // the rows of g filter rows: rows_box + g - 1 (a short last group copies fewer)
                const uint32_t a_bytes = (uint32_t)((p.rows_box + g - 1) * row_bytes);
                const uint32_t fb = smem_u32(&full_bar[slot]);
                mbar_arrive_expect_tx(fb, (uint32_t)(cgroups * p.S) * a_bytes + (uint32_t)(g * p.b_trip));
                uint8_t* a_dst = smem + slot * p.stage_bytes;
                const int64_t src_off = ((int64_t)(p0 + r0) * cgroups * p.S) * blk_stride + row * row_bytes;
                const uint8_t* src = p.xp + src_off;
                // (debug builds: a copy outside the staged operands is skipped; its stage then
                // never completes and the consumers' bounded wait reports it)
                for (int b = 0; b < cgroups * p.S; ++b)
                    if (in_range(src_off + b * blk_stride, p.xp_bytes) &&
                        in_range(src_off + b * blk_stride + a_bytes - 1, p.xp_bytes))
                        bulk_load(smem_u32(a_dst + b * p.a_blk), src + b * blk_stride, a_bytes, fb);
                const int64_t trip = ((int64_t)r0 * p.R[1] + r1) * p.R[2] + r2s;
                if (in_range(trip * p.b_trip, p.wp_bytes) && in_range(trip * p.b_trip + g * p.b_trip - 1, p.wp_bytes))
                    bulk_load(smem_u32(a_dst + p.a_region), p.wp + trip * p.b_trip, (uint32_t)(g * p.b_trip), fb);
                issued_mask |= 1u << slot;
                last_parity = (last_parity & ~(1u << slot)) | (ph << slot);
                if (++slot == SA) {
                    slot = 0;
                    ph ^= 1;
                }
                if (++grp == p.groups) {
                    grp = 0;
                    if (++r1 == p.R[1]) {
                        r1 = 0;
                        ++r0;
                    }
                }
            }
            // every copy this CTA issued must have landed before its shared memory goes away
            for (int s = 0; s < SA; ++s)
                if ((issued_mask >> s) & 1)
                    if (!mbar_wait(smem_u32(&full_bar[s]), (last_parity >> s) & 1, p.limit_ns))
                        ct_record_error(p.status, kDevTimeoutDrain, abort_flag);
        }
        __syncwarp();
    } else if (warp <= CT_MAX_ISSUERS) {
        // ---------------------------------------------------------------- MMA issuers
        // The (filter row, window) pairs of a stage are dealt round-robin to the issuers;
        // issuer i uses the accumulators i, i + issuers, ... in turn.  One thread issues
        // at best about one MMA per 55 cycles, while an MMA with N = 64 or 128 takes
        // 32 to 64, so several threads issue.
        if (lane == 0 && warp - 1 < p.issuers) {
            const int issuer = warp - 1;
            const int T = p.issuers;
            bool ok = true;
            const int ksteps = p.cin / 16;
            const int windows = p.R[3] + p.S - 1;
            // Descriptors hold the start address in 16-byte units in their low bits, so
            // moving an operand by n 16-byte rows is adding n to its descriptor (no carry:
            // shared-memory addresses stay below 2^18 bytes).
            const uint32_t a_cg2 = (uint32_t)(2 * p.S * p.a_blk) >> 4;            // next 16 channels of A
            const uint32_t b_cg2 = (uint32_t)(2 * p.nslices * p.cout * 16) >> 4;  // next 16 channels of B
            const uint32_t a_phase = (uint32_t)p.a_blk >> 4;                      // next phase of A
            const uint32_t a_row = (uint32_t)(p.I[3] / p.S);                      // next input row (r2 + 1)
            const uint32_t b_slice = (uint32_t)p.cout;                            // one weight slice
            const uint32_t b_r2 = (uint32_t)p.b_trip >> 4;                        // next filter triple
            const uint32_t acc_cols = (uint32_t)N;
            const uint32_t my_acc = (uint32_t)(p.nacc / T);
            uint32_t mma = 0, acc_j = 0;
            int slot = 0, grp = 0;
            uint32_t ph = 0;
            for (int st = 0; st < p.num_stages; ++st) {
                if (*abort_flag || !mbar_wait(smem_u32(&full_bar[slot]), ph, p.limit_ns, abort_flag)) {
                    ct_record_error(p.status, kDevTimeoutMma, abort_flag);
                    ok = false;
                    break;
                }
                tc_fence_after();
                const int g = min(p.g2, p.R[2] - grp * p.g2);
                const uint32_t a_st = smem_u32(smem + slot * p.stage_bytes);
                const uint64_t a_r = smem_desc(a_st + (uint32_t)(col0 / p.S) * 16, (uint32_t)(p.S * p.a_blk), 128,
                                               kLayoutNoSwizzle);
                // window 0 takes the slices from R3 + S - 2 on; window s starts s slices earlier
                const uint64_t b_r = smem_desc(a_st + p.a_region + (uint32_t)((p.R[3] + p.S - 2) * p.cout * 16),
                                               (uint32_t)(p.nslices * p.cout * 16), 128, kLayoutNoSwizzle);
                // pairs (rr, s), s fastest; this issuer starts at pair `issuer` and steps by T
                int rr = 0, s = issuer;
                while (s >= windows) {
                    s -= windows;
                    ++rr;
                }
                while (rr < g) {
                    // window s of filter row rr: phase s mod S, (s div S) entries on; B s slices earlier
                    const uint64_t a_w = a_r + (uint32_t)rr * a_row + (uint32_t)(s & (p.S - 1)) * a_phase +
                                         (uint32_t)(s >> p.s_log2);
                    const uint64_t b_w = b_r + (uint32_t)rr * b_r2 - (uint64_t)((uint32_t)s * b_slice);
                    for (int k = 0; k < ksteps; ++k) {
                        const uint32_t acc = mma >= my_acc ? 1u : 0u;  // first use overwrites
                        const uint32_t a_idx = (uint32_t)issuer + acc_j * (uint32_t)T;
                        umma_f16(tmem_base + a_idx * acc_cols, a_w + (uint32_t)k * a_cg2, b_w + (uint32_t)k * b_cg2,
                                 p.idesc, acc);
                        ++mma;
                        if (++acc_j == my_acc) acc_j = 0;
                    }
                    s += T;
                    while (s >= windows) {
                        s -= windows;
                        ++rr;
                    }
                }
                umma_commit(smem_u32(&empty_bar[slot]));  // stage free once these MMAs finish
                if (++slot == SA) {
                    slot = 0;
                    ph ^= 1;
                }
                if (++grp == p.groups) grp = 0;
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
            ok = mbar_wait_sleep(smem_u32(done_bar), 0, p.limit_ns, abort_flag, 1000);  // waits the whole main loop
            ok = __all_sync(0xffffffffu, ok);
            if (!ok && lane == 0) ct_record_error(p.status, kDevTimeoutEpilogue, abort_flag);
        }
        if (ok) {
            tc_fence_after();
            const int g = quarter * 32 + lane;  // tile row of this thread
            const int plane = p.I[2] * p.I[3];
            for (int c0 = 0; c0 < N; c0 += 16) {
                float acc[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) acc[i] = 0.f;
                for (int a = 0; a < p.nacc; ++a) {  // the accumulators that received MMAs, in order
                    if (!((p.acc_used >> a) & 1)) continue;
                    uint32_t v[16];
                    tmem_ld_32x32b_x16(tmem_base + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(a * N + c0), v);
                    tmem_ld_wait();
#pragma unroll
                    for (int i = 0; i < 16; ++i) acc[i] = __fadd_rn(acc[i], __uint_as_float(v[i]));
                }
                const int t = c0 / p.cout, o0 = c0 % p.cout;
                const int u = u0 + g * p.S + t;
                const int p1 = u / plane, rem = u - p1 * plane;
                const int p2 = rem / p.I[3], p3 = rem - p2 * p.I[3];
                if (p1 < p.P[1] && p2 < p.P[2] && p3 < p.P[3] && in_range(p0, p.P[0]) && in_range(o0 + 15, p.cout)) {
                    float* yrow = p.y + ((((int64_t)p0 * p.P[1] + p1) * p.P[2] + p2) * p.P[3] + p3) * p.cout + o0;
#pragma unroll
                    for (int i = 0; i < 16; i += 4)
                        *reinterpret_cast<float4*>(yrow + i) = make_float4(acc[i], acc[i + 1], acc[i + 2], acc[i + 3]);
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

// Plan of a launch: fills everything but the pointers.  Returns a gemm_status_t.
int plan_conv4d_tc(int64_t cin, const int64_t in[4], int64_t cout, const int64_t k[4], int S, ConvTcParams* out)
{
    if (cin % 16 != 0 || cout % 16 != 0 || cout < 16 || cout > 256 || cin > 2048) return GEMM_ERR_UNSUPPORTED;
    if ((S != 1 && S != 2 && S != 4) || S * cout > 256 || in[3] % S != 0) return GEMM_ERR_UNSUPPORTED;
    ConvTcParams p = {};
    p.cin = (int)cin;
    p.cout = (int)cout;
    p.S = S;
    for (int d = 0; d < 4; ++d) {
        if (in[d] > (1 << 20) || k[d] > in[d]) return GEMM_ERR_UNSUPPORTED;
        p.I[d] = (int)in[d];
        p.R[d] = (int)k[d];
        p.P[d] = (int)(in[d] - k[d] + 1);
    }
    const int64_t plane = in[2] * in[3];
    const int64_t U = (int64_t)p.P[1] * plane;
    const int64_t tile_pos = (int64_t)CT_G * S;
    const int64_t tiles = (U + tile_pos - 1) / tile_pos;
    const int64_t grid = tiles * p.P[0];
    if (U >= (1ll << 30) || grid >= (1ll << 31) || in[0] * in[1] * in[2] * in[3] >= (1ll << 31))
        return GEMM_ERR_UNSUPPORTED;
    p.U = (int)U;
    p.tiles_per_p0 = (int)tiles;
    // staged rows: a tile's positions plus the largest window shift R3 + S - 2, from the
    // tile's first row; the tile start within its row is a multiple of S below I3
    int64_t rows_box = 0;
    if (tiles <= 4096) {
        for (int64_t t = 0; t < tiles; ++t) {
            const int64_t span = ((t * tile_pos) % in[3]) + tile_pos + (k[3] + S - 2);
            const int64_t rows = (span + in[3] - 1) / in[3];
            if (rows > rows_box) rows_box = rows;
        }
    } else {
        rows_box = ((in[3] - S) + tile_pos + (k[3] + S - 2) + in[3] - 1) / in[3];
    }
    p.rows_box = (int)rows_box;
    // merged rows the last tile may reach: its first row, the largest tap row shift
    // (R1 - 1) I2 + R2 - 1, and the staged rows
    const int64_t last_row = (tiles - 1) * tile_pos / in[3] + (k[1] - 1) * in[2] + (k[2] - 1) + rows_box;
    if (last_row >= (1ll << 30)) return GEMM_ERR_UNSUPPORTED;
    p.xp_rows = (int)(last_row > in[1] * in[2] ? last_row : in[1] * in[2]);
    p.nslices = (int)(k[3] + 2 * S - 2);
    // the staging kernel's flat index: every staged 16-byte chunk in 31 bits
    const int64_t cgs = cin / 8, trips_all = k[0] * k[1] * k[2];
    const int64_t chunks = in[0] * in[1] * in[2] * in[3] * cgs +
                           in[0] * cgs * S * (p.xp_rows - in[1] * in[2]) * (in[3] / S) +
                           cout * trips_all * k[3] * cgs + trips_all * cgs * (2 * S - 2) * cout;
    if (chunks >= (1ll << 31) - (1ll << 20)) return GEMM_ERR_UNSUPPORTED;
    p.b_trip = (int)((cin / 8) * p.nslices * cout * 16);
    // MMA issuers: one per pair of TMEM accumulators' share, at most CT_MAX_ISSUERS
    const int N = S * p.cout;
    int nacc = CT_TMEM_COLS / N;
    if (nacc > CT_MAX_ACC) nacc = CT_MAX_ACC;
    p.issuers = nacc < CT_MAX_ISSUERS ? nacc : CT_MAX_ISSUERS;
    nacc -= nacc % p.issuers;
    p.nacc = nacc;
    const int64_t windows = k[3] + S - 1;
    // the most filter rows r2 per stage that leave room for three stages
    p.g2 = 0;
    for (int64_t g2 = k[2]; g2 >= 1 && p.g2 == 0; --g2) {
        const int64_t a_blk = (rows_box + g2 - 1) * (in[3] / S) * 16;
        const int64_t a_region = ((cin / 8) * S * a_blk + 1023) / 1024 * 1024;
        const int64_t stage = (a_region + g2 * p.b_trip + 1023) / 1024 * 1024;
        if (3 * stage > CT_SMEM_BUDGET) continue;
        p.g2 = (int)g2;
        p.a_blk = (int)a_blk;
        p.a_region = (int)a_region;
        p.stage_bytes = (int)stage;
    }
    if (p.g2 == 0) return GEMM_ERR_UNSUPPORTED;
    p.groups = (p.R[2] + p.g2 - 1) / p.g2;
    const int64_t nst = k[0] * k[1] * p.groups;
    if (nst >= (1 << 30) || k[0] * k[1] * k[2] >= (1 << 30)) return GEMM_ERR_UNSUPPORTED;
    p.num_stages = (int)nst;
    int ring = CT_SMEM_BUDGET / p.stage_bytes;
    if (ring > CT_MAX_STAGES) ring = CT_MAX_STAGES;
    if (ring > p.num_stages) ring = p.num_stages;
    p.nstages_ring = ring;
    // accumulator i + issuers j is written iff issuer i issues more than j MMAs; issuer i
    // takes (row, window) pairs i, i + issuers, ... of every stage
    p.acc_used = 0;
    for (int a = 0; a < nacc; ++a) {
        const int issuer = a % p.issuers, j = a / p.issuers;
        int64_t mine = 0;
        for (int grp = 0; grp < p.groups; ++grp) {
            const int64_t pairs = (int64_t)(p.R[2] - grp * p.g2 < p.g2 ? p.R[2] - grp * p.g2 : p.g2) * windows;
            mine += pairs > issuer ? (pairs - issuer + p.issuers - 1) / p.issuers : 0;
        }
        if (mine * k[0] * k[1] * (cin / 16) > j) p.acc_used |= 1u << a;
    }
    p.s_log2 = (S == 4) ? 2 : (S == 2) ? 1 : 0;
    p.tmem_cols = 32;
    while (p.tmem_cols < nacc * N) p.tmem_cols *= 2;
    *out = p;
    return GEMM_OK;
}

// Positions stacked along N: 2 when the shape allows it, else 1.
int choose_stack(int64_t cin, const int64_t in[4], int64_t cout, const int64_t k[4])
{
    ConvTcParams p;
    for (int S : {2, 1})
        if (plan_conv4d_tc(cin, in, cout, k, S, &p) == GEMM_OK) return S;
    return 0;
}

int64_t staged_input_bytes(const ConvTcParams& p)
{
    return (int64_t)p.I[0] * (p.cin / 8) * p.S * p.xp_rows * (p.I[3] / p.S) * 16;
}

}  // namespace

int64_t conv4d_tc_workspace(int64_t cin, const int64_t in[4], int64_t cout, const int64_t k[4], int S)
{
    ConvTcParams p;
    if (S <= 0) S = choose_stack(cin, in, cout, k);
    if (S <= 0 || plan_conv4d_tc(cin, in, cout, k, S, &p) != GEMM_OK) return -1;
    return staged_input_bytes(p) + (int64_t)p.R[0] * p.R[1] * p.R[2] * p.b_trip;
}

int launch_conv4d_tc(const void* x, int64_t cin, const int64_t in[4], const void* w, int64_t cout,
                     const int64_t k[4], float* y, bool bf16, int S, void* workspace, int num_sms, int* dev_status,
                     uint64_t limit_ns, int test_stall, cudaStream_t stream, int* launches)
{
    if (S <= 0) S = choose_stack(cin, in, cout, k);
    if (S <= 0) return GEMM_ERR_UNSUPPORTED;
    ConvTcParams p;
    const int rc = plan_conv4d_tc(cin, in, cout, k, S, &p);
    if (rc != GEMM_OK) return rc;
    const int64_t xb = staged_input_bytes(p);
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    p.xp = ws;
    p.wp = ws + xb;
    p.xp_bytes = xb;
    p.wp_bytes = (int64_t)p.R[0] * p.R[1] * p.R[2] * p.b_trip;
    p.idesc = conv_idesc(bf16, S * p.cout);
    p.y = y;
    p.status = dev_status;
    p.limit_ns = limit_ns;
    p.test_stall = test_stall;

    // one 16-byte chunk per thread where one resident wave holds them all (8 blocks of 256
    // threads per SM), a grid-stride loop beyond
    const int64_t cgs = cin / 8, trips_all = (int64_t)p.R[0] * p.R[1] * p.R[2];
    const int64_t chunks = (int64_t)p.I[0] * p.I[1] * p.I[2] * p.I[3] * cgs +
                           (int64_t)p.I[0] * cgs * S * (p.xp_rows - p.I[1] * p.I[2]) * (p.I[3] / S) +
                           (int64_t)cout * trips_all * p.R[3] * cgs + trips_all * cgs * (2 * S - 2) * cout;
    const int64_t blocks = std::max<int64_t>(1, std::min<int64_t>((chunks + 255) / 256, (int64_t)num_sms * 8));
    conv_tc_prepare_kernel<<<(unsigned)blocks, 256, 0, stream>>>(
        static_cast<const uint4*>(x), static_cast<const uint4*>(w), p, reinterpret_cast<uint4*>(ws),
        reinterpret_cast<uint4*>(ws + xb));
    if (cudaGetLastError() != cudaSuccess) return GEMM_ERR_CUDA;
    *launches += 1;

    const int smem = p.nstages_ring * p.stage_bytes + 1024 /*barriers*/ + 1024 /*alignment slack*/;
    if (cudaFuncSetAttribute(conv4d_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
        return GEMM_ERR_CUDA;
    // programmatic dependent launch: the CTAs set up their barriers and TMEM while the
    // staging kernel still runs; the producer waits for it before its first copy
    if (launch_dependent(conv4d_tc_kernel, dim3((unsigned)(p.tiles_per_p0 * p.P[0])), dim3(CT_THREADS), (size_t)smem,
                         stream, p) != cudaSuccess)
        return GEMM_ERR_CUDA;
    *launches += 1;
    return GEMM_OK;
}

}  // namespace gemm_gb300
