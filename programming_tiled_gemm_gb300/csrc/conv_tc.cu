// Valid 4-D cross-correlation on the tensor cores, channel-last bf16 / fp16 operands,
// computed by CTA pairs (tcgen05 cta_group::2) straight from the caller's tensors.
//
// "Three X: large convolutions in PyTorch for training", section "CUTLASS": the implicit
// GEMM runs best with 128-bit aligned tensors, channel and filter counts that are
// multiples of the MMA's K, and channel-last memory order.  With channels innermost, one
// filter tap (r0, r1, r2, r3) times 16 channels is one MMA's K, and the operand rows of
// that tap are input positions shifted by the tap:
//     y[p][o] = sum_{tap} sum_c x[p + tap][c] * w[o][tap][c].
//
// GEMM view.  For one i0-slab (output p0), input positions are numbered linearly over
// (i1, i2, i3): u = (i1 * I2 + i2) * I3 + i3; output position (p1, p2, p3) is u with
// p1 < P1, p2 < P2, p3 < P3, and tap (r1, r2, r3) of input plane i0 = p0 + r0 adds the
// shift (r1 * I2 + r2) * I3 + r3.  So the A operand of a tap is a run of consecutive
// positions, addressed by a shared-memory descriptor moved by the tap: no column matrix
// is built anywhere.  Positions u with p1 >= P1, p2 >= P2 or p3 >= P3 are computed too and
// never stored.
//
// MMA shape.  A CTA pair multiplies M = 256 positions (128 per CTA) at once.  C_out is often
// small (32), so S output positions are stacked along N: tile row g stands for positions
// u_g .. u_g + S - 1 (u_g = S g past the tile's start), and one MMA multiplies the input
// window at shift s by a B whose column block t' holds the weights of tap
// r3 = s - (S - 1) + t' (zero outside 0..R3-1): block t' accumulates the output at position
// u_g + S - 1 - t'.  Windows s < R3 + S - 1 cover every tap of every block.  N = S C_out
// columns are ordered (half h, block t', channel o % (C_out/2)): each CTA of the pair holds
// the weights of its half of the output channels only, so the pair reads every weight once.
//
// Data flow (no staging kernel, no workspace).  The Tensor Memory Accelerator loads, per
// pipeline stage (one (r0, r1), a group of g2 filter rows r2 and a group of 16-channel
// steps), each CTA's input rows and its half of the weights:
//   * input: x viewed as [i0][u / S][u % S][C] (phase split: window rows S positions
//     apart), one box of ROWS rows x 16 channels per (16-channel step, phase), in the
//     32-byte swizzle K-major layout (a row is one MMA's K).  Rows past the slab read zeros.
//     A window's descriptor starts at any row of a box: the swizzle is a function of the
//     shared-memory address, for the copy and for the MMA alike;
//   * weights: w viewed as [r0 r1 r2][r3][o][C], one box per 16-channel step of g2 filter
//     triples x (R3 + 2S - 2) slices x C_out/2 channels, its r3 range starting at -(S - 1):
//     the slices outside 0..R3-1 read zeros, which are the stacked blocks' padding.
//   With 16-byte rows of 8 channels (no swizzle) the copies took twice as many TMA rows and
//   the kernel ran 43.8 us instead of 37.5 us on the 16^4 x 16, 5^4 x 32 workload.
// Warp roles (416 threads per CTA): warp 0 = producer (both CTAs), warps 1..8 = MMA issuers
// (lane 0, even CTA only; warp 1 owns TMEM in both CTAs), warps 9..12 = epilogue (both CTAs,
// one per 32-lane TMEM quarter).  Once the MMAs are done, warps 1..8 read the accumulators
// with the epilogue warps: three warps per lane quarter, a third of the columns each.
//   * accumulation: each issuer's MMAs go round-robin to its share of up to 8 TMEM
//     accumulators; the tensor core's fp32 accumulator rounds toward zero, so shorter sums
//     per accumulator keep the error small; the epilogue adds them in fp32
//     round-to-nearest, in order.  Deterministic.
// K split.  With tiles for at most a quarter of the SMs, a tile is a cluster of four CTAs:
// two pairs, each over half of the stage sequence.  Each CTA's epilogue leaves its partial
// part (128 rows x N fp32) in its own shared memory (the operand ring, idle by then); after
// a cluster barrier each pair stores half of the columns, adding slot 0's part and slot 1's
// in that order, the other slot's read through distributed shared memory; a second cluster
// barrier keeps every part alive until it has been read.  Both barriers are reached by every
// thread on every path.  At 16^4 x 16 -> 32 channels, 5^4 filter this lets four positions
// stack along N (N = 128: MMAs at the full rate) on 144 CTAs: 29.3 us per call back to back
// against 35.1 us for two positions and one pair per tile.
// Every mbarrier wait is bounded (wall clock); on expiry the CTA records an error in the
// status word, waits (bounded) for its own copies and MMAs in flight, frees its TMEM and
// returns.
#include <algorithm>

#include "internal.h"
#include "ptx.h"

namespace gemm_gb300 {

GEMM_DEBUG_UNIT(conv_tc)

namespace {

constexpr int CT_ISSUERS_MAX = 8;   // warps whose lane 0 issues MMAs (even CTA)
constexpr int CT_THREADS = 32 * (1 + CT_ISSUERS_MAX + 4);
constexpr int CT_G = 128;           // tile rows per CTA (TMEM lanes); each stands for S positions
constexpr int CT_MAX_ACC = 8;       // TMEM accumulators (round-robin)
constexpr int CT_TMEM_COLS = 512;
constexpr int CT_SMEM_BUDGET = 200 * 1024;  // pipeline stages
constexpr int CT_MAX_STAGES = 8;
constexpr int CT_MAX_KS = 2;        // pairs per tile (K split over the stage sequence)

struct ConvTcParams {
    int cin, cout, S;
    int I[4], R[4], P[4];
    int tiles_per_p0;   // pair tiles (256 S positions each) per output slab
    int rows;           // input rows (u / S entries) per box: 128 + windows' reach + the group's r2 shifts
    int g2;             // filter rows r2 per stage
    int r2_groups;      // ceil(R2 / g2)
    int kq;             // 16-channel steps per stage
    int k_groups;       // cin / 16 / kq
    int nsl;            // weight slices per filter triple: R3 + 2S - 2
    int a_box;          // bytes of one input box (rows x 32, rounded up to 1024)
    int b_box;          // bytes of one weight box (g2 x nsl x C_out/2 x 32, rounded up to 1024)
    int a_region;       // input bytes per stage (kq S boxes)
    int tx_bytes;       // bytes one CTA's copies of a stage deliver
    int stage_bytes;    // kq (S a_box + b_box)
    int nstages_ring;
    int bar_offset;     // barriers after the operand ring (and after the K split's partial parts)
    int num_stages;     // R0 * R1 * r2_groups * k_groups
    int issuers;        // MMA-issuing threads (1 .. CT_ISSUERS_MAX)
    int nacc;           // TMEM accumulators (issuer i owns i, i + issuers, ...)
    int ks;             // pairs per tile (1 or 2): pair j of a tile's cluster runs stages
                        // [j n / ks, (j + 1) n / ks) and the pairs add their parts through
                        // distributed shared memory
    uint32_t acc_used[CT_MAX_KS];  // per K slot, bit a: accumulator a receives at least one MMA
    int tmem_cols;
    uint32_t idesc;
    float* y;
    int64_t ldy_cf;     // 0: y channel-last [P][C_out]; else y channel-first, y[o][p] at y + o ldy_cf + p
    int* status;
    uint64_t limit_ns;
    int test_stall;
};

// kind::f16 instruction descriptor: fp32 accumulator, A and B K-major, M = 256 (a CTA
// pair), N = n.
__host__ inline uint32_t conv_idesc(bool bf16, int n)
{
    return (1u << 4) | ((bf16 ? 1u : 0u) << 7) | ((bf16 ? 1u : 0u) << 10) | ((uint32_t)(n >> 3) << 17) |
           ((uint32_t)((2 * CT_G) >> 4) << 24);
}

__device__ __forceinline__ void ct_record_error(int* status, int code, volatile int* abort_flag)
{
    atomicCAS(status, 0, code);
    *abort_flag = 1;
}

__global__ void __launch_bounds__(CT_THREADS, 1)
conv4d_tc_pair_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW,
                      ConvTcParams p)
{
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    uint8_t* smem = smem_raw + ((1024 - (raw & 1023)) & 1023);
    const int SA = p.nstages_ring;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + p.bar_offset);
    uint64_t* full_bar = bars;             // [SA] both CTAs' copies of the stage landed (even CTA)
    uint64_t* empty_bar = bars + SA;       // [SA] MMAs reading the stage done (both CTAs)
    uint64_t* done_bar = bars + 2 * SA;    // all MMAs done (both CTAs)
    uint64_t* drain_bar = bars + 2 * SA + 1;
    uint64_t* never_bar = bars + 2 * SA + 2;  // never completes (test hook)
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bars + 2 * SA + 3);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);

    const int warp = threadIdx.x / 32;
    const int lane = threadIdx.x % 32;
    // a cluster is one tile: ks pairs of CTAs, pair j (cluster ranks 2j, 2j + 1) for K slot j
    const uint32_t crank = cluster_ctarank();
    const uint32_t rank = crank & 1u;          // CTA within the pair
    const uint32_t leader = crank & ~1u;       // the pair's even CTA (cluster rank)
    const uint16_t pair_mask = (uint16_t)(0x3u << leader);
    const int tile = blockIdx.x / (2 * p.ks), kslot = (int)(crank >> 1);
    const int p0 = tile / p.tiles_per_p0;
    const int u0 = (tile % p.tiles_per_p0) * 2 * CT_G * p.S;
    const int st_begin = (int)((int64_t)kslot * p.num_stages / p.ks);
    const int st_end = (int)((int64_t)(kslot + 1) * p.num_stages / p.ks);
    const int q_cta = u0 / p.S + (int)rank * CT_G;  // first input row (u / S) of this CTA's tile rows
    const int N = p.S * p.cout;
    const int half = p.cout / 2;

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
        prefetch_tensormap(&tmX);
        prefetch_tensormap(&tmW);
    }
    if (warp == 1) {
        tmem_alloc_pair(smem_u32(tmem_holder), (uint32_t)p.tmem_cols);
        tc_fence_before();
    }
    __syncthreads();
    cluster_sync_all();  // the peer's barriers and TMEM exist before anything targets them
    tc_fence_after();
    const uint32_t tmem_base = *tmem_holder;
    bool aborted = false;

    // Reading the accumulators (warps 1 .. 12, once the MMAs are done): thread = tile row of this
    // CTA in TMEM lane quarter `quarter`; columns in chunks of 16, the accumulators' parts of a
    // chunk added in order, then stored as groups of 8 columns.  Column
    // c = h (S C_out/2) + t' (C_out/2) + o_low is output channel h C_out/2 + o_low at position
    // ug + S - 1 - t'
    const int quarter = warp & 3;
    const int ug = u0 + ((int)rank * CT_G + quarter * 32 + lane) * p.S;  // this row's first position
    const int plane = p.I[2] * p.I[3];
    const uint32_t used = p.acc_used[kslot];
    float* const my_part = reinterpret_cast<float*>(smem) + quarter * N * 32;  // K split: [column][lane]
    // Warps 1..12 (the issuers' and the epilogue's) read the accumulators once the MMAs are
    // done: three warps per TMEM lane quarter, warp w takes the 16-column chunks
    // (w - 1) / 4, + 3, + 6, ...
    const int share = (warp - 1) / 4;
    bool part_ok = false;  // this warp saw the MMAs complete
    // a 16-column chunk of this row: the accumulators that received MMAs, added in order, four
    // TMEM loads per wait
    auto chunk_sum = [&](int c0, float (&acc)[16]) {
#pragma unroll
        for (int i = 0; i < 16; ++i) acc[i] = 0.f;
        const uint32_t lane_base = tmem_base + ((uint32_t)(quarter * 32) << 16) + (uint32_t)c0;
        for (int a0 = 0; a0 < p.nacc; a0 += 4) {
            uint32_t v[4][16];
#pragma unroll
            for (int b = 0; b < 4; ++b) {
                const int a = a0 + b;
                if (a < p.nacc && ((used >> a) & 1)) tmem_ld_32x32b_x16(lane_base + (uint32_t)(a * N), v[b]);
            }
            tmem_ld_wait();
#pragma unroll
            for (int b = 0; b < 4; ++b) {
                const int a = a0 + b;
                if (a >= p.nacc || !((used >> a) & 1)) continue;
#pragma unroll
                for (int i = 0; i < 16; ++i) acc[i] = __fadd_rn(acc[i], __uint_as_float(v[b][i]));
            }
        }
    };
    // columns c0 .. c0 + CW - 1 of this row to y, in groups of 8 (acc: float[16] or float[8])
    auto chunk_store = [&](int c0, const auto& acc) {
        constexpr int CW = sizeof(acc) / sizeof(acc[0]);
#pragma unroll
        for (int j = 0; j < CW; j += 8) {
            const int c = c0 + j;
            const int hh = c / (N / 2), cr = c - hh * (N / 2);
            const int tb = cr / half, o = hh * half + (cr - tb * half);
            const int u = ug + p.S - 1 - tb;
            const int p1 = u / plane, rem = u - p1 * plane;
            const int p2 = rem / p.I[3], p3 = rem - p2 * p.I[3];
            if (p1 < p.P[1] && p2 < p.P[2] && p3 < p.P[3] && in_range(p0, p.P[0]) && in_range(o + 7, p.cout)) {
                const int64_t pos = (((int64_t)p0 * p.P[1] + p1) * p.P[2] + p2) * p.P[3] + p3;
                if (p.ldy_cf == 0) {
                    float* yrow = p.y + pos * p.cout + o;
                    *reinterpret_cast<float4*>(yrow) = make_float4(acc[j], acc[j + 1], acc[j + 2], acc[j + 3]);
                    *reinterpret_cast<float4*>(yrow + 4) = make_float4(acc[j + 4], acc[j + 5], acc[j + 6], acc[j + 7]);
                } else {
                    float* ycol = p.y + (int64_t)o * p.ldy_cf + pos;
#pragma unroll
                    for (int e = 0; e < 8; ++e) ycol[(int64_t)e * p.ldy_cf] = acc[j + e];
                }
            }
        }
    };
    // this warp's chunks: stored to y, or with a K split left in shared memory as this CTA's
    // partial part (the operand ring, idle once the MMAs are done), [column][lane] so that a
    // warp's accesses are conflict-free 128-byte rows
    auto epilogue_share = [&]() {
        for (int c0 = 16 * share; c0 < N; c0 += 48) {
            float acc[16];
            chunk_sum(c0, acc);
            if (p.ks == 1) {
                chunk_store(c0, acc);
            } else {
#pragma unroll
                for (int i = 0; i < 16; ++i) my_part[(c0 + i) * 32 + lane] = acc[i];
            }
        }
    };
    if (warp == 0) {
        // ---------------------------------------------------------------- producer (both CTAs)
        if (lane == 0) {
            // after a programmatic launch (the channel-first re-layout): its output is complete
            // and visible before the first copy (a no-op after an ordinary launch)
            asm volatile("griddepcontrol.wait;" ::: "memory");
            uint32_t issued_mask = 0, last_parity = 0;
            // stage st = ((r0 R1 + r1) r2_groups + grp) k_groups + kg
            int kg = st_begin % p.k_groups, t = st_begin / p.k_groups;
            int grp = t % p.r2_groups;
            t /= p.r2_groups;
            int r1 = t % p.R[1], r0 = t / p.R[1];
            int slot = 0;
            uint32_t ph = 0;
            for (int st = st_begin; st < st_end; ++st) {
                if (!mbar_wait_cluster(smem_u32(&empty_bar[slot]), ph ^ 1, p.limit_ns, abort_flag)) {
                    ct_record_error(p.status, kDevTimeoutProducer, abort_flag);
                    aborted = true;
                    break;
                }
                const uint32_t fb_local = smem_u32(&full_bar[slot]);
                const uint32_t fb_even = mapa_shared(fb_local, leader);
                if (rank == 0) mbar_arrive_expect_tx(fb_local, 2u * (uint32_t)p.tx_bytes);
                const uint32_t st_base = smem_u32(smem + slot * p.stage_bytes);
                const int r2f = grp * p.g2;
                // input rows of filter row r2f: shift (r1 I2 + r2f) I3 positions, a multiple of S
                const int q0 = q_cta + (r1 * p.I[2] + r2f) * (p.I[3] / p.S);
                for (int kk = 0; kk < p.kq; ++kk) {
                    const int c16 = kg * p.kq + kk;  // 16-channel step
                    for (int ph_ = 0; ph_ < p.S; ++ph_)
                        tma_load_4d_pair(st_base + (uint32_t)((kk * p.S + ph_) * p.a_box), &tmX, fb_even, 16 * c16, ph_,
                                         q0, p0 + r0);
                    tma_load_4d_pair(st_base + (uint32_t)(p.a_region + kk * p.b_box), &tmW, fb_even, 16 * c16,
                                     (int)rank * half, -(p.S - 1), (r0 * p.R[1] + r1) * p.R[2] + r2f);
                }
                issued_mask |= 1u << slot;
                last_parity = (last_parity & ~(1u << slot)) | (ph << slot);
                if (++slot == SA) {
                    slot = 0;
                    ph ^= 1;
                }
                if (++kg == p.k_groups) {
                    kg = 0;
                    if (++grp == p.r2_groups) {
                        grp = 0;
                        if (++r1 == p.R[1]) {
                            r1 = 0;
                            ++r0;
                        }
                    }
                }
            }
            // every copy this CTA issued must have landed before its shared memory goes away
            // (the even CTA's full barriers count both CTAs' bytes)
            if (rank == 0)
                for (int s = 0; s < SA; ++s)
                    if ((issued_mask >> s) & 1)
                        if (!mbar_wait(smem_u32(&full_bar[s]), (last_parity >> s) & 1, p.limit_ns))
                            ct_record_error(p.status, kDevTimeoutDrain, abort_flag);
        }
        __syncwarp();
    } else if (warp <= CT_ISSUERS_MAX) {
        // ---------------------------------------------------------------- MMA issuers (even CTA)
        // The (filter row, window, channel step) triples of a stage are dealt to the issuers in
        // contiguous blocks; issuer i uses the accumulators i, i + issuers, ... in turn.  One
        // thread issues at best about one MMA per 55 cycles, so several threads issue.
        if (lane == 0 && rank == 0 && warp - 1 < p.issuers) {
            const int issuer = warp - 1;
            const int T = p.issuers;
            bool ok = true;
            const int windows = p.R[3] + p.S - 1;
            // Descriptors hold the start address in 16-byte units in their low bits, so moving
            // an operand by n 16-byte rows is adding n to its descriptor (no carry: shared-memory
            // addresses stay below 2^18 bytes).
            const uint32_t a_step = (uint32_t)(p.S * p.a_box) >> 4;      // next 16 channels of A
            const uint32_t b_step = (uint32_t)p.b_box >> 4;              // next 16 channels of B
            const uint32_t a_phase = (uint32_t)p.a_box >> 4;             // next phase of A
            const uint32_t a_row = 2;                                    // one 32-byte row
            const uint32_t a_r2 = (uint32_t)(p.I[3] / p.S) * a_row;      // next filter row r2: I3 / S rows
            const uint32_t b_slice = (uint32_t)(half * 32) >> 4;         // one weight slice (C_out/2 rows)
            const uint32_t b_r2 = (uint32_t)(p.nsl * half * 32) >> 4;    // next filter triple
            const uint32_t acc_cols = (uint32_t)N;
            const uint32_t my_acc = (uint32_t)(p.nacc / T);
            const int s_log2 = p.S == 4 ? 2 : p.S == 2 ? 1 : 0;
            uint32_t mma = 0, acc_j = 0;
            int slot = 0, grp = (st_begin / p.k_groups) % p.r2_groups;
            uint32_t ph = 0;
            for (int st = st_begin; st < st_end; ++st) {
                if (!mbar_wait_cluster(smem_u32(&full_bar[slot]), ph, p.limit_ns, abort_flag)) {
                    ct_record_error(p.status, kDevTimeoutMma, abort_flag);
                    ok = false;
                    break;
                }
                tc_fence_after();
                const int g = min(p.g2, p.R[2] - grp * p.g2);
                const uint32_t st_base = smem_u32(smem + slot * p.stage_bytes);
                // K-major, 32-byte swizzle: rows of 16 channels, 8-row atoms 256 bytes apart
                const uint64_t a_d = smem_desc(st_base, 16, 256, kLayoutSwizzle32);
                const uint64_t b_d = smem_desc(st_base + (uint32_t)p.a_region, 16, 256, kLayoutSwizzle32);
                // this issuer's MMAs: a contiguous block of the stage's (filter row rr, window s,
                // channel step k) triples, k fastest, walked by increments (a division or a long
                // carry chain per MMA costs the issuing thread most of its rate)
                const int n_st = g * windows * p.kq;
                const int lo = issuer * n_st / T, hi = (issuer + 1) * n_st / T;
                int rr = lo / (windows * p.kq);
                int s = (lo - rr * windows * p.kq) / p.kq;
                int k = lo - (rr * windows + s) * p.kq;
                for (int i = lo; i < hi; ++i) {
                    // window s of filter row rr: phase s mod S, rows (s div S) + rr I3 / S on;
                    // B: slices s .. s + S - 1 of triple rr
                    const uint64_t a_w = a_d + (uint32_t)(s & (p.S - 1)) * a_phase + (uint32_t)(s >> s_log2) * a_row +
                                         (uint32_t)rr * a_r2 + (uint32_t)k * a_step;
                    const uint64_t b_w = b_d + (uint32_t)rr * b_r2 + (uint32_t)s * b_slice + (uint32_t)k * b_step;
                    const uint32_t acc = mma >= my_acc ? 1u : 0u;  // first use overwrites
                    const uint32_t a_idx = (uint32_t)issuer + acc_j * (uint32_t)T;
                    umma_f16_pair(tmem_base + a_idx * acc_cols, a_w, b_w, p.idesc, acc);
                    ++mma;
                    if (++acc_j == my_acc) acc_j = 0;
                    if (++k == p.kq) {
                        k = 0;
                        if (++s == windows) {
                            s = 0;
                            ++rr;
                        }
                    }
                }
                umma_commit_mask(smem_u32(&empty_bar[slot]), pair_mask);  // stage free in both CTAs
                if (++slot == SA) {
                    slot = 0;
                    ph ^= 1;
                }
                if ((st + 1) % p.k_groups == 0 && ++grp == p.r2_groups) grp = 0;
            }
            if (ok) umma_commit_mask(smem_u32(done_bar), pair_mask);
            else aborted = true;
            // no MMA of this pair may still be running when TMEM and shared memory are released
            umma_commit_mask(smem_u32(drain_bar), pair_mask);
        }
        if (lane == 0 && warp - 1 < p.issuers) {
            // (the odd CTA's issuer warps wait here the whole main loop: sleep between polls)
            if (!mbar_wait_cluster_sleep(smem_u32(drain_bar), 0, p.limit_ns, nullptr, 1000)) {
                ct_record_error(p.status, kDevTimeoutDrain, abort_flag);
                aborted = true;
            }
        }
        __syncwarp();
        {
            // these warps take their share of the accumulators too (waiting, bounded, for the
            // MMAs; a timeout here is the epilogue's to report)
            bool ok = mbar_wait_cluster_sleep(smem_u32(done_bar), 0, p.limit_ns, abort_flag, 1000);
            ok = __all_sync(0xffffffffu, ok);
            if (ok) {
                tc_fence_after();
                part_ok = true;
                epilogue_share();
            }
        }
    } else {
        // ---------------------------------------------------------------- epilogue (both CTAs)
        bool ok = true;
        if (p.test_stall) {
            // test hook: a wait nothing will satisfy runs out and takes the abort path
            ok = mbar_wait(smem_u32(never_bar), 0, p.limit_ns);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok && lane == 0) ct_record_error(p.status, kDevTimeoutEpilogue, abort_flag);
        }
        if (ok) {
            // waits the whole main loop: sleep between polls
            ok = mbar_wait_cluster_sleep(smem_u32(done_bar), 0, p.limit_ns, abort_flag, 1000);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok && lane == 0) ct_record_error(p.status, kDevTimeoutEpilogue, abort_flag);
        }
        if (!ok) aborted = true;
        if (ok) {
            tc_fence_after();
            part_ok = true;
            epilogue_share();
        }
    }

    if (p.ks == 2) {
        // every CTA's part is in its shared memory (all threads of the cluster arrive, on every
        // path); then each slot's CTA adds the two parts of its rows for half of the columns,
        // slot 0's part + slot 1's part, reading the other slot's through distributed shared
        // memory, and stores y
        cluster_sync_all();
        if (part_ok) {
            // this warp's share of the slot's 8-column groups
            const uint32_t peer = crank ^ 2u;  // the same rows in the other slot's pair
            const int c_lo = kslot * (N / 2);
            for (int c0 = c_lo + 8 * share; c0 < c_lo + N / 2; c0 += 24) {
                float other[8], acc[8];
#pragma unroll
                for (int i = 0; i < 8; ++i)
                    other[i] = ld_shared_cluster_f32(mapa_shared(smem_u32(my_part + (c0 + i) * 32 + lane), peer));
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const float own = my_part[(c0 + i) * 32 + lane];
                    acc[i] = kslot == 0 ? __fadd_rn(own, other[i]) : __fadd_rn(other[i], own);
                }
                chunk_store(c0, acc);
            }
        }
    }

    // after an abort, give copies and MMAs already issued time to land before the pair's
    // shared memory and TMEM are released
    if (__syncthreads_or(aborted ? 1 : 0)) grace_period(2000000ull);
    tc_fence_before();
    __syncthreads();
    cluster_sync_all();  // no MMA, remote arrival or copy of the pair still targets this CTA
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc_pair(tmem_base, (uint32_t)p.tmem_cols);
    }
}

// Channel-first to channel-last re-layout of 16-bit tensors for the channel-first entry
// point: src [B][C][V] -> dst [B][V][Cp], channels C .. Cp-1 zero-filled (Cp a multiple of
// 16).  One launch does two independent jobs (the input, then the filters): the first
// `blocks0` blocks belong to the first job.  Within a job, row (b, 8-channel chunk) is split
// into blocks of 256 positions; a thread gathers the eight channels of one position (a
// warp's reads of one channel are 32 consecutive positions) and stores them as one 16-byte
// vector.
struct RelayoutJob {
    const uint16_t* src;
    uint16_t* dst;
    int64_t B, C, V, Cp;
    int64_t blocks_per_row;  // ceil(V / 256)
};

__global__ void __launch_bounds__(256) to_channel_last_kernel(RelayoutJob j0, RelayoutJob j1, int64_t blocks0)
{
    // the convolution launched next may set up (barriers, TMEM) now; its loads wait for this grid
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const bool first = blockIdx.x < blocks0;
    const RelayoutJob& j = first ? j0 : j1;
    const int64_t local = first ? (int64_t)blockIdx.x : (int64_t)blockIdx.x - blocks0;
    const int64_t row = local / j.blocks_per_row;
    const int64_t v = (local - row * j.blocks_per_row) * 256 + threadIdx.x;
    const int64_t chunks = j.Cp / 8;
    const int64_t b = row / chunks, c0 = (row - b * chunks) * 8;
    if (v >= j.V || b >= j.B) return;
    const uint16_t* s = j.src + b * j.C * j.V + v;
    uint16_t e[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int64_t c = c0 + i;
        e[i] = (c < j.C && in_range(b * j.C * j.V + c * j.V + v, j.B * j.C * j.V)) ? s[c * j.V] : (uint16_t)0;
    }
    if (!in_range(b * j.V * j.Cp + v * j.Cp + c0 + 7, j.B * j.V * j.Cp)) return;
    uint4 pk;
    pk.x = (uint32_t)e[0] | ((uint32_t)e[1] << 16);
    pk.y = (uint32_t)e[2] | ((uint32_t)e[3] << 16);
    pk.z = (uint32_t)e[4] | ((uint32_t)e[5] << 16);
    pk.w = (uint32_t)e[6] | ((uint32_t)e[7] << 16);
    *reinterpret_cast<uint4*>(j.dst + b * j.V * j.Cp + v * j.Cp + c0) = pk;
}

// Tensor maps over the caller's channel-last tensors (16-bit elements, box rows of 8
// channels = 16 bytes, no swizzle; out-of-range boxes read zeros).
//   x: [I0][I1 I2 I3 / S][S][C]  -> dims {C, S, I1 I2 I3 / S, I0}
//   w: [C_out][R0 R1 R2][R3][C]  -> dims {C, C_out, R3, R0 R1 R2} (C_out and r3 swapped, so
//      a box lands as [triple][r3][o][8 channels])
bool encode_conv_maps(CUtensorMap* tmX, CUtensorMap* tmW, const void* x, const void* w, bool bf16,
                      const ConvTcParams& p)
{
    auto enc = tensor_map_encoder();
    if (!enc) return false;
    const CUtensorMapDataType dt = bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    const cuuint64_t C = (cuuint64_t)p.cin, S = (cuuint64_t)p.S;
    const cuuint64_t plane = (cuuint64_t)p.I[1] * p.I[2] * p.I[3];
    cuuint64_t xd[4] = {C, S, plane / S, (cuuint64_t)p.I[0]};
    cuuint64_t xs[3] = {C * 2, S * C * 2, plane * C * 2};
    cuuint32_t xb[4] = {16, 1, (cuuint32_t)p.rows, 1};
    cuuint32_t es[4] = {1, 1, 1, 1};
    if (enc(tmX, dt, 4, const_cast<void*>(x), xd, xs, xb, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_32B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return false;
    const cuuint64_t R3 = (cuuint64_t)p.R[3], trips = (cuuint64_t)p.R[0] * p.R[1] * p.R[2];
    cuuint64_t wd[4] = {C, (cuuint64_t)p.cout, R3, trips};
    cuuint64_t ws[3] = {trips * R3 * C * 2, C * 2, R3 * C * 2};
    cuuint32_t wb[4] = {16, (cuuint32_t)(p.cout / 2), (cuuint32_t)p.nsl, (cuuint32_t)p.g2};
    return enc(tmW, dt, 4, const_cast<void*>(w), wd, ws, wb, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
               CU_TENSOR_MAP_SWIZZLE_32B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Stages in [a, b) whose filter-row group is gg; stage st has group (st / kg) % r2g.
int64_t stages_of_group(int64_t a, int64_t b, int64_t kg, int64_t r2g, int64_t gg)
{
    if (b <= a) return 0;
    auto blocks_below = [&](int64_t j) { return j / r2g + ((j % r2g) > gg ? 1 : 0); };  // j' < j with j' % r2g == gg
    const int64_t ja = a / kg, jb = (b - 1) / kg;  // first and last block of kg stages touched
    if (ja == jb) return (ja % r2g == gg) ? b - a : 0;
    int64_t n = 0;
    if (ja % r2g == gg) n += (ja + 1) * kg - a;
    if (jb % r2g == gg) n += b - jb * kg;
    n += (blocks_below(jb) - blocks_below(ja + 1)) * kg;
    return n;
}

// Tiling and pipeline of the convolution for stack S (GEMM_OK or GEMM_ERR_UNSUPPORTED).
// With tiles for at most a quarter of the SMs, the stage sequence of each tile is split
// over two pairs (K split, a cluster of four CTAs), so that the pairs fill the SMs.
int plan_conv4d_tc(int64_t cin, const int64_t in[4], int64_t cout, const int64_t k[4], int S, int num_sms,
                   int ks_opt, ConvTcParams* out)
{
    ConvTcParams p = {};
    if (cin % 16 || cout % 16 || S < 1 || in[3] % S || S * cout > 256) return GEMM_ERR_UNSUPPORTED;
    p.cin = (int)cin;
    p.cout = (int)cout;
    p.S = S;
    for (int d = 0; d < 4; ++d) {
        p.I[d] = (int)in[d];
        p.R[d] = (int)k[d];
        p.P[d] = (int)(in[d] - k[d] + 1);
    }
    const int64_t plane = in[1] * in[2] * in[3];
    if (plane * cin >= (1ll << 31) || in[0] * plane >= (1ll << 31) || k[0] * k[1] * k[2] * k[3] * cin >= (1ll << 31))
        return GEMM_ERR_UNSUPPORTED;
    // linear positions per slab that cover every valid (p1, p2, p3)
    const int64_t U = ((int64_t)(p.P[1] - 1) * in[2] + (p.P[2] - 1)) * in[3] + p.P[3];
    const int64_t per_tile = (int64_t)2 * CT_G * S;
    p.tiles_per_p0 = (int)((U + per_tile - 1) / per_tile);
    if ((int64_t)p.tiles_per_p0 * p.P[0] * 2 > 0x7fffffff) return GEMM_ERR_UNSUPPORTED;
    p.nsl = (int)(k[3] + 2 * S - 2);
    if (p.nsl > 256 || cout / 2 > 256) return GEMM_ERR_UNSUPPORTED;
    const int windows = (int)(k[3] + S - 1);
    const int ksteps = (int)(cin / 16);
    // the most filter rows r2 and then channel steps per stage that leave room for three
    // stages, with the input box at most 256 rows
    p.g2 = 0;
    for (int g2 = (int)k[2]; g2 >= 1 && p.g2 == 0; --g2) {
        const int64_t rows = CT_G + (windows - 1) / S + (int64_t)(g2 - 1) * (in[3] / S);
        if (rows > 256) continue;
        const int64_t rows8 = (rows + 7) / 8 * 8;
        for (int kq = ksteps; kq >= 1; --kq) {
            if (ksteps % kq) continue;
            // boxes start on 1024-byte boundaries (the swizzle pattern is a function of the
            // shared-memory address)
            const int64_t a_box = (rows8 * 32 + 1023) / 1024 * 1024;
            const int64_t b_box = ((int64_t)g2 * p.nsl * (cout / 2) * 32 + 1023) / 1024 * 1024;
            const int64_t stage = kq * S * a_box + kq * b_box;
            if (3 * stage > CT_SMEM_BUDGET) continue;
            p.g2 = g2;
            p.kq = kq;
            p.rows = (int)rows8;
            p.a_box = (int)a_box;
            p.b_box = (int)b_box;
            p.a_region = (int)(kq * S * a_box);
            p.tx_bytes = (int)(kq * S * rows8 * 32 + kq * (int64_t)g2 * p.nsl * (cout / 2) * 32);
            p.stage_bytes = (int)stage;
            break;
        }
    }
    if (p.g2 == 0) return GEMM_ERR_UNSUPPORTED;
    p.r2_groups = (p.R[2] + p.g2 - 1) / p.g2;
    p.k_groups = ksteps / p.kq;
    const int64_t nst = k[0] * k[1] * p.r2_groups * (int64_t)p.k_groups;
    if (nst >= (1 << 30)) return GEMM_ERR_UNSUPPORTED;
    p.num_stages = (int)nst;
    int ring = CT_SMEM_BUDGET / p.stage_bytes;
    if (ring > CT_MAX_STAGES) ring = CT_MAX_STAGES;
    if (ring > p.num_stages) ring = p.num_stages;
    p.nstages_ring = ring;
    // TMEM accumulators of N = S C_out columns, issuers dealt round-robin over them
    const int N = S * p.cout;
    int nacc = CT_TMEM_COLS / N;
    if (nacc > CT_MAX_ACC) nacc = CT_MAX_ACC;
    p.issuers = nacc < CT_ISSUERS_MAX ? nacc : CT_ISSUERS_MAX;
    nacc -= nacc % p.issuers;
    p.nacc = nacc;
    // K split: two pairs per tile (a cluster of four CTAs) when one pair per tile would leave
    // more than half the SMs idle, N is a multiple of 32 (each slot stores half the columns in
    // 16-column chunks) and there are at least two stages
    // (ks_opt: 0 choose, 1 one pair per tile, 2 two pairs per tile where the shape allows it)
    const int64_t tiles = (int64_t)p.tiles_per_p0 * p.P[0];
    const bool can_split = N % 32 == 0 && p.num_stages >= 2;
    if (ks_opt == 2 && !can_split) return GEMM_ERR_UNSUPPORTED;
    p.ks = ks_opt == 2 ? 2 : ks_opt == 1 ? 1 : (can_split && num_sms > 0 && 4 * tiles <= num_sms) ? 2 : 1;
    if (tiles * p.ks * 2 > 0x7fffffff) return GEMM_ERR_UNSUPPORTED;
    // the K split's partial parts (128 rows x N fp32) reuse the operand ring's shared memory,
    // which a short ring may not cover
    const int64_t ring_bytes = (int64_t)p.nstages_ring * p.stage_bytes;
    const int64_t part_bytes = p.ks == 2 ? (int64_t)CT_G * N * 4 : 0;
    p.bar_offset = (int)(ring_bytes > part_bytes ? ring_bytes : part_bytes);
    // accumulator i + issuers j of slot s is written iff issuer i issues more than j MMAs
    // in the slot's stages; issuer i takes MMAs [i n / issuers, (i + 1) n / issuers) of
    // every stage of n MMAs, and n depends on the stage's filter-row group
    for (int sl = 0; sl < CT_MAX_KS; ++sl) p.acc_used[sl] = 0;
    for (int sl = 0; sl < p.ks; ++sl) {
        const int64_t a0 = (int64_t)sl * nst / p.ks, b0 = (int64_t)(sl + 1) * nst / p.ks;
        for (int a = 0; a < nacc; ++a) {
            const int issuer = a % p.issuers, j = a / p.issuers;
            int64_t mine = 0;
            for (int grp = 0; grp < p.r2_groups; ++grp) {
                const int g = (p.R[2] - grp * p.g2) < p.g2 ? p.R[2] - grp * p.g2 : p.g2;
                const int64_t n = (int64_t)g * windows * p.kq;
                mine += stages_of_group(a0, b0, p.k_groups, p.r2_groups, grp) *
                        ((issuer + 1) * n / p.issuers - issuer * n / p.issuers);
            }
            if (mine > j) p.acc_used[sl] |= 1u << a;
        }
    }
    p.tmem_cols = 32;
    while (p.tmem_cols < nacc * N) p.tmem_cols *= 2;
    *out = p;
    return GEMM_OK;
}

// Positions stacked along N.  Four (N = 4 C_out, MMAs at the full rate from N = 128 on)
// when that plan, with its K split, fits the SMs in one wave and fills at least half of
// them: at 16^4 x 16 -> 32 channels, 5^4 filter, 29.3 us per call back to back against
// 35.1 us for two positions without a split, although the stacked zero blocks grow from 1/6
// to 3/8 of the products.
// Else two when the shape allows it, else one.
int choose_stack(int64_t cin, const int64_t in[4], int64_t cout, const int64_t k[4], int num_sms, int ks_opt)
{
    ConvTcParams p;
    if (plan_conv4d_tc(cin, in, cout, k, 4, num_sms, ks_opt, &p) == GEMM_OK) {
        const int64_t ctas = (int64_t)2 * p.ks * p.tiles_per_p0 * p.P[0];
        if (p.ks == 2 && ctas <= num_sms && 2 * ctas >= num_sms) return 4;
    }
    for (int S : {2, 1})
        if (plan_conv4d_tc(cin, in, cout, k, S, num_sms, ks_opt, &p) == GEMM_OK) return S;
    return 0;
}

}  // namespace

int conv4d_tc_supported(int64_t cin, const int64_t in[4], int64_t cout, const int64_t k[4], int S, int ks_opt,
                        int num_sms)
{
    ConvTcParams p;
    if (S <= 0) S = choose_stack(cin, in, cout, k, num_sms, ks_opt);
    if (S <= 0 || plan_conv4d_tc(cin, in, cout, k, S, num_sms, ks_opt, &p) != GEMM_OK) return GEMM_ERR_UNSUPPORTED;
    return GEMM_OK;  // the operands are read straight from the caller's tensors: no workspace
}

int launch_conv4d_tc(const void* x, int64_t cin, const int64_t in[4], const void* w, int64_t cout,
                     const int64_t k[4], float* y, int64_t ldy_cf, bool bf16, int S, int ks_opt, int num_sms,
                     int* dev_status, uint64_t limit_ns, int test_stall, bool programmatic, cudaStream_t stream,
                     int* launches)
{
    if (S <= 0) S = choose_stack(cin, in, cout, k, num_sms, ks_opt);
    if (S <= 0) return GEMM_ERR_UNSUPPORTED;
    ConvTcParams p;
    const int rc = plan_conv4d_tc(cin, in, cout, k, S, num_sms, ks_opt, &p);
    if (rc != GEMM_OK) return rc;
    p.idesc = conv_idesc(bf16, S * p.cout);
    p.y = y;
    p.ldy_cf = ldy_cf;
    p.status = dev_status;
    p.limit_ns = limit_ns;
    p.test_stall = test_stall;
    CUtensorMap tmX, tmW;
    if (!encode_conv_maps(&tmX, &tmW, x, w, bf16, p)) return GEMM_ERR_CUDA;
    const int smem = p.bar_offset + 1024 /*barriers*/ + 1024 /*alignment slack*/;
    if (cudaFuncSetAttribute(conv4d_tc_pair_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
        return GEMM_ERR_CUDA;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(2 * p.ks * p.tiles_per_p0 * p.P[0]), 1, 1);
    cfg.blockDim = dim3(CT_THREADS, 1, 1);
    cfg.dynamicSmemBytes = (size_t)smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2 * p.ks;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = programmatic ? 2 : 1;
    if (p.ks == 2 && ks_opt == 0) {
        // clusters of four CTAs of ~200 KiB each may not be placeable (a partitioned device):
        // then one pair per tile, clusters of two
        int clusters = 0;
        if (cudaOccupancyMaxActiveClusters(&clusters, conv4d_tc_pair_kernel, &cfg) != cudaSuccess || clusters < 1) {
            (void)cudaGetLastError();
            return launch_conv4d_tc(x, cin, in, w, cout, k, y, ldy_cf, bf16, S, 1, num_sms, dev_status, limit_ns,
                                    test_stall, programmatic, stream, launches);
        }
    }
    if (cudaLaunchKernelEx(&cfg, conv4d_tc_pair_kernel, tmX, tmW, p) != cudaSuccess) return GEMM_ERR_CUDA;
    *launches += 1;
    return GEMM_OK;
}

cudaError_t launch_to_channel_last(const void* x, int64_t C, int64_t V, void* xc, const void* w, int64_t B,
                                   int64_t T, void* wc, int64_t Cp, cudaStream_t stream)
{
    if (C <= 0 || V <= 0 || B <= 0 || T <= 0 || Cp < C || Cp % 16 != 0 ||
        ((reinterpret_cast<uintptr_t>(xc) | reinterpret_cast<uintptr_t>(wc)) & 15) != 0)
        return cudaErrorInvalidValue;
    RelayoutJob jx = {static_cast<const uint16_t*>(x), static_cast<uint16_t*>(xc), 1, C, V, Cp, (V + 255) / 256};
    RelayoutJob jw = {static_cast<const uint16_t*>(w), static_cast<uint16_t*>(wc), B, C, T, Cp, (T + 255) / 256};
    const int64_t bx = jx.blocks_per_row * (Cp / 8), bw = jw.blocks_per_row * B * (Cp / 8);
    if (bx + bw > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    to_channel_last_kernel<<<(unsigned)(bx + bw), 256, 0, stream>>>(jx, jw, bx);
    return cudaGetLastError();
}

}  // namespace gemm_gb300
