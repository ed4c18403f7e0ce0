// Valid 4-D cross-correlation as an implicit GEMM: the im2col matrix is never built.
//
// "Three X: large convolutions in PyTorch for training", sections "CUTLASS" and "What
// else had to change when using CUTLASS": implicit GEMM computes the convolution as the
// GEMM  y[o][p] = sum_k W[o][k] col[k][p]  but produces the needed elements of the
// column matrix from the input tensor on the fly (the "analytic" iterator recomputes
// input coordinates from the output position and the filter tap) instead of storing it.
// Here, with taps ordered (c, r0, r1, r2, r3) (r3 fastest) and output positions ordered
// (p0, p1, p2, p3) (p3 fastest):
//   col[(c,r0,r1,r2,r3)][(p0,p1,p2,p3)] = x[c][p0+r0][p1+r1][p2+r2][p3+r3]
//     = x[ tap_group_base(c,r0,r1,r2) + position_base(p0,p1,p2) + p3 + r3 ].
// A thread owns four adjacent positions of one p3-row and all 32 output channels.  For one
// tap group (c, r0, r1, r2) its R3 taps need x[base + p3 .. base + p3 + 3 + R3 - 1]: with
// R3 = 5 exactly eight consecutive floats that end inside the input row, two aligned float4
// loads shared by 5 x 4 x 32 fused multiply-adds (packed fma.rn.f32x2 on pairs of adjacent
// output channels, so the weights feed them as they are and only the eight input values are
// duplicated).  These window loads run two tap groups ahead of their use, in a ring of
// three register windows that continues across weight chunks, and the input offset of the
// next tap group is advanced incrementally (counters for r2, r1, r0, c) instead of being
// decoded with divisions.  Weights are staged in shared memory 24 tap groups at a time,
// double buffered: a chunk is loaded to registers while the previous one is multiplied.
// The grid is persistent over (position block, tap-group slice) items; slices write
// partial sums that the fixed-order split-K reduction adds, so results are deterministic.
// Shapes the R3 = 5 path does not cover (misaligned x, p3 extent not a multiple of 4,
// R3 other than 5, rows not 16-byte aligned) run a general kernel with scalar loads, two
// thread groups of 16 output channels and 40-tap weight chunks.
#include "internal.h"

namespace gemm_gb300 {

GEMM_DEBUG_UNIT(conv_implicit)

namespace {

constexpr int CI_COL_THREADS = 256;                 // threads across positions (4 each)
constexpr int CI_POS = 4 * CI_COL_THREADS;          // 1024 positions per item
constexpr int CI_MR = 32;                           // output channels per launch (max)
// general kernel: two thread groups of 16 output channels, 40-tap weight chunks
constexpr int CI_MSPLIT = 2;
constexpr int CI_THREADS = CI_COL_THREADS * CI_MSPLIT;
constexpr int CI_RT = CI_MR / CI_MSPLIT;
constexpr int CI_TAPS_PER_CHUNK = 40;
constexpr int CI_MAX_GROUPS_PER_CHUNK = 8;
constexpr int CI_MAX_R3 = CI_TAPS_PER_CHUNK;
// R3 = 5 kernel: one thread group of 32 output channels, 24 tap groups per weight chunk
constexpr int CI_VEC_R3 = 5;
constexpr int CI5_GPC = 24;  // a multiple of the three-window ring

struct ConvGeom {
    int cout, cin;
    int i0, i1, i2, i3;  // input extents
    int r0, r1, r2, r3;  // kernel extents
    int p0, p1, p2, p3;  // output extents
    int64_t npos;        // p0*p1*p2*p3
    int64_t ntaps;       // cin*r0*r1*r2*r3
    int ngroups;         // cin*r0*r1*r2 (tap groups)
    int64_t chan_stride; // i0*i1*i2*i3
};

struct ConvParams {
    ConvGeom g;
    const float* x;
    const float* w;   // [cout][ntaps]
    float* y;         // [cout][npos] with row stride ldy
    int64_t ldy;
    int groups_per_slice;
    int groups_per_chunk;  // min(8, 40 / r3)
    int nslice;
    int pos_blocks;
    int num_items;
    float* ws;        // [nslice][cout][npos] partials when nslice > 1
    int vec_out;
};

// input offset of tap group q = (c, r0, r1, r2) at output position (0, 0, 0, 0)
__device__ __forceinline__ int64_t group_base(const ConvGeom& g, int q)
{
    const int r2 = q % g.r2;
    int t = q / g.r2;
    const int r1 = t % g.r1;
    t /= g.r1;
    const int r0 = t % g.r0;
    const int c = t / g.r0;
    return (int64_t)c * g.chan_stride + (((int64_t)r0 * g.i1 + r1) * g.i2 + r2) * g.i3;
}

__global__ void __launch_bounds__(CI_THREADS, 1) conv4d_implicit_general_kernel(ConvParams p)
{
    // the split-K reduction launched next may start its blocks now; it waits for this grid
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    constexpr int W_PER_THREAD = (CI_TAPS_PER_CHUNK * CI_MR + CI_THREADS - 1) / CI_THREADS;
    __shared__ __align__(16) float wsm[2][CI_TAPS_PER_CHUNK][CI_MR];  // weights, [tap][out channel]
    __shared__ int64_t gbase[2][CI_MAX_GROUPS_PER_CHUNK];

    const ConvGeom& g = p.g;
    const int tid = threadIdx.x;
    const int ct = tid % CI_COL_THREADS;
    const int mg = tid / CI_COL_THREADS;
    const int m_base = mg * CI_RT;
    const int gpc = p.groups_per_chunk;
    const int ntap_chunk = gpc * g.r3;

    for (int item = blockIdx.x; item < p.num_items; item += gridDim.x) {
        const int pb = item % p.pos_blocks, sl = item / p.pos_blocks;
        const int q_begin = sl * p.groups_per_slice;
        const int q_end = min(g.ngroups, q_begin + p.groups_per_slice);

        // this thread's four positions n0 .. n0+3 (one p3-row when p3 % 4 == 0)
        const int64_t n0 = (int64_t)pb * CI_POS + ct * 4;
        const bool pos_ok = n0 < g.npos;
        int64_t pbase[4];  // input offset of position n0 + j at tap (0, 0, 0, 0, 0)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            int64_t n = n0 + j;
            if (n >= g.npos) n = g.npos - 1;  // clamped; never stored
            const int q3 = (int)(n % g.p3);
            int64_t t = n / g.p3;
            const int q2 = (int)(t % g.p2);
            t /= g.p2;
            const int q1 = (int)(t % g.p1);
            const int q0 = (int)(t / g.p1);
            pbase[j] = (((int64_t)q0 * g.i1 + q1) * g.i2 + q2) * g.i3 + q3;
        }

        // acc[mm][j] = output channels (m_base + 2mm, m_base + 2mm + 1) at position n0 + j
        float2 acc[CI_RT / 2][4];
#pragma unroll
        for (int m = 0; m < CI_RT / 2; ++m)
#pragma unroll
            for (int j = 0; j < 4; ++j) acc[m][j] = make_float2(0.f, 0.f);

        // weights of tap groups [qc, qc + gpc): loaded to registers one chunk ahead, then
        // stored to wsm[buf] (so the L2 latency overlaps the previous chunk's FMAs)
        float wreg[W_PER_THREAD];
        int64_t gb_reg = 0;
        // element e of a chunk = (tap e / 32, output channel e % 32): a warp stores one tap
        // row of 32 channels, conflict-free
        auto load_w = [&](int qc) {
#pragma unroll
            for (int i = 0; i < W_PER_THREAD; ++i) {
                const int e = tid + i * CI_THREADS;
                float v = 0.f;
                if (e < ntap_chunk * CI_MR) {
                    const int tap = e / CI_MR, m = e % CI_MR;
                    const int q = qc + tap / g.r3;
                    if (m < g.cout && q < q_end && in_range(m, g.cout) && in_range((int64_t)q * g.r3 + tap % g.r3, g.ntaps))
                        v = __ldg(p.w + (int64_t)m * g.ntaps + (int64_t)q * g.r3 + tap % g.r3);
                }
                wreg[i] = v;
            }
            if (tid < gpc) gb_reg = (qc + tid < q_end) ? group_base(g, qc + tid) : 0;
        };
        auto store_w = [&](int buf) {
#pragma unroll
            for (int i = 0; i < W_PER_THREAD; ++i) {
                const int e = tid + i * CI_THREADS;
                if (e < ntap_chunk * CI_MR) wsm[buf][e / CI_MR][e % CI_MR] = wreg[i];
            }
            if (tid < gpc) gbase[buf][tid] = gb_reg;
        };

        int buf = 0;
        load_w(q_begin);
        store_w(0);
        __syncthreads();
        for (int qc = q_begin; qc < q_end; qc += gpc) {
            const bool more = qc + gpc < q_end;
            if (more) load_w(qc + gpc);
            const int nq = min(gpc, q_end - qc);
            for (int qi = 0; qi < nq; ++qi) {
                const int64_t gb = gbase[buf][qi];
                for (int r3 = 0; r3 < g.r3; ++r3) {
                    float2 sd[4];
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const float s1 = (n0 + j < g.npos && in_range(gb + pbase[j] + r3, (int64_t)g.cin * g.chan_stride))
                                             ? __ldg(p.x + gb + pbase[j] + r3)
                                             : 0.f;
                        sd[j] = make_float2(s1, s1);
                    }
                    const float* wrow = &wsm[buf][qi * g.r3 + r3][m_base];
#pragma unroll
                    for (int m = 0; m < CI_RT; m += 4) {
                        const float4 w4 = *reinterpret_cast<const float4*>(wrow + m);
                        const float2 w01 = make_float2(w4.x, w4.y), w23 = make_float2(w4.z, w4.w);
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            acc[m / 2][j] = __ffma2_rn(w01, sd[j], acc[m / 2][j]);
                            acc[m / 2 + 1][j] = __ffma2_rn(w23, sd[j], acc[m / 2 + 1][j]);
                        }
                    }
                }
            }
            if (more) store_w(buf ^ 1);
            __syncthreads();  // next chunk's weights visible; this chunk's no longer read
            buf ^= 1;
        }

        if (pos_ok) {
            float* out;
            int64_t ldo;
            if (p.nslice > 1) {
                out = p.ws + (int64_t)sl * g.cout * g.npos;
                ldo = g.npos;
            } else {
                out = p.y;
                ldo = p.ldy;
            }
#pragma unroll
            for (int m = 0; m < CI_RT; ++m) {
                if (m_base + m >= g.cout) break;
                if (!in_range(m_base + m, g.cout) || !in_range(n0, g.npos)) break;
                float* dst = out + (int64_t)(m_base + m) * ldo + n0;
                float o[4];
#pragma unroll
                for (int j = 0; j < 4; ++j) o[j] = (m % 2 == 0) ? acc[m / 2][j].x : acc[m / 2][j].y;
                if (p.vec_out && n0 + 3 < g.npos) {
                    if (in_range(n0 + 3, g.npos)) *reinterpret_cast<float4*>(dst) = make_float4(o[0], o[1], o[2], o[3]);
                } else {
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        if (n0 + j < g.npos) dst[j] = o[j];
                }
            }
        }
    }
}

// R3 = 5, float4-aligned input rows: the window of four positions x five taps is two float4
// loads, issued two tap groups before their use
__global__ void __launch_bounds__(CI_COL_THREADS, 1) conv4d_implicit_r5_kernel(ConvParams p)
{
    // the split-K reduction launched next may start its blocks now; it waits for this grid
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    constexpr int THREADS = CI_COL_THREADS;
    constexpr int R3 = CI_VEC_R3;
    constexpr int TAPS = CI5_GPC * R3;
    constexpr int W_PER_THREAD = (TAPS * CI_MR + THREADS - 1) / THREADS;
    static_assert(CI5_GPC % 3 == 0, "the window ring is three deep");
    __shared__ __align__(16) float wsm[2][TAPS][CI_MR];  // weights, [tap][out channel]

    const ConvGeom& g = p.g;
    const int tid = threadIdx.x;
    const int64_t x_elems = (int64_t)g.cin * g.chan_stride;
    // input-offset steps when r2, r1 or r0 wraps around (the next tap group's counters)
    const int64_t d_r1 = (int64_t)(g.i2 - g.r2) * g.i3;
    const int64_t d_r0 = (int64_t)(g.i1 - g.r1) * g.i2 * g.i3;
    const int64_t d_c = g.chan_stride - (int64_t)g.r0 * g.i1 * g.i2 * g.i3;

    for (int item = blockIdx.x; item < p.num_items; item += gridDim.x) {
        const int pb = item % p.pos_blocks, sl = item / p.pos_blocks;
        const int q_begin = sl * p.groups_per_slice;
        const int q_end = min(g.ngroups, q_begin + p.groups_per_slice);

        // this thread's four positions n0 .. n0+3 lie in one p3-row (p3 % 4 == 0)
        const int64_t n0 = (int64_t)pb * CI_POS + tid * 4;
        const bool pos_ok = n0 < g.npos;
        int64_t pbase0;  // input offset of position n0 at tap (0, 0, 0, 0, 0)
        {
            const int64_t n = pos_ok ? n0 : 0;
            const int q3 = (int)(n % g.p3);
            int64_t t = n / g.p3;
            const int q2 = (int)(t % g.p2);
            t /= g.p2;
            const int q1 = (int)(t % g.p1);
            const int q0 = (int)(t / g.p1);
            pbase0 = (((int64_t)q0 * g.i1 + q1) * g.i2 + q2) * g.i3 + q3;
        }

        // acc[mm][j] = output channels (2mm, 2mm + 1) at position n0 + j
        float2 acc[CI_MR / 2][4];
#pragma unroll
        for (int m = 0; m < CI_MR / 2; ++m)
#pragma unroll
            for (int j = 0; j < 4; ++j) acc[m][j] = make_float2(0.f, 0.f);

        // the next tap group to load: its r2, r1, r0 counters and its window's input offset
        int wr2, wr1, wr0;
        {
            int t = q_begin;
            wr2 = t % g.r2;
            t /= g.r2;
            wr1 = t % g.r1;
            t /= g.r1;
            wr0 = t % g.r0;
        }
        int64_t wgb = group_base(g, q_begin) + pbase0;
        auto load_window = [&](float (&v)[8]) {
            if (pos_ok && in_range(wgb, x_elems) && in_range(wgb + 7, x_elems)) {
                const float4* src = reinterpret_cast<const float4*>(p.x + wgb);
                const float4 lo = __ldg(src);
                const float4 hi = __ldg(src + 1);
                v[0] = lo.x, v[1] = lo.y, v[2] = lo.z, v[3] = lo.w;
                v[4] = hi.x, v[5] = hi.y, v[6] = hi.z, v[7] = hi.w;
            } else {
#pragma unroll
                for (int j = 0; j < 8; ++j) v[j] = 0.f;
            }
            wgb += g.i3;
            if (++wr2 == g.r2) {
                wr2 = 0;
                wgb += d_r1;
                if (++wr1 == g.r1) {
                    wr1 = 0;
                    wgb += d_r0;
                    if (++wr0 == g.r0) {
                        wr0 = 0;
                        wgb += d_c;
                    }
                }
            }
        };

        // weights of tap groups [qc, qc + CI5_GPC); element e of a chunk = (tap e / 32, output
        // channel e % 32): a warp stores one tap row of 32 channels, conflict-free
        float wreg[W_PER_THREAD];
        auto load_w = [&](int qc) {
#pragma unroll
            for (int i = 0; i < W_PER_THREAD; ++i) {
                const int e = tid + i * THREADS;
                float v = 0.f;
                if (e < TAPS * CI_MR) {
                    const int tap = e / CI_MR, m = e % CI_MR;
                    const int q = qc + tap / R3;
                    const int64_t k = (int64_t)q * R3 + tap % R3;
                    if (m < g.cout && q < q_end && in_range(m, g.cout) && in_range(k, g.ntaps))
                        v = __ldg(p.w + (int64_t)m * g.ntaps + k);
                }
                wreg[i] = v;
            }
        };
        auto store_w = [&](int buf) {
#pragma unroll
            for (int i = 0; i < W_PER_THREAD; ++i) {
                const int e = tid + i * THREADS;
                if (e < TAPS * CI_MR) wsm[buf][e / CI_MR][e % CI_MR] = wreg[i];
            }
        };
        // the 5 taps x 4 positions x 32 channels of one tap group
        auto multiply = [&](const float (&v)[8], const float* wq) {
            float2 vd[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) vd[i] = make_float2(v[i], v[i]);
#pragma unroll
            for (int r3 = 0; r3 < R3; ++r3) {
                const float* wrow = wq + r3 * CI_MR;
#pragma unroll
                for (int m = 0; m < CI_MR; m += 4) {
                    const float4 w4 = *reinterpret_cast<const float4*>(wrow + m);
                    const float2 w01 = make_float2(w4.x, w4.y), w23 = make_float2(w4.z, w4.w);
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        acc[m / 2][j] = __ffma2_rn(w01, vd[r3 + j], acc[m / 2][j]);
                        acc[m / 2 + 1][j] = __ffma2_rn(w23, vd[r3 + j], acc[m / 2 + 1][j]);
                    }
                }
            }
        };

        int buf = 0;
        load_w(q_begin);
        store_w(0);
        __syncthreads();
        // windows of tap groups q, q + 1, q + 2 rotate through xa, xb, xc
        float xa[8], xb[8], xc[8];
        if (q_begin < q_end) load_window(xa);
        if (q_begin + 1 < q_end) load_window(xb);
        for (int qc = q_begin; qc < q_end; qc += CI5_GPC) {
            const bool more = qc + CI5_GPC < q_end;
            if (more) load_w(qc + CI5_GPC);
            const float* wc = &wsm[buf][0][0];
            for (int qi = 0; qi < CI5_GPC; qi += 3) {
                const int q = qc + qi;
                if (q >= q_end) break;
                if (q + 2 < q_end) load_window(xc);
                multiply(xa, wc + qi * R3 * CI_MR);
                if (q + 1 >= q_end) break;
                if (q + 3 < q_end) load_window(xa);
                multiply(xb, wc + (qi + 1) * R3 * CI_MR);
                if (q + 2 >= q_end) break;
                if (q + 4 < q_end) load_window(xb);
                multiply(xc, wc + (qi + 2) * R3 * CI_MR);
            }
            if (more) store_w(buf ^ 1);
            __syncthreads();  // next chunk's weights visible; this chunk's no longer read
            buf ^= 1;
        }

        if (pos_ok) {
            float* out;
            int64_t ldo;
            if (p.nslice > 1) {
                out = p.ws + (int64_t)sl * g.cout * g.npos;
                ldo = g.npos;
            } else {
                out = p.y;
                ldo = p.ldy;
            }
#pragma unroll
            for (int m = 0; m < CI_MR; ++m) {
                if (m >= g.cout) break;
                if (!in_range(m, g.cout) || !in_range(n0 + 3, g.npos)) break;
                float* dst = out + (int64_t)m * ldo + n0;
                float o[4];
#pragma unroll
                for (int j = 0; j < 4; ++j) o[j] = (m % 2 == 0) ? acc[m / 2][j].x : acc[m / 2][j].y;
                if (p.vec_out)
                    *reinterpret_cast<float4*>(dst) = make_float4(o[0], o[1], o[2], o[3]);
                else
#pragma unroll
                    for (int j = 0; j < 4; ++j) dst[j] = o[j];
            }
        }
    }
}

}  // namespace

int conv_implicit_auto_split(int64_t npos, int ngroups, int num_sms)
{
    const int64_t pbs = (npos + CI_POS - 1) / CI_POS;
    int64_t max_s = ngroups / 16;  // at least 16 tap groups per slice
    if (max_s < 1) max_s = 1;
    if (max_s > 1024) max_s = 1024;
    for (int64_t s = 1; s <= max_s; ++s) {
        const int64_t items = pbs * s;
        const int64_t waves = (items + num_sms - 1) / num_sms;
        if ((double)items / (double)(waves * num_sms) >= 0.92) return (int)s;
        if (items >= 4 * num_sms) return (int)s;
    }
    return (int)max_s;
}

cudaError_t launch_conv4d_implicit(const float* x, int64_t cin, const int64_t in[4], const float* w,
                                   int64_t cout, const int64_t k[4], float* y, int64_t ldy, int split,
                                   float* ws, int num_sms, cudaStream_t stream, int* launches)
{
    ConvParams p;
    ConvGeom& g = p.g;
    g.cout = (int)cout;
    g.cin = (int)cin;
    g.i0 = (int)in[0], g.i1 = (int)in[1], g.i2 = (int)in[2], g.i3 = (int)in[3];
    g.r0 = (int)k[0], g.r1 = (int)k[1], g.r2 = (int)k[2], g.r3 = (int)k[3];
    g.p0 = (int)(in[0] - k[0] + 1), g.p1 = (int)(in[1] - k[1] + 1), g.p2 = (int)(in[2] - k[2] + 1),
    g.p3 = (int)(in[3] - k[3] + 1);
    g.npos = (int64_t)g.p0 * g.p1 * g.p2 * g.p3;
    g.ntaps = cin * k[0] * k[1] * k[2] * k[3];
    g.ngroups = (int)(cin * k[0] * k[1] * k[2]);
    g.chan_stride = in[0] * in[1] * in[2] * in[3];
    p.x = x;
    p.w = w;
    p.y = y;
    p.ldy = ldy;
    if (g.r3 > CI_MAX_R3 || cout > CI_MR) return cudaErrorInvalidValue;
    p.groups_per_chunk = CI_TAPS_PER_CHUNK / g.r3 < CI_MAX_GROUPS_PER_CHUNK ? CI_TAPS_PER_CHUNK / g.r3
                                                                            : CI_MAX_GROUPS_PER_CHUNK;
    if (split < 1) split = 1;
    int gps = (g.ngroups + split - 1) / split;
    p.groups_per_slice = gps;
    p.nslice = (g.ngroups + gps - 1) / gps;
    p.pos_blocks = (int)((g.npos + CI_POS - 1) / CI_POS);
    const int64_t items = (int64_t)p.pos_blocks * p.nslice;
    if (items > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    p.num_items = (int)items;
    p.ws = ws;
    p.vec_out = (p.nslice > 1) ? (g.npos % 4 == 0)
                               : ((reinterpret_cast<uintptr_t>(y) & 15) == 0 && ldy % 4 == 0);
    // float4 gathers: 16-byte aligned x and rows, four positions per p3-row, R3 = 5
    const bool vec = (reinterpret_cast<uintptr_t>(x) & 15) == 0 && g.i3 % 4 == 0 && g.p3 % 4 == 0 &&
                     g.r3 == CI_VEC_R3;
    const int grid = (int)(items < num_sms ? items : num_sms);
    if (vec)
        conv4d_implicit_r5_kernel<<<grid, CI_COL_THREADS, 0, stream>>>(p);
    else
        conv4d_implicit_general_kernel<<<grid, CI_THREADS, 0, stream>>>(p);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    *launches += 1;
    if (p.nslice == 1) return cudaSuccess;
    *launches += 1;
    return launch_splitk_reduce(ws, p.nslice, cout, g.npos, y, ldy, num_sms, stream);
}

}  // namespace gemm_gb300
