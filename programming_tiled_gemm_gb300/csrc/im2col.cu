// Lowering of a valid 4-D cross-correlation to a GEMM operand (im2col in four dimensions).
//
// "Three X: large convolutions in PyTorch for training", section "CuBLAS": the
// convolution matrix has one column per application of the filter and one row per
// filter tap; PyTorch's im2col / vol2col kernels give one thread per element (a
// grid-stride loop) and compute from its position where the filter was applied; the
// 3-D version adds one index and one loop, and higher dimensions do the same again.
// Here: col[(c, r0, r1, r2, r3)][(p0, p1, p2, p3)] = x[c][p0+r0][p1+r1][p2+r2][p3+r3],
// both indices row-major.  Each thread writes four adjacent columns of one row with a
// single float4 store when the row is 16-byte aligned (the column count is a multiple of
// four); the writes are the whole cost (the input is small and stays in L2).  The
// element index is recovered from the position once per column (not once per element):
// the position's share of the source offset does not depend on the row.
#include "internal.h"

namespace gemm_gb300 {

GEMM_DEBUG_UNIT(im2col)

namespace {

struct Im2colGeom {
    int64_t nrows;             // cin*k0*k1*k2*k3
    int ncols;                 // p0*p1*p2*p3 (< 2^31, checked by the launcher)
    int k0, k1, k2, k3;        // kernel extents
    int in1, in2, in3;         // input extents (in0 only enters through the channel stride)
    int p1, p2, p3;            // output extents
    int64_t chan_stride;       // in0*in1*in2*in3
    int64_t x_elems;           // cin * chan_stride (index checks of debug builds)
};

// The position part of a column's source offset is the same for every row:
//   col[row][n] = x[base(row) + off(n)],  base(row) = c * chan_stride + tap offset,
//   off(n) = ((q0 * in1 + q1) * in2 + q2) * in3 + q3   for n = (q0, q1, q2, q3).
// A block owns IM_COLS consecutive columns: it computes their offsets once into shared
// memory and then walks rows (grid-stride over blockIdx.y), so the inner loop is a
// table lookup, four gathered loads (x stays in L2) and one streamed float4 store per
// thread, with no division.  The stores are the whole cost.
constexpr int IM_THREADS = 256;
constexpr int IM_COLS = 4 * IM_THREADS;

template <bool QUAD>
__global__ void __launch_bounds__(IM_THREADS) im2col4d_kernel(const float* __restrict__ x, Im2colGeom g,
                                                              float* __restrict__ col)
{
    __shared__ int off[IM_COLS];
    const int c0 = blockIdx.x * IM_COLS;
    for (int j = threadIdx.x; j < IM_COLS; j += IM_THREADS) {
        const int n = c0 + j;
        int o = 0;
        if (n < g.ncols) {
            const int q3 = n % g.p3;
            int u = n / g.p3;
            const int q2 = u % g.p2;
            u /= g.p2;
            const int q1 = u % g.p1;
            const int q0 = u / g.p1;
            o = ((q0 * g.in1 + q1) * g.in2 + q2) * g.in3 + q3;  // < in0*in1*in2*in3 < 2^31
        }
        off[j] = o;
    }
    __syncthreads();
    const int n0 = c0 + 4 * threadIdx.x;
    if (n0 >= g.ncols) return;
    const int4 o4 = *reinterpret_cast<const int4*>(&off[4 * threadIdx.x]);
    for (int64_t row = blockIdx.y; row < g.nrows; row += gridDim.y) {
        int64_t t = row;
        const int r3 = (int)(t % g.k3);
        t /= g.k3;
        const int r2 = (int)(t % g.k2);
        t /= g.k2;
        const int r1 = (int)(t % g.k1);
        t /= g.k1;
        const int r0 = (int)(t % g.k0);
        const int64_t c = t / g.k0;
        // input element of output position (0, 0, 0, 0) for this tap
        const int64_t xo = c * g.chan_stride + (((int64_t)r0 * g.in1 + r1) * g.in2 + r2) * g.in3 + r3;
        const float* xb = x + xo;
        float* dst = col + row * (int64_t)g.ncols + n0;
        if (!in_range(xo + o4.x, g.x_elems) || !in_range(xo + (n0 + 3 < g.ncols ? o4.w : o4.x), g.x_elems)) continue;
        if (QUAD) {
            if (!in_range(n0 + 3, g.ncols)) continue;
            float4 v;
            v.x = __ldg(xb + o4.x);
            v.y = __ldg(xb + o4.y);
            v.z = __ldg(xb + o4.z);
            v.w = __ldg(xb + o4.w);
            __stcs(reinterpret_cast<float4*>(dst), v);  // streamed: read later, L2 would not hold it
        } else {
            const int o[4] = {o4.x, o4.y, o4.z, o4.w};
            for (int j = 0; j < 4 && n0 + j < g.ncols; ++j) dst[j] = __ldg(xb + o[j]);
        }
    }
}

// The rows of one tap group (c, r0, r1, r2) differ only in r3, and the R3 source windows
// of a column quad overlap: with R3 = 5, p3 % 4 == 0, in3 % 4 == 0 and x 16-byte aligned,
// the quad's source for r3 = 0 is 16-byte aligned and x[.. + 0 .. 7] covers all five
// windows and ends at the input row's last element (q3 + 7 <= p3 - 4 + 7 = in3 - 1).  So a thread loads two float4s once and stores R3
// float4s, one per row of the group (rows are consecutive: r3 is the fastest tap index).
__global__ void __launch_bounds__(IM_THREADS) im2col4d_group_kernel(const float* __restrict__ x, Im2colGeom g,
                                                                    float* __restrict__ col)
{
    __shared__ int off[IM_COLS];
    const int c0 = blockIdx.x * IM_COLS;
    for (int j = threadIdx.x; j < IM_COLS; j += IM_THREADS) {
        const int n = c0 + j;
        int o = 0;
        if (n < g.ncols) {
            const int q3 = n % g.p3;
            int u = n / g.p3;
            const int q2 = u % g.p2;
            u /= g.p2;
            const int q1 = u % g.p1;
            const int q0 = u / g.p1;
            o = ((q0 * g.in1 + q1) * g.in2 + q2) * g.in3 + q3;
        }
        off[j] = o;
    }
    __syncthreads();
    const int n0 = c0 + 4 * threadIdx.x;
    if (n0 >= g.ncols) return;
    const int o = off[4 * threadIdx.x];  // the quad's four sources are consecutive
    const int64_t groups = g.nrows / g.k3;
    for (int64_t grp = blockIdx.y; grp < groups; grp += gridDim.y) {
        int64_t t = grp;
        const int r2 = (int)(t % g.k2);
        t /= g.k2;
        const int r1 = (int)(t % g.k1);
        t /= g.k1;
        const int r0 = (int)(t % g.k0);
        const int64_t c = t / g.k0;
        const int64_t xo = c * g.chan_stride + (((int64_t)r0 * g.in1 + r1) * g.in2 + r2) * g.in3 + o;
        if (!in_range(xo, g.x_elems) || !in_range(xo + 7, g.x_elems) || !in_range(grp * g.k3 + 4, g.nrows) ||
            !in_range(n0 + 3, g.ncols))
            continue;
        const float* src = x + xo;
        const float4 lo = __ldg(reinterpret_cast<const float4*>(src));
        const float4 hi = __ldg(reinterpret_cast<const float4*>(src + 4));
        const float v[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
        float* dst = col + grp * g.k3 * (int64_t)g.ncols + n0;
#pragma unroll
        for (int r3 = 0; r3 < 5; ++r3)
            __stcs(reinterpret_cast<float4*>(dst + r3 * (int64_t)g.ncols),
                   make_float4(v[r3], v[r3 + 1], v[r3 + 2], v[r3 + 3]));
    }
}

}  // namespace

cudaError_t launch_im2col4d(const float* x, int64_t cin, const int64_t in[4], const int64_t k[4],
                            float* col, int num_sms, cudaStream_t stream)
{
    const int64_t p0 = in[0] - k[0] + 1, p1 = in[1] - k[1] + 1, p2 = in[2] - k[2] + 1, p3 = in[3] - k[3] + 1;
    const int64_t ncols = p0 * p1 * p2 * p3;
    if (ncols >= (1ll << 31) - 4) return cudaErrorInvalidValue;
    Im2colGeom g;
    g.nrows = cin * k[0] * k[1] * k[2] * k[3];
    g.ncols = (int)ncols;
    g.k0 = (int)k[0], g.k1 = (int)k[1], g.k2 = (int)k[2], g.k3 = (int)k[3];
    g.in1 = (int)in[1], g.in2 = (int)in[2], g.in3 = (int)in[3];
    g.p1 = (int)p1, g.p2 = (int)p2, g.p3 = (int)p3;
    g.chan_stride = in[0] * in[1] * in[2] * in[3];
    if (g.chan_stride >= (1ll << 31)) return cudaErrorInvalidValue;  // 32-bit position offsets
    g.x_elems = cin * g.chan_stride;
    // blocks along x cover the columns once; along y they share the rows, about 16
    // blocks per SM in all
    const int64_t gx64 = (ncols + IM_COLS - 1) / IM_COLS;
    if (gx64 > 0x7fffffffLL) return cudaErrorInvalidValue;
    const unsigned gx = (unsigned)gx64;
    int64_t gy64 = (int64_t)(num_sms > 0 ? num_sms : 152) * 16 / gx64;
    if (gy64 < 1) gy64 = 1;
    if (gy64 > g.nrows) gy64 = g.nrows;
    if (gy64 > 65535) gy64 = 65535;
    const unsigned gy = (unsigned)gy64;
    const bool quad = (p3 % 4 == 0) && (reinterpret_cast<uintptr_t>(col) & 15) == 0;
    if (quad && k[3] == 5 && in[3] % 4 == 0 && (reinterpret_cast<uintptr_t>(x) & 15) == 0) {
        int64_t gy_g = (int64_t)(num_sms > 0 ? num_sms : 152) * 16 / gx64;
        const int64_t groups = g.nrows / g.k3;
        gy_g = gy_g < 1 ? 1 : (gy_g > groups ? groups : gy_g);
        if (gy_g > 65535) gy_g = 65535;
        im2col4d_group_kernel<<<dim3(gx, (unsigned)gy_g), IM_THREADS, 0, stream>>>(x, g, col);
        return cudaGetLastError();
    }
    if (quad)
        im2col4d_kernel<true><<<dim3(gx, gy), 256, 0, stream>>>(x, g, col);
    else
        im2col4d_kernel<false><<<dim3(gx, gy), 256, 0, stream>>>(x, g, col);
    return cudaGetLastError();
}

}  // namespace gemm_gb300
