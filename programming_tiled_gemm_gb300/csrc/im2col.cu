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
// four); the writes are the whole cost (the input is small and stays in L2).
#include "internal.h"

namespace gemm_gb300 {
namespace {

struct Im2colGeom {
    int64_t nrows;             // cin*k0*k1*k2*k3
    int ncols;                 // p0*p1*p2*p3 (< 2^31, checked by the launcher)
    int k0, k1, k2, k3;        // kernel extents
    int in1, in2, in3;         // input extents (in0 only enters through the channel stride)
    int p1, p2, p3;            // output extents
    int64_t chan_stride;       // in0*in1*in2*in3
};

// One block row per filter tap (c, r0, r1, r2, r3): the tap is decomposed once per block,
// the output position once per float4 of columns, all in 32-bit arithmetic.
// QUAD: p3 % 4 == 0, so four adjacent columns share (q0, q1, q2) and read four adjacent
// input elements.
template <bool QUAD>
__global__ void __launch_bounds__(256) im2col4d_kernel(const float* __restrict__ x, Im2colGeom g,
                                                       float* __restrict__ col)
{
    const int quads = (g.ncols + 3) / 4;
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
        const float* xb = x + c * g.chan_stride + (((int64_t)r0 * g.in1 + r1) * g.in2 + r2) * g.in3 + r3;
        float* dst_row = col + row * (int64_t)g.ncols;
        for (int qd = blockIdx.x * blockDim.x + threadIdx.x; qd < quads; qd += gridDim.x * blockDim.x) {
            const int n0 = qd * 4;
            if (QUAD) {
                const int q3 = n0 % g.p3;
                int u = n0 / g.p3;
                const int q2 = u % g.p2;
                u /= g.p2;
                const int q1 = u % g.p1;
                const int q0 = u / g.p1;
                const float* src = xb + (((int64_t)q0 * g.in1 + q1) * g.in2 + q2) * g.in3 + q3;
                float4 v;
                v.x = __ldg(src + 0);
                v.y = __ldg(src + 1);
                v.z = __ldg(src + 2);
                v.w = __ldg(src + 3);
                __stcs(reinterpret_cast<float4*>(dst_row + n0), v);  // streamed: read later, L2 would not hold it
            } else {
                for (int j = 0; j < 4 && n0 + j < g.ncols; ++j) {
                    const int n = n0 + j;
                    const int q3 = n % g.p3;
                    int u = n / g.p3;
                    const int q2 = u % g.p2;
                    u /= g.p2;
                    const int q1 = u % g.p1;
                    const int q0 = u / g.p1;
                    dst_row[n] = __ldg(xb + (((int64_t)q0 * g.in1 + q1) * g.in2 + q2) * g.in3 + q3);
                }
            }
        }
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
    const int quads = (g.ncols + 3) / 4;
    // a few thousand long-lived blocks: each thread walks several float4s of a row and
    // several rows (grid-stride in both directions)
    int64_t gx64 = (quads + 1023) / 1024;
    if (gx64 < 1) gx64 = 1;
    const unsigned gx = (unsigned)gx64;
    int64_t gy64 = (int64_t)(num_sms > 0 ? num_sms : 152) * 16 / gx64;
    if (gy64 < 1) gy64 = 1;
    if (gy64 > g.nrows) gy64 = g.nrows;
    if (gy64 > 65535) gy64 = 65535;
    const unsigned gy = (unsigned)gy64;
    const bool quad = (p3 % 4 == 0) && (reinterpret_cast<uintptr_t>(col) & 15) == 0;
    if (quad)
        im2col4d_kernel<true><<<dim3(gx, gy), 256, 0, stream>>>(x, g, col);
    else
        im2col4d_kernel<false><<<dim3(gx, gy), 256, 0, stream>>>(x, g, col);
    return cudaGetLastError();
}

}  // namespace gemm_gb300
