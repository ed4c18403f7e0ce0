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
    int64_t cin;
    int64_t in0, in1, in2, in3;
    int64_t k0, k1, k2, k3;
    int64_t p0, p1, p2, p3;
    int64_t ncols;  // p0*p1*p2*p3
    int64_t nrows;  // cin*k0*k1*k2*k3
};

__device__ __forceinline__ float im2col_value(const float* __restrict__ x, const Im2colGeom& g,
                                              int64_t xbase, int64_t n)
{
    // n -> (q0, q1, q2, q3), row-major over the output positions
    const int64_t q3 = n % g.p3;
    int64_t t = n / g.p3;
    const int64_t q2 = t % g.p2;
    t /= g.p2;
    const int64_t q1 = t % g.p1;
    const int64_t q0 = t / g.p1;
    return __ldg(x + xbase + ((q0 * g.in1 + q1) * g.in2 + q2) * g.in3 + q3);
}

template <bool VEC4>
__global__ void __launch_bounds__(256) im2col4d_kernel(const float* __restrict__ x, Im2colGeom g,
                                                       float* __restrict__ col)
{
    const int64_t quads = (g.ncols + 3) / 4;
    const int64_t total = g.nrows * quads;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; idx < total; idx += stride) {
        const int64_t row = idx / quads;
        const int64_t n0 = (idx - row * quads) * 4;
        // row -> (c, r0, r1, r2, r3)
        const int64_t r3 = row % g.k3;
        int64_t t = row / g.k3;
        const int64_t r2 = t % g.k2;
        t /= g.k2;
        const int64_t r1 = t % g.k1;
        t /= g.k1;
        const int64_t r0 = t % g.k0;
        const int64_t c = t / g.k0;
        // x index of output position (0,0,0,0) for this tap
        const int64_t xbase = (((c * g.in0 + r0) * g.in1 + r1) * g.in2 + r2) * g.in3 + r3;
        float* dst = col + row * g.ncols + n0;
        if (VEC4 && n0 + 3 < g.ncols) {
            float4 v;
            v.x = im2col_value(x, g, xbase, n0 + 0);
            v.y = im2col_value(x, g, xbase, n0 + 1);
            v.z = im2col_value(x, g, xbase, n0 + 2);
            v.w = im2col_value(x, g, xbase, n0 + 3);
            *reinterpret_cast<float4*>(dst) = v;
        } else {
            for (int j = 0; j < 4 && n0 + j < g.ncols; ++j) dst[j] = im2col_value(x, g, xbase, n0 + j);
        }
    }
}

}  // namespace

cudaError_t launch_im2col4d(const float* x, int64_t cin, const int64_t in[4], const int64_t k[4],
                            float* col, int num_sms, cudaStream_t stream)
{
    Im2colGeom g;
    g.cin = cin;
    g.in0 = in[0], g.in1 = in[1], g.in2 = in[2], g.in3 = in[3];
    g.k0 = k[0], g.k1 = k[1], g.k2 = k[2], g.k3 = k[3];
    g.p0 = in[0] - k[0] + 1, g.p1 = in[1] - k[1] + 1, g.p2 = in[2] - k[2] + 1, g.p3 = in[3] - k[3] + 1;
    g.ncols = g.p0 * g.p1 * g.p2 * g.p3;
    g.nrows = cin * k[0] * k[1] * k[2] * k[3];
    const int64_t total = g.nrows * ((g.ncols + 3) / 4);
    int64_t blocks = (total + 255) / 256;
    const int64_t cap = (int64_t)(num_sms > 0 ? num_sms : 152) * 16;  // grid-stride beyond this
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    const bool vec = (g.ncols % 4 == 0) && (reinterpret_cast<uintptr_t>(col) & 15) == 0;
    if (vec)
        im2col4d_kernel<true><<<(unsigned)blocks, 256, 0, stream>>>(x, g, col);
    else
        im2col4d_kernel<false><<<(unsigned)blocks, 256, 0, stream>>>(x, g, col);
    return cudaGetLastError();
}

}  // namespace gemm_gb300
