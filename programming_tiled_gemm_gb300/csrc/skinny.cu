// fp32 GEMM for few rows (M <= 32): a streaming kernel bound by reading B from HBM.
//
// With M this small every element of B is used M times, so the product is limited by
// how fast B streams from memory (16 rows: 8 flop per byte of B).  The kernel:
//  * gives each thread four adjacent columns (one float4 of a B row) and all M rows of
//    the output for them, so B is read exactly once, straight into registers, as
//    coalesced 512-byte warp loads ("CUDA overview: performance surprises", section
//    "Coalescing memory blocks": neighbouring threads take neighbouring elements);
//  * keeps a few B rows in flight per thread (a register ring) to cover memory latency;
//  * stages A (M x 64 per step) in shared memory with asynchronous copies, read back as
//    broadcast float4s, so the inner loop is an outer product of an A column with a B
//    float4, as in the register-blocked kernel of "Learning to develop for GPU with GEMM
//    as the example", section "Improving the solution and balancing memory work";
//  * splits K over grid.y when there are too few column blocks to fill the GPU
//    ("CUDA overview ...", section "Parallelism first"); partial products go to a
//    workspace and a fixed-order reduction writes C, so results are deterministic.
#include "internal.h"

namespace gemm_gb300 {

GEMM_DEBUG_UNIT(skinny)

namespace {

constexpr int kThreads = 256;
constexpr int kColsPerBlock = kThreads * 4;  // 1024 output columns per block
constexpr int KB = 64;                       // k rows of A staged per step

__device__ __forceinline__ void cp_async_4(void* smem, const void* gmem, int src_bytes)
{
    const uint32_t s = (uint32_t)__cvta_generic_to_shared(smem);
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;\n" ::"r"(s), "l"(gmem), "r"(src_bytes)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_1() { asm volatile("cp.async.wait_group 1;\n" ::: "memory"); }

template <int MR, int U, bool VEC>
__global__ void __launch_bounds__(kThreads, (MR <= 16) ? 2 : 1)
skinny_kernel(F32Args p, int64_t k_per_split, float* ws, int vec_out)
{
    static_assert(MR % 4 == 0 && KB % U == 0, "shape");
    __shared__ __align__(16) float As[2][KB][MR];  // As[kk][m] = A[m][k0 + kk]

    const int tid = threadIdx.x;
    const int64_t col = ((int64_t)blockIdx.x * kThreads + tid) * 4;
    const int64_t kbeg = (int64_t)blockIdx.y * k_per_split;
    const int64_t kend = min(p.K, kbeg + k_per_split);
    const bool col_ok = col < p.N;
    const bool col_full = col + 3 < p.N;

    float* out;
    int64_t ldo;
    if (gridDim.y > 1) {
        out = ws + (int64_t)blockIdx.y * p.M * p.N;
        ldo = p.N;
    } else {
        out = p.C;
        ldo = p.ldc;
    }

    // A[m][k0 .. k0+KB) -> As[buf][kk][m]; rows m >= M and k >= kend are zero-filled.
    auto stage_a = [&](int64_t k0, int buf) {
#pragma unroll
        for (int i = 0; i < (KB * MR + kThreads - 1) / kThreads; ++i) {
            const int e = tid + i * kThreads;
            if (e < KB * MR) {
                const int kk = e % KB, m = e / KB;
                const int64_t gk = k0 + kk;
                const bool ok = (m < p.M) && (gk < kend) && in_range(m, p.M) && in_range(gk, p.K);
                const float* src = ok ? (p.A + (int64_t)m * p.lda + gk) : p.A;
                cp_async_4(&As[buf][kk][m], src, ok ? 4 : 0);
            }
        }
    };

    auto load_b = [&](int64_t k) -> float4 {
        float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
        if (k < kend && col_ok && in_range(k, p.K) && in_range(col, p.N)) {
            const float* src = p.B + k * p.ldb + col;
            if (VEC && col_full) {
                v = __ldg(reinterpret_cast<const float4*>(src));
            } else {
                v.x = __ldg(src);
                if (col + 1 < p.N) v.y = __ldg(src + 1);
                if (col + 2 < p.N) v.z = __ldg(src + 2);
                if (col + 3 < p.N) v.w = __ldg(src + 3);
            }
        }
        return v;
    };

    float acc[MR][4];
#pragma unroll
    for (int m = 0; m < MR; ++m) acc[m][0] = acc[m][1] = acc[m][2] = acc[m][3] = 0.f;

    float4 breg[U];
    if (kbeg < kend) {
        stage_a(kbeg, 0);
        cp_async_commit();
#pragma unroll
        for (int u = 0; u < U; ++u) breg[u] = load_b(kbeg + u);
    }

    int buf = 0;
    for (int64_t k0 = kbeg; k0 < kend; k0 += KB) {
        if (k0 + KB < kend) stage_a(k0 + KB, buf ^ 1);
        cp_async_commit();
        cp_async_wait_1();
        __syncthreads();
        for (int kk = 0; kk < KB; kk += U) {
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const float4 b = breg[u];
                breg[u] = load_b(k0 + kk + u + U);
#pragma unroll
                for (int m = 0; m < MR; m += 4) {
                    const float4 a = *reinterpret_cast<const float4*>(&As[buf][kk + u][m]);
                    acc[m + 0][0] = fmaf(a.x, b.x, acc[m + 0][0]);
                    acc[m + 0][1] = fmaf(a.x, b.y, acc[m + 0][1]);
                    acc[m + 0][2] = fmaf(a.x, b.z, acc[m + 0][2]);
                    acc[m + 0][3] = fmaf(a.x, b.w, acc[m + 0][3]);
                    acc[m + 1][0] = fmaf(a.y, b.x, acc[m + 1][0]);
                    acc[m + 1][1] = fmaf(a.y, b.y, acc[m + 1][1]);
                    acc[m + 1][2] = fmaf(a.y, b.z, acc[m + 1][2]);
                    acc[m + 1][3] = fmaf(a.y, b.w, acc[m + 1][3]);
                    acc[m + 2][0] = fmaf(a.z, b.x, acc[m + 2][0]);
                    acc[m + 2][1] = fmaf(a.z, b.y, acc[m + 2][1]);
                    acc[m + 2][2] = fmaf(a.z, b.z, acc[m + 2][2]);
                    acc[m + 2][3] = fmaf(a.z, b.w, acc[m + 2][3]);
                    acc[m + 3][0] = fmaf(a.w, b.x, acc[m + 3][0]);
                    acc[m + 3][1] = fmaf(a.w, b.y, acc[m + 3][1]);
                    acc[m + 3][2] = fmaf(a.w, b.z, acc[m + 3][2]);
                    acc[m + 3][3] = fmaf(a.w, b.w, acc[m + 3][3]);
                }
            }
        }
        __syncthreads();  // every warp is done with As[buf] before it is refilled
        buf ^= 1;
    }

    if (!col_ok) return;
#pragma unroll
    for (int m = 0; m < MR; ++m) {
        if (m >= p.M || !in_range(m, p.M) || !in_range(col, p.N)) break;
        float* dst = out + (int64_t)m * ldo + col;
        if (vec_out && col_full) {
            *reinterpret_cast<float4*>(dst) = make_float4(acc[m][0], acc[m][1], acc[m][2], acc[m][3]);
        } else {
            dst[0] = acc[m][0];
            if (col + 1 < p.N) dst[1] = acc[m][1];
            if (col + 2 < p.N) dst[2] = acc[m][2];
            if (col + 3 < p.N) dst[3] = acc[m][3];
        }
    }
}

template <int MR>
cudaError_t launch_mr(const F32Args& a, int split, float* ws, int num_sms, cudaStream_t stream, int* launches)
{
    constexpr int U = 4;
    int64_t kps = (a.K + split - 1) / split;
    kps = (kps + KB - 1) / KB * KB;
    const int nsplit = (int)((a.K + kps - 1) / kps);
    const int64_t xblocks = (a.N + kColsPerBlock - 1) / kColsPerBlock;
    if (xblocks > 0x7fffffffLL || nsplit > 65535) return cudaErrorInvalidConfiguration;
    const bool vec_in = (reinterpret_cast<uintptr_t>(a.B) & 15) == 0 && a.ldb % 4 == 0;
    int vec_out;
    if (nsplit > 1)
        vec_out = (a.N % 4 == 0);
    else
        vec_out = (reinterpret_cast<uintptr_t>(a.C) & 15) == 0 && a.ldc % 4 == 0;
    dim3 grid((unsigned)xblocks, (unsigned)nsplit, 1);
    if (vec_in)
        skinny_kernel<MR, U, true><<<grid, kThreads, 0, stream>>>(a, kps, ws, vec_out);
    else
        skinny_kernel<MR, U, false><<<grid, kThreads, 0, stream>>>(a, kps, ws, vec_out);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    *launches += 1;
    if (nsplit == 1) return e;
    *launches += 1;
    return launch_splitk_reduce(ws, nsplit, a.M, a.N, a.C, a.ldc, num_sms, stream);
}

}  // namespace

int skinny_auto_split(const F32Args& a, int num_sms)
{
    const int64_t xblocks = (a.N + kColsPerBlock - 1) / kColsPerBlock;
    const int64_t resident = (a.M <= 16) ? 2 : 1;
    const int64_t target = (int64_t)num_sms * resident;
    int64_t s = (target + xblocks / 2) / xblocks;
    const int64_t max_s = (a.K + 4 * KB - 1) / (4 * KB);  // at least four A steps per split
    if (s > max_s) s = max_s;
    if (s > 1024) s = 1024;
    return (int)(s < 1 ? 1 : s);
}

cudaError_t launch_skinny(const F32Args& a, int split, float* ws, int num_sms, cudaStream_t stream,
                          int* launches)
{
    if (split < 1) split = 1;
    if (a.M <= 8) return launch_mr<8>(a, split, ws, num_sms, stream, launches);
    if (a.M <= 16) return launch_mr<16>(a, split, ws, num_sms, stream, launches);
    if (a.M <= 32) return launch_mr<32>(a, split, ws, num_sms, stream, launches);
    return cudaErrorInvalidValue;
}

}  // namespace gemm_gb300
