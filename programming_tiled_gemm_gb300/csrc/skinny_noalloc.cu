// Allocation-free entry point for the skinny fp32 GEMM (M <= 32).
//
// gemm_run keeps the skinny kernel's split-K partial sums in a workspace that the handle
// grows with cudaMalloc, and creating a handle allocates too.  This entry point runs the
// same kernel with no handle and no allocation: the partial sums live in a fixed array
// in device global memory that belongs to the library image itself.  The array is
// reserved on every GPU where the library's device code is loaded and stays reserved
// until the process exits.
//
// Host code cannot pass `g_skinny_scratch` to a kernel: in host code the name refers to
// a host-side shadow, not to device memory.  The device address is looked up once per
// device with cudaGetSymbolAddress while that device is current, and cached.
#include <mutex>

#include "internal.h"

namespace gemm_gb300 {
namespace {

constexpr int64_t kScratchFloats = int64_t(8) << 20;  // 8 Mi floats = 32 MiB
__device__ __align__(256) float g_skinny_scratch[kScratchFloats];

constexpr int kMaxDevices = 128;

struct DeviceScratch {
    float* ptr;
    int num_sms;
    bool ready;
};

DeviceScratch g_scratch[kMaxDevices];
std::mutex g_scratch_mutex;

// Look up (once per device) the device address of the scratch array and the SM count.
int scratch_for_current_device(DeviceScratch* out)
{
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return GEMM_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return GEMM_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    DeviceScratch& s = g_scratch[dev];
    if (!s.ready) {
        int major = 0, minor = 0, sms = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return GEMM_ERR_CUDA;
        if (major != 10 || minor != 3) return GEMM_ERR_UNSUPPORTED;
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_skinny_scratch) != cudaSuccess || p == nullptr) return GEMM_ERR_CUDA;
        s.ptr = static_cast<float*>(p);
        s.num_sms = sms;
        s.ready = true;
    }
    *out = s;
    return GEMM_OK;
}

}  // namespace
}  // namespace gemm_gb300

using namespace gemm_gb300;

extern "C" int gemm_run_f32_skinny_noalloc(int64_t M, int64_t N, int64_t K, const float* A, int64_t lda,
                                           const float* B, int64_t ldb, float* C, int64_t ldc, int split_k,
                                           void* stream)
{
    if (M < 0 || N < 0 || K < 0 || split_k < 0 || split_k > 1024) return GEMM_ERR_INVALID_ARG;
    if (M == 0 || N == 0) return GEMM_OK;
    if (!C || ldc < N) return GEMM_ERR_INVALID_ARG;
    if (K > 0 && (!A || !B || lda < K || ldb < N)) return GEMM_ERR_INVALID_ARG;
    if (M > 32) return GEMM_ERR_UNSUPPORTED;
    DeviceScratch s;
    int rc = scratch_for_current_device(&s);
    if (rc != GEMM_OK) return rc;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (K == 0)
        return cudaMemset2DAsync(C, (size_t)ldc * 4, 0, (size_t)N * 4, (size_t)M, st) == cudaSuccess ? GEMM_OK
                                                                                                    : GEMM_ERR_CUDA;
    F32Args a{M, N, K, A, lda, B, ldb, C, ldc};
    int split = split_k > 0 ? split_k : skinny_auto_split(a, s.num_sms);
    if ((int64_t)split > K) split = (int)K;
    // every split slice is fully written before it is summed: nothing needs clearing
    if (split > 1 && (int64_t)split * M * N > kScratchFloats) return GEMM_ERR_UNSUPPORTED;
    int launches = 0;
    return launch_skinny(a, split, s.ptr, s.num_sms, st, &launches) == cudaSuccess ? GEMM_OK : GEMM_ERR_CUDA;
}
