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
// a host-side shadow, not to device memory.  The device address is looked up with
// cudaGetSymbolAddress while that device is current, once per device and context, and
// cached together with the context's unique ID; a call from another context on that
// device (after cudaDeviceReset, or under a context the caller made current) looks the
// address up again instead of using a stale one.
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
    unsigned long long ctx_id;  // the context the address belongs to (0: unknown)
    bool ready;
};

DeviceScratch g_scratch[kMaxDevices];
std::mutex g_scratch_mutex;

// Unique ID of the calling thread's current CUDA context; 0 when there is none yet or it
// cannot be read.  IDs are never reused within a process.
unsigned long long current_context_id()
{
    static PFN_cuCtxGetCurrent_v4000 get_current = nullptr;
    static PFN_cuCtxGetId_v12000 get_id = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 4000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(f);
        f = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(f);
        (void)cudaGetLastError();
    });
    if (!get_current || !get_id) return 0;
    CUcontext ctx = nullptr;
    if (get_current(&ctx) != CUDA_SUCCESS || !ctx) return 0;
    unsigned long long id = 0;
    if (get_id(ctx, &id) != CUDA_SUCCESS) return 0;
    return id;
}

// A failed runtime query leaves the runtime's last error set; clear it so that a later
// launch check elsewhere in the library does not report it as its own.
int fail_cuda()
{
    (void)cudaGetLastError();
    return GEMM_ERR_CUDA;
}

// The device address of the scratch array and the SM count for the current device,
// looked up on the first call on each device and again whenever the current context is
// not the one the cached address was taken in.
int scratch_for_current_device(DeviceScratch* out)
{
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return fail_cuda();
    if (dev < 0 || dev >= kMaxDevices) return GEMM_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    DeviceScratch& s = g_scratch[dev];
    const unsigned long long id = current_context_id();
    if (!s.ready || id == 0 || id != s.ctx_id) {
        s.ready = false;
        int major = 0, minor = 0, sms = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return fail_cuda();
        if (major != 10 || minor != 3) return GEMM_ERR_UNSUPPORTED;
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_skinny_scratch) != cudaSuccess || p == nullptr) return fail_cuda();
        s.ptr = static_cast<float*>(p);
        s.num_sms = sms;
        s.ctx_id = current_context_id();  // the lookup has made the device's context current
        s.ready = true;
    }
    *out = s;
    return GEMM_OK;
}

}  // namespace
}  // namespace gemm_gb300

using namespace gemm_gb300;

static int run_noalloc(int64_t M, int64_t N, int64_t K, const float* A, int64_t lda, const float* B, int64_t ldb,
                       float* C, int64_t ldc, int split_k, void* stream)
{
    if (split_k < 0 || split_k > 1024) return GEMM_ERR_INVALID_ARG;
    const int rc0 = check_product_args(M, N, K, A, lda, B, ldb, C, ldc);
    if (rc0 != GEMM_OK) return rc0;
    if (M == 0 || N == 0) return GEMM_OK;
    if (M > 32 || beyond_kernel_limits(M, N, K, lda, ldb, ldc)) return GEMM_ERR_UNSUPPORTED;
    DeviceScratch s;
    int rc = scratch_for_current_device(&s);
    if (rc != GEMM_OK) return rc;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (K == 0)
        return cudaMemset2DAsync(C, (size_t)ldc * 4, 0, (size_t)N * 4, (size_t)M, st) == cudaSuccess ? GEMM_OK
                                                                                                    : fail_cuda();
    F32Args a{M, N, K, A, lda, B, ldb, C, ldc};
    int split = split_k > 0 ? split_k : skinny_auto_split(a, s.num_sms);
    if ((int64_t)split > K) split = (int)K;
    // every split slice is fully written before it is summed: nothing needs clearing
    // (compared by division: split * M * N itself may overflow for absurd N)
    if (split > 1 && N > kScratchFloats / ((int64_t)split * M)) {
        glog("gemm_run_f32_skinny_noalloc: split %d x M %lld x N %lld floats exceed the %lld-float scratch array", split,
             (long long)M, (long long)N, (long long)kScratchFloats);
        return GEMM_ERR_UNSUPPORTED;
    }
    glog("gemm_run_f32_skinny_noalloc %lldx%lldx%lld: skinny kernel (registers), split %d, scratch %lld floats",
         (long long)M, (long long)N, (long long)K, split, split > 1 ? (long long)split * M * N : 0ll);
    int launches = 0;
    return launch_skinny(a, split, s.ptr, s.num_sms, st, &launches) == cudaSuccess ? GEMM_OK : fail_cuda();
}

extern "C" int gemm_run_f32_skinny_noalloc(int64_t M, int64_t N, int64_t K, const float* A, int64_t lda,
                                           const float* B, int64_t ldb, float* C, int64_t ldc, int split_k,
                                           void* stream)
{
    const int rc = run_noalloc(M, N, K, A, lda, B, ldb, C, ldc, split_k, stream);
    if (rc != GEMM_OK)
        glog("gemm_run_f32_skinny_noalloc(M %lld, N %lld, K %lld, lda %lld, ldb %lld, ldc %lld, split %d) refused: %s (%d)",
             (long long)M, (long long)N, (long long)K, (long long)lda, (long long)ldb, (long long)ldc, split_k,
             gemm_status_string(rc), rc);
    return rc;
}
