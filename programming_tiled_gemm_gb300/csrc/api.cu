// Host side of the C ABI declared in include/gemm.h: handle, argument checks, kernel
// choice among this library's own kernels, workspace and staging buffers.
//
// The shape of the interface follows the host pipeline of "Learning to develop for GPU
// with GEMM as the example", section "Writing a GPU implementation of matrix
// multiplication" (set up device buffers once, pass (m, n, k, a, b, c) to the kernel,
// enqueue it on a queue, wait on an event): here a handle is created once, gemm_run
// enqueues on the caller's CUDA stream, and the caller synchronises as it wishes.
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <new>
#include <vector>

#include "internal.h"

using namespace gemm_gb300;

namespace gemm_gb300 {

bool log_enabled()
{
    static const bool on = [] {
        const char* v = getenv("GEMM_LOG");
        return v && strcmp(v, "1") == 0;
    }();
    return on;
}

void glog(const char* fmt, ...)
{
    if (!log_enabled()) return;
    va_list ap;
    va_start(ap, fmt);
    char line[512];
    vsnprintf(line, sizeof(line), fmt, ap);
    va_end(ap);
    fprintf(stderr, "[gemm] %s\n", line);
}

const char* dtype_name(int d) { return d == GEMM_F32 ? "f32" : d == GEMM_BF16 ? "bf16" : d == GEMM_F16 ? "f16" : "?"; }

int check_product_args(int64_t M, int64_t N, int64_t K, const void* A, int64_t lda, const void* B, int64_t ldb,
                       const void* C, int64_t ldc)
{
    if (M < 0 || N < 0 || K < 0) return GEMM_ERR_INVALID_ARG;
    if (M == 0 || N == 0) return GEMM_OK;
    if (!C || ldc < N) return GEMM_ERR_INVALID_ARG;
    if (K > 0) {
        if (!A || !B) return GEMM_ERR_INVALID_ARG;
        if (lda < K || ldb < N) return GEMM_ERR_INVALID_ARG;
    }
    // the largest element offsets must fit in int64 (they always do for real memory,
    // but reject nonsense before it reaches a kernel)
    const int64_t lim = (int64_t)1 << 46;
    if (M > lim / (ldc > 0 ? ldc : 1) || (K > 0 && (M > lim / lda || K > lim / ldb)))
        return GEMM_ERR_INVALID_ARG;
    return GEMM_OK;
}

// Every kernel indexes with 32-bit sizes and leading dimensions: larger ones are refused
// before anything is allocated or launched.
bool beyond_kernel_limits(int64_t M, int64_t N, int64_t K, int64_t lda, int64_t ldb, int64_t ldc)
{
    constexpr int64_t kLim32 = 0x7fffffffLL - 1024;
    return M > kLim32 || N > kLim32 || K > kLim32 || ldc > kLim32 || (K > 0 && (lda > kLim32 || ldb > kLim32));
}

}  // namespace gemm_gb300

struct gemm_ctx {
    int device = 0;
    int num_sms = 0;
    int* d_status = nullptr;  // device status word written by kernels with bounded waits
    float* workspace = nullptr;
    size_t workspace_bytes = 0;
    unsigned long long* tc_counters = nullptr;  // last-wave split counters of the tensor-core GEMM
    size_t tc_counters_bytes = 0;
    unsigned tc_seq = 0;  // tag of the last split tensor-core launch
    unsigned long long* f32_counters = nullptr;  // K-slice counters of the persistent fp32 GEMM
    size_t f32_counters_bytes = 0;
    unsigned f32_seq = 0;  // tag of the last split persistent fp32 launch
    void* host_stage = nullptr;  // gemm_run_host(_batch) device copies of A, B and C
    size_t host_stage_bytes = 0;
    float* product = nullptr;  // fp32 product for the generalised epilogue of fp32 inputs
    size_t product_bytes = 0;
    int opt_f32_kernel = 0;
    int opt_split_k = 0;
    int opt_tc_chunk = 0;  // tensor-core accumulation chunk in 64-wide k-blocks (0 = default)
    int opt_tc_pair = 0;   // tensor-core tile: 0 choose, 1 single CTA, 2 CTA pair
    int opt_test_stall = 0;  // test hook: kernels with bounded waits let one wait run out
    int opt_conv_stack = 0;  // tensor-core convolution: output positions stacked along N (0 = choose)
    int opt_conv_split = 0;  // tensor-core convolution: 0 choose, 1 one CTA pair per tile, 2 two pairs
    uint64_t wait_limit_ns = 2000000000ull;
    int64_t launches = 0;  // kernels launched through this handle
    // gemm_run_host pipeline: copy-in and copy-out streams and their events
    cudaStream_t s_in = nullptr, s_out = nullptr;
    static constexpr int kMaxChunks = 8;
    cudaEvent_t ev_start = nullptr, ev_done = nullptr;
    cudaEvent_t ev_a[kMaxChunks] = {}, ev_c[kMaxChunks] = {};
};

namespace {

class DeviceGuard {
  public:
    explicit DeviceGuard(int dev) : ok_(false), prev_(-1)
    {
        if (cudaGetDevice(&prev_) != cudaSuccess) prev_ = -1;
        ok_ = (prev_ == dev) || (cudaSetDevice(dev) == cudaSuccess);
    }
    ~DeviceGuard()
    {
        if (prev_ >= 0) cudaSetDevice(prev_);
    }
    bool ok() const { return ok_; }

  private:
    bool ok_;
    int prev_;
};

int from_cuda(cudaError_t e) { return e == cudaSuccess ? GEMM_OK : GEMM_ERR_CUDA; }

// Grow a device buffer to at least `bytes` (contents are not kept).
int ensure_buffer(void** buf, size_t* have, size_t bytes)
{
    if (*have >= bytes && *buf) return GEMM_OK;
    if (*buf) {
        cudaFree(*buf);  // implicit device synchronisation: no kernel still uses it
        *buf = nullptr;
        *have = 0;
    }
    size_t want = bytes < 256 ? 256 : bytes;
    if (cudaMalloc(buf, want) != cudaSuccess) {
        *buf = nullptr;
        (void)cudaGetLastError();  // an allocation failure is not sticky: keep it out of later launch checks
        return GEMM_ERR_CUDA;
    }
    *have = want;
    return GEMM_OK;
}

int check_common(gemm_handle_t h, int64_t M, int64_t N, int64_t K, const void* A, int64_t lda,
                 const void* B, int64_t ldb, const void* C, int64_t ldc, int dtype)
{
    if (!h) return GEMM_ERR_INVALID_ARG;
    if (M < 0 || N < 0 || K < 0) return GEMM_ERR_INVALID_ARG;
    if (dtype != GEMM_F32 && dtype != GEMM_BF16 && dtype != GEMM_F16) return GEMM_ERR_INVALID_ARG;
    return check_product_args(M, N, K, A, lda, B, ldb, C, ldc);
}

// Tagged arrival counters: a launch trusts only counts carrying its own tag, so the buffer
// is zeroed only when (re)allocated and when the tag wraps.
int tagged_counters(unsigned long long** buf, size_t* have, unsigned* seq, int64_t n, cudaStream_t s)
{
    const size_t bytes = (size_t)n * sizeof(unsigned long long);
    const bool fresh = !*buf || *have < bytes;
    int rc = ensure_buffer(reinterpret_cast<void**>(buf), have, bytes);
    if (rc != GEMM_OK) return rc;
    if (++*seq == 0) *seq = 1;
    if ((fresh || *seq == 1) && cudaMemsetAsync(*buf, 0, *have, s) != cudaSuccess) return GEMM_ERR_CUDA;
    return GEMM_OK;
}

int run_f32(gemm_handle_t h, const F32Args& a, cudaStream_t stream)
{
    int kernel = h->opt_f32_kernel;
    if (kernel == 0)
        kernel = (a.M <= 32) ? (skinny_tma_supported(a) ? 4 : 3)
                 : (a.M <= 64) ? 2
                               : (ffma_persistent_supported(a) ? 5 : 1);
    if ((kernel == 3 || kernel == 4) && a.M > 32) return GEMM_ERR_UNSUPPORTED;
    if (kernel == 4 && !skinny_tma_supported(a)) return GEMM_ERR_ALIGNMENT;
    if (kernel == 5) {
        if (!ffma_persistent_supported(a)) return GEMM_ERR_ALIGNMENT;
        const FfmaPlan pl = ffma_persistent_plan(a, h->opt_split_k, h->num_sms);
        if (pl.split > 1) {
            int rc = ensure_buffer(reinterpret_cast<void**>(&h->workspace), &h->workspace_bytes,
                                   (size_t)pl.ws_floats * sizeof(float));
            if (rc != GEMM_OK) return rc;
        }
        int rc = tagged_counters(&h->f32_counters, &h->f32_counters_bytes, &h->f32_seq, pl.counters, stream);
        if (rc != GEMM_OK) return rc;
        const uint32_t seq = h->f32_seq;
        glog("f32 %lldx%lldx%lld: persistent FFMA kernel (5), %lld tiles of 128x256, tiles from %lld in %d K slices, "
             "workspace %lld bytes", (long long)a.M, (long long)a.N, (long long)a.K, (long long)pl.tiles,
             (long long)pl.split_first, pl.split, (long long)(pl.ws_floats * 4));
        int n = 0;
        cudaError_t e = launch_ffma_persistent(a, pl, h->workspace, h->f32_counters, seq, h->num_sms, h->d_status,
                                               h->wait_limit_ns, h->opt_test_stall, stream, &n);
        h->launches += n;
        return from_cuda(e);
    }
    int split = h->opt_split_k;
    if (split == 0)
        split = (kernel == 4)   ? skinny_tma_auto_split(a, h->num_sms)
                : (kernel == 3) ? skinny_auto_split(a, h->num_sms)
                                : ffma_auto_split(a, kernel, h->num_sms);
    if ((int64_t)split > a.K) split = (int)(a.K > 0 ? a.K : 1);
    size_t need = (split > 1) ? (size_t)split * (size_t)a.M * (size_t)a.N * sizeof(float) : 0;
    if (kernel == 1) {
        const size_t rem = (size_t)ffma_remainder_workspace(a, kernel, split, h->num_sms) * sizeof(float);
        if (rem > need) need = rem;
    }
    if (need > 0) {
        int rc = ensure_buffer(reinterpret_cast<void**>(&h->workspace), &h->workspace_bytes, need);
        if (rc != GEMM_OK) return rc;
    }
    glog("f32 %lldx%lldx%lld: kernel %d (%s), split %d, workspace %zu bytes", (long long)a.M, (long long)a.N,
         (long long)a.K, kernel,
         kernel == 1 ? "tiled 128x256 FFMA" : kernel == 2 ? "tiled 64x128 FFMA" : kernel == 3 ? "skinny, registers"
                                                                                             : "skinny, TMA ring",
         split, need);
    cudaError_t e;
    int n = 0;
    if (kernel == 4)
        e = launch_skinny_tma(a, split, h->workspace, h->num_sms, h->d_status, h->wait_limit_ns, h->opt_test_stall,
                              stream, &n);
    else if (kernel == 3)
        e = launch_skinny(a, split, h->workspace, h->num_sms, stream, &n);
    else
        e = launch_ffma_tiled(a, kernel, split, h->workspace, h->num_sms, stream, &n);
    h->launches += n;
    return from_cuda(e);
}

}  // namespace

extern "C" {

static int gemm_create_impl(gemm_handle_t* out, int device)
{
    if (!out) return GEMM_ERR_INVALID_ARG;
    *out = nullptr;
    int count = 0;
    if (cudaGetDeviceCount(&count) != cudaSuccess) return GEMM_ERR_CUDA;
    if (device < 0 || device >= count) return GEMM_ERR_INVALID_ARG;
    int major = 0, minor = 0, sms = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, device) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, device) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device) != cudaSuccess)
        return GEMM_ERR_CUDA;
    if (major != 10 || minor != 3) return GEMM_ERR_UNSUPPORTED;  // kernels are built for sm_103a only
    DeviceGuard g(device);
    if (!g.ok()) return GEMM_ERR_CUDA;
    gemm_ctx* h = new (std::nothrow) gemm_ctx();
    if (!h) return GEMM_ERR_CUDA;
    h->device = device;
    h->num_sms = sms;
    if (cudaMalloc(&h->d_status, sizeof(int)) != cudaSuccess ||
        cudaMemset(h->d_status, 0, sizeof(int)) != cudaSuccess) {
        if (h->d_status) cudaFree(h->d_status);
        delete h;
        return GEMM_ERR_CUDA;
    }
    *out = h;
    return GEMM_OK;
}

int gemm_destroy(gemm_handle_t h)
{
    if (!h) return GEMM_OK;
    DeviceGuard g(h->device);
    cudaDeviceSynchronize();
    if (h->s_in) cudaStreamDestroy(h->s_in);
    if (h->s_out) cudaStreamDestroy(h->s_out);
    if (h->ev_start) cudaEventDestroy(h->ev_start);
    if (h->ev_done) cudaEventDestroy(h->ev_done);
    for (int i = 0; i < gemm_ctx::kMaxChunks; ++i) {
        if (h->ev_a[i]) cudaEventDestroy(h->ev_a[i]);
        if (h->ev_c[i]) cudaEventDestroy(h->ev_c[i]);
    }
    if (h->d_status) cudaFree(h->d_status);
    if (h->workspace) cudaFree(h->workspace);
    if (h->tc_counters) cudaFree(h->tc_counters);
    if (h->f32_counters) cudaFree(h->f32_counters);
    if (h->product) cudaFree(h->product);
    if (h->host_stage) cudaFree(h->host_stage);
    delete h;
    return GEMM_OK;
}

static int gemm_set_option_impl(gemm_handle_t h, int option, int64_t value)
{
    if (!h) return GEMM_ERR_INVALID_ARG;
    switch (option) {
    case GEMM_OPT_F32_KERNEL:
        if (value < 0 || value > 5) return GEMM_ERR_INVALID_ARG;
        h->opt_f32_kernel = (int)value;
        return GEMM_OK;
    case GEMM_OPT_SPLIT_K:
        if (value < 0 || value > 1024) return GEMM_ERR_INVALID_ARG;
        h->opt_split_k = (int)value;
        return GEMM_OK;
    case GEMM_OPT_TC_CHUNK:
        if (value < 0 || value > 4096) return GEMM_ERR_INVALID_ARG;
        h->opt_tc_chunk = (int)value;
        return GEMM_OK;
    case GEMM_OPT_TC_PAIR:
        if (value < 0 || value > 2) return GEMM_ERR_INVALID_ARG;
        h->opt_tc_pair = (int)value;
        return GEMM_OK;
    case GEMM_OPT_CONV_STACK:
        if (value != 0 && value != 1 && value != 2 && value != 4) return GEMM_ERR_INVALID_ARG;
        h->opt_conv_stack = (int)value;
        return GEMM_OK;
    case GEMM_OPT_CONV_SPLIT:
        if (value < 0 || value > 2) return GEMM_ERR_INVALID_ARG;
        h->opt_conv_split = (int)value;
        return GEMM_OK;
    case GEMM_OPT_TEST_STALL:
        if (value < 0 || value > 1) return GEMM_ERR_INVALID_ARG;
        h->opt_test_stall = (int)value;
        return GEMM_OK;
    case GEMM_OPT_WAIT_LIMIT_US:
        if (value < 0 || value > 60000000) return GEMM_ERR_INVALID_ARG;
        h->wait_limit_ns = value == 0 ? 2000000000ull : (uint64_t)value * 1000ull;
        return GEMM_OK;
    default:
        return GEMM_ERR_INVALID_ARG;
    }
}

static int gemm_run_ex_impl(gemm_handle_t h, int64_t M, int64_t N, int64_t K, float alpha, const void* A, int64_t lda,
                const void* B, int64_t ldb, float beta, void* C, int64_t ldc, gemm_dtype_t ab_dtype,
                gemm_dtype_t c_dtype, void* stream)
{
    int rc = check_common(h, M, N, K, A, lda, B, ldb, C, ldc, (int)ab_dtype);
    if (rc != GEMM_OK) return rc;
    if (c_dtype != GEMM_F32 && c_dtype != GEMM_BF16 && c_dtype != GEMM_F16) return GEMM_ERR_INVALID_ARG;
    if (M == 0 || N == 0) return GEMM_OK;
    if (beyond_kernel_limits(M, N, K, lda, ldb, ldc)) return GEMM_ERR_UNSUPPORTED;
    const size_t ces = (c_dtype == GEMM_F32) ? 4 : 2;
    if (reinterpret_cast<uintptr_t>(C) & (ces - 1)) return GEMM_ERR_ALIGNMENT;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (ab_dtype != GEMM_F32 && K > 0) {
        // TMA tensor maps: 16-byte aligned bases, row strides a multiple of 16 bytes.
        if ((reinterpret_cast<uintptr_t>(A) & 15) || (reinterpret_cast<uintptr_t>(B) & 15) || (lda % 8) ||
            (ldb % 8))
            return GEMM_ERR_ALIGNMENT;
    }
    DeviceGuard g(h->device);
    if (!g.ok()) return GEMM_ERR_CUDA;
    Epilogue epi;
    epi.alpha = alpha;
    epi.beta = beta;
    epi.c_dtype = (int)c_dtype;
    if (K == 0) {  // empty product: C = beta * C
        if (beta == 0.f) return from_cuda(cudaMemset2DAsync(C, (size_t)ldc * ces, 0, (size_t)N * ces, (size_t)M, s));
        cudaError_t e = launch_epilogue(nullptr, 0, C, ldc, M, N, epi, h->num_sms, s);
        if (e == cudaSuccess) h->launches += 1;
        return from_cuda(e);
    }
    if (ab_dtype == GEMM_F32) {
        if (epi.plain()) {
            F32Args a{M, N, K, static_cast<const float*>(A), lda, static_cast<const float*>(B), ldb,
                      static_cast<float*>(C), ldc};
            return run_f32(h, a, s);
        }
        // fp32 product into a handle buffer, then the epilogue pass
        rc = ensure_buffer(reinterpret_cast<void**>(&h->product), &h->product_bytes, (size_t)M * N * sizeof(float));
        if (rc != GEMM_OK) return rc;
        F32Args a{M, N, K, static_cast<const float*>(A), lda, static_cast<const float*>(B), ldb, h->product, N};
        rc = run_f32(h, a, s);
        if (rc != GEMM_OK) return rc;
        cudaError_t e = launch_epilogue(h->product, N, C, ldc, M, N, epi, h->num_sms, s);
        if (e == cudaSuccess) h->launches += 1;
        return from_cuda(e);
    }
    TcArgs t{M, N, K, A, lda, B, ldb, C, ldc, ab_dtype == GEMM_BF16 ? 1 : 0, h->opt_test_stall, epi};
    const TcWorkspace need = tc_workspace_need(t, h->num_sms, h->opt_tc_pair);
    if (need.counters > 0) {
        if (need.floats > 0) {
            rc = ensure_buffer(reinterpret_cast<void**>(&h->workspace), &h->workspace_bytes,
                               (size_t)need.floats * sizeof(float));
            if (rc != GEMM_OK) return rc;
            t.rem_ws = h->workspace;
        }
        // arrival counters and publication flags: zeroed when (re)allocated and when the
        // launch tag wraps; a launch trusts only values that carry its own tag
        const size_t cbytes = (size_t)need.counters * (sizeof(unsigned long long) + sizeof(uint32_t));
        const bool fresh = !h->tc_counters || h->tc_counters_bytes < cbytes;
        rc = ensure_buffer(reinterpret_cast<void**>(&h->tc_counters), &h->tc_counters_bytes, cbytes);
        if (rc != GEMM_OK) return rc;
        if (++h->tc_seq == 0) h->tc_seq = 1;
        if ((fresh || h->tc_seq == 1) && cudaMemsetAsync(h->tc_counters, 0, h->tc_counters_bytes, s) != cudaSuccess)
            return GEMM_ERR_CUDA;
        t.rem_cnt = h->tc_counters;
        t.rem_flag = reinterpret_cast<uint32_t*>(h->tc_counters + need.counters);
        t.rem_seq = h->tc_seq;
    }
    glog("%s %lldx%lldx%lld: tensor-core GEMM (tile option %d: 0 choose, 1 single CTA, 2 CTA pair), last-wave "
         "K-split workspace %lld floats and %lld counters, chunk %d k-blocks",
         dtype_name(ab_dtype), (long long)M, (long long)N, (long long)K, h->opt_tc_pair, (long long)need.floats,
         (long long)need.counters, h->opt_tc_chunk > 0 ? h->opt_tc_chunk : 16);
    int n = 0;
    int rc2 = launch_tc_gemm(t, h->num_sms, h->d_status, h->wait_limit_ns, h->opt_tc_chunk, h->opt_tc_pair, s, &n);
    h->launches += n;
    return rc2;
}

int gemm_run(gemm_handle_t h, int64_t M, int64_t N, int64_t K, const void* A, int64_t lda, const void* B,
             int64_t ldb, float* C, int64_t ldc, gemm_dtype_t dtype, void* stream)
{
    return gemm_run_ex(h, M, N, K, 1.f, A, lda, B, ldb, 0.f, C, ldc, dtype, GEMM_F32, stream);
}

}  // extern "C"

namespace {

// Row-pitched copy; one contiguous copy when both sides are dense.
cudaError_t copy_rows(void* dst, size_t dpitch, const void* src, size_t spitch, size_t width, size_t rows,
                      cudaMemcpyKind kind, cudaStream_t s)
{
    if (rows == 0 || width == 0) return cudaSuccess;
    if (dpitch == width && spitch == width) return cudaMemcpyAsync(dst, src, width * rows, kind, s);
    return cudaMemcpy2DAsync(dst, dpitch, src, spitch, width, rows, kind, s);
}

int ensure_pipeline(gemm_handle_t h)
{
    if (h->s_in) return GEMM_OK;
    if (cudaStreamCreateWithFlags(&h->s_in, cudaStreamNonBlocking) != cudaSuccess ||
        cudaStreamCreateWithFlags(&h->s_out, cudaStreamNonBlocking) != cudaSuccess ||
        cudaEventCreateWithFlags(&h->ev_start, cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&h->ev_done, cudaEventDisableTiming) != cudaSuccess)
        return GEMM_ERR_CUDA;
    for (int i = 0; i < gemm_ctx::kMaxChunks; ++i)
        if (cudaEventCreateWithFlags(&h->ev_a[i], cudaEventDisableTiming) != cudaSuccess ||
            cudaEventCreateWithFlags(&h->ev_c[i], cudaEventDisableTiming) != cudaSuccess)
            return GEMM_ERR_CUDA;
    return GEMM_OK;
}

// Device staging of one host problem: A, B and C with leading dimensions rounded up to
// multiples of 8 (16-bit) / 4 (fp32) elements, so every row is 16-byte aligned.
struct HostStage {
    int64_t lda_d, ldb_d, ldc_d;
    size_t a_off, b_off, c_off, bytes;  // offsets in the handle's staging buffer
};

HostStage host_stage_layout(const gemm_host_problem& q, size_t base)
{
    const size_t es = (q.dtype == GEMM_F32) ? 4 : 2;
    auto up = [](size_t v) { return (v + 255) / 256 * 256; };
    HostStage st;
    st.lda_d = (q.K + 7) / 8 * 8;
    st.ldb_d = (q.N + 7) / 8 * 8;
    st.ldc_d = (q.N + 3) / 4 * 4;
    st.a_off = base;
    st.b_off = st.a_off + up(q.K > 0 ? (size_t)q.M * st.lda_d * es : 0);
    st.c_off = st.b_off + up(q.K > 0 ? (size_t)q.K * st.ldb_d * es : 0);
    st.bytes = st.c_off + up((size_t)q.M * st.ldc_d * 4) - base;
    return st;
}

// Row chunks of one host problem, in order.
//   16-bit inputs are transfer-bound (the tensor cores outrun a ~200 GB/s host link):
//   2 to 4 chunks of >= 1024 rows, 4096 and more where M allows, so that each launch
//   keeps several waves of 256 x 256 tiles (measured at 8192^3: four 2048-row chunks
//   computed in 0.72 ms, one launch in 0.63 ms).
//   fp32 is compute-bound: one sixteenth of the rows (the first compute starts after B and
//   a short slice of A are in), seven sixteenths, three eighths, then one eighth (the
//   batch's last piece of work then has a small result to bring back).  Measured on the
//   bf16 8192^3 + fp32 4096^3 batch: 3.45 ms against 3.49 ms with a first chunk of 1/8.
std::vector<int64_t> host_chunk_rows(const gemm_host_problem& q)
{
    std::vector<int64_t> rows;
    if (q.M <= 0 || q.N <= 0) return rows;
    auto up256 = [](int64_t v) { return (v + 255) / 256 * 256; };
    if (q.K > 0 && q.dtype == GEMM_F32 && q.M >= 4096) {
        // 1/16, 7/16, 3/8 and the rest, each rounded up to 256 rows and cut to what is left
        const int64_t a = up256(q.M / 16), b = up256(q.M * 7 / 16), c = up256(q.M * 3 / 8);
        int64_t left = q.M;
        for (int64_t want : {a, b, c}) {
            const int64_t r = want < left ? want : left;
            if (r > 0) rows.push_back(r);
            left -= r;
        }
        if (left > 0) rows.push_back(left);
    } else if (q.K > 0 && q.dtype != GEMM_F32 && q.M >= 2048) {
        int64_t n = q.M / 4096;
        n = n < 2 ? 2 : (n > 4 ? 4 : n);
        const int64_t c = up256((q.M + n - 1) / n);
        for (int64_t m0 = 0; m0 < q.M; m0 += c) rows.push_back(q.M - m0 < c ? q.M - m0 : c);
    } else {
        rows = {q.M};
    }
    return rows;
}

// A problem whose estimated compute time exceeds its estimated transfer time (rates of
// this GPU's tensor / FP32 pipes and host link, for ordering only).
bool compute_bound(const gemm_host_problem& q)
{
    const double flops = 2.0 * (double)q.M * (double)q.N * (double)q.K;
    const double es = (q.dtype == GEMM_F32) ? 4.0 : 2.0;
    const double bytes = es * ((double)q.M * q.K + (double)q.K * q.N) + 4.0 * (double)q.M * q.N;
    const double t_compute = flops / ((q.dtype == GEMM_F32) ? 5.5e13 : 1.5e15);
    const double t_copy = bytes / 3.4e11;
    return t_compute >= t_copy;
}

struct HostChunk {
    int prob;
    int64_t m0, rows;
};

// Enqueue one row chunk: its A rows (and, before a problem's first chunk, all of B) go in
// on s_in, the chunk's product runs on `s` once they are in, and its C rows come back on
// s_out while later chunks compute.  Nothing waits on the host.
int enqueue_host_chunk(gemm_handle_t h, const gemm_host_problem& q, const HostStage& st, const HostChunk& c,
                       bool first, int ev, cudaStream_t s)
{
    const size_t es = (q.dtype == GEMM_F32) ? 4 : 2;
    uint8_t* base = static_cast<uint8_t*>(h->host_stage);
    uint8_t* Ad = base + st.a_off;
    uint8_t* Bd = base + st.b_off;
    float* Cd = reinterpret_cast<float*>(base + st.c_off);
    const uint8_t* Ah = static_cast<const uint8_t*>(q.A);
    if (q.K > 0) {
        if (first &&
            copy_rows(Bd, st.ldb_d * es, q.B, q.ldb * es, q.N * es, q.K, cudaMemcpyHostToDevice, h->s_in) != cudaSuccess)
            return GEMM_ERR_CUDA;
        if (copy_rows(Ad + c.m0 * st.lda_d * es, st.lda_d * es, Ah + c.m0 * q.lda * es, q.lda * es, q.K * es, c.rows,
                      cudaMemcpyHostToDevice, h->s_in) != cudaSuccess)
            return GEMM_ERR_CUDA;
    }
    if (cudaEventRecord(h->ev_a[ev], h->s_in) != cudaSuccess || cudaStreamWaitEvent(s, h->ev_a[ev], 0) != cudaSuccess)
        return GEMM_ERR_CUDA;
    const int rc = gemm_run(h, c.rows, q.N, q.K, Ad + c.m0 * st.lda_d * es, st.lda_d, Bd, st.ldb_d,
                            Cd + c.m0 * st.ldc_d, st.ldc_d, (gemm_dtype_t)q.dtype, s);
    if (rc != GEMM_OK) return rc;
    if (cudaEventRecord(h->ev_c[ev], s) != cudaSuccess || cudaStreamWaitEvent(h->s_out, h->ev_c[ev], 0) != cudaSuccess)
        return GEMM_ERR_CUDA;
    if (copy_rows(q.C + c.m0 * q.ldc, q.ldc * 4, Cd + c.m0 * st.ldc_d, st.ldc_d * 4, q.N * 4, c.rows,
                  cudaMemcpyDeviceToHost, h->s_out) != cudaSuccess)
        return GEMM_ERR_CUDA;
    return GEMM_OK;
}

// Run `count` host problems as one pipeline and wait for it.
int run_host_problems(gemm_handle_t h, int count, const gemm_host_problem* q, void* stream)
{
    for (int i = 0; i < count; ++i) {
        const int rc = check_common(h, q[i].M, q[i].N, q[i].K, q[i].A, q[i].lda, q[i].B, q[i].ldb, q[i].C, q[i].ldc,
                                    q[i].dtype);
        if (rc != GEMM_OK) return rc;
        if (q[i].M > 0 && q[i].N > 0 && beyond_kernel_limits(q[i].M, q[i].N, q[i].K, q[i].lda, q[i].ldb, q[i].ldc))
            return GEMM_ERR_UNSUPPORTED;
    }
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    DeviceGuard g(h->device);
    if (!g.ok()) return GEMM_ERR_CUDA;
    // every problem stages in its own region, so later problems' inputs travel while
    // earlier ones compute and drain
    size_t total = 0;
    for (int i = 0; i < count; ++i) total += host_stage_layout(q[i], total).bytes;
    int rc = ensure_buffer(&h->host_stage, &h->host_stage_bytes, total);
    if (rc != GEMM_OK) return rc;
    if ((rc = ensure_pipeline(h)) != GEMM_OK) return rc;
    if (cudaEventRecord(h->ev_start, s) != cudaSuccess || cudaStreamWaitEvent(h->s_in, h->ev_start, 0) != cudaSuccess ||
        cudaStreamWaitEvent(h->s_out, h->ev_start, 0) != cudaSuccess)
        return GEMM_ERR_CUDA;
    std::vector<HostStage> st(count);
    size_t off = 0;
    for (int i = 0; i < count; ++i) {
        st[i] = host_stage_layout(q[i], off);
        off += st[i].bytes;
    }
    // Chunk order on the compute stream: the compute-bound problems' chunks up to half of
    // their work, then the transfer-bound problems' chunks, then the rest.  The first
    // compute starts after a short upload, the transfer-bound chunks' copies hide under
    // compute on both sides, and the last chunk's result is short to bring back.  Chunks
    // of one problem keep their order (its B goes in before its first chunk).
    std::vector<HostChunk> cb, tb;
    double cb_work = 0.0;
    for (int i = 0; i < count; ++i) {
        const bool bound = compute_bound(q[i]);
        int64_t m0 = 0;
        for (const int64_t rows : host_chunk_rows(q[i])) {
            (bound ? cb : tb).push_back({i, m0, rows});
            if (bound) cb_work += (double)rows * (double)q[i].N * (double)q[i].K;
            m0 += rows;
        }
    }
    // compute-bound chunks up to half of their work go first, then the transfer-bound
    // ones, then the rest
    size_t first = 0;
    for (double done = 0.0; first < cb.size() && done < 0.5 * cb_work; ++first)
        done += (double)cb[first].rows * (double)q[cb[first].prob].N * (double)q[cb[first].prob].K;
    std::vector<HostChunk> order(cb.begin(), cb.begin() + first);
    order.insert(order.end(), tb.begin(), tb.end());
    order.insert(order.end(), cb.begin() + first, cb.end());
    std::vector<char> started(count, 0);
    for (size_t k = 0; k < order.size(); ++k) {
        const HostChunk& c = order[k];
        // an event pair is recorded, waited on, then reused: each wait takes the record
        // that precedes it
        rc = enqueue_host_chunk(h, q[c.prob], st[c.prob], c, !started[c.prob], (int)(k % gemm_ctx::kMaxChunks), s);
        if (rc != GEMM_OK) return rc;
        started[c.prob] = 1;
    }
    if (cudaEventRecord(h->ev_done, h->s_out) != cudaSuccess || cudaStreamWaitEvent(s, h->ev_done, 0) != cudaSuccess)
        return GEMM_ERR_CUDA;
    return from_cuda(cudaStreamSynchronize(s));
}

}  // namespace

extern "C" int gemm_run_host(gemm_handle_t h, int64_t M, int64_t N, int64_t K, const void* A, int64_t lda,
                             const void* B, int64_t ldb, float* C, int64_t ldc, gemm_dtype_t dtype, void* stream)
{
    const gemm_host_problem q = {M, N, K, A, lda, B, ldb, C, ldc, (int)dtype};
    return run_host_problems(h, 1, &q, stream);
}

extern "C" int gemm_run_host_batch(gemm_handle_t h, int count, const gemm_host_problem* problems, void* stream)
{
    if (!h || count < 0 || (count > 0 && !problems)) return GEMM_ERR_INVALID_ARG;
    if (count == 0) return GEMM_OK;
    return run_host_problems(h, count, problems, stream);
}

extern "C" {

static int conv4d_im2col_impl(gemm_handle_t h, const float* x, int64_t C_in, const int64_t in_dims[4],
                  const int64_t k_dims[4], float* col, void* stream)
{
    if (!h || !x || !col || !in_dims || !k_dims || C_in <= 0) return GEMM_ERR_INVALID_ARG;
    for (int d = 0; d < 4; ++d)
        if (in_dims[d] <= 0 || k_dims[d] <= 0 || k_dims[d] > in_dims[d] || in_dims[d] > (1 << 20))
            return GEMM_ERR_INVALID_ARG;
    if (C_in > (1 << 20)) return GEMM_ERR_INVALID_ARG;
    DeviceGuard g(h->device);
    if (!g.ok()) return GEMM_ERR_CUDA;
    cudaError_t e = launch_im2col4d(x, C_in, in_dims, k_dims, col, h->num_sms, reinterpret_cast<cudaStream_t>(stream));
    if (e == cudaSuccess) h->launches += 1;
    return from_cuda(e);
}

int64_t gemm_launch_count(gemm_handle_t h)
{
    return h ? h->launches : -1;
}

static int conv4d_forward_impl(gemm_handle_t h, const float* x, int64_t C_in, const int64_t in_dims[4], const float* w,
                   int64_t C_out, const int64_t k_dims[4], float* y, int64_t ldy, void* stream)
{
    if (!h || !x || !w || !y || !in_dims || !k_dims || C_in <= 0 || C_out <= 0) return GEMM_ERR_INVALID_ARG;
    int64_t npos = 1, taps = C_in;
    for (int d = 0; d < 4; ++d) {
        if (in_dims[d] <= 0 || k_dims[d] <= 0 || k_dims[d] > in_dims[d] || in_dims[d] > (1 << 20))
            return GEMM_ERR_INVALID_ARG;
        npos *= in_dims[d] - k_dims[d] + 1;
        taps *= k_dims[d];
    }
    if (ldy < npos || C_in > (1 << 20) || C_out > (1 << 20)) return GEMM_ERR_INVALID_ARG;
    if (k_dims[3] > 40 || npos >= (1ll << 40) || C_in * k_dims[0] * k_dims[1] * k_dims[2] >= (1ll << 31))
        return GEMM_ERR_UNSUPPORTED;
    DeviceGuard g(h->device);
    if (!g.ok()) return GEMM_ERR_CUDA;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const int ngroups = (int)(C_in * k_dims[0] * k_dims[1] * k_dims[2]);
    int split = h->opt_split_k > 0 ? h->opt_split_k : conv_implicit_auto_split(npos, ngroups, h->num_sms);
    if (split > ngroups) split = ngroups;
    const int64_t cblock = C_out < 32 ? C_out : 32;
    if (split > 1) {
        const size_t need = (size_t)split * (size_t)cblock * (size_t)npos * sizeof(float);
        int rc = ensure_buffer(reinterpret_cast<void**>(&h->workspace), &h->workspace_bytes, need);
        if (rc != GEMM_OK) return rc;
    }
    glog("conv4d_forward: implicit GEMM, %lld output positions, %d tap groups, split %d, workspace %lld bytes",
         (long long)npos, ngroups, split, split > 1 ? (long long)split * cblock * npos * 4 : 0ll);
    // output channels in blocks of 32 (rows of W and y)
    for (int64_t o0 = 0; o0 < C_out; o0 += 32) {
        const int64_t nc = (C_out - o0) < 32 ? (C_out - o0) : 32;
        int n = 0;
        cudaError_t e = launch_conv4d_implicit(x, C_in, in_dims, w + o0 * taps, nc, k_dims, y + o0 * ldy, ldy, split,
                                               h->workspace, h->num_sms, s, &n);
        h->launches += n;
        if (e != cudaSuccess) return GEMM_ERR_CUDA;
    }
    return GEMM_OK;
}

static int conv4d_forward_cl_impl(gemm_handle_t h, const void* x, int64_t C_in, const int64_t in_dims[4], const void* w,
                      int64_t C_out, const int64_t k_dims[4], float* y, int dtype, void* stream)
{
    if (!h || !x || !w || !y || !in_dims || !k_dims || C_in <= 0 || C_out <= 0) return GEMM_ERR_INVALID_ARG;
    if (dtype != GEMM_BF16 && dtype != GEMM_F16) return GEMM_ERR_INVALID_ARG;
    for (int d = 0; d < 4; ++d)
        if (in_dims[d] <= 0 || k_dims[d] <= 0 || k_dims[d] > in_dims[d] || in_dims[d] > (1 << 20))
            return GEMM_ERR_INVALID_ARG;
    if (C_in > (1 << 20) || C_out > (1 << 20)) return GEMM_ERR_INVALID_ARG;
    if (((reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(w) | reinterpret_cast<uintptr_t>(y)) & 15) != 0)
        return GEMM_ERR_ALIGNMENT;
    DeviceGuard g(h->device);
    if (!g.ok()) return GEMM_ERR_CUDA;
    int rc = conv4d_tc_supported(C_in, in_dims, C_out, k_dims, h->opt_conv_stack, h->opt_conv_split, h->num_sms);
    if (rc != GEMM_OK) return rc;
    glog("conv4d_forward_cl: tensor-core convolution on CTA pairs, no workspace (stack option %d, split option %d)",
         h->opt_conv_stack, h->opt_conv_split);
    int n = 0;
    rc = launch_conv4d_tc(x, C_in, in_dims, w, C_out, k_dims, y, 0, dtype == GEMM_BF16, h->opt_conv_stack,
                          h->opt_conv_split, h->num_sms, h->d_status, h->wait_limit_ns, h->opt_test_stall, false,
                          reinterpret_cast<cudaStream_t>(stream), &n);
    h->launches += n;
    return rc;
}

static int conv4d_forward_tc_impl(gemm_handle_t h, const void* x, int64_t C_in, const int64_t in_dims[4], const void* w,
                                  int64_t C_out, const int64_t k_dims[4], float* y, int64_t ldy, int dtype,
                                  void* stream)
{
    if (!h || !x || !w || !y || !in_dims || !k_dims || C_in <= 0 || C_out <= 0) return GEMM_ERR_INVALID_ARG;
    if (dtype != GEMM_BF16 && dtype != GEMM_F16) return GEMM_ERR_INVALID_ARG;
    int64_t V = 1, T = 1, npos = 1;
    for (int d = 0; d < 4; ++d) {
        if (in_dims[d] <= 0 || k_dims[d] <= 0 || k_dims[d] > in_dims[d] || in_dims[d] > (1 << 20))
            return GEMM_ERR_INVALID_ARG;
        // each factor is at most 2^20: stop before the products can leave 64 bits
        if (V > (1ll << 40) || T > (1ll << 40)) return GEMM_ERR_UNSUPPORTED;
        V *= in_dims[d];
        T *= k_dims[d];
        npos *= in_dims[d] - k_dims[d] + 1;
    }
    if (C_in > (1 << 20) || C_out > (1 << 20) || ldy < npos) return GEMM_ERR_INVALID_ARG;
    if (((reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(w)) & 1) != 0 ||
        (reinterpret_cast<uintptr_t>(y) & 3) != 0)
        return GEMM_ERR_ALIGNMENT;
    const int64_t Cp = (C_in + 15) / 16 * 16;  // channels padded to the MMA's K with zeros
    if (V > (1ll << 40) || T > (1ll << 40) || (double)V * Cp >= 9.0e15 || (double)C_out * T * Cp >= 9.0e15)
        return GEMM_ERR_UNSUPPORTED;
    if (conv4d_tc_supported(Cp, in_dims, C_out, k_dims, h->opt_conv_stack, h->opt_conv_split, h->num_sms) != GEMM_OK)
        return GEMM_ERR_UNSUPPORTED;
    DeviceGuard g(h->device);
    if (!g.ok()) return GEMM_ERR_CUDA;
    // channel-last copies of x and w in the workspace, each on a 256-byte boundary
    const size_t x_bytes = (size_t)(V * Cp * 2 + 255) / 256 * 256;
    const size_t w_bytes = (size_t)(C_out * T * Cp * 2);
    int rc = ensure_buffer(reinterpret_cast<void**>(&h->workspace), &h->workspace_bytes, x_bytes + w_bytes);
    if (rc != GEMM_OK) return rc;
    void* xc = h->workspace;
    void* wc = reinterpret_cast<uint8_t*>(h->workspace) + x_bytes;
    glog("conv4d_forward_tc: channel-first %s operands re-laid channel-last (C_in %lld padded to %lld), "
         "workspace %lld bytes, then the tensor-core convolution with channel-first output",
         dtype_name(dtype), (long long)C_in, (long long)Cp, (long long)(x_bytes + w_bytes));
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (launch_to_channel_last(x, C_in, V, xc, w, C_out, T, wc, Cp, s) != cudaSuccess) return GEMM_ERR_CUDA;
    h->launches += 1;
    int n = 0;
    rc = launch_conv4d_tc(xc, Cp, in_dims, wc, C_out, k_dims, y, ldy, dtype == GEMM_BF16, h->opt_conv_stack,
                          h->opt_conv_split, h->num_sms, h->d_status, h->wait_limit_ns, h->opt_test_stall, true, s, &n);
    h->launches += n;
    return rc;
}

int gemm_get_device_status(gemm_handle_t h, void* stream)
{
    if (!h) return GEMM_ERR_INVALID_ARG;
    DeviceGuard g(h->device);
    if (!g.ok()) return GEMM_ERR_CUDA;
    if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) return GEMM_ERR_CUDA;
    int v = 0;
    if (cudaMemcpy(&v, h->d_status, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return GEMM_ERR_CUDA;
    if (v != 0) {
        if (cudaMemset(h->d_status, 0, sizeof(int)) != cudaSuccess) return GEMM_ERR_CUDA;
        glog("gemm_get_device_status: a bounded wait ran out (device code %d)", v);
        return GEMM_ERR_DEVICE_TIMEOUT;
    }
#ifdef GEMM_DEBUG
    int bad = 0;
    for (auto take : {bounds_flag_take_ffma, bounds_flag_take_ffma_tma, bounds_flag_take_skinny,
                      bounds_flag_take_skinny_tma, bounds_flag_take_im2col, bounds_flag_take_conv_implicit,
                      bounds_flag_take_conv_tc, bounds_flag_take_tc_gemm}) {
        const int r = take();
        if (r < 0) return GEMM_ERR_CUDA;
        bad |= r;
    }
    if (bad) {
        glog("gemm_get_device_status: a kernel's index check failed (debug build)");
        return GEMM_ERR_DEVICE_BOUNDS;
    }
#endif
    return GEMM_OK;
}

const char* gemm_status_string(int status)
{
    switch (status) {
    case GEMM_OK: return "ok";
    case GEMM_ERR_INVALID_ARG: return "invalid argument";
    case GEMM_ERR_ALIGNMENT: return "misaligned pointer or leading dimension (16-bit inputs need 16-byte alignment)";
    case GEMM_ERR_UNSUPPORTED: return "unsupported device or size";
    case GEMM_ERR_CUDA: return "CUDA runtime error";
    case GEMM_ERR_DEVICE_TIMEOUT: return "a kernel gave up on a bounded wait; its output is invalid";
    case GEMM_ERR_DEVICE_BOUNDS: return "a kernel's index check failed and the access was skipped (debug build); its output is invalid";
    default: return "unknown status";
    }
}

}  // extern "C"

// Entry points: each forwards to its implementation above and, with GEMM_LOG=1, reports a
// refused call with its arguments.
extern "C" {

int gemm_create(gemm_handle_t* out, int device)
{
    const int rc = gemm_create_impl(out, device);
    if (rc != GEMM_OK) glog("gemm_create(device %d) refused: %s (%d)", device, gemm_status_string(rc), rc);
    else glog("gemm_create(device %d): %d SMs", device, (*out)->num_sms);
    return rc;
}

int gemm_set_option(gemm_handle_t h, int option, int64_t value)
{
    const int rc = gemm_set_option_impl(h, option, value);
    if (rc != GEMM_OK)
        glog("gemm_set_option(%d, %lld) refused: %s (%d)", option, (long long)value, gemm_status_string(rc), rc);
    return rc;
}

int gemm_run_ex(gemm_handle_t h, int64_t M, int64_t N, int64_t K, float alpha, const void* A, int64_t lda,
                const void* B, int64_t ldb, float beta, void* C, int64_t ldc, gemm_dtype_t ab_dtype,
                gemm_dtype_t c_dtype, void* stream)
{
    const int rc = gemm_run_ex_impl(h, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, ab_dtype, c_dtype, stream);
    if (rc != GEMM_OK)
        glog("gemm_run(%s, M %lld, N %lld, K %lld, lda %lld, ldb %lld, ldc %lld, A %p, B %p, C %p) refused: %s (%d)",
             dtype_name(ab_dtype), (long long)M, (long long)N, (long long)K, (long long)lda, (long long)ldb,
             (long long)ldc, A, B, C, gemm_status_string(rc), rc);
    return rc;
}

int conv4d_im2col(gemm_handle_t h, const float* x, int64_t C_in, const int64_t in_dims[4], const int64_t k_dims[4],
                  float* col, void* stream)
{
    const int rc = conv4d_im2col_impl(h, x, C_in, in_dims, k_dims, col, stream);
    if (rc != GEMM_OK) glog("conv4d_im2col(C_in %lld) refused: %s (%d)", (long long)C_in, gemm_status_string(rc), rc);
    return rc;
}

int conv4d_forward(gemm_handle_t h, const float* x, int64_t C_in, const int64_t in_dims[4], const float* w,
                   int64_t C_out, const int64_t k_dims[4], float* y, int64_t ldy, void* stream)
{
    const int rc = conv4d_forward_impl(h, x, C_in, in_dims, w, C_out, k_dims, y, ldy, stream);
    if (rc != GEMM_OK)
        glog("conv4d_forward(C_in %lld, C_out %lld, ldy %lld) refused: %s (%d)", (long long)C_in, (long long)C_out,
             (long long)ldy, gemm_status_string(rc), rc);
    return rc;
}

int conv4d_forward_cl(gemm_handle_t h, const void* x, int64_t C_in, const int64_t in_dims[4], const void* w,
                      int64_t C_out, const int64_t k_dims[4], float* y, int dtype, void* stream)
{
    const int rc = conv4d_forward_cl_impl(h, x, C_in, in_dims, w, C_out, k_dims, y, dtype, stream);
    if (rc != GEMM_OK)
        glog("conv4d_forward_cl(C_in %lld, C_out %lld, %s) refused: %s (%d)", (long long)C_in, (long long)C_out,
             dtype_name(dtype), gemm_status_string(rc), rc);
    return rc;
}

int conv4d_forward_tc(gemm_handle_t h, const void* x, int64_t C_in, const int64_t in_dims[4], const void* w,
                      int64_t C_out, const int64_t k_dims[4], float* y, int64_t ldy, int dtype, void* stream)
{
    const int rc = conv4d_forward_tc_impl(h, x, C_in, in_dims, w, C_out, k_dims, y, ldy, dtype, stream);
    if (rc != GEMM_OK)
        glog("conv4d_forward_tc(C_in %lld, C_out %lld, ldy %lld, %s) refused: %s (%d)", (long long)C_in,
             (long long)C_out, (long long)ldy, dtype_name(dtype), gemm_status_string(rc), rc);
    return rc;
}

}  // extern "C"
