// Internal declarations shared by the library's translation units (not installed).
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/gemm.h"

namespace gemm_gb300 {

// Device status word values written by kernels (0 = no error).
enum DeviceStatus : int {
    kDevOk = 0,
    kDevTimeoutProducer = 1,  // producer gave up waiting for a free pipeline stage
    kDevTimeoutMma = 2,       // MMA issuer gave up waiting for a full stage / free accumulator
    kDevTimeoutEpilogue = 3,  // epilogue gave up waiting for a finished accumulator
    kDevTimeoutDrain = 4      // a CTA gave up draining its own copies / MMAs before exit
};

// ------------------------------------------------------------------ host-side log
// With the environment variable GEMM_LOG=1 (read once per process) the library prints one
// line per call on stderr: the kernel it chose, its split of K, the workspace it uses, and
// the reason for every refused call.  Otherwise nothing is printed.
bool log_enabled();
void glog(const char* fmt, ...) __attribute__((format(printf, 1, 2)));

// ------------------------------------------------------------------ debug builds
// Built with -DGEMM_DEBUG (lib/libgemm_gb300_debug.so), every global access a kernel makes
// through an index it computed is checked against the extent of its operand first: a check
// that fails raises the bounds flag of the kernel's translation unit and the access is
// skipped (no trap, no assert; the thread carries on, so every barrier is still reached).
// gemm_get_device_status reads and clears the flags of all translation units and reports
// GEMM_ERR_DEVICE_BOUNDS.  The flags belong to the process and the device, not to a handle.
// In release builds in_range() is constant true and the checks compile away.
#ifdef GEMM_DEBUG
#define GEMM_DEBUG_UNIT(name)                                                                \
    __device__ int g_bounds_flag_##name;                                                     \
    int bounds_flag_take_##name()                                                            \
    {                                                                                        \
        int v = 0, z = 0;                                                                    \
        if (cudaMemcpyFromSymbol(&v, g_bounds_flag_##name, sizeof(int)) != cudaSuccess) {     \
            (void)cudaGetLastError();                                                        \
            return -1;                                                                       \
        }                                                                                    \
        if (v && cudaMemcpyToSymbol(g_bounds_flag_##name, &z, sizeof(int)) != cudaSuccess) { \
            (void)cudaGetLastError();                                                        \
            return -1;                                                                       \
        }                                                                                    \
        return v;                                                                            \
    }                                                                                        \
    static __device__ __forceinline__ bool in_range(int64_t i, int64_t n)                   \
    {                                                                                        \
        const bool ok = i >= 0 && i < n;                                                     \
        if (!ok) atomicExch(&g_bounds_flag_##name, 1);                                      \
        return ok;                                                                           \
    }
// The translation units with kernels (each uses GEMM_DEBUG_UNIT once).
int bounds_flag_take_ffma();
int bounds_flag_take_ffma_tma();
int bounds_flag_take_skinny();
int bounds_flag_take_skinny_tma();
int bounds_flag_take_im2col();
int bounds_flag_take_conv_implicit();
int bounds_flag_take_conv_tc();
int bounds_flag_take_tc_gemm();
#else
#define GEMM_DEBUG_UNIT(name) \
    static __device__ __forceinline__ constexpr bool in_range(int64_t, int64_t) { return true; }
#endif

// Output step of the generalised product: C = alpha * (A . B) + beta * C, C stored as
// fp32, bf16 or fp16 (a gemm_dtype_t); C is not read when beta == 0.
struct Epilogue {
    float alpha = 1.f, beta = 0.f;
    int c_dtype = 0;  // GEMM_F32, GEMM_BF16 or GEMM_F16
    bool plain() const { return alpha == 1.f && beta == 0.f && c_dtype == 0; }
};

// C = alpha * P + beta * C over an M x N fp32 product P (row stride ldp).
cudaError_t launch_epilogue(const float* P, int64_t ldp, void* C, int64_t ldc, int64_t M, int64_t N,
                            const Epilogue& epi, int num_sms, cudaStream_t stream);

// Argument checks every product entry point shares (sizes, pointers, leading dimensions
// and the int64 element-offset range).  GEMM_OK, or GEMM_ERR_INVALID_ARG.  M == 0 or
// N == 0 passes (nothing is done).
int check_product_args(int64_t M, int64_t N, int64_t K, const void* A, int64_t lda, const void* B, int64_t ldb,
                       const void* C, int64_t ldc);
// True when a size or leading dimension is beyond the kernels' 32-bit indexing.
bool beyond_kernel_limits(int64_t M, int64_t N, int64_t K, int64_t lda, int64_t ldb, int64_t ldc);

struct F32Args {
    int64_t M, N, K;
    const float* A;
    int64_t lda;
    const float* B;
    int64_t ldb;
    float* C;
    int64_t ldc;
};

// fp32 tiled FFMA GEMM (128x256 or 64x128 block tiles), optional split-K.
// With split > 1 the partial products go to `workspace` ([split][M][N], ld = N) and a
// fixed-order reduction writes C.  Returns a cudaError_t.
cudaError_t launch_ffma_tiled(const F32Args& a, int variant, int split, float* workspace,
                              int num_sms, cudaStream_t stream, int* launches);

// fp32 GEMM as one persistent launch fed by TMA (128 x 256 x 32 tiles, grouped raster,
// items handed out dynamically):
// a last, partial wave of tiles runs as K slices whose partial tiles the slice that
// finishes last adds in slice order.  Needs 16-byte aligned A and B with lda, ldb % 4 == 0.
struct FfmaPlan {
    int64_t tiles = 0, k_tiles = 0;
    int64_t split_first = 0;   // tiles [split_first, tiles) are cut into `split` K slices
    int split = 1;
    int64_t kt_per_slice = 0;  // 32-deep k-tiles per slice
    int64_t ws_floats = 0;     // partial-tile workspace the slices need
    int64_t counters = 0;      // tagged 64-bit counters: one per split tile, then the item counter
};
bool ffma_persistent_supported(const F32Args& a);
// split_opt > 0 forces that split on every tile.
FfmaPlan ffma_persistent_plan(const F32Args& a, int split_opt, int num_sms);
cudaError_t launch_ffma_persistent(const F32Args& a, const FfmaPlan& plan, float* ws, unsigned long long* cnt,
                                   uint32_t seq, int num_sms, int* dev_status, uint64_t limit_ns, int test_stall,
                                   cudaStream_t stream, int* launches);

// fp32 skinny streaming GEMM for M <= 32: B is read once, straight into registers.
cudaError_t launch_skinny(const F32Args& a, int split, float* workspace, int num_sms,
                          cudaStream_t stream, int* launches);

// fp32 skinny GEMM (M <= 32) with B streamed through a TMA ring in shared memory.
bool skinny_tma_supported(const F32Args& a);
int skinny_tma_auto_split(const F32Args& a, int num_sms);
cudaError_t launch_skinny_tma(const F32Args& a, int split, float* workspace, int num_sms, int* dev_status,
                              uint64_t limit_ns, int test_stall, cudaStream_t stream, int* launches);

// Launch `kern` as a programmatic dependent of the kernel before it on `stream`: its
// blocks may start once every block of that kernel has run griddepcontrol.launch_dependents
// (or it has finished); a kernel that reads what that one writes runs griddepcontrol.wait
// first.  Work queued after it still waits for both.
template <typename... KArgs, typename... Args>
cudaError_t launch_dependent(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                             Args... args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...);
}

// Fixed-order split-K reduction: C[m][n] = sum_{s=0..split-1} ws[s][m][n]; launched as a
// programmatic dependent of the kernel that wrote `ws` (it waits for that kernel before
// reading).
cudaError_t launch_splitk_reduce(const float* ws, int split, int64_t M, int64_t N, float* C,
                                 int64_t ldc, int num_sms, cudaStream_t stream);

// Every launcher adds the number of kernels it launched to *launches.

// The driver's cuTensorMapEncodeTiled (looked up once), or nullptr if unavailable.
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder();

// Workspace floats the 128x256 FFMA path needs to split the tiles of a last, partial wave
// along K (0 when it does not apply).
int64_t ffma_remainder_workspace(const F32Args& a, int variant, int split, int num_sms);

// Split factors the launchers would pick on their own (0 in the option = auto).
int ffma_auto_split(const F32Args& a, int variant, int num_sms);
int skinny_auto_split(const F32Args& a, int num_sms);

// 4-D valid cross-correlation lowering (im2col).
cudaError_t launch_im2col4d(const float* x, int64_t cin, const int64_t in[4], const int64_t k[4],
                            float* col, int num_sms, cudaStream_t stream);

// Valid 4-D cross-correlation on the tensor cores, channel-last 16-bit operands
// (conv4d_forward_cl), S output positions stacked along the MMA's N (0 = choose).
// Workspace bytes it needs (-1 if the shape is not supported).  Returns a gemm_status_t.
// GEMM_OK if the tensor-core convolution takes the shape (stack S, 0 = choose; K split
// ks_opt: 0 choose, 1 none, 2 over two pairs), else GEMM_ERR_UNSUPPORTED; it needs no
// workspace.
int conv4d_tc_supported(int64_t cin, const int64_t in[4], int64_t cout, const int64_t k[4], int S, int ks_opt,
                        int num_sms);
// y channel-last [P][C_out] when ldy_cf == 0, else channel-first (y[o][p] at y + o ldy_cf + p);
// `programmatic`: launched as a programmatic dependent of the kernel before it in the stream
int launch_conv4d_tc(const void* x, int64_t cin, const int64_t in[4], const void* w, int64_t cout,
                     const int64_t k[4], float* y, int64_t ldy_cf, bool bf16, int S, int ks_opt, int num_sms,
                     int* dev_status, uint64_t limit_ns, int test_stall, bool programmatic, cudaStream_t stream,
                     int* launches);
// 16-bit channel-first to channel-last copies, one launch: x [C][V] -> xc [V][Cp] and
// w [B][C][T] -> wc [B][T][Cp], channels C .. Cp-1 zero
cudaError_t launch_to_channel_last(const void* x, int64_t C, int64_t V, void* xc, const void* w, int64_t B,
                                   int64_t T, void* wc, int64_t Cp, cudaStream_t stream);

// Valid 4-D cross-correlation as an implicit GEMM (no column matrix), C_out <= 32 per
// launch.  y[o][p] at y + o*ldy + p; split > 1 uses `workspace` ([split][cout][npos]).
int conv_implicit_auto_split(int64_t npos, int ngroups, int num_sms);
cudaError_t launch_conv4d_implicit(const float* x, int64_t cin, const int64_t in[4], const float* w,
                                   int64_t cout, const int64_t k[4], float* y, int64_t ldy, int split,
                                   float* workspace, int num_sms, cudaStream_t stream, int* launches);

// bf16 / fp16 tensor-core GEMM (tcgen05 + TMA + TMEM), persistent.
struct TcArgs {
    int64_t M, N, K;
    const void* A;
    int64_t lda;
    const void* B;
    int64_t ldb;
    void* C;         // fp32, bf16 or fp16 per epi.c_dtype
    int64_t ldc;
    int is_bf16;     // 1 = bf16, 0 = fp16
    int test_stall;  // test hook: make a bounded wait run out (exercises the timeout path)
    Epilogue epi;
    // CTA-pair kernel, K split of the last wave's tiles (sizes from tc_workspace_need;
    // null: no split)
    float* rem_ws = nullptr;                  // partial tiles (when TcWorkspace::floats > 0)
    unsigned long long* rem_cnt = nullptr;    // arrival counters, zeroed when allocated
    uint32_t* rem_flag = nullptr;             // publication flags, as many, zeroed when allocated
    unsigned rem_seq = 0;                     // a nonzero tag no earlier launch on them used
};
struct TcWorkspace {
    int64_t floats = 0;    // partial-tile floats
    int64_t counters = 0;  // 64-bit arrival counters, and as many 32-bit flags
};
// What launch_tc_gemm with these arguments would use to split its last wave (zero: none).
TcWorkspace tc_workspace_need(const TcArgs& a, int num_sms, int pair_mode);
// Returns GEMM_OK or a negative gemm_status_t.
// kc_blocks: 64-wide k-blocks per accumulation chunk (0 = default 16).
// pair_mode: 0 = choose, 1 = single-CTA 128 x 256 tiles, 2 = CTA-pair 256 x 256 tiles.
// With pair_mode 0, M <= 128 and tiles that fill under half the SMs, K is split into
// slices run by the CTAs of one cluster per tile (no workspace).
int launch_tc_gemm(const TcArgs& a, int num_sms, int* dev_status, uint64_t wait_limit_ns, int kc_blocks,
                   int pair_mode, cudaStream_t stream, int* launches);

}  // namespace gemm_gb300
