/*
 * gemm.h -- C ABI of the GB300 (sm_103a) dense GEMM library.
 *
 * The operation is the matrix product of "Learning to develop for GPU with GEMM as the
 * example", section "Matrix product": C (M x N) = A (M x K) . B (K x N), where each
 * element of C is the sum over k of A[i][k] * B[k][j].  That section's "generalised"
 * form (section "Generalised matrix multiplication GEMM") also scales the product and
 * adds a scaled accumulator; this library computes the plain product (alpha = 1,
 * beta = 0) and OVERWRITES C.
 *
 * Layout: row-major throughout, with leading dimensions counted in elements:
 *     A[i][k] = A[i*lda + k],  B[k][j] = B[k*ldb + j],  C[i][j] = C[i*ldc + j].
 * The page's own examples are column-major; a column-major caller gets its product by
 * swapping the operands (C^T = B^T . A^T) and passing the same pointers.
 *
 * Input types: fp32 (FFMA path), bf16 or fp16 (tensor-core path).  C is always fp32,
 * accumulated in fp32.
 *
 * Memory ownership: A, B, C, x, col are caller-owned device pointers on the handle's
 * device (any allocation the CUDA runtime can address from that device), except in
 * gemm_run_host where they are host pointers.  The library never frees caller memory.
 * The handle owns a small device status word, a split-K workspace (grown on demand,
 * stream-ordered) and host-call staging buffers; gemm_destroy frees them.
 *
 * Streams: calls taking `stream` enqueue on that cudaStream_t (NULL = the legacy
 * default stream) and return without waiting, except gemm_run_host and
 * gemm_get_device_status, which synchronise the stream.  The returned status covers
 * argument checks and launch errors only; errors raised later on the device (a
 * bounded wait that ran out) are reported by gemm_get_device_status.
 *
 * Threads: a handle is not thread-safe.  Use one handle per host thread, or serialise
 * calls.  Calls on one handle from different streams must not overlap in time when
 * they use the split-K workspace (fp32 shapes with small M or few output tiles; bf16 /
 * fp16 shapes whose last wave of 256 x 256 tiles is cut along K).
 *
 * Errors: every entry point returns a gemm_status_t (0 = success, negative = error)
 * and writes nothing when it fails its argument checks.
 */
#ifndef GEMM_GB300_H
#define GEMM_GB300_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct gemm_ctx* gemm_handle_t; /* opaque, owned by the library */

typedef enum {
    GEMM_F32 = 0,  /* fp32 inputs, register-blocked FFMA kernels */
    GEMM_BF16 = 1, /* bf16 inputs, tcgen05 tensor cores, fp32 accumulate */
    GEMM_F16 = 2   /* fp16 inputs, tcgen05 tensor cores, fp32 accumulate */
} gemm_dtype_t;

typedef enum {
    GEMM_OK = 0,
    GEMM_ERR_INVALID_ARG = -1,    /* null handle/pointer, negative size, ld < cols, ... */
    GEMM_ERR_ALIGNMENT = -2,      /* bf16/fp16: base not 16-byte aligned or ld*2 % 16 != 0 */
    GEMM_ERR_UNSUPPORTED = -3,    /* device is not sm_103, or a size beyond a kernel limit */
    GEMM_ERR_CUDA = -4,           /* a CUDA runtime call or a launch failed */
    GEMM_ERR_DEVICE_TIMEOUT = -5, /* a kernel's bounded wait ran out (see gemm_get_device_status) */
    GEMM_ERR_DEVICE_BOUNDS = -6   /* debug library only: a kernel's index check failed and the access was
                                     skipped (see gemm_get_device_status) */
} gemm_status_t;

/* Create a handle bound to CUDA device `device`.  Queries the SM count, allocates the
 * device status word.  The caller's current device is restored before returning.
 * Fails with GEMM_ERR_UNSUPPORTED unless the device is compute capability 10.3.
 * The handle is the set-up step of the host program in "Learning to develop for GPU with
 * GEMM as the example", section "Writing a GPU implementation of matrix multiplication"
 * (its part on initialising the device: a device chosen by index and a context built on
 * it; the command queue there is the caller's CUDA stream here), and it owns the extra
 * memory that "Three X: large convolutions in PyTorch for training", section "How to call
 * a convolution in the CUTLASS library", has the caller query and provide before the
 * operation is initialised (here it is sized and grown by the library). */
int gemm_create(gemm_handle_t* out, int device);

/* Destroy a handle and free the memory it owns (not caller memory).  The handle's
 * streams must be idle (the call synchronises the device).  NULL is a no-op.
 * The end of the life cycle whose start is gemm_create: the device objects of "Learning
 * to develop for GPU with GEMM as the example", section "Writing a GPU implementation of
 * matrix multiplication", and the workspace of "Three X: large convolutions in PyTorch for
 * training", section "How to call a convolution in the CUTLASS library". */
int gemm_destroy(gemm_handle_t h);

/* C = A . B (alpha = 1, beta = 0; C is overwritten, never read): the product of
 * "Learning to develop for GPU with GEMM as the example", section "Matrix product", with
 * the argument list (m, n, k, a, b, c) that section "Writing a GPU implementation of
 * matrix multiplication" hands its kernel, plus leading dimensions, the type and a
 * stream in place of the command queue.
 *   M, N, K  >= 0.  M == 0 or N == 0: nothing is done.  K == 0: C is set to zero.
 *   lda >= K, ldb >= N, ldc >= N (elements).  Rows may be padded; padding is never
 *   read or written.  Every size and leading dimension must stay below 2^31 - 1024
 *   (the kernels index in 32 bits), else GEMM_ERR_UNSUPPORTED before anything is
 *   allocated or launched.
 *   dtype GEMM_F32: A, B are float*; any alignment (16-byte aligned bases and ld % 4
 *   == 0 take the vectorised loads).
 *   dtype GEMM_BF16 / GEMM_F16: A, B are 16-bit; A, B must be 16-byte aligned and
 *   lda, ldb multiples of 8 elements (TMA tensor-map rules), else GEMM_ERR_ALIGNMENT.
 *   C (float*) needs no alignment beyond 4 bytes.
 *   stream: cudaStream_t (NULL = legacy default stream).  Asynchronous.
 * Kernel choice is by shape and dtype among this library's own kernels only.  Results
 * are deterministic: the same call on the same device repeats its result bit for bit
 * (every split of K adds its slices in a fixed order). */
int gemm_run(gemm_handle_t h, int64_t M, int64_t N, int64_t K,
             const void* A, int64_t lda, const void* B, int64_t ldb,
             float* C, int64_t ldc, gemm_dtype_t dtype, void* stream);

/* The generalised product of "Learning to develop for GPU with GEMM as the example",
 * section "Generalised matrix multiplication GEMM" (a weighted product added to a
 * weighted accumulator):
 *     C = alpha * (A . B) + beta * C,
 * with C stored as c_dtype (GEMM_F32, GEMM_BF16 or GEMM_F16; rounded to nearest even)
 * and read only when beta != 0 (the BLAS convention: with beta == 0, C may hold
 * anything, NaN included).  The product accumulates in fp32 as in gemm_run; the
 * epilogue computes alpha * p in fp32, then fma(beta, c, .) in fp32, then converts.
 * Tensor-core products (bf16 / fp16 inputs) apply it as they store C; fp32 inputs
 * store their fp32 product in a handle-owned buffer (M x N floats, grown on demand)
 * and apply it in one more pass.  C must be aligned to its element size; other
 * arguments and errors as in gemm_run.  gemm_run is this call with alpha = 1,
 * beta = 0, c_dtype = GEMM_F32. */
int gemm_run_ex(gemm_handle_t h, int64_t M, int64_t N, int64_t K, float alpha,
                const void* A, int64_t lda, const void* B, int64_t ldb, float beta,
                void* C, int64_t ldc, gemm_dtype_t ab_dtype, gemm_dtype_t c_dtype, void* stream);

/* The same product with A, B and C in HOST memory (pageable or pinned): the whole host
 * program of "Learning to develop for GPU with GEMM as the example", section "Writing a
 * GPU implementation of matrix multiplication" (copy the inputs to device buffers,
 * enqueue the kernel, read the result back), with the copies overlapped with compute.  A and B are
 * copied into handle-owned device buffers and C is copied back, on two internal
 * streams ordered after the work already queued on `stream`; the product runs on
 * `stream`.  Large products are pipelined over row chunks (a multiple of 256 rows;
 * up to 8 chunks of >= 1024 rows for 16-bit inputs, 2 chunks of >= 2048 rows for fp32):
 * A chunk i+1 travels while chunk i computes, and C chunk i travels back while chunk
 * i+1 computes.  Overlap needs
 * pinned host memory; pageable memory is copied through the driver's staging.
 * Returns after `stream` has been synchronised.  Leading dimensions as in gemm_run. */
int gemm_run_host(gemm_handle_t h, int64_t M, int64_t N, int64_t K,
                  const void* A, int64_t lda, const void* B, int64_t ldb,
                  float* C, int64_t ldc, gemm_dtype_t dtype, void* stream);

/* One product of gemm_run_host_batch: the arguments of gemm_run_host. */
typedef struct gemm_host_problem {
    int64_t M, N, K;
    const void* A;
    int64_t lda;
    const void* B;
    int64_t ldb;
    float* C;
    int64_t ldc;
    int dtype; /* gemm_dtype_t of A and B */
} gemm_host_problem;

/* Several host-memory products as one pipeline (the host program of "Learning to develop
 * for GPU with GEMM as the example", section "Writing a GPU implementation of matrix
 * multiplication", run for a list of products): each is staged in its own region of the
 * handle's device buffer and split into row chunks as in gemm_run_host.  The chunks run
 * on `stream` with half of the compute-bound products' chunks first, the transfer-bound
 * products' chunks next and the rest last (chunks of one product in order), so copies in
 * both directions hide under compute.  Each C is the same as gemm_run_host's.
 * Every problem is checked before anything is queued (the first failing check is
 * returned and nothing runs).  Returns after `stream` has been synchronised.
 * count == 0 is a no-op. */
int gemm_run_host_batch(gemm_handle_t h, int count, const gemm_host_problem* problems, void* stream);

/* Lowering of a valid (no padding, stride 1, dilation 1) 4-D cross-correlation to a
 * GEMM operand, as in "Three X: large convolutions in PyTorch for training", section
 * "CuBLAS" (im2col / vol2col, extended by one spatial dimension):
 *   x   : fp32 [C_in][in[0]][in[1]][in[2]][in[3]], contiguous, device memory.
 *   col : fp32 [C_in*k0*k1*k2*k3][P0*P1*P2*P3], contiguous, device memory, where
 *         Pd = in[d] - k[d] + 1.  Row (c, r0, r1, r2, r3) row-major; column = output
 *         position (p0, p1, p2, p3) row-major.
 *         col[row][col] = x[c][p0+r0][p1+r1][p2+r2][p3+r3].
 * With weights W as the row-major [C_out][C_in*k0*k1*k2*k3] matrix, gemm_run(W, col)
 * gives the output [C_out][P0*P1*P2*P3].  Asynchronous on `stream`.
 * GEMM_ERR_INVALID_ARG if any extent is <= 0 or k[d] > in[d]. */
int conv4d_im2col(gemm_handle_t h, const float* x, int64_t C_in, const int64_t in_dims[4],
                  const int64_t k_dims[4], float* col, void* stream);

/* The same valid 4-D cross-correlation computed directly, as an implicit GEMM: the
 * column matrix of conv4d_im2col is never stored ("Three X: large convolutions in
 * PyTorch for training", sections "CUTLASS" and "What else had to change when using
 * CUTLASS": the operand tile is gathered from the input on the fly).
 *   x : fp32 [C_in][in[0]][in[1]][in[2]][in[3]], contiguous, device memory.
 *   w : fp32 [C_out][C_in][k[0]][k[1]][k[2]][k[3]], contiguous, device memory.
 *   y : fp32 output, y[o][p] at y + o*ldy + p, p the row-major output position over
 *       (P0, P1, P2, P3), Pd = in[d] - k[d] + 1; ldy >= P0*P1*P2*P3.  Overwritten.
 * fp32 FMAs, accumulation order over taps (c, r0, r1, r2, r3) in slices added in fixed
 * order: results are deterministic and agree with gemm_run(W, im2col(x)) within fp32
 * rounding.  Asynchronous on `stream`; uses the handle's split-K workspace.
 * GEMM_ERR_INVALID_ARG for bad extents or pointers; GEMM_ERR_UNSUPPORTED if k[3] > 40. */
int conv4d_forward(gemm_handle_t h, const float* x, int64_t C_in, const int64_t in_dims[4], const float* w,
                   int64_t C_out, const int64_t k_dims[4], float* y, int64_t ldy, void* stream);

/* The same valid 4-D cross-correlation on the tensor cores, with 16-bit channel-last
 * operands ("Three X: large convolutions in PyTorch for training", section "CUTLASS":
 * the tensor-core implicit GEMM wants 128-bit aligned tensors, channel counts that are
 * multiples of the MMA's K and channel-last memory order).
 *   x : [in[0]][in[1]][in[2]][in[3]][C_in], bf16 or fp16 (`dtype`), contiguous, device.
 *   w : [C_out][k[0]][k[1]][k[2]][k[3]][C_in], the same type, contiguous, device.
 *   y : fp32 [P0][P1][P2][P3][C_out], contiguous, device, Pd = in[d] - k[d] + 1;
 *       overwritten.  y[p][o] = sum over taps r and channels c of x[p + r][c] * w[o][r][c].
 * Products of 16-bit values are exact in fp32; the tensor core accumulates in fp32, with
 * consecutive MMAs (16 channels of one window of taps) going round-robin to up to 8
 * partial sums that are added in fp32 round-to-nearest, in order.  Deterministic.
 * Asynchronous on `stream`.  One launch on CTA pairs (tcgen05 cta_group::2), reading x and w
 * straight from the caller's tensors with the Tensor Memory Accelerator; no workspace.  When
 * the tiles would fill at most a quarter of the SMs, two pairs (one cluster of four CTAs)
 * share each tile, each over half of K, and add their partial tiles through distributed
 * shared memory in a fixed order (deterministic).
 * x, w and y must be 16-byte aligned (GEMM_ERR_ALIGNMENT).
 * GEMM_ERR_INVALID_ARG for bad extents, pointers or dtype (GEMM_BF16 or GEMM_F16 only);
 * GEMM_ERR_UNSUPPORTED unless C_in % 16 == 0, C_out % 16 == 0, S * C_out <= 256,
 * in[3] % S == 0, three pipeline stages of one filter triple (r0, r1, r2) and one 16-channel
 * step fit in shared memory, and the input rows of one stage (128 + (k[3] + S - 2) / S)
 * are at most 256. */
int conv4d_forward_cl(gemm_handle_t h, const void* x, int64_t C_in, const int64_t in_dims[4], const void* w,
                      int64_t C_out, const int64_t k_dims[4], float* y, int dtype, void* stream);

/* The tensor-core convolution for 16-bit operands in PyTorch's channel-first order
 * ("Three X: large convolutions in PyTorch for training", section "CUTLASS", its closing
 * part on memory layout: PyTorch keeps channels outermost, so the channel-last operands
 * the tensor-core implicit GEMM wants are produced by transposing the input and the
 * filters first).
 *   x : [C_in][in[0]][in[1]][in[2]][in[3]], bf16 or fp16 (`dtype`), contiguous, device.
 *   w : [C_out][C_in][k[0]][k[1]][k[2]][k[3]], the same type, contiguous, device.
 *   y : fp32 output, y[o][p] at y + o*ldy + p (the layout of conv4d_forward), p the
 *       row-major output position over (P0, P1, P2, P3), Pd = in[d] - k[d] + 1;
 *       ldy >= P0*P1*P2*P3.  Overwritten.
 * Two launches on `stream`: one kernel re-lays x and w channel-last into the handle's
 * workspace (V*Cp + C_out*T*Cp 16-bit values, V = in[0]*..*in[3], T = k[0]*..*k[3],
 * Cp = C_in rounded up to a multiple of 16, the added channels zero), then the kernel of
 * conv4d_forward_cl, launched as its programmatic dependent (its set-up overlaps the
 * re-layout; its first copy waits for it), runs on those copies and stores y
 * channel-first.  Results equal
 * conv4d_forward_cl's on the re-laid operands, bit for bit.
 * x and w must be 2-byte aligned and y 4-byte aligned (GEMM_ERR_ALIGNMENT).
 * GEMM_ERR_INVALID_ARG for bad extents, pointers, ldy or dtype (GEMM_BF16 or GEMM_F16);
 * GEMM_ERR_UNSUPPORTED when conv4d_forward_cl would refuse C_in = Cp (C_out % 16 != 0,
 * S * C_out > 256, a stage that does not fit) or the copies' sizes leave 64 bits;
 * GEMM_ERR_CUDA if the workspace cannot be allocated. */
int conv4d_forward_tc(gemm_handle_t h, const void* x, int64_t C_in, const int64_t in_dims[4], const void* w,
                      int64_t C_out, const int64_t k_dims[4], float* y, int64_t ldy, int dtype, void* stream);

/* Synchronise `stream`, then read and clear the handle's device status word (and, in the
 * debug library, the kernels' bounds-check flags).  This is
 * the wait of "Learning to develop for GPU with GEMM as the example", section "Writing a
 * GPU implementation of matrix multiplication" (its part on launching the kernel: the host
 * waits on an event for the enqueued kernel), extended with the kernel's own report.
 * Returns GEMM_OK, or GEMM_ERR_DEVICE_TIMEOUT if a kernel launched through this
 * handle gave up on a bounded wait since the last call (its output is then invalid),
 * GEMM_ERR_DEVICE_BOUNDS (debug library, lib/libgemm_gb300_debug.so, built with
 * -DGEMM_DEBUG) if a kernel of this process found a computed global index outside its
 * operand since the last call and skipped that access (the output is then invalid; these
 * flags are per process and device, not per handle), or GEMM_ERR_CUDA if the stream
 * reports an error.
 * Debugging aids: the environment variable GEMM_LOG=1 makes the library print, on stderr,
 * one line per call with the kernel it chose, its split of K and the workspace it uses,
 * and the reason for every refused call; any other value (or none) prints nothing. */
int gemm_get_device_status(gemm_handle_t h, void* stream);

/* Tuning and test options (see GEMM_OPT_*).  Values outside the documented range are
 * rejected with GEMM_ERR_INVALID_ARG.  Defaults are restored by passing 0.
 * The choices "Three X: large convolutions in PyTorch for training", section "How to
 * call a convolution in the CUTLASS library", makes when it builds the operation's type
 * (which tile iterator, which epilogue), made here at run time on a handle. */
typedef enum {
    GEMM_OPT_F32_KERNEL = 1, /* 0 auto, 1 tiled 128x256 FFMA (one launch per wave kind), 2 tiled 64x128 FFMA,
                                3 skinny streaming from registers (M<=32), 4 skinny streaming through a TMA
                                ring (M<=32; B 16-byte aligned with ldb % 4 == 0, else GEMM_ERR_ALIGNMENT),
                                5 persistent 128x256 FFMA fed by TMA, one launch per product (A and B
                                16-byte aligned with lda, ldb % 4 == 0, else GEMM_ERR_ALIGNMENT).  Auto:
                                M<=32 skinny (4, else 3), M<=64 2, else 5 when its alignment holds, else 1 */
    GEMM_OPT_SPLIT_K = 2,    /* 0 auto, else the split-K factor for fp32 kernels (1..1024) */
    GEMM_OPT_WAIT_LIMIT_US = 3, /* 0 default (2 s), else the bounded-wait limit of device waits in microseconds */
    GEMM_OPT_TC_CHUNK = 4,      /* 0 default (16), else the tensor-core accumulation chunk in 64-wide k-blocks
                                   (1..4096): the tensor core's fp32 accumulator is restarted every chunk and
                                   chunk sums are added in fp32 round-to-nearest */
    GEMM_OPT_TC_PAIR = 5,       /* tensor-core tiles: 0 choose (default: pairs when M > 128; for M <= 128 with
                                   128x256 tiles that fill under half the SMs, K split into 2 to 16 slices,
                                   one CTA each, on a cluster per tile that adds the fp32 partial tiles in
                                   slice order through distributed shared memory), 1 one CTA per
                                   128x256 tile, 2 a pair of CTAs (cluster of two) per 256x256 tile.  Any
                                   other value (3 included) is GEMM_ERR_INVALID_ARG */
    GEMM_OPT_TEST_STALL = 6,    /* test hook for failure detection, 0 (default) or 1: the kernels with
                                   bounded waits (tensor-core GEMMs and convolution, TMA skinny GEMM, persistent
                                   fp32 GEMM) first wait on a
                                   barrier nothing arrives on; the wait runs out after the wait limit, the
                                   kernel drains its copies and MMAs, frees its tensor memory, returns,
                                   and gemm_get_device_status reports GEMM_ERR_DEVICE_TIMEOUT.  C is not
                                   written.  No fault, trap or unbounded wait is involved. */
    GEMM_OPT_CONV_STACK = 7,    /* tensor-core convolution (conv4d_forward_cl, conv4d_forward_tc): output
                                   positions stacked along the MMA's N, 0 choose (default: 4 when that plan,
                                   with its K split over two CTA pairs per tile, fills between half and all
                                   of the SMs in one wave; else 2 when in[3] is even and 2*C_out <= 256;
                                   else 1), or 1, 2, 4 */
    GEMM_OPT_CONV_SPLIT = 8     /* tensor-core convolution: K split over CTA pairs, 0 choose (default: two
                                   pairs per tile when the tiles would fill at most a quarter of the SMs),
                                   1 one pair per tile, 2 two pairs per tile (GEMM_ERR_UNSUPPORTED from the
                                   convolution when S*C_out is not a multiple of 32 or there is a single
                                   pipeline stage) */
} gemm_option_t;
int gemm_set_option(gemm_handle_t h, int option, int64_t value);

/* Number of kernels launched through this handle since it was created (a cumulative
 * count kept on the host; -1 for a NULL handle).  Zero-size calls launch nothing.
 * It counts the kernel enqueues of "Learning to develop for GPU with GEMM as the
 * example", section "Writing a GPU implementation of matrix multiplication" (its part on
 * launching the kernel). */
int64_t gemm_launch_count(gemm_handle_t h);

/* fp32 C = A . B for M <= 32 (the skinny streaming kernel) WITHOUT ALLOCATING.
 *
 * The pages have no counterpart to this entry point; it exists for callers that must
 * not allocate device memory: code that runs inside another framework's memory
 * manager (which already owns the device memory and forbids or cannot satisfy
 * cudaMalloc), or a latency-critical path where cudaMalloc / cudaFree would
 * synchronise the device.  Such a caller cannot create a gemm handle either (that
 * allocates), so this call takes no handle and runs on the calling thread's current
 * device, on `stream` (NULL = legacy default stream), asynchronously.
 *
 * The split-K partial sums live in a file-scope device array of 8,388,608 floats
 * (32 MiB) inside the library; every GPU that loads the library's device code holds
 * it until the process exits.  The call never calls cudaMalloc, cudaFree or any
 * allocating library routine.
 *   - The FIRST call on each device looks up that array's device address
 *     (cudaGetSymbolAddress, which may load the library's device code); make that
 *     first call before any stream capture.  The address is cached with the unique ID
 *     of the context it was taken in, and a call made under another context of that
 *     device (after cudaDeviceReset, or with a context the caller made current) looks
 *     it up again: such a call is a first call too.
 *   - All calls share the one array and it keeps the last call's contents: two
 *     calls that can run at the same time on the GPU (different streams, or
 *     different host threads) race on it and both results are then undefined.
 *     Serialise them on one stream.  Nothing needs clearing between calls: every
 *     partial sum is written before it is read.
 * It runs the register-streaming skinny kernel, the one gemm_run runs for M <= 32 with
 * GEMM_OPT_F32_KERNEL = 3.  Arguments as in gemm_run with dtype GEMM_F32; split_k = 0
 * picks the split gemm_run picks for that kernel (results are then bit-identical to
 * gemm_run with that option; gemm_run's default TMA-fed kernel agrees within fp32
 * rounding), 1..1024 forces one.  Errors: GEMM_ERR_INVALID_ARG for bad arguments (gemm_run's
 * checks), GEMM_ERR_UNSUPPORTED for M > 32, for sizes beyond the kernels' 32-bit indexing
 * (as gemm_run), for a device that is not sm_103, or when split * M * N exceeds the
 * 8,388,608-float scratch array (the size limit); nothing is written then. */
int gemm_run_f32_skinny_noalloc(int64_t M, int64_t N, int64_t K, const float* A, int64_t lda,
                                const float* B, int64_t ldb, float* C, int64_t ldc, int split_k,
                                void* stream);

/* Static string describing a status code: the outcome of a step of the host program of
 * "Learning to develop for GPU with GEMM as the example", section "Writing a GPU
 * implementation of matrix multiplication" (device set-up, argument checks, the enqueue,
 * the wait). */
const char* gemm_status_string(int status);

#ifdef __cplusplus
}
#endif

#endif /* GEMM_GB300_H */
