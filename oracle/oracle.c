/*
 * CPU oracle for the GEMM library.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path links, loads or calls this
 * file: only the test suite, the smoke check and the benchmark's CPU-baseline leg do.
 * It shares no source, header, table or helper with the CUDA library; the two meet
 * only through seeded inputs that the test harness hands to both.
 *
 * What it computes, and where the pages define it:
 *
 *   oracle_gemm          C[i][j] = sum_{k=0..K-1} A[i][k] * B[k][j]
 *       "Learning to develop for GPU with GEMM as the example", section "Matrix
 *       product": each element of C is the sum of products of a row of A with a
 *       column of B; the CPU version there is three nested loops.  The page's loop is
 *       column-major and accumulates into a zeroed C; this restatement is row-major
 *       (A[i*lda+k], B[k*ldb+j], C[i*ldc+j]) and overwrites C, which is the same
 *       result.  The sum runs over k in ascending order, in double precision, with the
 *       multiply and the add rounded separately (built with -ffp-contract=off).
 *       The loops over i and j only name independent elements, so the code walks
 *       them as i, k, j to stream rows of B; every C[i][j] still sees exactly the
 *       additions 0 + A[i][0]B[0][j] + A[i][1]B[1][j] + ... in that order, so the
 *       result is bit-identical to the i, j, k nesting.
 *
 *   oracle_gemm_general  the "generalised" product of the same page, section "Generalised
 *       matrix multiplication GEMM": a weighted product added to a weighted accumulator,
 *         D[i][j] = alpha * (sum_k A[i][k] * B[k][j]) + beta * C[i][j],
 *       with the sum exactly as in oracle_gemm and C not read when beta == 0 (the usual
 *       BLAS convention); double precision throughout, each operation rounded once.
 *
 *   oracle_gemm_entries  the same sum for a list of (i, j) pairs, with B given by
 *       an arbitrary element stride pair so a transposed copy can be streamed.
 *
 *   oracle_conv4d_direct valid (no padding, stride 1, dilation 1) 4-D
 *       cross-correlation, written as its nested loops:
 *         y[o][p0][p1][p2][p3] = sum_c sum_{r0..r3} w[o][c][r0][r1][r2][r3]
 *                                       * x[c][p0+r0][p1+r1][p2+r2][p3+r3]
 *       "Three X: large convolutions in PyTorch for training", sections "Why we need
 *       high-dimensional convolution" (N-D inputs) and "CuBLAS" (PyTorch-style
 *       convolution, output extent in - k + 1 at stride 1 without padding).
 *       The summation order is c, r0, r1, r2, r3 ascending.
 *
 *   oracle_im2col4d      the lowering of the same convolution to a matrix: one column
 *       per filter application, one row per (c, r0, r1, r2, r3) filter tap, columns
 *       ordered row-major over the output positions (p0, p1, p2, p3).
 *       "Three X ...", section "CuBLAS" (im2col / vol2col: every column of the
 *       convolution matrix is one application of the filter; higher dimensions add
 *       one index and one loop each).
 *
 * Threads: a static partition of output rows over pthreads; each element's sum is
 * computed by one thread in the order stated above, so the result does not depend on
 * the thread count.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_MAX_THREADS 256

typedef void (*row_fn)(void* ctx, int64_t lo, int64_t hi);

typedef struct {
    row_fn fn;
    void* ctx;
    int64_t lo, hi;
} slice_t;

static void* run_slice(void* p)
{
    slice_t* s = (slice_t*)p;
    s->fn(s->ctx, s->lo, s->hi);
    return NULL;
}

/* Split [0, n) into nthreads contiguous slices and run fn on each. */
static int parallel_rows(row_fn fn, void* ctx, int64_t n, int nthreads)
{
    if (nthreads < 1) nthreads = 1;
    if (nthreads > ORACLE_MAX_THREADS) nthreads = ORACLE_MAX_THREADS;
    if ((int64_t)nthreads > n) nthreads = (int)(n > 0 ? n : 1);
    if (nthreads == 1) {
        fn(ctx, 0, n);
        return 0;
    }
    pthread_t tid[ORACLE_MAX_THREADS];
    slice_t sl[ORACLE_MAX_THREADS];
    int started = 0;
    for (int t = 0; t < nthreads; ++t) {
        sl[t].fn = fn;
        sl[t].ctx = ctx;
        sl[t].lo = n * t / nthreads;
        sl[t].hi = n * (t + 1) / nthreads;
        if (pthread_create(&tid[t], NULL, run_slice, &sl[t]) != 0) {
            /* fall back to running the slice on this thread */
            run_slice(&sl[t]);
            tid[t] = 0;
        } else {
            ++started;
        }
    }
    for (int t = 0; t < nthreads; ++t)
        if (tid[t]) pthread_join(tid[t], NULL);
    (void)started;
    return 0;
}

/* ------------------------------------------------------------------------- GEMM */

typedef struct {
    int64_t N, K;
    const float* A;
    int64_t lda;
    const float* B;
    int64_t ldb;
    double* C;
    int64_t ldc;
} gemm_ctx_t;

static void gemm_rows(void* p, int64_t lo, int64_t hi)
{
    const gemm_ctx_t* g = (const gemm_ctx_t*)p;
    for (int64_t i = lo; i < hi; ++i) {
        double* c = g->C + i * g->ldc;
        for (int64_t j = 0; j < g->N; ++j) c[j] = 0.0;
        for (int64_t k = 0; k < g->K; ++k) {
            const double a = (double)g->A[i * g->lda + k];
            const float* b = g->B + k * g->ldb;
            for (int64_t j = 0; j < g->N; ++j) {
                const double prod = a * (double)b[j];
                c[j] = c[j] + prod;
            }
        }
    }
}

int oracle_gemm(int64_t M, int64_t N, int64_t K, const float* A, int64_t lda,
                const float* B, int64_t ldb, double* C, int64_t ldc, int nthreads)
{
    if (M < 0 || N < 0 || K < 0) return -1;
    if (M == 0 || N == 0) return 0;
    if (ldc < N || (K > 0 && (lda < K || ldb < N))) return -1;
    gemm_ctx_t g = {N, K, A, lda, B, ldb, C, ldc};
    return parallel_rows(gemm_rows, &g, M, nthreads);
}

int oracle_gemm_general(int64_t M, int64_t N, int64_t K, double alpha, const float* A, int64_t lda,
                        const float* B, int64_t ldb, double beta, const double* C, int64_t ldc, double* D,
                        int64_t ldd, int nthreads)
{
    if (M < 0 || N < 0 || K < 0) return -1;
    if (M == 0 || N == 0) return 0;
    if (beta != 0.0 && (!C || ldc < N)) return -1;
    int rc = oracle_gemm(M, N, K, A, lda, B, ldb, D, ldd, nthreads);
    if (rc != 0) return rc;
    for (int64_t i = 0; i < M; ++i)
        for (int64_t j = 0; j < N; ++j) {
            const double prod = alpha * D[i * ldd + j];
            D[i * ldd + j] = (beta != 0.0) ? prod + beta * C[i * ldc + j] : prod;
        }
    return 0;
}

typedef struct {
    int64_t K;
    const float* A;
    int64_t lda;
    const float* B;
    int64_t b_sk, b_sj; /* B[k][j] = B[k*b_sk + j*b_sj] */
    const int64_t* rows;
    const int64_t* cols;
    double* out;
} entries_ctx_t;

static void entry_range(void* p, int64_t lo, int64_t hi)
{
    const entries_ctx_t* e = (const entries_ctx_t*)p;
    for (int64_t t = lo; t < hi; ++t) {
        const int64_t i = e->rows[t], j = e->cols[t];
        double acc = 0.0;
        for (int64_t k = 0; k < e->K; ++k) {
            const double prod = (double)e->A[i * e->lda + k] * (double)e->B[k * e->b_sk + j * e->b_sj];
            acc = acc + prod;
        }
        e->out[t] = acc;
    }
}

int oracle_gemm_entries(int64_t M, int64_t N, int64_t K, const float* A, int64_t lda,
                        const float* B, int64_t b_sk, int64_t b_sj, int64_t n,
                        const int64_t* rows, const int64_t* cols, double* out, int nthreads)
{
    if (M < 0 || N < 0 || K < 0 || n < 0) return -1;
    for (int64_t t = 0; t < n; ++t)
        if (rows[t] < 0 || rows[t] >= M || cols[t] < 0 || cols[t] >= N) return -1;
    entries_ctx_t e = {K, A, lda, B, b_sk, b_sj, rows, cols, out};
    return parallel_rows(entry_range, &e, n, nthreads);
}

/* ------------------------------------------------------------------ convolution */

typedef struct {
    int64_t Cin, Cout;
    int64_t in[4], ks[4], out[4];
    const float* x;
    const float* w;
    double* y;
} conv_ctx_t;

static int64_t out_extent(int64_t in, int64_t k) { return in - k + 1; }

static void conv_rows(void* p, int64_t lo, int64_t hi)
{
    const conv_ctx_t* c = (const conv_ctx_t*)p;
    const int64_t I0 = c->in[0], I1 = c->in[1], I2 = c->in[2], I3 = c->in[3];
    const int64_t R0 = c->ks[0], R1 = c->ks[1], R2 = c->ks[2], R3 = c->ks[3];
    const int64_t P0 = c->out[0], P1 = c->out[1], P2 = c->out[2], P3 = c->out[3];
    /* one "row" = one (output channel, p0) pair */
    for (int64_t row = lo; row < hi; ++row) {
        const int64_t o = row / P0, p0 = row % P0;
        for (int64_t p1 = 0; p1 < P1; ++p1)
            for (int64_t p2 = 0; p2 < P2; ++p2)
                for (int64_t p3 = 0; p3 < P3; ++p3) {
                    double acc = 0.0;
                    for (int64_t ci = 0; ci < c->Cin; ++ci)
                        for (int64_t r0 = 0; r0 < R0; ++r0)
                            for (int64_t r1 = 0; r1 < R1; ++r1)
                                for (int64_t r2 = 0; r2 < R2; ++r2)
                                    for (int64_t r3 = 0; r3 < R3; ++r3) {
                                        const int64_t widx =
                                            ((((o * c->Cin + ci) * R0 + r0) * R1 + r1) * R2 + r2) * R3 + r3;
                                        const int64_t xidx =
                                            (((ci * I0 + (p0 + r0)) * I1 + (p1 + r1)) * I2 + (p2 + r2)) * I3 + (p3 + r3);
                                        const double prod = (double)c->w[widx] * (double)c->x[xidx];
                                        acc = acc + prod;
                                    }
                    c->y[(((o * P0 + p0) * P1 + p1) * P2 + p2) * P3 + p3] = acc;
                }
    }
}

int oracle_conv4d_direct(int64_t Cin, const int64_t in[4], int64_t Cout, const int64_t ks[4],
                         const float* x, const float* w, double* y, int nthreads)
{
    conv_ctx_t c;
    if (Cin <= 0 || Cout <= 0) return -1;
    c.Cin = Cin;
    c.Cout = Cout;
    for (int d = 0; d < 4; ++d) {
        if (in[d] <= 0 || ks[d] <= 0 || ks[d] > in[d]) return -1;
        c.in[d] = in[d];
        c.ks[d] = ks[d];
        c.out[d] = out_extent(in[d], ks[d]);
    }
    c.x = x;
    c.w = w;
    c.y = y;
    return parallel_rows(conv_rows, &c, Cout * c.out[0], nthreads);
}

int oracle_im2col4d(int64_t Cin, const int64_t in[4], const int64_t ks[4], const float* x,
                    float* col)
{
    int64_t out[4];
    if (Cin <= 0) return -1;
    for (int d = 0; d < 4; ++d) {
        if (in[d] <= 0 || ks[d] <= 0 || ks[d] > in[d]) return -1;
        out[d] = out_extent(in[d], ks[d]);
    }
    const int64_t ncols = out[0] * out[1] * out[2] * out[3];
    int64_t r = 0; /* row of the column matrix = filter tap (c, r0, r1, r2, r3) */
    for (int64_t ci = 0; ci < Cin; ++ci)
        for (int64_t r0 = 0; r0 < ks[0]; ++r0)
            for (int64_t r1 = 0; r1 < ks[1]; ++r1)
                for (int64_t r2 = 0; r2 < ks[2]; ++r2)
                    for (int64_t r3 = 0; r3 < ks[3]; ++r3, ++r) {
                        int64_t n = 0; /* column = output position, row-major */
                        for (int64_t p0 = 0; p0 < out[0]; ++p0)
                            for (int64_t p1 = 0; p1 < out[1]; ++p1)
                                for (int64_t p2 = 0; p2 < out[2]; ++p2)
                                    for (int64_t p3 = 0; p3 < out[3]; ++p3, ++n) {
                                        const int64_t xidx =
                                            (((ci * in[0] + (p0 + r0)) * in[1] + (p1 + r1)) * in[2] + (p2 + r2)) * in[3] + (p3 + r3);
                                        col[r * ncols + n] = x[xidx];
                                    }
                    }
    return 0;
}
