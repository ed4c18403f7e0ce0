// fp32 GEMM on the FP32 pipe: a register-blocked FFMA kernel with shared-memory tiles.
//
// Design (from "Learning to develop for GPU with GEMM as the example"):
//  * section "Making the GPU implementation better": the K loop is split into tiles that
//    are first staged in shared memory by the whole block, then multiplied;
//  * section "How loading into local memory is organised": each thread copies its part of
//    the tile, a barrier separates copying from use;
//  * section "Why does tiling work?": neighbouring threads read neighbouring addresses
//    (128-byte transactions) -- here every global access is a float4;
//  * section "Improving the solution and balancing memory work": every thread owns a 2-D
//    block of accumulators (TM x TN; the page's WPTM x WPTN = 8 x 8, here 8 x 16) and runs
//    an outer product per k from registers: one A value times a row of B values, no
//    shuffles;
//  * section "How to do even better": rectangular tiles, A stored transposed (k-major)
//    in shared memory, rows padded against bank conflicts.
// What differs from the page: the tile is 128 x 256 x 16 (or 64 x 128 x 16) for 256
// threads, global loads for tile t+1 are in flight while tile t is multiplied (two
// shared buffers, one barrier per tile), M/N/K tails are predicated (zero fill), and an
// optional split of K over grid.z with a fixed-order reduction fills the GPU when there
// are few output tiles.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "internal.h"

namespace gemm_gb300 {

GEMM_DEBUG_UNIT(ffma)

namespace {

constexpr int kThreads = 256;
constexpr int kGroupM = 8;  // output-tile rows per raster group (L2 reuse of B columns)

// Sizes and leading dimensions arrive as 32-bit values (the host keeps them below 2^31),
// so that the compiler can keep the load-address arithmetic in 32 bits; they are widened
// into `p` only where addresses are formed.
template <int BM, int BN, int BK, int TM, int TN, bool VEC>
__global__ void __launch_bounds__(kThreads, 2)
ffma_tiled_kernel(const float* __restrict__ A, int lda, const float* __restrict__ B, int ldb, float* __restrict__ C,
                  int ldc, int M, int N, int K, int k_per_split, int m_tiles, int n_tiles, float* __restrict__ ws,
                  int vec_out)
{
    const struct {
        const float* A;
        int64_t lda;
        const float* B;
        int64_t ldb;
        float* C;
        int64_t ldc, M, N, K;
    } p = {A, lda, B, ldb, C, ldc, M, N, K};
    constexpr int TY = BM / TM;  // thread rows
    constexpr int TX = BN / TN;  // thread columns
    static_assert(TY * TX == kThreads, "tile/thread mismatch");
    static_assert(TM % 4 == 0 && TN % 4 == 0 && BK % 4 == 0, "float4 fragments");
    constexpr int AS_LD = BM + 4;  // padded row of the k-major A tile
    constexpr int A_CNT = BM * BK / 4, B_CNT = BN * BK / 4;  // float4s per tile
    constexpr int A_IT = (A_CNT + kThreads - 1) / kThreads;
    constexpr int B_IT = (B_CNT + kThreads - 1) / kThreads;

    __shared__ __align__(16) float As[2][BK][AS_LD];
    __shared__ __align__(16) float Bs[2][BK][BN];

    const int tid = threadIdx.x;

    // Grouped raster: kGroupM consecutive tile rows sweep the tile columns together.
    const int pid = blockIdx.x;
    const int width = kGroupM * n_tiles;
    const int group = pid / width;
    const int first_m = group * kGroupM;
    const int gsize = min(m_tiles - first_m, kGroupM);
    const int mt = first_m + (pid % width) % gsize;
    const int nt = (pid % width) / gsize;
    const int64_t m0 = (int64_t)mt * BM, n0 = (int64_t)nt * BN;

    const int64_t kbeg = (int64_t)blockIdx.z * k_per_split;
    const int64_t kend = min(p.K, kbeg + k_per_split);

    float* out;
    int64_t ldo;
    if (gridDim.z > 1) {
        out = ws + (int64_t)blockIdx.z * p.M * p.N;
        ldo = p.N;
    } else {
        out = p.C;
        ldo = p.ldc;
    }

    float4 a_st[A_IT], b_st[B_IT];

    auto load_tiles = [&](int64_t k0) {
#pragma unroll
        for (int i = 0; i < A_IT; ++i) {
            const int f = tid + i * kThreads;
            float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
            if (f < A_CNT) {
                const int row = f / (BK / 4);
                const int kq = (f % (BK / 4)) * 4;
                const int64_t gm = m0 + row, gk = k0 + kq;
                if (gm < p.M && in_range(gm, p.M)) {
                    const float* src = p.A + gm * p.lda + gk;
                    if (VEC && gk + 3 < kend) {
                        if (in_range(gk + 3, p.K)) v = __ldg(reinterpret_cast<const float4*>(src));
                    } else {
                        if (gk + 0 < kend) v.x = __ldg(src + 0);
                        if (gk + 1 < kend) v.y = __ldg(src + 1);
                        if (gk + 2 < kend) v.z = __ldg(src + 2);
                        if (gk + 3 < kend) v.w = __ldg(src + 3);
                    }
                }
            }
            a_st[i] = v;
        }
#pragma unroll
        for (int i = 0; i < B_IT; ++i) {
            const int f = tid + i * kThreads;
            float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
            if (f < B_CNT) {
                const int krow = f / (BN / 4);
                const int nq = (f % (BN / 4)) * 4;
                const int64_t gk = k0 + krow, gn = n0 + nq;
                if (gk < kend && in_range(gk, p.K)) {
                    const float* src = p.B + gk * p.ldb + gn;
                    if (VEC && gn + 3 < p.N) {
                        if (in_range(gn + 3, p.N)) v = __ldg(reinterpret_cast<const float4*>(src));
                    } else {
                        if (gn + 0 < p.N) v.x = __ldg(src + 0);
                        if (gn + 1 < p.N) v.y = __ldg(src + 1);
                        if (gn + 2 < p.N) v.z = __ldg(src + 2);
                        if (gn + 3 < p.N) v.w = __ldg(src + 3);
                    }
                }
            }
            b_st[i] = v;
        }
    };

    auto store_tiles = [&](int buf) {
#pragma unroll
        for (int i = 0; i < A_IT; ++i) {
            const int f = tid + i * kThreads;
            if (f < A_CNT) {
                const int row = f / (BK / 4);
                const int kq = (f % (BK / 4)) * 4;
                As[buf][kq + 0][row] = a_st[i].x;  // transposed: A tile stored k-major
                As[buf][kq + 1][row] = a_st[i].y;
                As[buf][kq + 2][row] = a_st[i].z;
                As[buf][kq + 3][row] = a_st[i].w;
            }
        }
#pragma unroll
        for (int i = 0; i < B_IT; ++i) {
            const int f = tid + i * kThreads;
            if (f < B_CNT) {
                const int krow = f / (BN / 4);
                const int nq = (f % (BN / 4)) * 4;
                *reinterpret_cast<float4*>(&Bs[buf][krow][nq]) = b_st[i];
            }
        }
    };

    float acc[TM][TN];
#pragma unroll
    for (int i = 0; i < TM; ++i)
#pragma unroll
        for (int j = 0; j < TN; ++j) acc[i][j] = 0.f;

    const int ty = tid / TX, tx = tid % TX;
    const int64_t ktiles = (kend > kbeg) ? (kend - kbeg + BK - 1) / BK : 0;

    if (ktiles > 0) {
        load_tiles(kbeg);
        store_tiles(0);
        __syncthreads();
    }
    for (int64_t kt = 0; kt < ktiles; ++kt) {
        const int buf = (int)(kt & 1);
        if (kt + 1 < ktiles) load_tiles(kbeg + (kt + 1) * BK);  // in flight during the FFMAs
#pragma unroll
        for (int k = 0; k < BK; ++k) {
            float af[TM], bf[TN];
#pragma unroll
            for (int a = 0; a < TM / 4; ++a) {
                const float4 t = *reinterpret_cast<const float4*>(&As[buf][k][ty * 4 + a * TY * 4]);
                af[a * 4 + 0] = t.x;
                af[a * 4 + 1] = t.y;
                af[a * 4 + 2] = t.z;
                af[a * 4 + 3] = t.w;
            }
#pragma unroll
            for (int b = 0; b < TN / 4; ++b) {
                const float4 t = *reinterpret_cast<const float4*>(&Bs[buf][k][tx * 4 + b * TX * 4]);
                bf[b * 4 + 0] = t.x;
                bf[b * 4 + 1] = t.y;
                bf[b * 4 + 2] = t.z;
                bf[b * 4 + 3] = t.w;
            }
#pragma unroll
            for (int i = 0; i < TM; ++i)
#pragma unroll
                for (int j = 0; j < TN; ++j) acc[i][j] = fmaf(af[i], bf[j], acc[i][j]);
        }
        if (kt + 1 < ktiles) store_tiles(buf ^ 1);
        __syncthreads();
    }

    // Epilogue: each thread writes its (TM/4) x (TN/4) blocks of 4 x 4 as float4 rows.
#pragma unroll
    for (int a = 0; a < TM / 4; ++a) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int64_t gm = m0 + ty * 4 + a * TY * 4 + i;
            if (gm >= p.M || !in_range(gm, p.M)) continue;
            float* row = out + gm * ldo;
#pragma unroll
            for (int b = 0; b < TN / 4; ++b) {
                const int64_t gn = n0 + tx * 4 + b * TX * 4;
                const float* v = &acc[a * 4 + i][b * 4];
                if (vec_out && gn + 3 < p.N) {
                    if (in_range(gn + 3, p.N)) *reinterpret_cast<float4*>(row + gn) = make_float4(v[0], v[1], v[2], v[3]);
                } else {
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        if (gn + j < p.N) row[gn + j] = v[j];
                }
            }
        }
    }
}

// 128 x 256 x 16 block tile, 256 threads as 2 x 4 warps of 64 x 64; inside a warp the
// lanes form an 8 x 4 grid and each owns 8 rows x 16 columns: rows ty*4 + {0,32} + {0..3},
// columns tx*4 + {0,16,32,48} + {0..3}.  Every fragment read is one shared-memory
// wavefront and every float4 store row is 64 contiguous bytes per 4 lanes.  The packed
// FMAs pair columns: one duplicated A value per row serves 8 of them, so the register
// moves that build the (a, a) pairs cost 1 per 8 packed FMAs (1 per 4 with 8 columns per
// thread: 58.6 against 63.0 TFLOP/s at 8192^3).
// Two instantiations: EDGE = false for tiles wholly inside M x N with K a multiple of 16
// and aligned operands (no predicates, running pointers), EDGE = true for everything
// else (predicated, zero-filled loads).  The host launches the interior tiles and the
// L-shaped edge region separately.  One block per SM (~254 registers, 48.6 KiB of
// dynamic shared memory).
constexpr int W_BM = 128, W_BN = 256, W_BK = 16;
constexpr int W_AS_LD = W_BM + 4;  // padded row of the k-major A tile
constexpr int W_SMEM_BYTES = (2 * W_BK * W_AS_LD + 2 * W_BK * W_BN) * 4;

// A last, partial wave of interior tiles leaves SMs idle for a whole tile time.  Its tiles
// can instead run cut along K into `rs` pieces (K slices of one tile, summed in fixed order
// afterwards): the remainder then takes ceil(rem * rs / slots) / rs tile times.  Returns the
// remainder tile count and the split (rs = 1, rem = 0 when it does not pay).
void remainder_plan(int64_t interior, int64_t slots, int64_t K, int* rem_out, int* rs_out)
{
    *rem_out = 0;
    *rs_out = 1;
    if (slots <= 0 || interior <= slots) return;
    const int64_t rem = interior % slots;
    if (rem == 0) return;
    double best_t = 1.0;
    int best_rs = 1;
    for (int rs = 2; rs <= 8; ++rs) {
        if (K / rs < 32 * W_BK) break;  // keep at least 32 k-tiles per piece
        const double t = (double)((rem * rs + slots - 1) / slots) / rs;
        if (t < best_t - 1e-9) {
            best_t = t;
            best_rs = rs;
        }
    }
    if (best_t > 0.85) return;
    *rem_out = (int)rem;
    *rs_out = best_rs;
}

struct TileMap {
    int mode;        // 0: grouped raster over rows x cols tiles; 1: L-shaped edge region
    int rows, cols;  // mode 0: tile grid; mode 1: full tile rows / cols (interior extent)
    int m_tiles, n_tiles;
    int first = 0;    // index of the block's tile = first + blockIdx.x
    int compact = 0;  // split-K partials go to a per-tile workspace [split][blocks][BM*BN]
};

__device__ __forceinline__ void map_tile(const TileMap& t, int pid, int& mt, int& nt)
{
    if (t.mode == 0) {
        const int width = kGroupM * t.cols;
        const int group = pid / width;
        const int first_m = group * kGroupM;
        const int gsize = min(t.rows - first_m, kGroupM);
        mt = first_m + (pid % width) % gsize;
        nt = (pid % width) / gsize;
    } else {
        const int bottom = (t.m_tiles - t.rows) * t.n_tiles;  // partial tile rows, all columns
        if (pid < bottom) {
            mt = t.rows + pid / t.n_tiles;
            nt = pid % t.n_tiles;
        } else {
            const int j = pid - bottom, w = t.n_tiles - t.cols;  // partial columns, full rows
            mt = j / w;
            nt = t.cols + j % w;
        }
    }
}

// Sizes and leading dimensions come as 32-bit scalars (the host keeps them below 2^31),
// widened where addresses are formed: with 64-bit leading dimensions the same body
// measured 20 % slower (50.2 against 63.0 TFLOP/s at 8192^3; the address arithmetic of
// the loads can no longer stay in 32 bits).
template <bool EDGE>
__global__ void __launch_bounds__(kThreads, 1)
ffma_warptile_kernel(const float* __restrict__ A, int lda_, const float* __restrict__ B, int ldb_,
                     float* __restrict__ C, int ldc_, int M, int N, int K, int k_per_split, TileMap tmap,
                     float* __restrict__ ws, int vec_in, int vec_out)
{
    // a programmatic dependent launched next (the last wave's K slices, or the reduction,
    // which waits for this grid) may start as SMs free up
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int64_t lda = lda_, ldb = ldb_, ldc = ldc_;
    extern __shared__ __align__(16) float w_smem[];
    float (*As)[W_BK][W_AS_LD] = reinterpret_cast<float (*)[W_BK][W_AS_LD]>(w_smem);
    float (*Bs)[W_BK][W_BN] = reinterpret_cast<float (*)[W_BK][W_BN]>(w_smem + 2 * W_BK * W_AS_LD);

    const int tid = threadIdx.x;
    int mt, nt;
    map_tile(tmap, tmap.first + blockIdx.x, mt, nt);
    const int64_t m0 = (int64_t)mt * W_BM, n0 = (int64_t)nt * W_BN;
    const int kbeg = (int)blockIdx.z * k_per_split;  // < K
    const int kend = (int)min((int64_t)K, (int64_t)kbeg + k_per_split);

    // global -> register staging: A float4s at (row a_row, k a_kq) and (a_row, a_kq + 8);
    // B float4s at (k b_k + 4 h, cols b_nq..+3), h = 0..3
    const int a_row = tid % W_BM, a_kq = (tid / W_BM) * 4;
    const int b_k = tid / 64, b_nq = (tid % 64) * 4;
    const bool a_ok = !EDGE || (m0 + a_row) < M;
    const float* a_cur = A + (a_ok ? (m0 + a_row) : 0) * lda + kbeg + a_kq;
    const float* b_cur = B + (int64_t)(kbeg + b_k) * ldb + n0 + b_nq;
    const int64_t b_step = 4 * ldb;

    float4 ra[2], rb[4];
    int k_next = kbeg;  // k of the tile the next load() fetches
    auto load = [&]() {
        if constexpr (!EDGE) {
            // (the index checks compile away outside debug builds)
            if (in_range(m0 + a_row, M) && in_range(k_next + a_kq + 11, K)) {
                ra[0] = __ldg(reinterpret_cast<const float4*>(a_cur));
                ra[1] = __ldg(reinterpret_cast<const float4*>(a_cur + 8));
            }
            if (in_range(k_next + b_k + 12, K) && in_range(n0 + b_nq + 3, N))
#pragma unroll
                for (int h = 0; h < 4; ++h) rb[h] = __ldg(reinterpret_cast<const float4*>(b_cur + h * b_step));
            k_next += W_BK;
        } else {
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
                const int gk = k_next + a_kq + h * 8;
                if (a_ok) {
                    const float* src = a_cur + h * 8;
                    if (vec_in && gk + 3 < kend) {
                        v = __ldg(reinterpret_cast<const float4*>(src));
                    } else {
                        if (gk + 0 < kend) v.x = __ldg(src + 0);
                        if (gk + 1 < kend) v.y = __ldg(src + 1);
                        if (gk + 2 < kend) v.z = __ldg(src + 2);
                        if (gk + 3 < kend) v.w = __ldg(src + 3);
                    }
                }
                ra[h] = v;
            }
#pragma unroll
            for (int h = 0; h < 4; ++h) {
                float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
                const int bk = k_next + b_k + h * 4;
                const int64_t gn = n0 + b_nq;
                if (bk < kend) {
                    const float* src = b_cur + h * b_step;
                    if (vec_in && gn + 3 < N) {
                        v = __ldg(reinterpret_cast<const float4*>(src));
                    } else {
                        if (gn + 0 < N) v.x = __ldg(src + 0);
                        if (gn + 1 < N) v.y = __ldg(src + 1);
                        if (gn + 2 < N) v.z = __ldg(src + 2);
                        if (gn + 3 < N) v.w = __ldg(src + 3);
                    }
                }
                rb[h] = v;
            }
            k_next += W_BK;
        }
        a_cur += W_BK;
        b_cur += 4 * b_step;
    };
    auto store = [&](int buf) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            // a warp holds 32 consecutive rows of one k: conflict-free transposed stores
            As[buf][a_kq + h * 8 + 0][a_row] = ra[h].x;
            As[buf][a_kq + h * 8 + 1][a_row] = ra[h].y;
            As[buf][a_kq + h * 8 + 2][a_row] = ra[h].z;
            As[buf][a_kq + h * 8 + 3][a_row] = ra[h].w;
        }
#pragma unroll
        for (int h = 0; h < 4; ++h) *reinterpret_cast<float4*>(&Bs[buf][b_k + h * 4][b_nq]) = rb[h];
    };

    const int warp = tid / 32, lane = tid % 32;
    const int wm = warp / 4, wn = warp % 4;  // 2 x 4 warps
    const int ty = lane / 4, tx = lane % 4;  // 8 x 4 lanes
    const int a_frag = wm * 64 + ty * 4;     // rows a_frag + {0..3}, a_frag + 32 + {0..3}
    const int b_frag = wn * 64 + tx * 4;     // cols b_frag + 16 h + {0..3}, h = 0..3

    // acc[i][jj] holds columns (2jj, 2jj+1) of this thread's 16 in accumulator row i: the
    // outer product runs as packed fp32 FMAs (fma.rn.f32x2, two independent
    // round-to-nearest FMAs per issue)
    float2 acc[8][8];
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[i][j] = make_float2(0.f, 0.f);

    const int ktiles = (kend > kbeg) ? (kend - kbeg + W_BK - 1) / W_BK : 0;
    if (ktiles > 0) {
        load();
        store(0);
        __syncthreads();
    }
    for (int kt = 0; kt < ktiles; ++kt) {
        const int buf = kt & 1;
        if (kt + 1 < ktiles) load();  // in flight during the FFMAs below
#pragma unroll
        for (int k = 0; k < W_BK; ++k) {
            const float4 a0 = *reinterpret_cast<const float4*>(&As[buf][k][a_frag]);
            const float4 a1 = *reinterpret_cast<const float4*>(&As[buf][k][a_frag + 32]);
            float2 bp[8];
#pragma unroll
            for (int h = 0; h < 4; ++h) {
                const float4 b = *reinterpret_cast<const float4*>(&Bs[buf][k][b_frag + 16 * h]);
                bp[2 * h] = make_float2(b.x, b.y);
                bp[2 * h + 1] = make_float2(b.z, b.w);
            }
            const float af[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const float2 ai = make_float2(af[i], af[i]);
#pragma unroll
                for (int j = 0; j < 8; ++j) acc[i][j] = __ffma2_rn(ai, bp[j], acc[i][j]);
            }
        }
        if (kt + 1 < ktiles) store(buf ^ 1);
        __syncthreads();
    }

    // output rows: C, or a split-K partial (a full M x N slice, or one BM x BN tile);
    // element (gm, gn) lives at out[(gm - row0) * ldo + (gn - col0)].  (Worked out only
    // now, so that none of it stays live in registers through the main loop.)
    float* out;
    int64_t ldo, row0 = 0, col0 = 0;
    if (tmap.compact) {
        out = ws + ((int64_t)blockIdx.z * gridDim.x + blockIdx.x) * (W_BM * W_BN);
        ldo = W_BN;
        row0 = m0;
        col0 = n0;
    } else if (gridDim.z > 1) {
        out = ws + (int64_t)blockIdx.z * M * N;
        ldo = N;
    } else {
        out = C;
        ldo = ldc;
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int64_t gm = m0 + a_frag + (i / 4) * 32 + (i % 4);
        if (EDGE && gm >= M) continue;
        if (!in_range(gm, M)) continue;
        float* row = out + (gm - row0) * ldo - col0;
#pragma unroll
        for (int h = 0; h < 4; ++h) {
            const int64_t gn = n0 + b_frag + h * 16;
            const float v[4] = {acc[i][2 * h].x, acc[i][2 * h].y, acc[i][2 * h + 1].x, acc[i][2 * h + 1].y};
            if ((vec_out || tmap.compact) && (!EDGE || gn + 3 < N)) {
                if (in_range(gn + 3, N)) *reinterpret_cast<float4*>(row + gn) = make_float4(v[0], v[1], v[2], v[3]);
            } else {
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    if (gn + j < N) row[gn + j] = v[j];
            }
        }
    }
}

// Fixed-order sum of per-tile split-K partials (compact layout [split][tiles][BM*BN]):
// C[tile element] = part 0 + part 1 + ... for the tiles first .. first + ntiles - 1.
__global__ void __launch_bounds__(256)
splitk_reduce_tiles_kernel(const float* __restrict__ ws, int split, TileMap tmap, int ntiles, float* __restrict__ C,
                           int64_t ldc, int M, int N)
{
    asm volatile("griddepcontrol.wait;" ::: "memory");  // the partials' writer has finished
    constexpr int TILE = W_BM * W_BN;
    const int64_t total = (int64_t)ntiles * TILE / 4;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t q = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; q < total; q += stride) {
        const int64_t e = q * 4;
        const int t = (int)(e / TILE);
        const int w = (int)(e % TILE);
        float4 s = *reinterpret_cast<const float4*>(ws + e);
        for (int z = 1; z < split; ++z) {
            const float4 v = *reinterpret_cast<const float4*>(ws + (int64_t)z * ntiles * TILE + e);
            s.x += v.x, s.y += v.y, s.z += v.z, s.w += v.w;
        }
        int mt, nt;
        map_tile(tmap, tmap.first + t, mt, nt);
        const int64_t r = (int64_t)mt * W_BM + w / W_BN, c = (int64_t)nt * W_BN + w % W_BN;
        if (!in_range(r, M) || !in_range(c + 3, N)) continue;
        float* dst = C + r * ldc + c;
        dst[0] = s.x, dst[1] = s.y, dst[2] = s.z, dst[3] = s.w;
    }
}

// Fixed-order sum of split-K partials: C[m][n] = ws[0][m][n] + ws[1][m][n] + ...
__global__ void __launch_bounds__(256)
splitk_reduce_kernel(const float* __restrict__ ws, int split, int64_t M, int64_t N,
                     float* __restrict__ C, int64_t ldc)
{
    asm volatile("griddepcontrol.wait;" ::: "memory");  // the partials' writer has finished
    const int64_t total = M * N;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; idx < total; idx += stride) {
        const int64_t m = idx / N, n = idx - m * N;
        if (!in_range(m, M) || !in_range(n, N)) continue;
        float s = ws[idx];
        for (int z = 1; z < split; ++z) s += ws[(int64_t)z * total + idx];
        C[m * ldc + n] = s;
    }
}

// The same sum for rows of a multiple of four floats: four adjacent outputs per thread and
// the partials of four slices in flight at once; the additions keep the slice order.
__global__ void __launch_bounds__(256)
splitk_reduce4_kernel(const float* __restrict__ ws, int split, int64_t M, int64_t N,
                      float* __restrict__ C, int64_t ldc)
{
    asm volatile("griddepcontrol.wait;" ::: "memory");  // the partials' writer has finished
    const int64_t total = M * N;
    const int64_t n4 = N / 4;
    const int64_t quads = M * n4;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t q = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; q < quads; q += stride) {
        const int64_t m = q / n4, n = (q - m * n4) * 4;
        if (!in_range(m, M) || !in_range(n + 3, N)) continue;
        const float* src = ws + q * 4;
        float4 s = __ldcs(reinterpret_cast<const float4*>(src));
        int z = 1;
        for (; z + 4 <= split; z += 4) {
            float4 v[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) v[u] = __ldcs(reinterpret_cast<const float4*>(src + (int64_t)(z + u) * total));
#pragma unroll
            for (int u = 0; u < 4; ++u) s.x += v[u].x, s.y += v[u].y, s.z += v[u].z, s.w += v[u].w;
        }
        for (; z < split; ++z) {
            const float4 v = __ldcs(reinterpret_cast<const float4*>(src + (int64_t)z * total));
            s.x += v.x, s.y += v.y, s.z += v.z, s.w += v.w;
        }
        *reinterpret_cast<float4*>(C + m * ldc + n) = s;
    }
}

// C = alpha * P + beta * C (C unread when beta == 0), stored as fp32, bf16 or fp16.
// P == nullptr stands for a zero product.
template <int CT>
__global__ void __launch_bounds__(256)
epilogue_kernel(const float* __restrict__ P, int64_t ldp, void* C, int64_t ldc, int64_t M, int64_t N, float alpha,
                float beta)
{
    const int64_t total = M * N;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; idx < total; idx += stride) {
        const int64_t m = idx / N, n = idx - m * N;
        if (!in_range(m, M) || !in_range(n, N)) continue;
        float v = P ? alpha * P[m * ldp + n] : 0.f;  // no P: an empty product (K == 0)
        const int64_t c = m * ldc + n;
        if (CT == GEMM_F32) {
            float* out = static_cast<float*>(C);
            if (beta != 0.f) v = fmaf(beta, out[c], v);
            out[c] = v;
        } else if (CT == GEMM_BF16) {
            __nv_bfloat16* out = static_cast<__nv_bfloat16*>(C);
            if (beta != 0.f) v = fmaf(beta, __bfloat162float(out[c]), v);
            out[c] = __float2bfloat16_rn(v);
        } else {
            __half* out = static_cast<__half*>(C);
            if (beta != 0.f) v = fmaf(beta, __half2float(out[c]), v);
            out[c] = __float2half_rn(v);
        }
    }
}

template <int BM, int BN, int BK, int TM, int TN>
cudaError_t launch_variant(const F32Args& a, int split, float* ws, cudaStream_t stream, int* launches)
{
    const int64_t m_tiles = (a.M + BM - 1) / BM, n_tiles = (a.N + BN - 1) / BN;
    // the kernel takes sizes and leading dimensions as 32-bit values
    if (m_tiles * n_tiles > 0x7fffffffLL || a.M > 0x7fffffffLL || a.N > 0x7fffffffLL || a.K > 0x7fffffffLL - BK ||
        a.lda > 0x7fffffffLL || a.ldb > 0x7fffffffLL || a.ldc > 0x7fffffffLL)
        return cudaErrorInvalidConfiguration;
    int64_t kps = (a.K + split - 1) / split;
    kps = (kps + BK - 1) / BK * BK;  // every split but the last starts on a tile boundary
    const int nsplit = (int)((a.K + kps - 1) / kps);
    const bool vec_in = ((reinterpret_cast<uintptr_t>(a.A) | reinterpret_cast<uintptr_t>(a.B)) & 15) == 0 &&
                        a.lda % 4 == 0 && a.ldb % 4 == 0;
    int vec_out;
    if (nsplit > 1)
        vec_out = (a.N % 4 == 0);
    else
        vec_out = (reinterpret_cast<uintptr_t>(a.C) & 15) == 0 && a.ldc % 4 == 0;
    dim3 grid((unsigned)(m_tiles * n_tiles), 1, (unsigned)nsplit);
    if (vec_in)
        ffma_tiled_kernel<BM, BN, BK, TM, TN, true><<<grid, kThreads, 0, stream>>>(
            a.A, (int)a.lda, a.B, (int)a.ldb, a.C, (int)a.ldc, (int)a.M, (int)a.N, (int)a.K, (int)kps, (int)m_tiles,
            (int)n_tiles, ws, vec_out);
    else
        ffma_tiled_kernel<BM, BN, BK, TM, TN, false><<<grid, kThreads, 0, stream>>>(
            a.A, (int)a.lda, a.B, (int)a.ldb, a.C, (int)a.ldc, (int)a.M, (int)a.N, (int)a.K, (int)kps, (int)m_tiles,
            (int)n_tiles, ws, vec_out);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    *launches += 1;
    if (nsplit == 1) return e;
    *launches += 1;
    return launch_splitk_reduce(ws, nsplit, a.M, a.N, a.C, a.ldc, 0, stream);
}

cudaError_t launch_warptile(const F32Args& a, int split, float* ws, int remainder_split, int num_sms,
                            cudaStream_t stream, int* launches)
{
    const int64_t m_tiles64 = (a.M + W_BM - 1) / W_BM, n_tiles64 = (a.N + W_BN - 1) / W_BN;
    // the kernel takes sizes and leading dimensions as 32-bit values
    if (m_tiles64 * n_tiles64 > 0x7fffffffLL || a.M > 0x7fffffffLL || a.N > 0x7fffffffLL ||
        a.K > 0x7fffffffLL - W_BK || a.lda > 0x7fffffffLL || a.ldb > 0x7fffffffLL || a.ldc > 0x7fffffffLL)
        return cudaErrorInvalidConfiguration;
    int64_t kps = (a.K + split - 1) / split;
    kps = (kps + W_BK - 1) / W_BK * W_BK;
    const int nsplit = (int)((a.K + kps - 1) / kps);
    const int vec_in = ((reinterpret_cast<uintptr_t>(a.A) | reinterpret_cast<uintptr_t>(a.B)) & 15) == 0 &&
                       a.lda % 4 == 0 && a.ldb % 4 == 0;
    int vec_out;
    if (nsplit > 1)
        vec_out = (a.N % 4 == 0);
    else
        vec_out = (reinterpret_cast<uintptr_t>(a.C) & 15) == 0 && a.ldc % 4 == 0;
    for (auto kern : {ffma_warptile_kernel<false>, ffma_warptile_kernel<true>})
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, W_SMEM_BYTES) != cudaSuccess)
            return cudaGetLastError();
    const int m_tiles = (int)m_tiles64, n_tiles = (int)n_tiles64;
    const int m_full = (int)(a.M / W_BM), n_full = (int)(a.N / W_BN);
    const bool fast_ok = vec_in && (a.K % W_BK == 0);
    const int interior = fast_ok ? m_full * n_full : 0;
    const int64_t edge = (int64_t)m_tiles * n_tiles - interior;
    if (interior > 0) {
        // whole waves as usual; the tiles of a last, partial wave (if any) are cut along
        // K so that they fill the GPU's block slots (one per SM; remainder_plan)
        int rem = 0, rs = 1;
        if (nsplit == 1 && remainder_split) remainder_plan(interior, num_sms, a.K, &rem, &rs);
        const int main_tiles = interior - rem;
        TileMap t{0, m_full, n_full, m_tiles, n_tiles};
        if (main_tiles > 0) {
            ffma_warptile_kernel<false><<<dim3(main_tiles, 1, nsplit), kThreads, W_SMEM_BYTES, stream>>>(
                a.A, (int)a.lda, a.B, (int)a.ldb, a.C, (int)a.ldc, (int)a.M, (int)a.N, (int)a.K, (int)kps, t, ws, vec_in, vec_out);
            cudaError_t e = cudaGetLastError();
            if (e != cudaSuccess) return e;
            *launches += 1;
        }
        if (rem > 0) {
            int64_t rkps = (a.K + rs - 1) / rs;
            rkps = (rkps + W_BK - 1) / W_BK * W_BK;
            const int rsplit = (int)((a.K + rkps - 1) / rkps);
            TileMap tr = t;
            tr.first = main_tiles;
            tr.compact = 1;
            // the K slices read nothing the full waves write (their partials go to the
            // workspace), so they start on SMs as the last full wave drains
            cudaError_t e = launch_dependent(ffma_warptile_kernel<false>, dim3(rem, 1, rsplit), dim3(kThreads),
                                             W_SMEM_BYTES, stream, a.A, (int)a.lda, a.B, (int)a.ldb, a.C, (int)a.ldc,
                                             (int)a.M, (int)a.N, (int)a.K, (int)rkps, tr, ws, vec_in, vec_out);
            if (e != cudaSuccess) return e;
            int64_t blocks = (int64_t)rem * W_BM * W_BN / 4 / 256;
            if (blocks < 1) blocks = 1;
            e = launch_dependent(splitk_reduce_tiles_kernel, dim3((unsigned)blocks), dim3(256), 0, stream, ws, rsplit,
                                 tr, rem, a.C, a.ldc, (int)a.M, (int)a.N);
            if (e != cudaSuccess) return e;
            *launches += 2;
        }
    }
    if (edge > 0) {
        TileMap t = fast_ok ? TileMap{1, m_full, n_full, m_tiles, n_tiles} : TileMap{0, m_tiles, n_tiles, m_tiles, n_tiles};
        ffma_warptile_kernel<true><<<dim3((unsigned)edge, 1, nsplit), kThreads, W_SMEM_BYTES, stream>>>(
            a.A, (int)a.lda, a.B, (int)a.ldb, a.C, (int)a.ldc, (int)a.M, (int)a.N, (int)a.K, (int)kps, t, ws, vec_in, vec_out);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
        *launches += 1;
    }
    if (nsplit == 1) return cudaSuccess;
    *launches += 1;
    return launch_splitk_reduce(ws, nsplit, a.M, a.N, a.C, a.ldc, 0, stream);
}

}  // namespace

int64_t ffma_remainder_workspace(const F32Args& a, int variant, int split, int num_sms)
{
    // floats of workspace the remainder-wave split needs (0 when it does not apply)
    if (variant == 2 || split > 1) return 0;
    const bool vec_in = ((reinterpret_cast<uintptr_t>(a.A) | reinterpret_cast<uintptr_t>(a.B)) & 15) == 0 &&
                        a.lda % 4 == 0 && a.ldb % 4 == 0;
    if (!vec_in || a.K % W_BK) return 0;
    int rem = 0, rs = 1;
    remainder_plan((a.M / W_BM) * (a.N / W_BN), num_sms, a.K, &rem, &rs);
    return (int64_t)rem * rs * W_BM * W_BN;
}

int ffma_auto_split(const F32Args& a, int variant, int num_sms)
{
    const int BM = (variant == 2) ? 64 : W_BM, BN = (variant == 2) ? 128 : W_BN, BK = 16;
    const int64_t tiles = ((a.M + BM - 1) / BM) * ((a.N + BN - 1) / BN);
    const int64_t capacity = (int64_t)num_sms * 2;  // two resident blocks per SM
    if (tiles >= capacity) return 1;
    int64_t s = capacity / tiles;
    const int64_t max_s = a.K / (BK * 16);  // keep at least 16 K tiles per split
    if (s > max_s) s = max_s;
    return (int)(s < 1 ? 1 : s);
}

cudaError_t launch_ffma_tiled(const F32Args& a, int variant, int split, float* ws, int num_sms,
                              cudaStream_t stream, int* launches)
{
    if (split < 1) split = 1;
    if (variant == 2) return launch_variant<64, 128, 16, 4, 8>(a, split, ws, stream, launches);
    return launch_warptile(a, split, ws, 1, num_sms, stream, launches);
}

cudaError_t launch_epilogue(const float* P, int64_t ldp, void* C, int64_t ldc, int64_t M, int64_t N,
                            const Epilogue& epi, int num_sms, cudaStream_t stream)
{
    const int64_t total = M * N;
    int64_t blocks = (total + 255) / 256;
    const int64_t cap = (int64_t)(num_sms > 0 ? num_sms : 152) * 8;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    if (epi.c_dtype == GEMM_BF16)
        epilogue_kernel<GEMM_BF16><<<(unsigned)blocks, 256, 0, stream>>>(P, ldp, C, ldc, M, N, epi.alpha, epi.beta);
    else if (epi.c_dtype == GEMM_F16)
        epilogue_kernel<GEMM_F16><<<(unsigned)blocks, 256, 0, stream>>>(P, ldp, C, ldc, M, N, epi.alpha, epi.beta);
    else
        epilogue_kernel<GEMM_F32><<<(unsigned)blocks, 256, 0, stream>>>(P, ldp, C, ldc, M, N, epi.alpha, epi.beta);
    return cudaGetLastError();
}

cudaError_t launch_splitk_reduce(const float* ws, int split, int64_t M, int64_t N, float* C,
                                 int64_t ldc, int num_sms, cudaStream_t stream)
{
    const bool vec4 = N % 4 == 0 && ldc % 4 == 0 &&
                      ((reinterpret_cast<uintptr_t>(ws) | reinterpret_cast<uintptr_t>(C)) & 15) == 0;
    const int64_t total = vec4 ? M * (N / 4) : M * N;
    int64_t blocks = (total + 255) / 256;
    const int64_t cap = (int64_t)(num_sms > 0 ? num_sms : 152) * 8;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    if (vec4)
        return launch_dependent(splitk_reduce4_kernel, dim3((unsigned)blocks), dim3(256), 0, stream, ws, split, M, N,
                                C, ldc);
    return launch_dependent(splitk_reduce_kernel, dim3((unsigned)blocks), dim3(256), 0, stream, ws, split, M, N, C,
                            ldc);
}

}  // namespace gemm_gb300
