/*
 * CPU oracle for the fused GEMM + reduce-scatter (GEMM+RS) hot path.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg may load this code.  The product path (the
 * CUDA library) never calls it, and this file shares no code, header, table
 * or helper with the product path.
 *
 * What it computes (the plain definition, no blocking and no reordering):
 *
 *   Y[m, n] = fold_{r = 0 .. W-1}  p_r[m, n]
 *   p_r[m, n] = fp32( alpha * S_r[m, n] + beta * C[m, n] )
 *   S_r[m, n] = sum_{k = 0 .. K/W - 1}  A_r[m, k] * B_r[k, n]
 *
 * - The W logical tensor-parallel ranks each hold a K-shard:
 *   A_r = A[r] of shape [M][K/W] and B_r = B[r] of shape [K/W][N], both bf16.
 *   This is the row-parallel second FFN GEMM whose output feeds a
 *   reduce-scatter ("flux实现：sm80 gemm+rs", opening paragraph; "flux精读" §3).
 * - The epilogue computes alpha*acc, then beta*C + (alpha*acc), per rank
 *   ("flux实现：sm80 gemm+rs", section "custom_evt_d()": EVT_Compute0 and
 *   EVT_Compute1).  The C term is applied by every rank.  When beta == 0, C is
 *   not read at all.
 * - Chunk c of the output is rows [c*M/W, (c+1)*M/W).  Rank c keeps chunk c,
 *   and the other W-1 chunks go to the other ranks ("flux实现：sm80 gemm+rs",
 *   section "gemmrs版本的swizzle如何编排").  Y holds all W chunks in row order.
 * - The page gives no summation order.  The reading taken here: S_r is
 *   accumulated in double with k ascending.  alpha*S_r + beta*C is evaluated in
 *   double and rounded once to fp32.  The W partials are folded in fp32 in rank
 *   order: y = p_0, then y = y + p_r for r = 1 .. W-1.  A bf16 output is the
 *   round-to-nearest-even of y.
 *
 * The swizzle (oracle_chunk_order, oracle_tile_chunk) is what the pages fix
 * of the tile order and no more: each rank's chunk order, remote chunks first
 * and the local chunk last ("flux实现：sm80 gemm+rs", section
 * "gemmrs版本的swizzle如何编排"), each rank offset by its rank so that no two
 * ranks write the same chunk at the same step ("flux精读" §4.1), and the
 * chunk each row tile goes to.
 *
 * Build: gcc -O2 -ffp-contract=off -fopenmp -shared -fPIC.  FP contraction
 * stays off so that the result is the same on x86-64 and aarch64.
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* bf16 is the upper 16 bits of an IEEE binary32 value. */
static float bf16_to_float(uint16_t h)
{
    uint32_t u = ((uint32_t)h) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* Round an fp32 value to bf16, to nearest with ties to even.  NaN stays NaN
 * (quiet).  A finite value that rounds past the largest bf16 becomes inf. */
static uint16_t float_to_bf16_rne(float f)
{
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    if ((u & 0x7f800000u) == 0x7f800000u && (u & 0x007fffffu) != 0u)
        return (uint16_t)((u >> 16) | 0x0040u);
    uint32_t lower = u & 0xffffu;
    uint32_t upper = u >> 16;
    if (lower > 0x8000u || (lower == 0x8000u && (upper & 1u)))
        upper += 1u;
    return (uint16_t)upper;
}

void oracle_bf16_from_float(const float *x, uint16_t *out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = float_to_bf16_rne(x[i]);
}

void oracle_float_from_bf16(const uint16_t *x, float *out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = bf16_to_float(x[i]);
}

/*
 * Computes the rows listed in `rows` (all M rows in order when rows == NULL)
 * of Y.  A is [W][M][K/W] bf16, B is [W][K/W][N] bf16, C is [M][N] bf16
 * (ignored when beta == 0; may be NULL then).  The output is [n_rows][N]:
 * y_f32 when y_is_bf16 == 0, else y_bf16.
 *
 * split = 0: the fold over the ranks is one level, y = p_0, then y = y + p_r.
 * 0 < split < W: two levels ("flux实现：sm80 gemm+rs", section "2D Ring优化": the
 * ranks form two groups, each keeps its own partial sum, and the two are
 * added last): y0 = fold of p_0 .. p_{split-1} and y1 = fold of
 * p_split .. p_{W-1}, each in rank order, then y = y0 + y1.
 * Returns 0, or -1 on bad arguments.
 */
static int gemm_rs_impl(int W, int64_t M, int64_t N, int64_t K, float alpha, float beta,
                        const uint16_t *A, const uint16_t *B, const uint16_t *C, int y_is_bf16,
                        const int64_t *rows, int64_t n_rows, float *y_f32, uint16_t *y_bf16,
                        int n_threads, int split)
{
    if (split < 0 || split >= W)
        split = 0;
    if (W < 1 || M < 0 || N < 0 || K < 0 || K % W != 0 || M % W != 0)
        return -1;
    if (beta != 0.0f && C == NULL)
        return -1;
    if (rows == NULL)
        n_rows = M;
    const int64_t Kpr = K / W;
    int bad = 0;
#ifdef _OPENMP
    if (n_threads > 0)
        omp_set_num_threads(n_threads);
#else
    (void)n_threads;
#endif

#pragma omp parallel
    {
        double *s = (double *)malloc((size_t)(N > 0 ? N : 1) * sizeof(double));
        float *y = (float *)malloc((size_t)(N > 0 ? N : 1) * sizeof(float));
        float *y1 = (float *)malloc((size_t)(N > 0 ? N : 1) * sizeof(float));
        if (s == NULL || y == NULL || y1 == NULL) {
#pragma omp atomic write
            bad = 1;
        } else {
#pragma omp for schedule(dynamic, 1)
            for (int64_t ii = 0; ii < n_rows; ++ii) {
                const int64_t m = rows ? rows[ii] : ii;
                if (m < 0 || m >= M) {
#pragma omp atomic write
                    bad = 1;
                    continue;
                }
                for (int r = 0; r < W; ++r) {
                    /* S_r[m, :] with k ascending for every n. */
                    for (int64_t n = 0; n < N; ++n)
                        s[n] = 0.0;
                    const uint16_t *arow = A + ((int64_t)r * M + m) * Kpr;
                    for (int64_t k = 0; k < Kpr; ++k) {
                        const double a = (double)bf16_to_float(arow[k]);
                        const uint16_t *brow = B + ((int64_t)r * Kpr + k) * N;
                        for (int64_t n = 0; n < N; ++n)
                            s[n] += a * (double)bf16_to_float(brow[n]);
                    }
                    /* p_r = fp32(alpha*S_r + beta*C), then the rank-order fold. */
                    for (int64_t n = 0; n < N; ++n) {
                        double v = (double)alpha * s[n];
                        if (beta != 0.0f)
                            v += (double)beta * (double)bf16_to_float(C[m * N + n]);
                        const float p = (float)v;
                        if (split > 0 && r >= split) {      /* the second group's own sum */
                            if (r == split)
                                y1[n] = p;
                            else
                                y1[n] = y1[n] + p;
                        } else if (r == 0) {
                            y[n] = p;
                        } else {
                            y[n] = y[n] + p;
                        }
                    }
                }
                if (split > 0)
                    for (int64_t n = 0; n < N; ++n)
                        y[n] = y[n] + y1[n];
                for (int64_t n = 0; n < N; ++n) {
                    if (y_is_bf16)
                        y_bf16[ii * N + n] = float_to_bf16_rne(y[n]);
                    else
                        y_f32[ii * N + n] = y[n];
                }
            }
        }
        free(s);
        free(y);
        free(y1);
    }
    return bad ? -1 : 0;
}

int oracle_gemm_rs(int W, int64_t M, int64_t N, int64_t K, float alpha, float beta,
                   const uint16_t *A, const uint16_t *B, const uint16_t *C,
                   int y_is_bf16, const int64_t *rows, int64_t n_rows,
                   float *y_f32, uint16_t *y_bf16, int n_threads)
{
    return gemm_rs_impl(W, M, N, K, alpha, beta, A, B, C, y_is_bf16, rows, n_rows, y_f32, y_bf16,
                        n_threads, 0);
}

/* The two-level fold: ranks [0, split) and [split, W) (see gemm_rs_impl). */
int oracle_gemm_rs_two_level(int W, int64_t M, int64_t N, int64_t K, float alpha, float beta,
                             const uint16_t *A, const uint16_t *B, const uint16_t *C,
                             int y_is_bf16, const int64_t *rows, int64_t n_rows,
                             float *y_f32, uint16_t *y_bf16, int n_threads, int split)
{
    return gemm_rs_impl(W, M, N, K, alpha, beta, A, B, C, y_is_bf16, rows, n_rows, y_f32, y_bf16,
                        n_threads, split);
}

/*
 * Row m of the output belongs to chunk m / R (R = M/W rows per chunk) at row
 * m % R inside it.  Writes both for every m in [0, M).
 */
int oracle_row_chunk(int W, int64_t M, int32_t *chunk, int64_t *row_in_chunk)
{
    if (W < 1 || M % W != 0)
        return -1;
    const int64_t R = M / W;
    for (int64_t m = 0; m < M; ++m) {
        chunk[m] = (int32_t)(m / R);
        row_in_chunk[m] = m % R;
    }
    return 0;
}

/*
 * The rank-offset swizzle, as the pages define it: the order in which each
 * rank writes the W chunks of its output.  Rank r computes the remote chunks
 * first and its own chunk r last ("flux实现：sm80 gemm+rs", section
 * "gemmrs版本的swizzle如何编排"), and each rank starts one chunk further on
 * than the rank before it, so that at no step do two ranks write the same
 * chunk ("flux精读" §4.1, where rank 1 writes ranks 1..7 and then 0).  Joined,
 * the two passages give chunk (r + 1 + s) mod W at step s = 0 .. W-1.
 *
 * The pages fix nothing finer than this: not the order of the tiles inside a
 * chunk, nor how the W ranks share one device.  Those are the library's
 * choices, and the tests check them against this order and the properties
 * the pages state, not against an enumeration here.
 *
 * Writes out[r*W + s] for r, s = 0 .. W-1.  Returns 0, or -1 on bad arguments.
 */
int oracle_chunk_order(int W, int32_t *out)
{
    if (W < 1 || out == NULL)
        return -1;
    for (int r = 0; r < W; ++r) {
        /* remote chunks in rank order after r, wrapping, then r itself */
        int c = r;
        for (int s = 0; s < W; ++s) {
            c = (c + 1 == W) ? 0 : c + 1;
            out[r * W + s] = c;
        }
    }
    return 0;
}

/*
 * The chunk a row tile of BM rows is sent to.  The pages' unit of
 * communication is one output tile ("flux实现：sm80 gemm+rs": the scatter
 * store goes through a ReduceScatterOp over kM x kN tiles) and a chunk is
 * M/W contiguous rows; where a tile straddles two chunks the reading taken
 * is that it goes with the chunk of its first row.  Writes out[mt] for
 * mt = 0 .. ceil(M/BM)-1.  Returns the number of row tiles, -1 on bad
 * arguments, or -2 if cap is too small.
 */
int64_t oracle_tile_chunk(int W, int64_t M, int BM, int32_t *out, int64_t cap)
{
    if (W < 1 || M < 1 || BM < 1 || M % W != 0 || out == NULL)
        return -1;
    const int64_t nM = (M + BM - 1) / BM;
    if (cap < nM)
        return -2;
    const int64_t R = M / W;
    for (int64_t mt = 0; mt < nM; ++mt) {
        const int64_t first_row = mt * BM;
        out[mt] = (int32_t)(first_row / R);
    }
    return nM;
}
