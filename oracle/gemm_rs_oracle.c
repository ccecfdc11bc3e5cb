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
 * The tile schedule (oracle_schedule) is written out from the swizzle rule
 * ("flux实现：sm80 gemm+rs", section "gemmrs版本的swizzle如何编排": remote
 * chunks first, the local chunk last; "flux精读" §4.1: each rank is offset
 * by its rank so that no two ranks write the same chunk at the same step).
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
 * The tile schedule, built by enumeration:
 *  - Output tiles are (mt, nt) with mt < ceil(M/BM) and nt < ceil(N/BN).
 *  - A tile belongs to the chunk of its first row: key(mt) = (mt*BM) / R.
 *  - Rank r visits chunks in the order (r+1+s) mod W for s = 0 .. W-1, so its
 *    own chunk r comes last.
 *  - The column tiles form groups of G consecutive tiles (G <= 0 or G >= nN: a
 *    single group).  For each group, in order, the rank runs all W steps.
 *    Inside a group of gn tiles the rank starts at the group's tile
 *    ((W-r) mod W)*gn/W and wraps around within the group.  In a step, the
 *    chunk's row tiles (ascending) are split into row groups of RG tiles
 *    (RG <= 0: the whole chunk).  Each row group is one forward sweep over the
 *    group's column tiles.  For each column tile a sweep takes the row group's
 *    tiles in ascending order.
 *  - seq == 0: the W ranks run side by side: entry p*W + r of the global order
 *    is the p-th tile of rank r.  seq != 0: for each column group in turn, the
 *    ranks run one after another: the group's block of the global order holds
 *    rank 0's tiles of the group (its nM*gn entries in its own order), then
 *    rank 1's, and so on.
 * Writes (r, mt, nt) triples to out[3*g .. 3*g+2].  Returns the number of
 * entries W*nM*nN, -1 on bad arguments, or -2 if cap (in entries) is too small.
 */
int64_t oracle_schedule(int W, int64_t M, int64_t N, int BM, int BN, int G, int RG, int seq,
                        int32_t *out, int64_t cap)
{
    if (W < 1 || M < 1 || N < 1 || BM < 1 || BN < 1 || M % W != 0)
        return -1;
    const int64_t R = M / W;
    const int64_t nM = (M + BM - 1) / BM;
    const int64_t nN = (N + BN - 1) / BN;
    const int64_t T = nM * nN;
    if (cap < W * T)
        return -2;
    int32_t *list = (int32_t *)malloc((size_t)T * 2 * sizeof(int32_t));
    int64_t *rows = (int64_t *)malloc((size_t)nM * sizeof(int64_t));
    if (list == NULL || rows == NULL) {
        free(list);
        free(rows);
        return -1;
    }
    const int64_t group = (G <= 0 || G >= nN) ? nN : G;
    for (int r = 0; r < W; ++r) {
        int64_t p = 0;
        for (int64_t g0 = 0; g0 < nN; g0 += group) {
            const int64_t gn = (nN - g0 < group) ? nN - g0 : group;
            const int64_t rot = ((int64_t)((W - r) % W) * gn) / W;
            for (int s = 0; s < W; ++s) {
                const int64_t c = (r + 1 + s) % W;
                /* the chunk's row tiles, ascending */
                int64_t n_rows = 0;
                for (int64_t mt = 0; mt < nM; ++mt)
                    if ((mt * BM) / R == c)
                        rows[n_rows++] = mt;
                const int64_t rgs = (RG <= 0 || RG > n_rows) ? n_rows : RG;
                for (int64_t r0 = 0; r0 < n_rows; r0 += rgs) {
                    const int64_t r1 = (r0 + rgs < n_rows) ? r0 + rgs : n_rows;
                    for (int64_t j = 0; j < gn; ++j) {
                        const int64_t nt = g0 + (j + rot) % gn;
                        for (int64_t i = r0; i < r1; ++i) {
                            list[2 * p] = (int32_t)rows[i];
                            list[2 * p + 1] = (int32_t)nt;
                            ++p;
                        }
                    }
                }
            }
        }
        if (p != T) {
            free(list);
            free(rows);
            return -1;
        }
        for (int64_t q = 0; q < T; ++q) {
            int64_t g = q * W + r;
            if (seq) {
                const int64_t k = q / (nM * group);            /* column group of entry q */
                const int64_t gn = (nN - k * group < group) ? nN - k * group : group;
                g = k * W * nM * group + r * nM * gn + (q - k * nM * group);
            }
            out[3 * g] = r;
            out[3 * g + 1] = list[2 * q];
            out[3 * g + 2] = list[2 * q + 1];
        }
    }
    free(list);
    free(rows);
    return W * T;
}
