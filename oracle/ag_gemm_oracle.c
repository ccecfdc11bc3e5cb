/*
 * CPU oracle for the fused all-gather + GEMM (AG+GEMM) path: the first GEMM
 * of a tensor-parallel FFN, whose input rows are all-gathered from the ranks.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite and the benchmark's CPU
 * baseline may load this code.  The product path never calls it, and this
 * file shares no code with the product path.
 *
 * What it computes (the plain definition):
 *
 *   H_r[m, n] = out( fp32( alpha * sum_{k = 0 .. K-1} X[m, k] * B1_r[k, n] ) )
 *
 * - X is [M][K] bf16, the concatenation of the W row chunks X_c = rows
 *   [c*M/W, (c+1)*M/W) that the W ranks hold before the all-gather.  Every
 *   rank multiplies the whole gathered X ("flux精读" §3 Design: the AG of the
 *   input rows ahead of the GEMM; "通信 overlap 实现", section "Flux 的 tile 级融合
 *   解决了什么？": AG+GEMM, prologue fusion).
 * - B1_r = B1[r] is rank r's [K][N] column shard of the weight (bf16).
 * - The sum is accumulated in double with k ascending, alpha * sum is rounded
 *   once to fp32, and a bf16 output is the round-to-nearest-even of that.
 *   The pages give no summation order; this is the reading taken.
 * - H is [W][M][N]: rank r's full-M output of its columns.
 *
 * The chunk order (oracle_ag_chunk_order) is written out from the same pages:
 * a thread block waits for its tile's signal in the order the tiles are sent
 * ("flux精读" §3, the AllGather GEMM paragraph), and a rank starts with the
 * rows it already holds ("flux精读" §4.1: each rank starts at its own chunk).
 *
 * Build: with gemm_rs_oracle.c, gcc -O2 -ffp-contract=off -fopenmp -shared.
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

static float ag_bf16_to_float(uint16_t h)
{
    uint32_t u = ((uint32_t)h) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* Round to bf16, to nearest with ties to even; NaN stays a quiet NaN. */
static uint16_t ag_float_to_bf16(float f)
{
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    if ((u & 0x7f800000u) == 0x7f800000u && (u & 0x007fffffu) != 0)
        return (uint16_t)((u >> 16) | 0x0040u);
    const uint32_t lsb = (u >> 16) & 1u;
    u += 0x7fffu + lsb;
    return (uint16_t)(u >> 16);
}

/*
 * X: bf16 bits [M][K].  B1: bf16 bits [W][K][N].  rows: NULL for all M rows,
 * else n_rows row indices; the output then holds those rows only, in that
 * order: [W][n_rows][N].  Exactly one of out_f32 (y_bf16 == 0) and out_bf16
 * is written.  Returns 0, or -1 on bad arguments.
 */
int oracle_ag_gemm(int W, int64_t M, int64_t N, int64_t K, float alpha, const uint16_t *X,
                   const uint16_t *B1, int y_bf16, const int64_t *rows, int64_t n_rows,
                   float *out_f32, uint16_t *out_bf16)
{
    if (W < 1 || M < 0 || N < 0 || K < 0 || X == NULL || B1 == NULL)
        return -1;
    if ((y_bf16 && out_bf16 == NULL) || (!y_bf16 && out_f32 == NULL))
        return -1;
    const int64_t nr = rows ? n_rows : M;
    for (int64_t i = 0; i < nr; ++i)
        if (rows && (rows[i] < 0 || rows[i] >= M))
            return -1;
#pragma omp parallel for collapse(2) schedule(dynamic, 1)
    for (int r = 0; r < W; ++r) {
        for (int64_t i = 0; i < nr; ++i) {
            const int64_t m = rows ? rows[i] : i;
            const uint16_t *xr = X + m * K;
            const uint16_t *b = B1 + (int64_t)r * K * N;
            double *acc = (double *)calloc((size_t)(N > 0 ? N : 1), sizeof(double));
            for (int64_t k = 0; k < K; ++k) {
                const double xv = (double)ag_bf16_to_float(xr[k]);
                const uint16_t *brow = b + k * N;
                for (int64_t n = 0; n < N; ++n)
                    acc[n] += xv * (double)ag_bf16_to_float(brow[n]);
            }
            const int64_t o = ((int64_t)r * nr + i) * N;
            for (int64_t n = 0; n < N; ++n) {
                const float v = (float)((double)alpha * acc[n]);
                if (y_bf16)
                    out_bf16[o + n] = ag_float_to_bf16(v);
                else
                    out_f32[o + n] = v;
            }
            free(acc);
        }
    }
    return 0;
}

/*
 * The order in which rank r consumes the W chunks of the gathered rows: its
 * own chunk first, then the others in rank order after it, wrapping:
 * (r + s) mod W at step s = 0 .. W-1 ("flux精读" §4.1: each rank starts at
 * its own chunk, as printed for ranks 0 and 1; §3: the GEMM blocks take their
 * tiles in the order the chunks are sent).  The order of the tiles inside a
 * chunk and how the ranks share one device are the library's choices; the
 * tests check them against this order.
 *
 * Writes out[r*W + s].  Returns 0, or -1 on bad arguments.
 */
int oracle_ag_chunk_order(int W, int32_t *out)
{
    if (W < 1 || out == NULL)
        return -1;
    for (int r = 0; r < W; ++r)
        for (int s = 0; s < W; ++s)
            out[r * W + s] = (r + s) % W;
    return 0;
}
