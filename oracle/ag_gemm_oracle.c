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
 * The tile order (oracle_ag_schedule) is written out from the same pages: a
 * thread block waits for its tile's signal in the order the tiles are sent
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
 * The AG+GEMM tile order, built by enumeration:
 *  - Output tiles of rank r are (mt, nt) with mt < M/BM and nt < ceil(N/BN);
 *    a row tile lies in one chunk (BM divides M/W): chunk(mt) = mt*BM / (M/W).
 *  - Rank r takes its chunks in the order (r+s) mod W, s = 0 .. W-1: the rows
 *    it holds first, then the chunks in the order they are sent to it.
 *  - Inside a chunk, for each column tile, the chunk's row tiles ascending.
 *  - The ranks run one after another: entry r*T + p is rank r's p-th tile
 *    (T = tiles per rank).
 * Writes (r, mt, nt) triples.  Returns W*T, -1 on bad arguments, or -2 if
 * cap (in entries) is too small.
 */
int64_t oracle_ag_schedule(int W, int64_t M, int64_t N, int BM, int BN, int32_t *out, int64_t cap)
{
    if (W < 1 || M < 1 || N < 1 || BM < 1 || BN < 1 || M % W != 0 || (M / W) % BM != 0)
        return -1;
    const int64_t R = M / W;
    const int64_t cnt = R / BM; /* row tiles per chunk */
    const int64_t nN = (N + BN - 1) / BN;
    const int64_t T = (M / BM) * nN;
    if (cap < W * T)
        return -2;
    int64_t g = 0;
    for (int r = 0; r < W; ++r)
        for (int s = 0; s < W; ++s) {
            const int64_t c = (r + s) % W;
            for (int64_t nt = 0; nt < nN; ++nt)
                for (int64_t i = 0; i < cnt; ++i) {
                    out[3 * g] = r;
                    out[3 * g + 1] = (int32_t)(c * cnt + i);
                    out[3 * g + 2] = (int32_t)nt;
                    ++g;
                }
        }
    return g;
}
