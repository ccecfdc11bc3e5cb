/*
 * C ABI of the fused all-gather + GEMM (AG+GEMM): the first GEMM of a
 * tensor-parallel FFN, whose input rows are all-gathered from the ranks
 * before the GEMM ("flux精读" §3 Design, the AllGather GEMM paragraph;
 * "通信 overlap 实现", section "Flux 的 tile 级融合解决了什么？": AG+GEMM, prologue
 * fusion).  Its output H_r is the A_r of the GEMM+RS in gemm_rs.h.
 *
 * W logical ranks run on one GPU.  Rank r holds row chunk r of X (rows
 * [r*M/W, (r+1)*M/W)) and the column shard B1_r of the weight:
 *
 *     H_r = alpha * X @ B1_r      for r = 0 .. W-1
 *
 * where X is the all-gather of the W chunks.  One kernel emulates the ranks:
 * copy warps deliver each remote chunk into rank r's gather buffer and raise a
 * 32-bit signal per (rank, chunk) when it is complete; each GEMM tile waits
 * (bounded) for the signal of its chunk, in the order the chunks are sent,
 * and a rank's own chunk needs no wait ("flux精读" §4.1: each rank starts at
 * its own chunk).  The launch is cooperative: all CTAs are resident.
 *
 * Types, error codes and the stream handle are those of gemm_rs.h, and
 * gemm_rs_last_error() returns the message of a failing call here too.
 */
#ifndef AG_GEMM_H
#define AG_GEMM_H

#include "gemm_rs.h"

#ifdef __cplusplus
extern "C" {
#endif

typedef struct ag_gemm_s *ag_gemm_t;

/*
 * Device workspace for a shape, in bytes (0 for an unsupported shape): a
 * 256-byte status word, the W*W chunk signals, and the gather buffers
 * [W][M][K] bf16.
 *   M  rows of X and of every H_r; M must be a multiple of 256*W (each
 *      256-row tile lies in one chunk)
 *   N  columns of each rank's shard B1_r and of H_r; a multiple of 8
 *   K  columns of X, rows of B1_r; a multiple of 8
 *   W  ranks, 1 .. 16
 */
GEMM_RS_API size_t ag_gemm_workspace_bytes(int64_t M, int64_t N, int64_t K, int W);

/*
 * Create a handle for one shape.  `workspace` is caller-owned device memory of
 * at least ag_gemm_workspace_bytes(), 256-byte aligned; its status word and
 * signals are zeroed on `stream` (asynchronously).  y_dtype is GEMM_RS_BF16
 * or GEMM_RS_FP32.  Returns ERR_ARG, ERR_SHAPE, ERR_ALIGN, ERR_WORKSPACE,
 * ERR_UNSUPPORTED (not sm_103) or ERR_CUDA.
 */
GEMM_RS_API int ag_gemm_create(ag_gemm_t *out, int64_t M, int64_t N, int64_t K, int W, float alpha,
                               gemm_rs_dtype y_dtype, void *workspace, size_t workspace_bytes,
                               gemm_rs_stream_t stream);

/*
 * One call, asynchronous on `stream`.
 *   X   device, bf16 [M][K] row-major: the W row chunks, chunk c = rows
 *       [c*M/W, (c+1)*M/W); 16-byte aligned.
 *   B1  device, bf16 [W][K][N] row-major (N contiguous): rank r's shard.
 *   H   device, [W][M][N] in y_dtype: H_r = alpha * X @ B1_r; every element
 *       is written.
 * The gather buffers in the workspace are rewritten on every call.  Returns
 * ERR_ARG / ERR_ALIGN for bad pointers and ERR_CUDA if the launch fails.  A
 * device-side timeout is reported by ag_gemm_status.
 */
GEMM_RS_API int ag_gemm_run(ag_gemm_t h, const void *X, const void *B1, void *H,
                            gemm_rs_stream_t stream);

/* Synchronise `stream`, then read and clear the status word: GEMM_RS_OK or
 * GEMM_RS_ERR_TIMEOUT (or, in the checked build, GEMM_RS_ERR_BOUNDS).  After
 * a timeout call ag_gemm_reset. */
GEMM_RS_API int ag_gemm_status(ag_gemm_t h, gemm_rs_stream_t stream);

/* Zero the status word and the chunk signals (one memset on `stream`). */
GEMM_RS_API int ag_gemm_reset(ag_gemm_t h, gemm_rs_stream_t stream);

/* Free the handle's host state; NULL is a no-op. */
GEMM_RS_API int ag_gemm_destroy(ag_gemm_t h);

/*
 * The tile order, as int32 triples (r, mt, nt) of 256x256 tiles, into host
 * memory `out` (capacity `cap` triples): the ranks one after another; rank r
 * takes its chunks in the order (r+s) mod W, s = 0 .. W-1 (its own first);
 * inside a chunk, column tiles outer and the chunk's 256-row tiles inner.
 * Worker b of G workers (CTA pairs) processes entries b, b+G, ...  Returns the
 * number of entries or a negative error code.
 */
GEMM_RS_API int64_t ag_gemm_schedule(int64_t M, int64_t N, int W, int32_t *out, int64_t cap);

/* Launch plan (host outputs; any pointer may be NULL): grid (CTAs), stages,
 * slice_rows (rows per copy slice) and slices (per chunk). */
GEMM_RS_API int ag_gemm_get_plan(ag_gemm_t h, int *grid, int *stages, int *slice_rows, int *slices);

/* Device wait limit in SM cycles (default 2^32). */
GEMM_RS_API int ag_gemm_set_timeout_cycles(ag_gemm_t h, uint64_t cycles);

/* Debug flags for ag_gemm_set_debug. */
enum {
    /* The copy warps deliver nothing, so every wait for a remote chunk runs
     * out: this exercises the timeout path on the GPU without a fault.  Use
     * only together with a short ag_gemm_set_timeout_cycles. */
    AG_GEMM_DEBUG_SKIP_COPIES = 1
};

/* Record the device tile order (`record`: device int32 [entries][4],
 * (r, mt, nt, worker) per entry, or NULL) and set debug flags. */
GEMM_RS_API int ag_gemm_set_debug(ag_gemm_t h, int32_t *record, int flags);

/* The handle's shape and output dtype (host outputs; any pointer may be NULL). */
GEMM_RS_API int ag_gemm_get_shape(ag_gemm_t h, int64_t *M, int64_t *N, int64_t *K, int *W,
                                  int *y_dtype);

/*
 * The tensor-parallel FFN on one GPU, both halves fused with their collective
 * ("通信 overlap 实现", the passage on why AG and RS cannot simply be issued
 * asynchronously: the AG output is the GEMM input and the GEMM output is the
 * RS input, so the chain is split into tile-level steps):
 *
 *     H_r = alpha1 * X @ B1_r                    (ag, bf16 output)
 *     Y   = sum_r (alpha2 * H_r @ B2_r + beta * C)   (rs, chunk c = rows of chunk c)
 *
 * Two launches on `stream`: the AG+GEMM, then the GEMM+RS with A = H.  No
 * activation is applied between them.  `ag` must have a bf16 output and `rs`
 * the matching shape: same M and W, rs K = W * (ag N).  Pointers as in
 * ag_gemm_run (X, B1, H) and gemm_rs_run (B2 = its B, C, Y).
 */
GEMM_RS_API int ffn_tp_run(ag_gemm_t ag, gemm_rs_t rs, const void *X, const void *B1, void *H,
                           const void *B2, const void *C, void *Y, gemm_rs_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* AG_GEMM_H */
