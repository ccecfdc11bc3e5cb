/*
 * gemm_rs.h: C ABI of the fused GEMM + reduce-scatter (GEMM+RS) library
 * for GB300 (sm_103a).
 *
 * OPERATION
 *   Y_c = sum over r = 0 .. W-1 of (alpha * A_r * B_r + beta * C)[rows of chunk c]
 *
 *   This is the second GEMM of a tensor-parallel FFN, whose epilogue writes
 *   into the reduce-scatter buffers instead of a plain output
 *   ("flux实现：sm80 gemm+rs", opening paragraph; "flux精读" §3 Design).
 *   - The W logical ranks each hold one K-shard: A_r = A[r] is [M][K/W] and
 *     B_r = B[r] is [K/W][N].  All W shards live in one GPU's memory.
 *   - The output Y is [M][N], made of W chunks of R = M/W contiguous rows.
 *     Rank c keeps chunk c, and the other W-1 chunks go to the other ranks
 *     ("flux实现：sm80 gemm+rs", section "gemmrs版本的swizzle如何编排").
 *   - Each rank's epilogue forms alpha*acc + beta*C ("flux实现：sm80 gemm+rs",
 *     section "custom_evt_d()": EVT_Compute0 = alpha*acc, EVT_Compute1 =
 *     beta*C + EVT_Compute0).  So beta*C is added once per rank: the result
 *     is alpha * sum_r(A_r B_r) + W * beta * C.  C is never read when
 *     beta == 0.
 *   - The partials are fp32 and are summed in fp32 in a fixed order, so
 *     results are bit-identical from run to run: rank order
 *     ((p_0 + p_1) + p_2) + ... by default (see GEMM_RS_REDUCE_* for the
 *     orders of the other modes).  A bf16 Y is rounded to nearest even.
 *
 *   One call runs one fused kernel.  Each output tile's partials meet in
 *   workspace slots keyed to the tile's chunk, coordinated by 32-bit state
 *   words per output tile ("flux实现：sm80 gemm+rs", section "evt_store_d()": a
 *   globally unique id per tile and a barrier flag per tile; "flux精读" §4.2:
 *   signals are 32-bit contiguous memory that lives as long as the op).  In
 *   the pages' design (GEMM_RS_REDUCE_LAST_ARRIVER) every rank stores its
 *   partial and the last rank to arrive reduces the tile; by default
 *   (GEMM_RS_REDUCE_CHAIN) each rank adds its partial onto a running sum as it
 *   lands and the last one writes Y.  Either way the tile's state words end
 *   at zero, so no memset, separate reduce kernel or host sync runs between
 *   calls (the page's reduce buffer had to start zeroed and its clear cost tens
 *   of microseconds: "flux实现：sm80 gemm+rs", section "自己的类flux实现").
 *
 * CONVENTIONS
 *   - Every function returns GEMM_RS_OK (0) or a negative GEMM_RS_ERR_* code.
 *     gemm_rs_last_error() then gives a message (per calling thread).  No C++
 *     exception crosses this boundary.
 *   - Pointers marked "device" are CUDA device addresses.  Pointers marked
 *     "host" are ordinary host memory.
 *   - The caller owns all device memory: A, B, C, Y and the workspace.  The
 *     library never allocates device memory.
 *   - A handle owns host state only (shape, TMA descriptors, launch plan).
 *   - gemm_rs_stream_t is a cudaStream_t.  NULL means the legacy default
 *     stream.  The calls that run on a stream are asynchronous, except
 *     gemm_rs_status, which synchronises the stream.
 *   - A handle's workspace holds the tile counters.  Two runs of one handle
 *     must not overlap in time: use one stream per handle, or order the
 *     streams.
 */
#ifndef GEMM_RS_H
#define GEMM_RS_H

#include <stddef.h>
#include <stdint.h>

#if defined(GEMM_RS_BUILD) && defined(__GNUC__)
#define GEMM_RS_API __attribute__((visibility("default")))
#else
#define GEMM_RS_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef struct gemm_rs_s *gemm_rs_t;
typedef struct CUstream_st *gemm_rs_stream_t; /* == cudaStream_t */

typedef enum {
    GEMM_RS_BF16 = 0,
    GEMM_RS_FP32 = 1
} gemm_rs_dtype;

enum {
    GEMM_RS_OK = 0,
    GEMM_RS_ERR_ARG = -1,         /* NULL handle or pointer, bad enum value, W out of range */
    GEMM_RS_ERR_SHAPE = -2,       /* M % W, K % W, (K/W) % 8, N % 8, negative or too-large size */
    GEMM_RS_ERR_ALIGN = -3,       /* a device pointer not 16-byte (workspace: 256-byte) aligned */
    GEMM_RS_ERR_CUDA = -4,        /* a CUDA runtime/driver call failed (message has the detail) */
    GEMM_RS_ERR_TIMEOUT = -5,     /* a device-side wait ran past its cycle limit */
    GEMM_RS_ERR_UNSUPPORTED = -6, /* dtype combination or device (needs sm_103) not supported */
    GEMM_RS_ERR_WORKSPACE = -7,   /* workspace smaller than gemm_rs_workspace_bytes() */
    GEMM_RS_ERR_BOUNDS = -8       /* checked build only (libgemm_rs_checked.so, compiled with
                                     GEMM_RS_CHECKED): an access of the epilogue or a fold
                                     outside its buffer was caught and skipped */
};

/* How the W partials of an output tile are reduced (gemm_rs_set_reduce_mode). */
enum {
    /* Default.  The ranks fold into the tile in the order in which the
     * schedule brings them to it (a fixed order per tile: rank order 0..W-1
     * when the ranks run one after another, the order of their steps when they
     * run side by side).  The rank whose turn it is adds its accumulator
     * straight from TMEM onto the running sum.  A rank that is early stores its
     * partial, and the current owner of the fold picks it up.  The last rank
     * writes Y.  The reduction overlaps the GEMM. */
    GEMM_RS_REDUCE_CHAIN = 0,
    /* Every rank stores its partial.  The last rank to arrive at a tile folds
     * all W partials in rank order 0 .. W-1 and writes Y. */
    GEMM_RS_REDUCE_LAST_ARRIVER = 1,
    /* The two-level reduction of a multi-node reduce-scatter, as one GPU sees
     * it ("flux实现：sm80 gemm+rs", section "2D Ring优化": the partial sums of
     * the ranks of one node meet first, and the nodes' sums meet after that).
     * The ranks form two groups, [0, h) and [h, W) with h = ceil(W/2).  Each
     * group folds its ranks in rank order as in CHAIN, into a running sum of
     * its own.  The group that finishes second writes
     * Y = (sum of group 0) + (sum of group 1).  W = 1 is CHAIN. */
    GEMM_RS_REDUCE_TWO_LEVEL = 2
};

/* The order in which the W logical ranks' tiles run (gemm_rs_set_schedule). */
enum {
    GEMM_RS_RANKS_DEFAULT = 0,     /* the library's choice: SEQUENTIAL */
    GEMM_RS_RANKS_SEQUENTIAL = 1,  /* rank 0's tiles, then rank 1's, ...: one rank's
                                      operands are live at a time */
    GEMM_RS_RANKS_INTERLEAVED = 2  /* the W ranks side by side, as W GPUs would run */
};

/* Debug flags for gemm_rs_set_debug. */
enum {
    /* The TMA producer issues no loads, so the MMA warp's wait on the first
     * stage runs out.  This exercises the timeout path on the GPU without a
     * fault.  Use only together with a short gemm_rs_set_timeout_cycles. */
    GEMM_RS_DEBUG_STALL_PRODUCER = 1,
    /* gemm_rs_run_streamed issues its copies but not the ready words that
     * follow them, so the kernel's wait for the first rank's operands runs
     * out (with a short gemm_rs_set_timeout_cycles): the timeout path of the
     * streamed call, without a fault. */
    GEMM_RS_DEBUG_SKIP_READY = 2
};

/*
 * Bytes of device workspace that a handle with this shape needs.  This
 * covers every tile width the library may pick.  Layout (internal, for
 * information):
 *   [0, 256)   device status word
 *   flags      three uint32 state words per output tile (ceil(M/128) x ceil(N/64) tiles
 *              max): a chain state or arrival counter per rank group, and a group count
 *   partials   fp32 partial tiles, one per (output tile, rank), grouped by the chunk
 *              that owns the tile's first row: W * ceil(M/128)*128 * ceil(N/256)*256 * 4 bytes
 * Returns 0 for invalid arguments (same checks as gemm_rs_create).
 */
GEMM_RS_API size_t gemm_rs_workspace_bytes(int64_t M, int64_t N, int64_t K, int W);

/*
 * Create a handle for one problem shape.
 *   M, N      output rows and columns.  M % W == 0 and N % 8 == 0.  M = 0 or
 *             N = 0 gives an empty problem: run() then returns at once.
 *   K         TOTAL reduction length.  Each rank holds K/W of it.  K % W == 0
 *             and (K/W) % 8 == 0.  K = 0 gives Y = W * beta * C.
 *   W         logical tensor-parallel ranks, 1 .. 16.
 *   alpha, beta  epilogue scalars (see OPERATION).
 *   ab_dtype  GEMM_RS_BF16 (A and B).
 *   c_dtype   GEMM_RS_BF16.
 *   y_dtype   GEMM_RS_BF16 or GEMM_RS_FP32.
 *   workspace device, caller-owned, 256-byte aligned, at least
 *             gemm_rs_workspace_bytes(M, N, K, W) bytes, workspace_bytes = its size.
 *             It must stay valid until gemm_rs_destroy.  Its contents
 *             belong to the library while the handle lives.
 *   stream    create() zeroes the status word and the tile counters once, on this
 *             stream, with one cudaMemsetAsync.  Later runs never clear them again.
 * Fails with ERR_ARG / ERR_SHAPE / ERR_ALIGN / ERR_WORKSPACE / ERR_UNSUPPORTED /
 * ERR_CUDA.  On failure *out is set to NULL.
 */
GEMM_RS_API int gemm_rs_create(gemm_rs_t *out, int64_t M, int64_t N, int64_t K, int W,
                   float alpha, float beta, gemm_rs_dtype ab_dtype,
                   gemm_rs_dtype c_dtype, gemm_rs_dtype y_dtype,
                   void *workspace, size_t workspace_bytes, gemm_rs_stream_t stream);

/*
 * Run the fused kernel once.  It is asynchronous on `stream`: no host sync
 * and no memset.
 *   A  device, bf16 [W][M][K/W] row-major (K contiguous), 16-byte aligned.
 *   B  device, bf16 [W][K/W][N] row-major (N contiguous), 16-byte aligned.
 *   C  device, bf16 [M][N], 16-byte aligned.  May be NULL when beta == 0, and
 *      is not read then.
 *   Y  device, [M][N] in y_dtype, 16-byte aligned.  Rows [c*M/W, (c+1)*M/W)
 *      are chunk c.  Every element is written.
 * A and B may change between calls.  Their TMA descriptors are re-encoded on
 * the host when the pointers change.  Returns ERR_ARG / ERR_ALIGN for bad
 * pointers and ERR_CUDA if the launch fails.  A device-side timeout is not
 * seen here: call gemm_rs_status.
 * The launch uses programmatic stream serialization: the kernel may start its
 * shared-memory and TMEM set-up while the previous kernel on `stream` is
 * still finishing, and waits for that kernel to complete (griddepcontrol.wait)
 * before its first global memory access, so every read and write is ordered
 * after the earlier work on the stream as for any launch.  Calls issued back
 * to back overlap by that set-up; an event recorded between them removes the
 * overlap.
 */
GEMM_RS_API int gemm_rs_run(gemm_rs_t h, const void *A, const void *B, const void *C, void *Y,
                gemm_rs_stream_t stream);

/*
 * gemm_rs_run with the inputs still in host memory: the host-to-device copies
 * overlap the kernel.  The pages overlap a GEMM with the communication of its
 * operands at tile granularity (the all-gather feeding the GEMM's tiles in the
 * order they are sent, "flux精读" §3); here the transfer is the one from the
 * host, and the unit is one rank's operands.
 *   A_host, B_host, C_host  host, pinned (page-locked) copies of A, B and C in
 *                           the layouts of gemm_rs_run; C_host may be NULL when
 *                           beta == 0.
 *   Y_host                  host, pinned, [M][N] in y_dtype: receives Y.
 *   A, B, C, Y              device buffers as for gemm_rs_run; A, B and C are
 *                           overwritten with the host copies.
 *   stream                  the kernel and the copy of Y back run on it.
 *   copy_stream             a second stream (not stream, not the legacy NULL
 *                           stream) for the host-to-device copies.
 * On copy_stream the call first waits for this handle's previous streamed
 * kernel (so a streamed call never overwrites operands that the previous one
 * still reads; other work that reads A, B or C must be ordered before this call
 * by the caller), then copies C, and then rank by rank A_r and B_r, each
 * followed by a 32-bit
 * ready word in the workspace (a stream memory operation, after a memory
 * fence).  The kernel's TMA producer waits, bounded, for rank r's word before
 * it loads rank r's first tile, and the epilogue for C's word before it reads
 * C, so with the ranks one after another rank r computes while rank r+1 is
 * still being copied.  Asynchronous: Y_host is complete once `stream` has
 * reached this point.  Errors as for gemm_rs_run, plus ERR_ARG for a NULL
 * host pointer or copy_stream == stream; a wait that runs out is reported by
 * gemm_rs_status like any other timeout.
 */
GEMM_RS_API int gemm_rs_run_streamed(gemm_rs_t h, const void *A_host, const void *B_host,
                                     const void *C_host, void *Y_host, void *A, void *B, void *C,
                                     void *Y, gemm_rs_stream_t stream,
                                     gemm_rs_stream_t copy_stream);

/* Free the handle's host state.  Does not touch device memory.  NULL is a no-op. */
GEMM_RS_API int gemm_rs_destroy(gemm_rs_t h);

/* Message for the last failing call on this thread ("" if none).  The string
 * stays valid until the next failing call on this thread. */
GEMM_RS_API const char *gemm_rs_last_error(void);

/*
 * Synchronise `stream`, then read and clear the handle's device status
 * word.  Returns GEMM_RS_OK, or GEMM_RS_ERR_TIMEOUT if a kernel of this
 * handle gave up on a wait since the last check.  After a timeout, Y of that
 * run is incomplete and the tile counters may be non-zero: call
 * gemm_rs_reset before the next run.  The checked build can also return
 * GEMM_RS_ERR_BOUNDS (see the error codes).
 */
GEMM_RS_API int gemm_rs_status(gemm_rs_t h, gemm_rs_stream_t stream);

/* Zero the status word and the tile counters again (one cudaMemsetAsync on
 * `stream`).  Needed only after a timeout. */
GEMM_RS_API int gemm_rs_reset(gemm_rs_t h, gemm_rs_stream_t stream);

/*
 * The global tile order of the fused kernel, written to host memory `out` as
 * int32 triples (r, mt, nt) for entries g = 0 .. W*nM*nN-1, where
 * nM = ceil(M/bm) and nN = ceil(N/bn).  With bm = 256 (the CTA-pair kernel) a
 * row tile is 256 rows.  Worker b of G workers (CTAs, or CTA pairs)
 * processes entries b, b+G, b+2G, ...
 *   - Rank r visits its chunks in the order (r+1+s) mod W, s = 0 .. W-1:
 *     the remote chunks first and its own chunk r last
 *     ("flux实现：sm80 gemm+rs", section "gemmrs版本的swizzle如何编排").
 *     Each rank's start is offset by its rank ("flux精读" §4.1), so when the
 *     ranks run side by side the W ranks target W different chunks at every
 *     step.
 *   - A row tile belongs to the chunk of its first row.
 *   - The column tiles are split into groups of `colgroup` consecutive tiles
 *     (0 or >= nN: one group).  For each group, the rank runs all W steps.
 *     Inside a group of gn tiles the rank starts at the group's tile
 *     ((W-r) mod W)*gn/W and wraps around within the group.  In a step, the
 *     chunk's row tiles (ascending) are split into row groups of `rowgroup`
 *     tiles (0: the whole chunk).  Each row group is one forward sweep over
 *     the column group's tiles.  For each column tile a sweep takes the row
 *     group's tiles in ascending order.
 *   - rank_order GEMM_RS_RANKS_INTERLEAVED: entry p*W + r is rank r's p-th
 *     tile (the ranks advance side by side).  GEMM_RS_RANKS_SEQUENTIAL or
 *     GEMM_RS_RANKS_DEFAULT: entry r*T + p is rank r's p-th tile, T = nM*nN
 *     (one rank after another).
 * `cap` is the capacity of `out` in triples.  Returns the number of entries,
 * or a negative error code (ERR_SHAPE if cap is too small).
 */
GEMM_RS_API int64_t gemm_rs_schedule(int64_t M, int64_t N, int W, int bm, int bn, int colgroup,
                                     int rowgroup, int rank_order, int32_t *out, int64_t cap);

/*
 * Launch plan of the handle (host outputs; any pointer may be NULL):
 *   bm, bn   the output tile (bm = 128; bn = 256, 128 or 64)
 *   stages   depth of the TMA -> MMA shared-memory ring
 *   grid     CTAs launched (persistent: one per SM, at most one per work item)
 *   colgroup, rowgroup, rank_order  the schedule in effect (see gemm_rs_set_schedule;
 *                       rank_order is GEMM_RS_RANKS_SEQUENTIAL or _INTERLEAVED)
 *   reduce_mode         GEMM_RS_REDUCE_* in effect
 */
GEMM_RS_API int gemm_rs_get_plan(gemm_rs_t h, int *bm, int *bn, int *stages, int *grid,
                                 int *colgroup, int *rowgroup, int *rank_order, int *reduce_mode);

/* The handle's shape and output dtype (host outputs; any pointer may be NULL). */
GEMM_RS_API int gemm_rs_get_shape(gemm_rs_t h, int64_t *M, int64_t *N, int64_t *K, int *W,
                                  int *y_dtype);

/* Override the tile width (bn = 256, 128 or 64) of the single-CTA kernel
 * (bm = 128).  Returns ERR_ARG for any other value. */
GEMM_RS_API int gemm_rs_set_tile_n(gemm_rs_t h, int bn);

/* Override the output tile.  (128, 64|128|256) runs the single-CTA kernel.
 * (256, 256) runs the CTA-pair kernel: a cluster of two CTAs shares one 256x256
 * tile.  Each CTA loads its own 128 rows of A and 128 columns of B, and one
 * tcgen05.mma.cta_group::2 computes the pair's product.  The default is the pair
 * kernel when there are at least four 256x256 rank-tiles per SM pair, otherwise
 * the widest single-CTA tile with at least four work items per SM (one work item
 * per SM when M fits in one 128-row tile). */
GEMM_RS_API int gemm_rs_set_tile(gemm_rs_t h, int bm, int bn);

/* Schedule (see gemm_rs_schedule).  "Live ranks" below is 1 for the
 * sequential rank order and W for the interleaved one.
 *   colgroup    column tiles per column group.  0 (the default) = the
 *               library's choice.  Ranks one after another: two groups when
 *               that keeps a group's fp32 running sums (M x its columns)
 *               within 40 MB, else one.  Ranks side by side: 1, 2, 4 or 8
 *               groups, whichever a model of the operand bytes read from DRAM
 *               favours (A rows are read once per group; a group's B panels of
 *               the W ranks are read once when they fit in about 64 MB, else
 *               once per step), keeping groups large enough that a tile's
 *               contributions arrive in step order.
 *   rowgroup    row tiles per column sweep.  0 (the default) = the library's
 *               choice: the chunk's row tiles in the fewest groups of
 *               near-equal size that each keep at most 64 MB of A rows of the
 *               live ranks.  Smaller groups re-read B once per sweep.
 *   rank_order  GEMM_RS_RANKS_* (0: the default, SEQUENTIAL).
 * Returns ERR_ARG for negative values or an unknown rank order. */
GEMM_RS_API int gemm_rs_set_schedule(gemm_rs_t h, int colgroup, int rowgroup, int rank_order);

/* Select the reduction (GEMM_RS_REDUCE_*).  All give Y within the stated
 * tolerances of each other.  Each is bit-identical from run to run.  They
 * differ in summation order: rank order 0..W-1 for LAST_ARRIVER, the
 * schedule's arrival order for CHAIN (the same rank order with the default
 * sequential ranks), rank order within each of the two groups for TWO_LEVEL.
 * CHAIN and TWO_LEVEL add the middle positions to the running sum in L2
 * (red.add.f32), which flushes subnormal sums to zero.  ERR_ARG for other
 * values. */
GEMM_RS_API int gemm_rs_set_reduce_mode(gemm_rs_t h, int mode);

/* Device wait limit in SM clock cycles (default 2^32, about two seconds).  A
 * wait that runs past it sets the status word and lets the kernel exit. */
GEMM_RS_API int gemm_rs_set_timeout_cycles(gemm_rs_t h, uint64_t cycles);

/*
 * Debug hooks.
 *   record  device int32 buffer of 4 * W*nM*nN entries, or NULL.  When set,
 *           each run writes (r, mt, nt, cta) for every entry g that it
 *           processes, at record[4g .. 4g+3].
 *   flags   GEMM_RS_DEBUG_* bits (0 = none).
 */
GEMM_RS_API int gemm_rs_set_debug(gemm_rs_t h, int32_t *record, int flags);

/*
 * Baseline only (not the fused path): the separate reduce step of an
 * unfused GEMM+RS, which runs after W per-rank GEMMs.
 *   partials  device, [W][M][N], fp32 (partial_dtype = GEMM_RS_FP32) or bf16
 *   C         device bf16 [M][N], or NULL when beta == 0
 *   Y         device [M][N] in y_dtype
 * Y = fold over r in rank order of fp32(alpha * partials[r] + beta * C), with
 * the same rounding as the fused path.  Asynchronous on `stream`.
 * Pointers must be 16-byte aligned, and N % 8 == 0.
 */
GEMM_RS_API int gemm_rs_reduce_partials(const void *partials, gemm_rs_dtype partial_dtype, const void *C,
                            void *Y, int64_t M, int64_t N, int W, float alpha, float beta,
                            gemm_rs_dtype y_dtype, gemm_rs_stream_t stream);

/*
 * Size of the static device scratch used by gemm_rs_run_noalloc: 64 MiB.  It holds
 * the status word, the tile counters and the fp32 partial tiles, laid out as in the
 * workspace of gemm_rs_create.  A shape fits if gemm_rs_workspace_bytes(M, N, K, W)
 * is at most this size.
 */
#define GEMM_RS_NOALLOC_SCRATCH_BYTES (64u * 1024u * 1024u)

/*
 * gemm_rs_run without a handle and without a workspace: this call allocates
 * nothing.  (The pages have no counterpart.  This is a convenience of this
 * library.)
 *
 * Some callers cannot call cudaMalloc and have no workspace to hand over.
 * Examples: a plugin inside a host application that owns every device
 * allocation, or a latency-critical path where an allocation, which may
 * synchronise the device, is not allowed.  This entry point runs the same fused
 * kernel.  Its scratch (status word, tile counters, partial tiles) is a
 * file-scope device array of GEMM_RS_NOALLOC_SCRATCH_BYTES, which every GPU that
 * loads this library holds until the process exits.  The call makes no
 * cudaMalloc or cudaFree and calls no allocating library routine.
 *
 *   M, N, K, W, alpha, beta, y_dtype   as for gemm_rs_create (A, B and C are bf16).
 *   A, B, C, Y                         as for gemm_rs_run (device, 16-byte aligned).
 *   stream                             the call is asynchronous on this stream.
 *
 * - The first call in a context does a one-time set-up there (kernel
 *   attributes).  Every call looks up the scratch array's device address with
 *   cudaGetSymbolAddress (no allocation).  Make the first call before any
 *   stream capture begins.
 * - Each call clears the status word and the tile counters with one
 *   cudaMemsetAsync on `stream`.  The scratch keeps the previous call's
 *   contents otherwise.
 * - Every call on a device shares the one scratch array.  Calls that overlap
 *   on the GPU (different streams, or host threads with no ordering between
 *   them) race on it and give wrong results.  Order them on one stream.
 * - The scratch address is looked up on every call, in the calling thread's
 *   current CUDA context, so callers that own several contexts on one device
 *   get the array of the context they run in.  The kernel attributes are set
 *   once per context.
 * - A shape whose gemm_rs_workspace_bytes exceeds GEMM_RS_NOALLOC_SCRATCH_BYTES
 *   is rejected with GEMM_RS_ERR_WORKSPACE.  Other errors are as for
 *   gemm_rs_create and gemm_rs_run.  A device-side timeout leaves its code in
 *   the scratch's status word until the next call clears it: read it with
 *   gemm_rs_noalloc_status before the next call.
 */
GEMM_RS_API int gemm_rs_run_noalloc(int64_t M, int64_t N, int64_t K, int W, float alpha,
                                    float beta, gemm_rs_dtype y_dtype, const void *A,
                                    const void *B, const void *C, void *Y,
                                    gemm_rs_stream_t stream);

/*
 * GEMM_RS_NOALLOC_SCRATCH_BYTES as compiled into this library (the size of its
 * static scratch), for callers and bindings that do not read this header.
 * (Part of the no-alloc entry point; the pages have no counterpart.)
 */
GEMM_RS_API size_t gemm_rs_noalloc_scratch_bytes(void);

/*
 * The outcome of the last gemm_rs_run_noalloc call in the current context, for
 * callers without a handle (the pages have no counterpart).  Waits for `stream` (the stream of that call),
 * reads the status word of the static scratch, and clears it.  Allocates
 * nothing (the word is copied into a host variable).  Returns GEMM_RS_OK,
 * GEMM_RS_ERR_TIMEOUT (a device wait ran out; Y is not valid),
 * GEMM_RS_ERR_BOUNDS (checked build only) or GEMM_RS_ERR_CUDA.  The next
 * gemm_rs_run_noalloc clears the word too, so call this in between.
 */
GEMM_RS_API int gemm_rs_noalloc_status(gemm_rs_stream_t stream);

/* Library version string. */
GEMM_RS_API const char *gemm_rs_version(void);

#ifdef __cplusplus
}
#endif

#endif /* GEMM_RS_H */
