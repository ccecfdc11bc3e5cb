// Host side of the C ABI declared in include/gemm_rs.h: argument checks, the
// workspace layout, TMA descriptors, the launch plan and the launch.  No
// exception crosses the boundary; errors come back as codes, and the
// message is kept per thread.
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <cuda.h>
#include <cuda_runtime.h>
#include <mutex>
#include <new>
#include <string>

#include "api_common.cuh"
#include "gemm_rs.h"
#include "gemm_rs_kernel.cuh"
#include "reduce_baseline.cuh"
#include "schedule.cuh"

namespace {

using namespace gemm_rs_host;

constexpr size_t kStatusBytes = 256;
constexpr int64_t kMaxDim = (int64_t(1) << 31) - 1;

struct Layout {
    size_t flags_off, flags_bytes, part_off, part_bytes, total;
};

Layout layout_for(int64_t M, int64_t N, int W)
{
    Layout L;
    const int64_t nM = cdiv(M, gemm_rs::kBM);
    L.flags_off = kStatusBytes;
    // three state words per output tile: the chain (or arrival counter) of
    // ranks [0, W) or of the first group of the two-level fold, the second
    // group's chain, and the count of groups done
    L.flags_bytes = round_up(static_cast<size_t>(3 * nM * cdiv(N, 64)) * sizeof(uint32_t), 256);
    L.part_off = L.flags_off + L.flags_bytes;
    L.part_bytes = static_cast<size_t>(W) * static_cast<size_t>(nM) * gemm_rs::kBM *
                   static_cast<size_t>(cdiv(N, 256) * 256) * sizeof(float);
    L.total = L.part_off + L.part_bytes;
    return L;
}

int check_shape(int64_t M, int64_t N, int64_t K, int W)
{
    if (W < 1 || W > 16)
        return fail(GEMM_RS_ERR_ARG, "W = %d is outside 1..16", W);
    if (M < 0 || N < 0 || K < 0)
        return fail(GEMM_RS_ERR_SHAPE, "negative size (M=%lld N=%lld K=%lld)", (long long)M,
                    (long long)N, (long long)K);
    if (M > kMaxDim || N > kMaxDim || K > kMaxDim)
        return fail(GEMM_RS_ERR_SHAPE, "size above 2^31-1");
    if (M % W != 0)
        return fail(GEMM_RS_ERR_SHAPE, "M = %lld is not a multiple of W = %d (chunks are M/W rows)",
                    (long long)M, W);
    if (K % W != 0)
        return fail(GEMM_RS_ERR_SHAPE, "K = %lld is not a multiple of W = %d", (long long)K, W);
    if ((K / W) % 8 != 0)
        return fail(GEMM_RS_ERR_SHAPE, "K/W = %lld is not a multiple of 8 (16-byte TMA row stride)",
                    (long long)(K / W));
    if (N % 8 != 0)
        return fail(GEMM_RS_ERR_SHAPE, "N = %lld is not a multiple of 8 (16-byte rows)",
                    (long long)N);
    if (cdiv(M, 128) * cdiv(N, 64) >= (int64_t(1) << 25))
        return fail(GEMM_RS_ERR_SHAPE, "more than 2^25 output tiles");
    return GEMM_RS_OK;
}

struct DeviceInfo {
    int dev = 0;
    int sms = 0;
    int pair_clusters = 0; // CTA pairs of the pair kernel that fit on the device at once
};
ContextCache<DeviceInfo> g_dev;

template <int BN>
cudaError_t set_kernel_attrs()
{
    return cudaFuncSetAttribute(gemm_rs::gemm_rs_fused_kernel<BN>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize,
                                gemm_rs::smem_bytes<BN>());
}

cudaError_t set_pair_kernel_attrs()
{
    return cudaFuncSetAttribute(gemm_rs::gemm_rs_pair_kernel<256>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize,
                                gemm_rs::smem_bytes_pair<256>());
}

// Once per CUDA context: check the device, set the kernels' shared-memory
// attributes and count the co-resident CTA pairs.
int setup_device(DeviceInfo &d)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return cuda_fail(e, "cudaGetDevice");
    int major = 0, minor = 0;
    if ((e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess)
        return cuda_fail(e, "cudaDeviceGetAttribute(major)");
    if ((e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess)
        return cuda_fail(e, "cudaDeviceGetAttribute(minor)");
    if (major != 10 || minor != 3)
        return fail(GEMM_RS_ERR_UNSUPPORTED,
                    "device %d has compute capability %d.%d; this library is built for sm_103a",
                    dev, major, minor);
    d.dev = dev;
    if ((e = cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
        return cuda_fail(e, "cudaDeviceGetAttribute(SM count)");
    if ((e = set_kernel_attrs<256>()) != cudaSuccess ||
        (e = set_kernel_attrs<128>()) != cudaSuccess ||
        (e = set_kernel_attrs<64>()) != cudaSuccess || (e = set_pair_kernel_attrs()) != cudaSuccess)
        return cuda_fail(e, "cudaFuncSetAttribute(max dynamic shared memory)");
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * (d.sms / 2), 1, 1);
    cfg.blockDim = dim3(gemm_rs::kThreads, 1, 1);
    cfg.dynamicSmemBytes = gemm_rs::smem_bytes_pair<256>();
    int clusters = 0;
    if ((e = cudaOccupancyMaxActiveClusters(&clusters, gemm_rs::gemm_rs_pair_kernel<256>, &cfg)) !=
        cudaSuccess)
        return cuda_fail(e, "cudaOccupancyMaxActiveClusters(pair kernel)");
    d.pair_clusters = clusters > 0 ? clusters : 1;
    return GEMM_RS_OK;
}

int prepare_device(int *dev_out, int *sms_out, int *pair_clusters_out = nullptr)
{
    DeviceInfo d;
    const int rc = g_dev.get(&d, setup_device);
    if (rc != GEMM_RS_OK)
        return rc;
    *dev_out = d.dev;
    *sms_out = d.sms;
    if (pair_clusters_out)
        *pair_clusters_out = d.pair_clusters;
    return GEMM_RS_OK;
}

// The error a non-zero status word reports (the word is then cleared by the caller).
int status_word_error(uint32_t word)
{
    if (word == gemm_rs::kStatusOutOfBounds)
        return fail(GEMM_RS_ERR_BOUNDS,
                    "checked build: an access outside its buffer was caught and skipped");
    static const char *role[] = {"?", "TMA producer", "MMA issuer", "epilogue", "reducer"};
    return fail(GEMM_RS_ERR_TIMEOUT, "device wait timed out in the %s (status %u)",
                role[word < 5 ? word : 0], word);
}

int stages_for(int bm, int bn)
{
    if (bm == 2 * gemm_rs::kBM)
        return gemm_rs::PairCfg<256>::kStages;
    switch (bn) {
    case 256: return gemm_rs::TileCfg<256>::kStages;
    case 128: return gemm_rs::TileCfg<128>::kStages;
    default: return gemm_rs::TileCfg<64>::kStages;
    }
}

// The widest tile that still gives at least four work items per SM.
int pick_bn(int64_t M, int64_t N, int W, int sms)
{
    const int64_t nM = cdiv(M, gemm_rs::kBM);
    // With a single row tile the call streams B once and re-reads the small A
    // for every tile: wide tiles cut the A share of each stage, and one wave
    // of work items is enough.
    const int64_t waves = nM == 1 ? 1 : 4;
    for (int bn : {256, 128}) {
        if (static_cast<int64_t>(W) * nM * cdiv(N, bn) >= waves * sms)
            return bn;
    }
    return 64;
}

// Launch plan: the CTA-pair kernel (256 x 256 tiles) when there are at least
// four pair tiles per SM pair, otherwise the single-CTA kernel with the widest
// tile that still gives at least four work items per SM (one when M is a
// single row tile).
void pick_tile(int64_t M, int64_t N, int W, int sms, int *bm, int *bn)
{
    const int64_t pairs = static_cast<int64_t>(W) * cdiv(M, 2 * gemm_rs::kBM) * cdiv(N, 256);
    if (M > gemm_rs::kBM && pairs >= 4LL * (sms / 2)) {
        *bm = 2 * gemm_rs::kBM;
        *bn = 256;
        return;
    }
    *bm = gemm_rs::kBM;
    *bn = pick_bn(M, N, W, sms);
}

// Row tiles per column sweep.  A sweep keeps its row tiles' A rows live in
// L2 for every live rank (1 when the ranks run one after another, W when they
// run side by side), so bound them to about 64 MB across the live ranks.
// Returns the chunk's row tile count (one sweep per step) when that fits.
int pick_rowgroup(int64_t M, int64_t Kpr, int W, int bm, int live)
{
    // row tiles keyed to one chunk: at most ceil(R/bm), plus one when R is ragged
    const int64_t R = M / W;
    const int64_t rows_per_chunk = cdiv(R, bm) + (R % bm != 0 ? 1 : 0);
    const int64_t panel = static_cast<int64_t>(bm) * Kpr * 2 * live;
    if (panel <= 0 || rows_per_chunk <= 1)
        return static_cast<int>(rows_per_chunk > 0 ? rows_per_chunk : 1);
    // The A rows live across the live ranks' sweeps stay within about half of L2.
    const int64_t budget = int64_t(64) << 20;
    int64_t rg = budget / panel;
    if (rg < 1)
        rg = 1;
    if (rg >= rows_per_chunk)
        return static_cast<int>(rows_per_chunk);
    // Balanced groups: as many as the budget needs, of near-equal size.
    const int64_t groups = cdiv(rows_per_chunk, rg);
    return static_cast<int>(cdiv(rows_per_chunk, groups));
}

// Column tiles per group when the caller leaves it to the library.
//
// Ranks side by side (live = W): the model counts the operand bytes read from
// DRAM.  With k column groups, the A rows of every chunk are read once per
// group (k * |A|).  The B panels of one group are read once if the W ranks'
// panels of a group fit in about 64 MB of L2, and once per step (W * |B|)
// otherwise.  k = 1, 2, 4, 8 are tried and the least traffic wins (a tie keeps
// fewer groups).  A group must also hold enough tiles that consecutive
// contributions to one output tile lie at least 1.25 waves of workers apart,
// so that they arrive in step order.
//
// Ranks one after another (live = 1): one group.  One rank's operands stay in
// L2 through its pass whatever the group.  Two groups would keep half the
// running sums (M x half the columns, fp32) live across the W passes, for the
// price of reading A twice, but timed in interleaved rounds they were no
// faster at W=8 M=N=4096 (32 MB of sums per group) and 11-14 % slower with
// the MMA loop that issues one multicast commit per stage.
int pick_colgroup(int64_t M, int64_t N, int64_t Kpr, int W, int bm, int bn, int64_t workers,
                  int live)
{
    const int64_t nN = cdiv(N, bn);
    const int64_t nMs = cdiv(M, bm);
    if (live == 1)
        return static_cast<int>(nN);
    const double a_bytes = 2.0 * W * M * Kpr;
    const double b_bytes = 2.0 * W * Kpr * N;
    const double budget = 64.0 * (1 << 20);
    int64_t best = nN;
    double best_cost = 0.0;
    int64_t prev = -1;
    for (int k = 1; k <= 8; k *= 2) {
        const int64_t G = cdiv(nN, k);
        if (G == prev)
            break;
        prev = G;
        const double sep = static_cast<double>(nMs) * G * (W - 1) / W; // work items apart
        if (k > 1 && sep < 1.25 * static_cast<double>(workers))
            break;
        const double b_live = 2.0 * live * Kpr * G * bn;
        const double cost = a_bytes * static_cast<double>(cdiv(nN, G)) + b_bytes * (b_live <= budget ? 1 : W);
        if (k == 1 || cost < best_cost) {
            best = G;
            best_cost = cost;
        }
    }
    return static_cast<int>(best);
}

} // namespace

struct gemm_rs_s {
    int64_t M, N, K, Kpr;
    int W;
    float alpha, beta;
    gemm_rs_dtype y_dtype;
    uint8_t *ws;
    Layout L;
    int device, sms, pair_clusters, bm, bn;
    int colgroup; // 0: the default (pick_colgroup)
    int rowgroup; // 0: the default (pick_rowgroup)
    int rank_order; // GEMM_RS_RANKS_*
    int reduce_mode; // GEMM_RS_REDUCE_* (default CHAIN)
    CUtensorMap tmA, tmB;
    const void *tmA_ptr, *tmB_ptr;
    int tmB_atoms, tmB_4d; // the B map's atoms per load, and whether it is 4D
    unsigned long long timeout;
    int32_t *record;
    int debug_flags;
    // gemm_rs_run_streamed: the call index its ready words carry, and an event
    // after its latest kernel (the next call's copies wait for it)
    uint32_t stream_epoch;
    cudaEvent_t streamed_done;
    bool streamed_pending;
};

namespace {

// Launch with programmatic stream serialization: the kernel's CTAs may start
// (and set up shared memory and TMEM) while the previous kernel on the stream
// finishes; each kernel waits (griddepcontrol.wait) before it touches global
// memory.  With a non-kernel predecessor the launch is ordered as usual.
template <typename Kern>
cudaError_t launch_overlapped(Kern kernel, int grid, int smem, cudaStream_t s, const CUtensorMap &tmA,
                              const CUtensorMap &tmB, const gemm_rs::KernelArgs &a)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
    cfg.blockDim = dim3(gemm_rs::kThreads, 1, 1);
    cfg.dynamicSmemBytes = static_cast<size_t>(smem);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, tmA, tmB, a);
}

// Workers of the launch: CTA pairs for the 256-row tile, CTAs otherwise.
int64_t workers_of(const gemm_rs_s *h)
{
    const int64_t total = static_cast<int64_t>(h->W) * cdiv(h->M, h->bm) * cdiv(h->N, h->bn);
    const int64_t cap = h->bm == 2 * gemm_rs::kBM ? h->pair_clusters : h->sms;
    return total < cap ? total : cap;
}

bool sequential(const gemm_rs_s *h) { return h->rank_order != GEMM_RS_RANKS_INTERLEAVED; }

// Ranks whose operands are live at once.
int live_ranks(const gemm_rs_s *h) { return sequential(h) ? 1 : h->W; }

int rowgroup_of(const gemm_rs_s *h)
{
    return h->rowgroup > 0 ? h->rowgroup : pick_rowgroup(h->M, h->Kpr, h->W, h->bm, live_ranks(h));
}

int colgroup_of(const gemm_rs_s *h)
{
    const int64_t nN = cdiv(h->N, h->bn);
    if (h->colgroup > 0)
        return static_cast<int>(h->colgroup < nN ? h->colgroup : nN);
    return pick_colgroup(h->M, h->N, h->Kpr, h->W, h->bm, h->bn, workers_of(h), live_ranks(h));
}

} // namespace

extern "C" {

#ifdef GEMM_RS_CHECKED
const char *gemm_rs_version(void) { return "gemm_rs 0.1 (sm_103a, tcgen05, checked)"; }
#else
const char *gemm_rs_version(void) { return "gemm_rs 0.1 (sm_103a, tcgen05)"; }
#endif

const char *gemm_rs_last_error(void) { return g_err.c_str(); }

size_t gemm_rs_workspace_bytes(int64_t M, int64_t N, int64_t K, int W)
{
    if (check_shape(M, N, K, W) != GEMM_RS_OK)
        return 0;
    return layout_for(M, N, W).total;
}

int gemm_rs_create(gemm_rs_t *out, int64_t M, int64_t N, int64_t K, int W, float alpha, float beta,
                   gemm_rs_dtype ab_dtype, gemm_rs_dtype c_dtype, gemm_rs_dtype y_dtype,
                   void *workspace, size_t workspace_bytes, gemm_rs_stream_t stream)
{
    if (out == nullptr)
        return fail(GEMM_RS_ERR_ARG, "out is NULL");
    *out = nullptr;
    int rc = check_shape(M, N, K, W);
    if (rc != GEMM_RS_OK)
        return rc;
    if (ab_dtype != GEMM_RS_BF16)
        return fail(GEMM_RS_ERR_UNSUPPORTED, "A/B dtype must be GEMM_RS_BF16");
    if (c_dtype != GEMM_RS_BF16)
        return fail(GEMM_RS_ERR_UNSUPPORTED, "C dtype must be GEMM_RS_BF16");
    if (y_dtype != GEMM_RS_BF16 && y_dtype != GEMM_RS_FP32)
        return fail(GEMM_RS_ERR_UNSUPPORTED, "Y dtype must be GEMM_RS_BF16 or GEMM_RS_FP32");
    if (!(alpha == alpha) || !(beta == beta))
        return fail(GEMM_RS_ERR_ARG, "alpha and beta must not be NaN");
    const Layout L = layout_for(M, N, W);
    if (workspace == nullptr)
        return fail(GEMM_RS_ERR_ARG, "workspace is NULL");
    if (!aligned(workspace, 256))
        return fail(GEMM_RS_ERR_ALIGN, "workspace must be 256-byte aligned");
    if (workspace_bytes < L.total)
        return fail(GEMM_RS_ERR_WORKSPACE, "workspace has %zu bytes, needs %zu", workspace_bytes,
                    L.total);
    int dev = 0, sms = 0, pair_clusters = 0;
    if ((rc = prepare_device(&dev, &sms, &pair_clusters)) != GEMM_RS_OK)
        return rc;
    cudaError_t e = cudaMemsetAsync(workspace, 0, L.part_off, reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess)
        return cuda_fail(e, "cudaMemsetAsync(status and tile counters)");
    gemm_rs_s *h = new (std::nothrow) gemm_rs_s();
    if (h == nullptr)
        return fail(GEMM_RS_ERR_ARG, "out of host memory");
    h->M = M;
    h->N = N;
    h->K = K;
    h->Kpr = K / W;
    h->W = W;
    h->alpha = alpha;
    h->beta = beta;
    h->y_dtype = y_dtype;
    h->ws = static_cast<uint8_t *>(workspace);
    h->L = L;
    h->device = dev;
    h->sms = sms;
    h->pair_clusters = pair_clusters;
    pick_tile(M, N, W, sms, &h->bm, &h->bn);
    h->colgroup = 0;
    h->rowgroup = 0;
    h->rank_order = GEMM_RS_RANKS_DEFAULT;
    h->reduce_mode = GEMM_RS_REDUCE_CHAIN;
    h->tmA_ptr = h->tmB_ptr = nullptr;
    h->tmB_atoms = 0;
    h->tmB_4d = 0;
    h->timeout = 1ull << 32;
    h->record = nullptr;
    h->debug_flags = 0;
    h->stream_epoch = 0;
    h->streamed_done = nullptr;
    h->streamed_pending = false;
    *out = h;
    return GEMM_RS_OK;
}

int gemm_rs_destroy(gemm_rs_t h)
{
    if (h != nullptr && h->streamed_done != nullptr)
        cudaEventDestroy(h->streamed_done);
    delete h;
    return GEMM_RS_OK;
}

int gemm_rs_get_plan(gemm_rs_t h, int *bm, int *bn, int *stages, int *grid, int *colgroup,
                     int *rowgroup, int *rank_order, int *reduce_mode)
{
    if (h == nullptr)
        return fail(GEMM_RS_ERR_ARG, "handle is NULL");
    const int64_t total = static_cast<int64_t>(h->W) * cdiv(h->M, h->bm) * cdiv(h->N, h->bn);
    if (bm)
        *bm = h->bm;
    if (bn)
        *bn = h->bn;
    if (stages)
        *stages = stages_for(h->bm, h->bn);
    if (colgroup)
        *colgroup = colgroup_of(h);
    if (rowgroup)
        *rowgroup = rowgroup_of(h);
    if (rank_order)
        *rank_order = sequential(h) ? GEMM_RS_RANKS_SEQUENTIAL : GEMM_RS_RANKS_INTERLEAVED;
    if (reduce_mode)
        *reduce_mode = h->reduce_mode;
    if (grid) {
        if (h->bm == 2 * gemm_rs::kBM) {
            const int64_t pairs = h->pair_clusters;
            *grid = static_cast<int>(2 * (total < pairs ? total : pairs));
        } else {
            *grid = static_cast<int>(total < h->sms ? total : h->sms);
        }
    }
    return GEMM_RS_OK;
}

int gemm_rs_get_shape(gemm_rs_t h, int64_t *M, int64_t *N, int64_t *K, int *W, int *y_dtype)
{
    if (h == nullptr)
        return fail(GEMM_RS_ERR_ARG, "handle is NULL");
    if (M)
        *M = h->M;
    if (N)
        *N = h->N;
    if (K)
        *K = h->K;
    if (W)
        *W = h->W;
    if (y_dtype)
        *y_dtype = h->y_dtype;
    return GEMM_RS_OK;
}

int gemm_rs_set_tile_n(gemm_rs_t h, int bn)
{
    if (h == nullptr)
        return fail(GEMM_RS_ERR_ARG, "handle is NULL");
    if (bn != 64 && bn != 128 && bn != 256)
        return fail(GEMM_RS_ERR_ARG, "tile width %d is not 64, 128 or 256", bn);
    h->bm = gemm_rs::kBM;
    h->bn = bn;
    return GEMM_RS_OK;
}

int gemm_rs_set_tile(gemm_rs_t h, int bm, int bn)
{
    if (h == nullptr)
        return fail(GEMM_RS_ERR_ARG, "handle is NULL");
    const bool single = bm == gemm_rs::kBM && (bn == 64 || bn == 128 || bn == 256);
    const bool pair = bm == 2 * gemm_rs::kBM && bn == 256;
    if (!single && !pair)
        return fail(GEMM_RS_ERR_ARG, "tile %dx%d is not 128x{64,128,256} or 256x256", bm, bn);
    h->bm = bm;
    h->bn = bn;
    return GEMM_RS_OK;
}

int gemm_rs_set_schedule(gemm_rs_t h, int colgroup, int rowgroup, int rank_order)
{
    if (h == nullptr)
        return fail(GEMM_RS_ERR_ARG, "handle is NULL");
    if (colgroup < 0 || rowgroup < 0)
        return fail(GEMM_RS_ERR_ARG, "column group %d / row group %d is negative", colgroup,
                    rowgroup);
    if (rank_order < GEMM_RS_RANKS_DEFAULT || rank_order > GEMM_RS_RANKS_INTERLEAVED)
        return fail(GEMM_RS_ERR_ARG, "unknown rank order %d", rank_order);
    h->colgroup = colgroup;
    h->rowgroup = rowgroup;
    h->rank_order = rank_order;
    return GEMM_RS_OK;
}

int gemm_rs_set_reduce_mode(gemm_rs_t h, int mode)
{
    if (h == nullptr)
        return fail(GEMM_RS_ERR_ARG, "handle is NULL");
    if (mode != GEMM_RS_REDUCE_CHAIN && mode != GEMM_RS_REDUCE_LAST_ARRIVER &&
        mode != GEMM_RS_REDUCE_TWO_LEVEL)
        return fail(GEMM_RS_ERR_ARG, "unknown reduce mode %d", mode);
    h->reduce_mode = mode;
    return GEMM_RS_OK;
}

int gemm_rs_set_timeout_cycles(gemm_rs_t h, uint64_t cycles)
{
    if (h == nullptr)
        return fail(GEMM_RS_ERR_ARG, "handle is NULL");
    if (cycles == 0)
        return fail(GEMM_RS_ERR_ARG, "timeout must be positive");
    h->timeout = cycles;
    return GEMM_RS_OK;
}

int gemm_rs_set_debug(gemm_rs_t h, int32_t *record, int flags)
{
    if (h == nullptr)
        return fail(GEMM_RS_ERR_ARG, "handle is NULL");
    if (flags & ~(GEMM_RS_DEBUG_STALL_PRODUCER | GEMM_RS_DEBUG_SKIP_READY))
        return fail(GEMM_RS_ERR_ARG, "unknown debug flags 0x%x", flags);
    if (record != nullptr && !aligned(record, 16))
        return fail(GEMM_RS_ERR_ALIGN, "record buffer must be 16-byte aligned");
    h->record = record;
    h->debug_flags = flags;
    return GEMM_RS_OK;
}

} // extern "C"

namespace {

// One launch of the fused kernel for gemm_rs_run and gemm_rs_run_streamed.
// ready: NULL, or the ready words the kernel waits on before it reads the
// inputs (rank r's A_r and B_r, then C), which reach `epoch` when they land.
int run_impl(gemm_rs_t h, const void *A, const void *B, const void *C, void *Y,
             gemm_rs_stream_t stream, const uint32_t *ready, uint32_t epoch)
{
    if (h == nullptr)
        return fail(GEMM_RS_ERR_ARG, "handle is NULL");
    if (h->M == 0 || h->N == 0)
        return GEMM_RS_OK;
    if (Y == nullptr)
        return fail(GEMM_RS_ERR_ARG, "Y is NULL");
    if (!aligned(Y, 16))
        return fail(GEMM_RS_ERR_ALIGN, "Y must be 16-byte aligned");
    if (h->beta != 0.0f) {
        if (C == nullptr)
            return fail(GEMM_RS_ERR_ARG, "C is NULL but beta != 0");
        if (!aligned(C, 16))
            return fail(GEMM_RS_ERR_ALIGN, "C must be 16-byte aligned");
    }
    if (h->Kpr > 0) {
        if (A == nullptr || B == nullptr)
            return fail(GEMM_RS_ERR_ARG, "A or B is NULL");
        if (!aligned(A, 16) || !aligned(B, 16))
            return fail(GEMM_RS_ERR_ALIGN, "A and B must be 16-byte aligned");
        int rc;
        if (A != h->tmA_ptr) {
            // A: [W][M][K/W] -> dims {K/W, M, W}, box {64, 128, 1}
            if ((rc = encode_3d(&h->tmA, A, h->Kpr, h->M, h->W, gemm_rs::kBK, gemm_rs::kBM)) != GEMM_RS_OK)
                return rc;
            h->tmA_ptr = A;
        }
        // B: [W][K/W][N] as 4D {64, K/W, N/64, W} with one box per stage (the
        // CTA's 64-column atoms: BN/64, or 2 for a CTA of a 256-column pair
        // tile), or as 3D {N, K/W, W} with 64x64 boxes when N % 64 != 0
        const int atoms = h->bm == 2 * gemm_rs::kBM ? 2 : h->bn / 64;
        if (B != h->tmB_ptr || atoms != h->tmB_atoms) {
            h->tmB_ptr = nullptr;
            if ((rc = encode_b(&h->tmB, B, h->N, h->Kpr, h->W, atoms, &h->tmB_4d)) != GEMM_RS_OK)
                return rc;
            h->tmB_ptr = B;
            h->tmB_atoms = atoms;
        }
    }
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return cuda_fail(e, "cudaGetDevice");
    if (dev != h->device)
        return fail(GEMM_RS_ERR_ARG, "handle was created on device %d, current device is %d",
                    h->device, dev);

    gemm_rs::KernelArgs a{};
    a.W = h->W;
    a.M = static_cast<int>(h->M);
    a.N = static_cast<int>(h->N);
    a.nM = static_cast<int>(cdiv(h->M, gemm_rs::kBM));
    a.nN = static_cast<int>(cdiv(h->N, h->bn));
    a.nK = static_cast<int>(cdiv(h->Kpr, gemm_rs::kBK));
    a.nMs = static_cast<int>(cdiv(h->M, h->bm));
    a.colgroup = colgroup_of(h);
    a.rowgroup = rowgroup_of(h);
    a.chain = h->reduce_mode != GEMM_RS_REDUCE_LAST_ARRIVER ? 1 : 0;
    // two groups of ranks, [0, ceil(W/2)) and [ceil(W/2), W)
    a.split = (h->reduce_mode == GEMM_RS_REDUCE_TWO_LEVEL && h->W > 1) ? (h->W + 1) / 2 : 0;
    a.seq = sequential(h) ? 1 : 0;
    // Sequential ranks reach a tile a rank's pass apart, and a single row tile
    // brings all positions at once: neither gains from waiting for a turn.
    a.chain_wait = (!a.seq && a.nMs > 1) ? 16384 : 0;
    a.R = h->M / h->W;
    a.total = static_cast<int64_t>(h->W) * a.nMs * a.nN;
    a.alpha = h->alpha;
    a.beta = h->beta;
    a.C = h->beta != 0.0f ? static_cast<const uint16_t *>(C) : nullptr;
    a.Y = Y;
    a.y_fp32 = h->y_dtype == GEMM_RS_FP32 ? 1 : 0;
    a.part = reinterpret_cast<float *>(h->ws + h->L.part_off);
    a.flags = reinterpret_cast<uint32_t *>(h->ws + h->L.flags_off);
    a.part_floats = static_cast<int64_t>(h->L.part_bytes / sizeof(float));
    a.nflags = static_cast<int64_t>(h->L.flags_bytes / sizeof(uint32_t));
    a.status = reinterpret_cast<uint32_t *>(h->ws);
    a.record = h->record;
    a.timeout = h->timeout;
    a.stall_producer = (h->debug_flags & GEMM_RS_DEBUG_STALL_PRODUCER) ? 1 : 0;
    a.b4d = h->Kpr > 0 ? h->tmB_4d : 0;
    a.ready = ready;
    a.epoch = epoch;

    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (h->bm == 2 * gemm_rs::kBM) {
        const int64_t pairs = h->pair_clusters;
        const int grid = static_cast<int>(2 * (a.total < pairs ? a.total : pairs));
        e = launch_overlapped(gemm_rs::gemm_rs_pair_kernel<256>, grid,
                              gemm_rs::smem_bytes_pair<256>(), s, h->tmA, h->tmB, a);
        if (e != cudaSuccess)
            return cuda_fail(e, "launch of the fused GEMM+RS pair kernel");
        return GEMM_RS_OK;
    }
    const int grid = static_cast<int>(a.total < h->sms ? a.total : h->sms);
    switch (h->bn) {
    case 256:
        e = launch_overlapped(gemm_rs::gemm_rs_fused_kernel<256>, grid, gemm_rs::smem_bytes<256>(), s,
                              h->tmA, h->tmB, a);
        break;
    case 128:
        e = launch_overlapped(gemm_rs::gemm_rs_fused_kernel<128>, grid, gemm_rs::smem_bytes<128>(), s,
                              h->tmA, h->tmB, a);
        break;
    default:
        e = launch_overlapped(gemm_rs::gemm_rs_fused_kernel<64>, grid, gemm_rs::smem_bytes<64>(), s,
                              h->tmA, h->tmB, a);
        break;
    }
    if (e != cudaSuccess)
        return cuda_fail(e, "launch of the fused GEMM+RS kernel");
    return GEMM_RS_OK;
}

// Ready words of the streamed call: 32-bit words inside the workspace's
// 256-byte status block, from byte 128 (W <= 16 ranks and C: at most 68 bytes).
constexpr size_t kReadyOff = 128;

using WriteValue32 = CUresult (*)(CUstream, CUdeviceptr, cuuint32_t, unsigned int);

// cuStreamWriteValue32 from the driver, looked up once.
int get_write_value(WriteValue32 *out)
{
    static WriteValue32 fn = nullptr;
    if (fn == nullptr) {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        cudaError_t e = cudaGetDriverEntryPointByVersion("cuStreamWriteValue32", &p, 12000,
                                                         cudaEnableDefault, &q);
        if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || p == nullptr)
            return fail(GEMM_RS_ERR_CUDA, "cuStreamWriteValue32 is not available from the driver");
        fn = reinterpret_cast<WriteValue32>(p);
    }
    *out = fn;
    return GEMM_RS_OK;
}

} // namespace

extern "C" {

int gemm_rs_run(gemm_rs_t h, const void *A, const void *B, const void *C, void *Y,
                gemm_rs_stream_t stream)
{
    return run_impl(h, A, B, C, Y, stream, nullptr, 0);
}

int gemm_rs_run_streamed(gemm_rs_t h, const void *A_host, const void *B_host, const void *C_host,
                         void *Y_host, void *A, void *B, void *C, void *Y, gemm_rs_stream_t stream,
                         gemm_rs_stream_t copy_stream)
{
    if (h == nullptr)
        return fail(GEMM_RS_ERR_ARG, "handle is NULL");
    if (copy_stream == nullptr || copy_stream == stream)
        return fail(GEMM_RS_ERR_ARG, "copy_stream must be a stream of its own, not stream or NULL");
    if (Y_host == nullptr || (h->Kpr > 0 && (A_host == nullptr || B_host == nullptr)) ||
        (h->beta != 0.0f && C_host == nullptr))
        return fail(GEMM_RS_ERR_ARG, "a host buffer is NULL");
    if (h->M == 0 || h->N == 0)
        return GEMM_RS_OK;
    if (Y == nullptr || (h->Kpr > 0 && (A == nullptr || B == nullptr)) ||
        (h->beta != 0.0f && C == nullptr))
        return fail(GEMM_RS_ERR_ARG, "a device buffer is NULL");
    WriteValue32 write_value;
    int rc = get_write_value(&write_value);
    if (rc != GEMM_RS_OK)
        return rc;
    cudaStream_t cs = reinterpret_cast<cudaStream_t>(copy_stream);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e;
    if (h->streamed_done == nullptr &&
        (e = cudaEventCreateWithFlags(&h->streamed_done, cudaEventDisableTiming)) != cudaSuccess)
        return cuda_fail(e, "cudaEventCreateWithFlags");
    // the previous streamed kernel of this handle no longer reads A, B and C
    if (h->streamed_pending && (e = cudaStreamWaitEvent(cs, h->streamed_done, 0)) != cudaSuccess)
        return cuda_fail(e, "cudaStreamWaitEvent(copy stream)");
    if (++h->stream_epoch == 0)
        h->stream_epoch = 1;
    const uint32_t epoch = h->stream_epoch;
    uint32_t *ready = reinterpret_cast<uint32_t *>(h->ws + kReadyOff);
    const bool skip = (h->debug_flags & GEMM_RS_DEBUG_SKIP_READY) != 0;
    auto mark = [&](int i) -> int {
        if (skip)
            return GEMM_RS_OK;
        const CUresult r = write_value(reinterpret_cast<CUstream>(cs),
                                       reinterpret_cast<CUdeviceptr>(ready + i), epoch, 0);
        return r == CUDA_SUCCESS ? GEMM_RS_OK
                                 : fail(GEMM_RS_ERR_CUDA, "cuStreamWriteValue32 failed (CUresult %d)",
                                        (int)r);
    };
    // C first (every rank's epilogue reads it), then rank by rank
    if (h->beta != 0.0f) {
        if ((e = cudaMemcpyAsync(C, C_host, static_cast<size_t>(h->M * h->N) * 2,
                                 cudaMemcpyHostToDevice, cs)) != cudaSuccess)
            return cuda_fail(e, "cudaMemcpyAsync(C)");
        if ((rc = mark(h->W)) != GEMM_RS_OK)
            return rc;
    }
    const size_t a_rank = static_cast<size_t>(h->M * h->Kpr) * 2;
    const size_t b_rank = static_cast<size_t>(h->Kpr * h->N) * 2;
    for (int r = 0; r < h->W; ++r) {
        if (h->Kpr > 0) {
            if ((e = cudaMemcpyAsync(static_cast<uint8_t *>(A) + r * a_rank,
                                     static_cast<const uint8_t *>(A_host) + r * a_rank, a_rank,
                                     cudaMemcpyHostToDevice, cs)) != cudaSuccess ||
                (e = cudaMemcpyAsync(static_cast<uint8_t *>(B) + r * b_rank,
                                     static_cast<const uint8_t *>(B_host) + r * b_rank, b_rank,
                                     cudaMemcpyHostToDevice, cs)) != cudaSuccess)
                return cuda_fail(e, "cudaMemcpyAsync(A_r, B_r)");
        }
        if ((rc = mark(r)) != GEMM_RS_OK)
            return rc;
    }
    if ((rc = run_impl(h, A, B, h->beta != 0.0f ? C : nullptr, Y, stream, ready, epoch)) != GEMM_RS_OK)
        return rc;
    if ((e = cudaEventRecord(h->streamed_done, s)) != cudaSuccess)
        return cuda_fail(e, "cudaEventRecord");
    h->streamed_pending = true;
    const size_t y_bytes = static_cast<size_t>(h->M * h->N) * (h->y_dtype == GEMM_RS_FP32 ? 4 : 2);
    if ((e = cudaMemcpyAsync(Y_host, Y, y_bytes, cudaMemcpyDeviceToHost, s)) != cudaSuccess)
        return cuda_fail(e, "cudaMemcpyAsync(Y)");
    return GEMM_RS_OK;
}

int gemm_rs_status(gemm_rs_t h, gemm_rs_stream_t stream)
{
    if (h == nullptr)
        return fail(GEMM_RS_ERR_ARG, "handle is NULL");
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    uint32_t word = 0;
    cudaError_t e = cudaMemcpyAsync(&word, h->ws, sizeof word, cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess)
        e = cudaStreamSynchronize(s);
    if (e != cudaSuccess)
        return cuda_fail(e, "reading the status word");
    if (word == 0)
        return GEMM_RS_OK;
    e = cudaMemsetAsync(h->ws, 0, sizeof word, s);
    if (e == cudaSuccess)
        e = cudaStreamSynchronize(s);
    if (e != cudaSuccess)
        return cuda_fail(e, "clearing the status word");
    return status_word_error(word);
}

int gemm_rs_reset(gemm_rs_t h, gemm_rs_stream_t stream)
{
    if (h == nullptr)
        return fail(GEMM_RS_ERR_ARG, "handle is NULL");
    cudaError_t e = cudaMemsetAsync(h->ws, 0, h->L.part_off, reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess)
        return cuda_fail(e, "cudaMemsetAsync(status and tile counters)");
    return GEMM_RS_OK;
}

int64_t gemm_rs_schedule(int64_t M, int64_t N, int W, int bm, int bn, int colgroup, int rowgroup,
                         int rank_order, int32_t *out, int64_t cap)
{
    if (W < 1 || W > 16)
        return fail(GEMM_RS_ERR_ARG, "W = %d is outside 1..16", W);
    if (M < 1 || N < 1 || M % W != 0)
        return fail(GEMM_RS_ERR_SHAPE, "need M, N >= 1 and M %% W == 0");
    if ((bm != gemm_rs::kBM && bm != 2 * gemm_rs::kBM) || (bn != 64 && bn != 128 && bn != 256))
        return fail(GEMM_RS_ERR_ARG, "tile %dx%d is not a tile of this library", bm, bn);
    if (out == nullptr)
        return fail(GEMM_RS_ERR_ARG, "out is NULL");
    if (colgroup < 0 || rowgroup < 0)
        return fail(GEMM_RS_ERR_ARG, "column group %d / row group %d is negative", colgroup,
                    rowgroup);
    if (rank_order < GEMM_RS_RANKS_DEFAULT || rank_order > GEMM_RS_RANKS_INTERLEAVED)
        return fail(GEMM_RS_ERR_ARG, "unknown rank order %d", rank_order);
    const int nN = static_cast<int>(cdiv(N, bn));
    const int nMs = static_cast<int>(cdiv(M, bm));
    const gemm_rs::Sched s{W, nMs, nN, bm == gemm_rs::kBM ? 7 : 8, M / W,
                           (colgroup == 0 || colgroup > nN) ? nN : colgroup,
                           rowgroup == 0 ? nMs : rowgroup,
                           rank_order == GEMM_RS_RANKS_INTERLEAVED ? 0 : 1};
    const int64_t total = static_cast<int64_t>(W) * s.nM * s.nN;
    if (cap < total)
        return fail(GEMM_RS_ERR_SHAPE, "cap %lld < %lld entries", (long long)cap, (long long)total);
    for (int64_t g = 0; g < total; ++g) {
        int r, mt, nt;
        gemm_rs::decode_tile(s, g, r, mt, nt);
        out[3 * g] = r;
        out[3 * g + 1] = mt;
        out[3 * g + 2] = nt;
    }
    return total;
}

int gemm_rs_reduce_partials(const void *partials, gemm_rs_dtype partial_dtype, const void *C,
                            void *Y, int64_t M, int64_t N, int W, float alpha, float beta,
                            gemm_rs_dtype y_dtype, gemm_rs_stream_t stream)
{
    if (W < 1 || W > 16)
        return fail(GEMM_RS_ERR_ARG, "W = %d is outside 1..16", W);
    if (M < 0 || N < 0 || N % 8 != 0)
        return fail(GEMM_RS_ERR_SHAPE, "need M, N >= 0 and N %% 8 == 0");
    if ((partial_dtype != GEMM_RS_BF16 && partial_dtype != GEMM_RS_FP32) ||
        (y_dtype != GEMM_RS_BF16 && y_dtype != GEMM_RS_FP32))
        return fail(GEMM_RS_ERR_UNSUPPORTED, "unknown dtype");
    if (M == 0 || N == 0)
        return GEMM_RS_OK;
    if (partials == nullptr || Y == nullptr || (beta != 0.0f && C == nullptr))
        return fail(GEMM_RS_ERR_ARG, "NULL partials, Y, or C with beta != 0");
    if (!aligned(partials, 16) || !aligned(Y, 16) || (beta != 0.0f && !aligned(C, 16)))
        return fail(GEMM_RS_ERR_ALIGN, "pointers must be 16-byte aligned");
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess)
        e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess)
        return cuda_fail(e, "querying the device");
    gemm_rs::ReduceArgs a{partials, partial_dtype == GEMM_RS_BF16 ? 1 : 0,
                          beta != 0.0f ? static_cast<const uint16_t *>(C) : nullptr, Y,
                          y_dtype == GEMM_RS_FP32 ? 1 : 0, M, N, W, alpha, beta};
    const int64_t groups = M * (N / 8);
    int64_t blocks = (groups + 255) / 256;
    if (blocks > int64_t(sms) * 8)
        blocks = int64_t(sms) * 8;
    e = gemm_rs::launch_reduce_partials(a, static_cast<int>(blocks),
                                        reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess)
        return cuda_fail(e, "launch of the baseline reduce kernel");
    return GEMM_RS_OK;
}

} // extern "C"

// ------------------------------------------------------------------------------------------
// Entry point that allocates nothing: gemm_rs_run_noalloc.
//
// Some callers cannot call cudaMalloc and have no workspace to hand over.  Examples: a
// plugin inside a host application that owns every device allocation, or a
// latency-critical path where an allocation, which may synchronise the device, is not
// allowed.  For them, the fused kernel's scratch (status word, tile counters and fp32
// partial tiles) lives in the file-scope array below.  Every GPU that loads this library
// holds the array until the process exits.  The caller still passes A, B, C and Y.
namespace {

constexpr size_t kNoAllocScratchBytes = size_t(GEMM_RS_NOALLOC_SCRATCH_BYTES);
__device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];

// With the current context's set-up done: the device address of g_noalloc_scratch
// in that context.  In host code the array's name is only a host-side stand-in,
// so the address comes from cudaGetSymbolAddress, looked up on every call (it
// allocates nothing, and a cached address could belong to another context).
int noalloc_device(int *dev_out, uint8_t **scratch_out, int *sms_out)
{
    int dev = 0, sms = 0;
    int rc = prepare_device(&dev, &sms);
    if (rc != GEMM_RS_OK)
        return rc;
    void *p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess)
        return cuda_fail(e, "cudaGetSymbolAddress(static scratch)");
    if (!aligned(p, 256))
        return fail(GEMM_RS_ERR_ALIGN, "static scratch is not 256-byte aligned");
    *dev_out = dev;
    *scratch_out = static_cast<uint8_t *>(p);
    *sms_out = sms;
    return GEMM_RS_OK;
}

} // namespace

extern "C" int gemm_rs_run_noalloc(int64_t M, int64_t N, int64_t K, int W, float alpha, float beta,
                                   gemm_rs_dtype y_dtype, const void *A, const void *B,
                                   const void *C, void *Y, gemm_rs_stream_t stream)
{
    int rc = check_shape(M, N, K, W);
    if (rc != GEMM_RS_OK)
        return rc;
    if (y_dtype != GEMM_RS_BF16 && y_dtype != GEMM_RS_FP32)
        return fail(GEMM_RS_ERR_UNSUPPORTED, "Y dtype must be GEMM_RS_BF16 or GEMM_RS_FP32");
    if (!(alpha == alpha) || !(beta == beta))
        return fail(GEMM_RS_ERR_ARG, "alpha and beta must not be NaN");
    const Layout L = layout_for(M, N, W);
    if (L.total > kNoAllocScratchBytes)
        return fail(GEMM_RS_ERR_WORKSPACE,
                    "this shape needs %zu bytes of scratch; the static scratch of "
                    "gemm_rs_run_noalloc holds %zu (use gemm_rs_create with a workspace)",
                    L.total, kNoAllocScratchBytes);
    if (M == 0 || N == 0)
        return GEMM_RS_OK;
    if (Y == nullptr)
        return fail(GEMM_RS_ERR_ARG, "Y is NULL");
    if (!aligned(Y, 16))
        return fail(GEMM_RS_ERR_ALIGN, "Y must be 16-byte aligned");
    if (beta != 0.0f && (C == nullptr || !aligned(C, 16)))
        return fail(C == nullptr ? GEMM_RS_ERR_ARG : GEMM_RS_ERR_ALIGN,
                    "C must be non-NULL and 16-byte aligned when beta != 0");
    const int64_t Kpr = K / W;
    CUtensorMap tmA, tmB;
    std::memset(&tmA, 0, sizeof tmA);
    std::memset(&tmB, 0, sizeof tmB);
    if (Kpr > 0) {
        if (A == nullptr || B == nullptr)
            return fail(GEMM_RS_ERR_ARG, "A or B is NULL");
        if (!aligned(A, 16) || !aligned(B, 16))
            return fail(GEMM_RS_ERR_ALIGN, "A and B must be 16-byte aligned");
        if ((rc = encode_3d(&tmA, A, Kpr, M, W, gemm_rs::kBK, gemm_rs::kBM)) != GEMM_RS_OK)
            return rc;
    }
    int dev = 0, sms = 0;
    uint8_t *scratch = nullptr;
    if ((rc = noalloc_device(&dev, &scratch, &sms)) != GEMM_RS_OK)
        return rc;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    // The array keeps the previous call's contents: the status word and the tile
    // counters must start at zero.  The partial slots need no clearing, because every
    // slot a call reads is written earlier in the same call.
    cudaError_t e = cudaMemsetAsync(scratch, 0, L.part_off, s);
    if (e != cudaSuccess)
        return cuda_fail(e, "cudaMemsetAsync(static scratch counters)");

    const int bn = pick_bn(M, N, W, sms);
    int b4d = 0;
    if (Kpr > 0 && (rc = encode_b(&tmB, B, N, Kpr, W, bn / 64, &b4d)) != GEMM_RS_OK)
        return rc;
    gemm_rs::KernelArgs a{};
    a.W = W;
    a.M = static_cast<int>(M);
    a.N = static_cast<int>(N);
    a.nM = static_cast<int>(cdiv(M, gemm_rs::kBM));
    a.nN = static_cast<int>(cdiv(N, bn));
    a.nK = static_cast<int>(cdiv(Kpr, gemm_rs::kBK));
    a.nMs = a.nM;
    a.colgroup = a.nN;
    a.rowgroup = a.nM;
    a.chain = 1;
    a.seq = 1;
    a.chain_wait = 0;
    a.split = 0;
    a.R = M / W;
    a.total = static_cast<int64_t>(W) * a.nM * a.nN;
    a.alpha = alpha;
    a.beta = beta;
    a.C = beta != 0.0f ? static_cast<const uint16_t *>(C) : nullptr;
    a.Y = Y;
    a.y_fp32 = y_dtype == GEMM_RS_FP32 ? 1 : 0;
    a.part = reinterpret_cast<float *>(scratch + L.part_off);
    a.flags = reinterpret_cast<uint32_t *>(scratch + L.flags_off);
    a.part_floats = static_cast<int64_t>(L.part_bytes / sizeof(float));
    a.nflags = static_cast<int64_t>(L.flags_bytes / sizeof(uint32_t));
    a.status = reinterpret_cast<uint32_t *>(scratch);
    a.record = nullptr;
    a.timeout = 1ull << 32;
    a.stall_producer = 0;
    a.b4d = b4d;
    const int grid = static_cast<int>(a.total < sms ? a.total : sms);
    switch (bn) {
    case 256:
        gemm_rs::gemm_rs_fused_kernel<256>
            <<<grid, gemm_rs::kThreads, gemm_rs::smem_bytes<256>(), s>>>(tmA, tmB, a);
        break;
    case 128:
        gemm_rs::gemm_rs_fused_kernel<128>
            <<<grid, gemm_rs::kThreads, gemm_rs::smem_bytes<128>(), s>>>(tmA, tmB, a);
        break;
    default:
        gemm_rs::gemm_rs_fused_kernel<64>
            <<<grid, gemm_rs::kThreads, gemm_rs::smem_bytes<64>(), s>>>(tmA, tmB, a);
        break;
    }
    e = cudaGetLastError();
    if (e != cudaSuccess)
        return cuda_fail(e, "launch of the fused GEMM+RS kernel (no-alloc entry point)");
    return GEMM_RS_OK;
}

extern "C" size_t gemm_rs_noalloc_scratch_bytes(void) { return kNoAllocScratchBytes; }

extern "C" int gemm_rs_noalloc_status(gemm_rs_stream_t stream)
{
    int dev = 0, sms = 0;
    uint8_t *scratch = nullptr;
    int rc = noalloc_device(&dev, &scratch, &sms);
    if (rc != GEMM_RS_OK)
        return rc;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    uint32_t word = 0;
    cudaError_t e = cudaMemcpyAsync(&word, scratch, sizeof word, cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess)
        e = cudaStreamSynchronize(s);
    if (e != cudaSuccess)
        return cuda_fail(e, "reading the static scratch's status word");
    if (word == 0)
        return GEMM_RS_OK;
    e = cudaMemsetAsync(scratch, 0, sizeof word, s);
    if (e == cudaSuccess)
        e = cudaStreamSynchronize(s);
    if (e != cudaSuccess)
        return cuda_fail(e, "clearing the static scratch's status word");
    return status_word_error(word);
}
