// Host side of the AG+GEMM C ABI declared in include/ag_gemm.h: argument
// checks, the workspace layout, TMA descriptors, the plan and the cooperative
// launch.  Errors come back as codes; the message is kept per thread and read
// with gemm_rs_last_error().
#include <cstring>
#include <cuda.h>
#include <cuda_runtime.h>
#include <mutex>
#include <new>

#include "ag_gemm.h"
#include "ag_gemm_kernel.cuh"
#include "api_common.cuh"

namespace {

using namespace gemm_rs_host;

constexpr size_t kAgStatusBytes = 256;
constexpr int kAgTile = 256; // output tiles are 256 x 256 (CTA pairs)

struct AgLayout {
    size_t ready_off, g_off, total;
};

AgLayout ag_layout(int64_t M, int64_t K, int W)
{
    AgLayout L;
    L.ready_off = kAgStatusBytes;
    L.g_off = L.ready_off + round_up(static_cast<size_t>(W) * W * sizeof(uint32_t), 256);
    L.total = L.g_off + round_up(static_cast<size_t>(W) * M * K * 2, 256);
    return L;
}

int ag_check_shape(int64_t M, int64_t N, int64_t K, int W)
{
    if (W < 1 || W > 16)
        return fail(GEMM_RS_ERR_ARG, "W = %d is outside 1..16", W);
    if (M < 1 || N < 1 || K < 1)
        return fail(GEMM_RS_ERR_SHAPE, "M, N and K must be positive");
    if (M > (int64_t(1) << 30) || N > (int64_t(1) << 30) || K > (int64_t(1) << 30))
        return fail(GEMM_RS_ERR_SHAPE, "size above 2^30");
    if (M % (static_cast<int64_t>(kAgTile) * W) != 0)
        return fail(GEMM_RS_ERR_SHAPE,
                    "M = %lld is not a multiple of 256*W = %d (a 256-row tile must lie in one chunk)",
                    (long long)M, kAgTile * W);
    if (K % 8 != 0 || N % 8 != 0)
        return fail(GEMM_RS_ERR_SHAPE, "K and N must be multiples of 8 (16-byte TMA rows)");
    // the kernel decodes its work items in 32-bit arithmetic
    if (static_cast<int64_t>(W) * (M / kAgTile) * ((N + kAgTile - 1) / kAgTile) >= (int64_t(1) << 31))
        return fail(GEMM_RS_ERR_SHAPE, "more than 2^31 work items");
    return GEMM_RS_OK;
}

// Rows per copy slice: about 64 KB per slice, a power of two that divides the
// chunk (M/W is a multiple of 256).
int ag_slice_rows(int64_t K)
{
    int rows = 256;
    while (rows > 1 && static_cast<int64_t>(rows) * K * 2 > (int64_t(64) << 10))
        rows /= 2;
    return rows;
}

struct AgDevice {
    int dev = 0;
    int clusters = 0;
};
ContextCache<AgDevice> g_ag_dev;

// Once per CUDA context: check the device, set the kernel's shared-memory
// attribute and count the co-resident CTA pairs.
int ag_setup(AgDevice &d)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return cuda_fail(e, "cudaGetDevice");
    int major = 0, minor = 0;
    cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    if (major != 10 || minor != 3)
        return fail(GEMM_RS_ERR_UNSUPPORTED,
                    "device %d has compute capability %d.%d; this library is built for sm_103a", dev,
                    major, minor);
    int sms = 0;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
        return cuda_fail(e, "cudaDeviceGetAttribute(SM count)");
    if ((e = cudaFuncSetAttribute(gemm_rs::ag_gemm_pair_kernel<256>,
                                  cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  gemm_rs::smem_bytes_pair<256>())) != cudaSuccess)
        return cuda_fail(e, "cudaFuncSetAttribute(AG kernel shared memory)");
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * (sms / 2), 1, 1);
    cfg.blockDim = dim3(gemm_rs::kThreads, 1, 1);
    cfg.dynamicSmemBytes = gemm_rs::smem_bytes_pair<256>();
    int clusters = 0;
    if ((e = cudaOccupancyMaxActiveClusters(&clusters, gemm_rs::ag_gemm_pair_kernel<256>, &cfg)) !=
        cudaSuccess)
        return cuda_fail(e, "cudaOccupancyMaxActiveClusters(AG kernel)");
    d.dev = dev;
    d.clusters = clusters > 0 ? clusters : 1;
    return GEMM_RS_OK;
}

int ag_prepare(int *dev_out, int *clusters_out)
{
    AgDevice d;
    const int rc = g_ag_dev.get(&d, ag_setup);
    if (rc != GEMM_RS_OK)
        return rc;
    *dev_out = d.dev;
    *clusters_out = d.clusters;
    return GEMM_RS_OK;
}

} // namespace

struct ag_gemm_s {
    int64_t M, N, K;
    int W;
    float alpha;
    gemm_rs_dtype y_dtype;
    uint8_t *ws;
    AgLayout L;
    int device, clusters;
    int slice_rows, nslices;
    uint32_t epoch;
    CUtensorMap tmX, tmG, tmB;
    const void *tmX_ptr, *tmB_ptr;
    int tmB_4d; // B1's map is 4D (N % 64 == 0)
    unsigned long long timeout;
    int32_t *record;
    int debug_flags;
};

extern "C" {

size_t ag_gemm_workspace_bytes(int64_t M, int64_t N, int64_t K, int W)
{
    if (ag_check_shape(M, N, K, W) != GEMM_RS_OK)
        return 0;
    return ag_layout(M, K, W).total;
}

int ag_gemm_create(ag_gemm_t *out, int64_t M, int64_t N, int64_t K, int W, float alpha,
                   gemm_rs_dtype y_dtype, void *workspace, size_t workspace_bytes,
                   gemm_rs_stream_t stream)
{
    if (out == nullptr)
        return fail(GEMM_RS_ERR_ARG, "out is NULL");
    *out = nullptr;
    int rc = ag_check_shape(M, N, K, W);
    if (rc != GEMM_RS_OK)
        return rc;
    if (y_dtype != GEMM_RS_BF16 && y_dtype != GEMM_RS_FP32)
        return fail(GEMM_RS_ERR_UNSUPPORTED, "H dtype must be GEMM_RS_BF16 or GEMM_RS_FP32");
    if (!(alpha == alpha))
        return fail(GEMM_RS_ERR_ARG, "alpha must not be NaN");
    const AgLayout L = ag_layout(M, K, W);
    if (workspace == nullptr)
        return fail(GEMM_RS_ERR_ARG, "workspace is NULL");
    if (!aligned(workspace, 256))
        return fail(GEMM_RS_ERR_ALIGN, "workspace must be 256-byte aligned");
    if (workspace_bytes < L.total)
        return fail(GEMM_RS_ERR_WORKSPACE, "workspace of %zu bytes is below the %zu needed",
                    workspace_bytes, L.total);
    int dev = 0, clusters = 0;
    if ((rc = ag_prepare(&dev, &clusters)) != GEMM_RS_OK)
        return rc;
    cudaError_t e = cudaMemsetAsync(workspace, 0, L.g_off, reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess)
        return cuda_fail(e, "cudaMemsetAsync(status and chunk signals)");
    ag_gemm_s *h = new (std::nothrow) ag_gemm_s();
    if (h == nullptr)
        return fail(GEMM_RS_ERR_ARG, "out of host memory");
    h->M = M;
    h->N = N;
    h->K = K;
    h->W = W;
    h->alpha = alpha;
    h->y_dtype = y_dtype;
    h->ws = static_cast<uint8_t *>(workspace);
    h->L = L;
    h->device = dev;
    h->clusters = clusters;
    h->slice_rows = ag_slice_rows(K);
    h->nslices = static_cast<int>(M / W / h->slice_rows);
    h->epoch = 0;
    h->tmX_ptr = h->tmB_ptr = nullptr;
    h->tmB_4d = 0;
    h->timeout = 1ull << 32;
    h->record = nullptr;
    h->debug_flags = 0;
    // The gather buffers live in the workspace: G = [W][M][K], box {64, 128, 1}.
    if ((rc = encode_3d(&h->tmG, h->ws + L.g_off, static_cast<uint64_t>(K), static_cast<uint64_t>(M),
                        static_cast<uint64_t>(W), gemm_rs::kBK, gemm_rs::kBM)) != GEMM_RS_OK) {
        delete h;
        return rc;
    }
    *out = h;
    return GEMM_RS_OK;
}

int ag_gemm_run(ag_gemm_t h, const void *X, const void *B1, void *H, gemm_rs_stream_t stream)
{
    if (h == nullptr)
        return fail(GEMM_RS_ERR_ARG, "handle is NULL");
    if (X == nullptr || B1 == nullptr || H == nullptr)
        return fail(GEMM_RS_ERR_ARG, "X, B1 and H must not be NULL");
    if (!aligned(X, 16) || !aligned(B1, 16) || !aligned(H, 16))
        return fail(GEMM_RS_ERR_ALIGN, "X, B1 and H must be 16-byte aligned");
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return cuda_fail(e, "cudaGetDevice");
    if (dev != h->device)
        return fail(GEMM_RS_ERR_ARG, "handle was created on device %d, current device is %d",
                    h->device, dev);
    int rc;
    if (X != h->tmX_ptr) {
        // X: [M][K] as a 3-D map {K, M, 1}, box {64, 128, 1}
        if ((rc = encode_3d(&h->tmX, X, static_cast<uint64_t>(h->K), static_cast<uint64_t>(h->M), 1,
                            gemm_rs::kBK, gemm_rs::kBM)) != GEMM_RS_OK)
            return rc;
        h->tmX_ptr = X;
    }
    if (B1 != h->tmB_ptr) {
        // B1: [W][K][N] as 4D {64, K, N/64, W} with one box of a CTA's two
        // 64-column atoms per stage, or 3D {N, K, W} with 64x64 boxes when
        // N % 64 != 0
        h->tmB_ptr = nullptr;
        if ((rc = encode_b(&h->tmB, B1, static_cast<uint64_t>(h->N), static_cast<uint64_t>(h->K),
                           static_cast<uint64_t>(h->W), 2, &h->tmB_4d)) != GEMM_RS_OK)
            return rc;
        h->tmB_ptr = B1;
    }

    gemm_rs::AgArgs a;
    a.W = h->W;
    a.M = static_cast<int>(h->M);
    a.N = static_cast<int>(h->N);
    a.K = static_cast<int>(h->K);
    a.nK = static_cast<int>(cdiv(h->K, gemm_rs::kBK));
    a.nMs = static_cast<int>(h->M / kAgTile);
    a.nN = static_cast<int>(cdiv(h->N, kAgTile));
    a.R = static_cast<int>(h->M / h->W);
    a.cntp = a.R / kAgTile;
    a.total = static_cast<int64_t>(h->W) * a.nMs * a.nN;
    a.alpha = h->alpha;
    a.H = H;
    a.y_fp32 = h->y_dtype == GEMM_RS_FP32 ? 1 : 0;
    a.X = static_cast<const uint16_t *>(X);
    a.G = reinterpret_cast<uint16_t *>(h->ws + h->L.g_off);
    a.ready = reinterpret_cast<uint32_t *>(h->ws + h->L.ready_off);
    a.status = reinterpret_cast<uint32_t *>(h->ws);
    a.record = h->record;
    a.slice_rows = h->slice_rows;
    a.nslices = h->nslices;
    a.epoch = ++h->epoch;
    a.timeout = h->timeout;
    a.skip_copies = (h->debug_flags & AG_GEMM_DEBUG_SKIP_COPIES) ? 1 : 0;
    a.b4d = h->tmB_4d;

    const int64_t pairs = h->clusters;
    const int grid = static_cast<int>(2 * (a.total < pairs ? a.total : pairs));
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
    cfg.blockDim = dim3(gemm_rs::kThreads, 1, 1);
    cfg.dynamicSmemBytes = gemm_rs::smem_bytes_pair<256>();
    cfg.stream = reinterpret_cast<cudaStream_t>(stream);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative; // every CTA resident: they wait on each other's copies
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, gemm_rs::ag_gemm_pair_kernel<256>, h->tmX, h->tmG, h->tmB, a);
    if (e != cudaSuccess) {
        --h->epoch;
        return cuda_fail(e, "launch of the AG+GEMM kernel");
    }
    return GEMM_RS_OK;
}

int ag_gemm_status(ag_gemm_t h, gemm_rs_stream_t stream)
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
    if (word == gemm_rs::kStatusOutOfBounds)
        return fail(GEMM_RS_ERR_BOUNDS,
                    "checked build: an access outside its buffer was caught and skipped");
    return fail(GEMM_RS_ERR_TIMEOUT, "device wait timed out in the AG+GEMM kernel (status %u)", word);
}

int ag_gemm_reset(ag_gemm_t h, gemm_rs_stream_t stream)
{
    if (h == nullptr)
        return fail(GEMM_RS_ERR_ARG, "handle is NULL");
    cudaError_t e = cudaMemsetAsync(h->ws, 0, h->L.g_off, reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess)
        return cuda_fail(e, "cudaMemsetAsync(status and chunk signals)");
    h->epoch = 0;
    return GEMM_RS_OK;
}

int ag_gemm_destroy(ag_gemm_t h)
{
    delete h;
    return GEMM_RS_OK;
}

int64_t ag_gemm_schedule(int64_t M, int64_t N, int W, int32_t *out, int64_t cap)
{
    int rc = ag_check_shape(M, N, 8, W);
    if (rc != GEMM_RS_OK)
        return rc;
    if (out == nullptr)
        return fail(GEMM_RS_ERR_ARG, "out is NULL");
    gemm_rs::AgArgs a = {};
    a.W = W;
    a.nMs = static_cast<int>(M / kAgTile);
    a.nN = static_cast<int>(cdiv(N, kAgTile));
    a.R = static_cast<int>(M / W);
    a.cntp = a.R / kAgTile;
    a.total = static_cast<int64_t>(W) * a.nMs * a.nN;
    if (cap < a.total)
        return fail(GEMM_RS_ERR_SHAPE, "cap %lld < %lld entries", (long long)cap, (long long)a.total);
    for (int64_t g = 0; g < a.total; ++g) {
        int r, mt2, nt, c;
        gemm_rs::ag_decode(a, g, r, mt2, nt, c);
        out[3 * g] = r;
        out[3 * g + 1] = mt2;
        out[3 * g + 2] = nt;
    }
    return a.total;
}

int ag_gemm_get_plan(ag_gemm_t h, int *grid, int *stages, int *slice_rows, int *slices)
{
    if (h == nullptr)
        return fail(GEMM_RS_ERR_ARG, "handle is NULL");
    const int64_t total = static_cast<int64_t>(h->W) * (h->M / kAgTile) * cdiv(h->N, kAgTile);
    if (grid)
        *grid = static_cast<int>(2 * (total < h->clusters ? total : h->clusters));
    if (stages)
        *stages = gemm_rs::PairCfg<256>::kStages;
    if (slice_rows)
        *slice_rows = h->slice_rows;
    if (slices)
        *slices = h->nslices;
    return GEMM_RS_OK;
}

int ag_gemm_set_timeout_cycles(ag_gemm_t h, uint64_t cycles)
{
    if (h == nullptr)
        return fail(GEMM_RS_ERR_ARG, "handle is NULL");
    if (cycles == 0)
        return fail(GEMM_RS_ERR_ARG, "the wait limit must be positive");
    h->timeout = cycles;
    return GEMM_RS_OK;
}

int ag_gemm_set_debug(ag_gemm_t h, int32_t *record, int flags)
{
    if (h == nullptr)
        return fail(GEMM_RS_ERR_ARG, "handle is NULL");
    if (flags & ~AG_GEMM_DEBUG_SKIP_COPIES)
        return fail(GEMM_RS_ERR_ARG, "unknown debug flags 0x%x", flags);
    h->record = record;
    h->debug_flags = flags;
    return GEMM_RS_OK;
}

int ag_gemm_get_shape(ag_gemm_t h, int64_t *M, int64_t *N, int64_t *K, int *W, int *y_dtype)
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

int ffn_tp_run(ag_gemm_t ag, gemm_rs_t rs, const void *X, const void *B1, void *H, const void *B2,
               const void *C, void *Y, gemm_rs_stream_t stream)
{
    if (ag == nullptr || rs == nullptr)
        return fail(GEMM_RS_ERR_ARG, "both handles are needed");
    int64_t rM = 0, rK = 0;
    int rW = 0;
    int rc = gemm_rs_get_shape(rs, &rM, nullptr, &rK, &rW, nullptr);
    if (rc != GEMM_RS_OK)
        return rc;
    if (ag->y_dtype != GEMM_RS_BF16)
        return fail(GEMM_RS_ERR_UNSUPPORTED, "the AG+GEMM output feeds the GEMM+RS: it must be bf16");
    if (rM != ag->M || rW != ag->W || rK != static_cast<int64_t>(ag->W) * ag->N)
        return fail(GEMM_RS_ERR_SHAPE,
                    "GEMM+RS shape (M=%lld, K=%lld, W=%d) does not continue the AG+GEMM "
                    "(M=%lld, N=%lld per rank, W=%d)",
                    (long long)rM, (long long)rK, rW, (long long)ag->M, (long long)ag->N, ag->W);
    if ((rc = ag_gemm_run(ag, X, B1, H, stream)) != GEMM_RS_OK)
        return rc;
    return gemm_rs_run(rs, H, B2, C, Y, stream);
}

} // extern "C"
