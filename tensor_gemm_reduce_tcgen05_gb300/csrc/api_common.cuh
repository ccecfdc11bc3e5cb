// Host helpers shared by the C ABI's translation units: the per-thread error
// message that gemm_rs_last_error returns, error codes from CUDA calls, and
// TMA descriptor encoding.  Host code only.
#pragma once

#include <cstdarg>
#include <cstdint>
#include <cstdio>
#include <cuda.h>
#include <cuda_runtime.h>
#include <mutex>
#include <string>

#include "gemm_rs.h"

namespace gemm_rs_host {

// The message for the last failing call on this thread (one object for the
// whole library: an inline variable).
inline thread_local std::string g_err;

inline int fail(int code, const char *fmt, ...)
{
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    g_err = buf;
    return code;
}

inline int cuda_fail(cudaError_t e, const char *what)
{
    return fail(GEMM_RS_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

inline size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

inline int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

inline bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

using EncodeTiled = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                 const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                 const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                 CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// cuTensorMapEncodeTiled from the driver, looked up once.
inline int get_encoder(EncodeTiled *out)
{
    static EncodeTiled fn = nullptr;
    if (fn == nullptr) {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                                         cudaEnableDefault, &q);
        if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || p == nullptr)
            return fail(GEMM_RS_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
        fn = reinterpret_cast<EncodeTiled>(p);
    }
    *out = fn;
    return GEMM_RS_OK;
}

// The calling thread's current CUDA context (a driver handle), for caches of
// per-context set-up.  cuCtxGetCurrent comes from the driver, looked up once.
inline int current_context(void **out)
{
    using GetCurrent = CUresult (*)(CUcontext *);
    static GetCurrent fn = nullptr;
    if (fn == nullptr) {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        cudaError_t e = cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000,
                                                         cudaEnableDefault, &q);
        if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || p == nullptr)
            return fail(GEMM_RS_ERR_CUDA, "cuCtxGetCurrent is not available from the driver");
        fn = reinterpret_cast<GetCurrent>(p);
    }
    CUcontext ctx = nullptr;
    const CUresult r = fn(&ctx);
    if (r != CUDA_SUCCESS || ctx == nullptr)
        return fail(GEMM_RS_ERR_CUDA, "no current CUDA context (CUresult %d)", (int)r);
    *out = ctx;
    return GEMM_RS_OK;
}

// Per-context set-up (kernel attributes, occupancy), keyed by the driver's
// context handle: a host application may run several contexts on one device,
// and each needs the kernels' attributes set in it.  A small table; when it
// is full the oldest entry is replaced.  Lookups hold the table's mutex.
template <typename T>
struct ContextCache {
    static constexpr int kEntries = 32;
    struct Entry {
        void *ctx = nullptr;
        T info{};
    };
    Entry e[kEntries];
    int next = 0;
    std::mutex mu;

    // The entry of the current context, set up by setup(T&) (an int-returning
    // callable) the first time; its return code is passed on.
    template <typename F>
    int get(T *out, F setup)
    {
        void *ctx = nullptr;
        int rc = current_context(&ctx);
        if (rc != GEMM_RS_OK)
            return rc;
        std::lock_guard<std::mutex> lock(mu);
        for (int i = 0; i < kEntries; ++i)
            if (e[i].ctx == ctx) {
                *out = e[i].info;
                return GEMM_RS_OK;
            }
        T info{};
        if ((rc = setup(info)) != GEMM_RS_OK)
            return rc;
        e[next].ctx = ctx;
        e[next].info = info;
        next = (next + 1) % kEntries;
        *out = info;
        return GEMM_RS_OK;
    }
};

// 3-D bf16 tensor map {d0, d1, d2} (d0 contiguous), box {b0, b1, 1}, 128-byte
// swizzle, zero fill outside the tensor.
inline int encode_3d(CUtensorMap *map, const void *ptr, uint64_t d0, uint64_t d1, uint64_t d2,
                     uint32_t b0, uint32_t b1)
{
    EncodeTiled enc;
    int rc = get_encoder(&enc);
    if (rc != GEMM_RS_OK)
        return rc;
    const cuuint64_t dims[3] = {d0, d1, d2};
    const cuuint64_t strides[2] = {d0 * 2, d0 * d1 * 2};
    const cuuint32_t box[3] = {b0, b1, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(ptr), dims, strides,
                     box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
        return fail(GEMM_RS_ERR_CUDA, "cuTensorMapEncodeTiled failed (CUresult %d)", (int)r);
    return GEMM_RS_OK;
}

// B [W][K/W][N] bf16 as a 4D tensor {64, K/W, N/64, W}: column n = 64*a + j
// is (j, a), so a box {64, 64, atoms, 1} is `atoms` consecutive 64-column
// swizzle atoms of one 64-row k-block, laid out one after another (each 64
// rows x 128 bytes, 128-byte swizzled), exactly as `atoms` 3D boxes would
// be.  Needs N % 64 == 0; a box past the last atom reads zeros.
inline int encode_b4d(CUtensorMap *map, const void *ptr, uint64_t N, uint64_t Kpr, uint64_t W,
                      uint32_t atoms)
{
    EncodeTiled enc;
    int rc = get_encoder(&enc);
    if (rc != GEMM_RS_OK)
        return rc;
    const cuuint64_t dims[4] = {64, Kpr, N / 64, W};
    const cuuint64_t strides[3] = {N * 2, 128, Kpr * N * 2};
    const cuuint32_t box[4] = {64, 64, atoms, 1};
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(ptr), dims, strides,
                     box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
        return fail(GEMM_RS_ERR_CUDA, "cuTensorMapEncodeTiled (4D B) failed (CUresult %d)", (int)r);
    return GEMM_RS_OK;
}

// The B tensor map of a launch: 4D with one box per stage when N is a
// multiple of 64 (atoms = the 64-column atoms a CTA loads per stage), else
// 3D with one 64-column box per atom.  Returns the `b4d` kernel argument
// through *b4d.
inline int encode_b(CUtensorMap *map, const void *ptr, uint64_t N, uint64_t Kpr, uint64_t W,
                    uint32_t atoms, int *b4d)
{
    if (N % 64 == 0) {
        *b4d = 1;
        return encode_b4d(map, ptr, N, Kpr, W, atoms);
    }
    *b4d = 0;
    return encode_3d(map, ptr, N, Kpr, W, 64, 64);
}

} // namespace gemm_rs_host
