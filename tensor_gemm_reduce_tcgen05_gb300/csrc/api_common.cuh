// Host helpers shared by the C ABI's translation units: the per-thread error
// message that gemm_rs_last_error returns, error codes from CUDA calls, and
// TMA descriptor encoding.  Host code only.
#pragma once

#include <cstdarg>
#include <cstdint>
#include <cstdio>
#include <cuda.h>
#include <cuda_runtime.h>
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

} // namespace gemm_rs_host
