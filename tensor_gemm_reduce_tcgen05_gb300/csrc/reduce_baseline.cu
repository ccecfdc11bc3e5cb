// The separate reduce step of the UNFUSED GEMM+RS baseline.  It runs after W
// per-rank GEMMs have written full [M][N] partials.  This is the
// "GEMM, then a collective" arrangement that tile-level fusion replaces
// ("flux精读" §2 Motivation; "通信 overlap 实现", section "Flux 的 tile
// 级融合解决了什么？").  It is used only to measure that baseline.  The
// fused path does not call it.
//
// Y[m, n] = fold over r in rank order of fp32(alpha * P_r[m, n] + beta * C[m, n]).
// Each thread handles 8 consecutive columns.  The grid is a multiple of the
// SM count and strides over the output.  The kernel is bound by HBM bandwidth.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cstdint>

#include "reduce_baseline.cuh"

namespace gemm_rs {
namespace {

__device__ __forceinline__ void load8(const ReduceArgs &a, int64_t off, float (&v)[8])
{
    if (a.p_bf16) {
        const uint4 u = __ldcs(reinterpret_cast<const uint4 *>(static_cast<const uint16_t *>(a.P) + off));
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            v[2 * e] = __uint_as_float(w[e] << 16);
            v[2 * e + 1] = __uint_as_float(w[e] & 0xffff0000u);
        }
    } else {
        const float4 *p = reinterpret_cast<const float4 *>(static_cast<const float *>(a.P) + off);
        const float4 x = __ldcs(p), y = __ldcs(p + 1);
        v[0] = x.x; v[1] = x.y; v[2] = x.z; v[3] = x.w;
        v[4] = y.x; v[5] = y.y; v[6] = y.z; v[7] = y.w;
    }
}

__global__ void __launch_bounds__(256) reduce_partials_kernel(const ReduceArgs a)
{
    const int64_t groups = a.M * (a.N / 8);
    const int64_t plane = a.M * a.N;
    for (int64_t gi = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; gi < groups;
         gi += int64_t(gridDim.x) * blockDim.x) {
        const int64_t off = gi * 8;
        float c[8] = {0, 0, 0, 0, 0, 0, 0, 0};
        if (a.beta != 0.0f) {
            const uint4 u = __ldg(reinterpret_cast<const uint4 *>(a.C + off));
            const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                c[2 * e] = __uint_as_float(w[e] << 16);
                c[2 * e + 1] = __uint_as_float(w[e] & 0xffff0000u);
            }
        }
        float y[8];
        for (int r = 0; r < a.W; ++r) {
            float v[8];
            load8(a, r * plane + off, v);
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                float p = a.alpha * v[e];
                if (a.beta != 0.0f)
                    p = fmaf(a.beta, c[e], p);
                y[e] = (r == 0) ? p : y[e] + p;
            }
        }
        if (a.y_fp32) {
            float4 *yp = reinterpret_cast<float4 *>(static_cast<float *>(a.Y) + off);
            yp[0] = make_float4(y[0], y[1], y[2], y[3]);
            yp[1] = make_float4(y[4], y[5], y[6], y[7]);
        } else {
            uint4 w;
            __nv_bfloat162 h0 = __floats2bfloat162_rn(y[0], y[1]);
            __nv_bfloat162 h1 = __floats2bfloat162_rn(y[2], y[3]);
            __nv_bfloat162 h2 = __floats2bfloat162_rn(y[4], y[5]);
            __nv_bfloat162 h3 = __floats2bfloat162_rn(y[6], y[7]);
            w.x = *reinterpret_cast<uint32_t *>(&h0);
            w.y = *reinterpret_cast<uint32_t *>(&h1);
            w.z = *reinterpret_cast<uint32_t *>(&h2);
            w.w = *reinterpret_cast<uint32_t *>(&h3);
            *reinterpret_cast<uint4 *>(static_cast<uint16_t *>(a.Y) + off) = w;
        }
    }
}

} // namespace

cudaError_t launch_reduce_partials(const ReduceArgs &a, int blocks, cudaStream_t stream)
{
    reduce_partials_kernel<<<blocks, 256, 0, stream>>>(a);
    return cudaGetLastError();
}

} // namespace gemm_rs
