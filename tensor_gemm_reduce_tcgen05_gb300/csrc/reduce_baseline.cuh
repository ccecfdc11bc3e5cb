// Declarations shared by the baseline reduce kernel and the C-ABI host code.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace gemm_rs {

struct ReduceArgs {
    const void *P;      // [W][M][N] partials, fp32 or bf16
    int p_bf16;
    const uint16_t *C;  // bf16 [M][N] or NULL when beta == 0
    void *Y;
    int y_fp32;
    int64_t M, N;
    int W;
    float alpha, beta;
};

cudaError_t launch_reduce_partials(const ReduceArgs &a, int blocks, cudaStream_t stream);

} // namespace gemm_rs
