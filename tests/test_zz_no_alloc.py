"""The entry point that allocates nothing (gemm_rs_run_noalloc).

Some callers cannot call cudaMalloc and have no workspace to hand the
library.  Examples: a plugin whose host application owns every device
allocation, or a latency-critical path where an allocation is not allowed.
gemm_rs_run_noalloc serves them.  It runs the same fused kernel with its
scratch in a static device array of a fixed size.  This test calls it
through the C ABI, twice in a row, and checks each output against the
handle-based entry point (gemm_rs_create + gemm_rs_run) on the same inputs,
within the tolerances the other parity tests use.  Both paths run the same
kernel, so the outputs are also expected to match bit for bit.  It also checks
the claim in the name: once the first call has done its set-up, further calls
leave torch's allocator and the device's free memory where they were, and the
status query (which reads the scratch's status word) reports success.

This file is collected last on purpose.  It must pass both on its own in a
fresh process and after every other test.
"""
import numpy as np
import pytest
import torch

from helpers import assert_close, inputs, to_np_y

pytestmark = pytest.mark.gpu


def _y(M, N, y_dtype):
    Y = torch.empty((M, N), dtype=torch.bfloat16 if y_dtype == "bf16" else torch.float32,
                    device="cuda:0")
    Y.view(torch.uint8).fill_(0xFF)  # NaN: every element must be written
    return Y


@pytest.mark.parametrize("W,M,N,Kpr,alpha,beta,y_dtype", [
    (4, 512, 520, 200, 0.5, 1.0, "bf16"),   # ragged N and K, bias-like C
    (8, 64, 1024, 192, 1.0, 0.0, "fp32"),   # 8-row chunks inside one row tile
])
def test_noalloc_matches_handle_path_on_two_calls_in_a_row(W, M, N, Kpr, alpha, beta, y_dtype):
    from tensor_gemm_reduce_tcgen05_gb300 import binding as b
    A, B, C = inputs(W, M, N, Kpr, "normal", c_dist="normal1" if beta != 0 else None)
    dev = torch.device("cuda", 0)
    Ad, Bd = A.to(dev), B.to(dev)
    Cd = None if C is None else C.to(dev)
    K = W * Kpr
    assert b.gemm_rs_workspace_bytes(M, N, K, W) <= b.gemm_rs_noalloc_scratch_bytes()

    op = b.GemmRS(M, N, K, W, alpha, beta, y_dtype, device=dev)
    ref = to_np_y(op.run(Ad, Bd, Cd))
    torch.cuda.synchronize()
    assert op.status() == 0

    code = b.GEMM_RS_BF16 if y_dtype == "bf16" else b.GEMM_RS_FP32
    stream = torch.cuda.current_stream(dev).cuda_stream
    Ys = [_y(M, N, y_dtype) for _ in range(2)]
    torch.cuda.synchronize()
    for call in range(2):
        Y = Ys[call]
        if call == 1:
            # the first call did the set-up; from here on nothing may allocate
            torch.cuda.synchronize()
            torch_before = (torch.cuda.memory_allocated(dev), torch.cuda.memory_reserved(dev))
            free_before = torch.cuda.mem_get_info(dev)[0]
        b.gemm_rs_run_noalloc(M, N, K, W, alpha, beta, code, Ad.data_ptr(), Bd.data_ptr(),
                              0 if Cd is None else Cd.data_ptr(), Y.data_ptr(), stream)
        assert b.gemm_rs_noalloc_status(stream) == b.GEMM_RS_OK
        if call == 1:
            assert (torch.cuda.memory_allocated(dev), torch.cuda.memory_reserved(dev)) == torch_before
            # cudaMemGetInfo: no device allocation behind torch's back either
            assert torch.cuda.mem_get_info(dev)[0] >= free_before - (1 << 20)
        torch.cuda.synchronize()
        y = to_np_y(Y)
        assert_close(y, ref, y_dtype, f"no-alloc call {call}")
        np.testing.assert_array_equal(y, ref)


def test_noalloc_rejects_shapes_beyond_its_scratch():
    from tensor_gemm_reduce_tcgen05_gb300 import binding as b
    W, M, N, K = 8, 4096, 4096, 8 * 64
    assert b.gemm_rs_workspace_bytes(M, N, K, W) > b.gemm_rs_noalloc_scratch_bytes()
    Y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda:0")
    A = torch.zeros((W, M, K // W), dtype=torch.bfloat16, device="cuda:0")
    B = torch.zeros((W, K // W, N), dtype=torch.bfloat16, device="cuda:0")
    with pytest.raises(b.GemmRSError) as e:
        b.gemm_rs_run_noalloc(M, N, K, W, 1.0, 0.0, b.GEMM_RS_BF16, A.data_ptr(), B.data_ptr(),
                              0, Y.data_ptr(), 0)
    assert e.value.code == b.GEMM_RS_ERR_WORKSPACE
    assert "static scratch" in b.gemm_rs_last_error()
