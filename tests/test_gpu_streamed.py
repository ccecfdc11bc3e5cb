"""gemm_rs_run_streamed: host inputs copied rank by rank on a copy stream while
the kernel consumes the ranks that have landed.

Integer inputs make every sum exact, so each call must equal the oracle bit for
bit, also when the host inputs change from call to call (every call's kernel
must wait for its own copies, not see the previous call's operands).  Normal
inputs must equal gemm_rs_run on the same data bit for bit (same kernel).  A
streamed call whose ready words never come times out cleanly, and the handle
then runs exactly again after gemm_rs_reset.
"""
import numpy as np
import pytest
import torch

from helpers import assert_close, inputs, oracle_y, to_np_y

pytestmark = pytest.mark.gpu


def _pinned(t):
    return t.contiguous().pin_memory()


def _streamed(op, A, B, C, y_dtype, Ad, Bd, Cd, stream, copy_stream):
    from tensor_gemm_reduce_tcgen05_gb300 import binding as b
    Y_host = torch.empty((op.M, op.N), dtype=torch.bfloat16 if y_dtype == "bf16" else torch.float32,
                         pin_memory=True)
    Y_host.view(torch.uint8).fill_(0xFF)
    op.run_streamed(_pinned(A), _pinned(B), None if C is None else _pinned(C), Y_host, Ad, Bd, Cd,
                    stream=stream, copy_stream=copy_stream)
    torch.cuda.synchronize()
    assert op.status(stream) == b.GEMM_RS_OK
    return to_np_y(Y_host)


@pytest.mark.parametrize("W,M,N,Kpr,tile,order,beta", [
    (8, 2048, 1024, 128, (256, 256), 1, 0.5),   # CTA pairs, ranks one after another, with C
    (4, 512, 520, 200, (128, 256), 1, 0.0),     # single-CTA kernel, ragged N and K
    (3, 300, 520, 64, (128, 128), 2, 0.5),      # ranks side by side
    (1, 256, 256, 64, (256, 256), 1, 0.0),      # W = 1
])
def test_streamed_calls_bit_exact_with_changing_inputs(W, M, N, Kpr, tile, order, beta):
    from tensor_gemm_reduce_tcgen05_gb300 import binding as b
    dev = torch.device("cuda", 0)
    op = b.GemmRS(M, N, W * Kpr, W, 1.0, beta, "fp32", device=dev, tile_m=tile[0], tile_n=tile[1])
    b.gemm_rs_set_schedule(op.handle, 0, 0, order)
    stream = torch.cuda.current_stream(dev)
    copy_stream = torch.cuda.Stream(device=dev)
    Ad = torch.empty((W, M, Kpr), dtype=torch.bfloat16, device=dev)
    Bd = torch.empty((W, Kpr, N), dtype=torch.bfloat16, device=dev)
    Cd = torch.empty((M, N), dtype=torch.bfloat16, device=dev) if beta != 0 else None
    for call in range(3):
        A, B, C = inputs(W, M, N, Kpr, "int", c_dist="int" if beta != 0 else None,
                         seeds=(10 + call, 20 + call, 30 + call))
        y = _streamed(op, A, B, C, "fp32", Ad, Bd, Cd, stream, copy_stream)
        np.testing.assert_array_equal(y, oracle_y(A, B, C, 1.0, beta, "fp32"), f"call {call}")
        assert int(op.flags_view().abs().sum()) == 0


@pytest.mark.parametrize("y_dtype", ["bf16", "fp32"])
def test_streamed_equals_run_on_normal_inputs(y_dtype):
    from tensor_gemm_reduce_tcgen05_gb300 import binding as b
    W, M, N, Kpr = 8, 4096, 2048, 256
    dev = torch.device("cuda", 0)
    A, B, C = inputs(W, M, N, Kpr, "normal", c_dist="normal1")
    op = b.GemmRS(M, N, W * Kpr, W, 0.5, 1.0, y_dtype, device=dev)
    stream = torch.cuda.current_stream(dev)
    copy_stream = torch.cuda.Stream(device=dev)
    Ad, Bd, Cd = A.to(dev), B.to(dev), C.to(dev)
    ref = to_np_y(op.run(Ad, Bd, Cd))
    torch.cuda.synchronize()
    A2, B2, C2 = (torch.empty_like(t) for t in (Ad, Bd, Cd))
    y = _streamed(op, A, B, C, y_dtype, A2, B2, C2, stream, copy_stream)
    np.testing.assert_array_equal(y, ref)
    rows = np.arange(0, M, 97)
    assert_close(y[rows], oracle_y(A, B, C, 0.5, 1.0, y_dtype, rows=rows), y_dtype, "streamed")


@pytest.mark.parametrize("tile", [(128, 256), (256, 256)])
def test_streamed_wait_times_out_and_recovers(tile):
    """The copies are issued but their ready words are not: the producers'
    bounded waits run out, the status reports a timeout, and after a reset the
    next streamed call is exact."""
    from tensor_gemm_reduce_tcgen05_gb300 import binding as b
    W, M, N, Kpr = 4, 1024, 512, 64
    dev = torch.device("cuda", 0)
    A, B, C = inputs(W, M, N, Kpr, "int", c_dist="int")
    op = b.GemmRS(M, N, W * Kpr, W, 1.0, 0.5, "fp32", device=dev, tile_m=tile[0], tile_n=tile[1])
    stream = torch.cuda.current_stream(dev)
    copy_stream = torch.cuda.Stream(device=dev)
    Ad = torch.empty((W, M, Kpr), dtype=torch.bfloat16, device=dev)
    Bd = torch.empty((W, Kpr, N), dtype=torch.bfloat16, device=dev)
    Cd = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    b.gemm_rs_set_timeout_cycles(op.handle, 1 << 22)
    b.gemm_rs_set_debug(op.handle, 0, b.GEMM_RS_DEBUG_SKIP_READY)
    Y_host = torch.empty((M, N), dtype=torch.float32, pin_memory=True)
    op.run_streamed(_pinned(A), _pinned(B), _pinned(C), Y_host, Ad, Bd, Cd, stream=stream,
                    copy_stream=copy_stream)
    torch.cuda.synchronize()
    assert op.status(stream) == b.GEMM_RS_ERR_TIMEOUT
    op.reset(stream)
    b.gemm_rs_set_debug(op.handle, 0, 0)
    b.gemm_rs_set_timeout_cycles(op.handle, 1 << 32)
    y = _streamed(op, A, B, C, "fp32", Ad, Bd, Cd, stream, copy_stream)
    np.testing.assert_array_equal(y, oracle_y(A, B, C, 1.0, 0.5, "fp32"))


def test_streamed_rejects_bad_streams_and_buffers():
    """The copy stream must be a stream of its own, and every host buffer the
    call needs must be given; the checks fail before anything is enqueued."""
    from tensor_gemm_reduce_tcgen05_gb300 import binding as b
    W, M, N, Kpr = 2, 256, 256, 64
    dev = torch.device("cuda", 0)
    op = b.GemmRS(M, N, W * Kpr, W, 1.0, 0.5, "fp32", device=dev)
    A = torch.zeros((W, M, Kpr), dtype=torch.bfloat16, pin_memory=True)
    B = torch.zeros((W, Kpr, N), dtype=torch.bfloat16, pin_memory=True)
    C = torch.zeros((M, N), dtype=torch.bfloat16, pin_memory=True)
    Yh = torch.empty((M, N), dtype=torch.float32, pin_memory=True)
    Ad, Bd, Cd, Y = A.to(dev), B.to(dev), C.to(dev), op.new_output()
    s = torch.cuda.Stream(device=dev)
    L = b.lib()
    args = [A.data_ptr(), B.data_ptr(), C.data_ptr(), Yh.data_ptr(), Ad.data_ptr(), Bd.data_ptr(),
            Cd.data_ptr(), Y.data_ptr()]
    assert L.gemm_rs_run_streamed(op.handle, *args, s.cuda_stream, s.cuda_stream) == b.GEMM_RS_ERR_ARG
    assert L.gemm_rs_run_streamed(op.handle, *args, s.cuda_stream, None) == b.GEMM_RS_ERR_ARG
    no_c = list(args)
    no_c[2] = None  # beta != 0 needs C_host
    other = torch.cuda.Stream(device=dev)
    assert L.gemm_rs_run_streamed(op.handle, *no_c, s.cuda_stream, other.cuda_stream) == \
        b.GEMM_RS_ERR_ARG
    assert "host buffer" in b.gemm_rs_last_error()
