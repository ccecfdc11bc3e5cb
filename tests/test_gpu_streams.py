"""Stream use of the C ABI: a run captured in a CUDA graph and replayed, and
two handles running at the same time on two streams.  The call makes no host
sync and no memset, and each handle's state lives in its own workspace, so
both must give the eager single-stream results bit for bit."""
import numpy as np
import pytest
import torch

from helpers import inputs, oracle_y, to_np_y

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("mode", [0, 1, 2])
@pytest.mark.parametrize("W,M,N,Kpr", [(4, 1024, 2560, 128), (8, 64, 1024, 192)])
def test_cuda_graph_capture_and_replay(W, M, N, Kpr, mode):
    """Three calls captured in one graph (A, B changing between them through
    copies inside the graph), replayed five times: every replay is exact and
    leaves the state words at 0."""
    from tensor_gemm_reduce_tcgen05_gb300 import binding as b
    dev = torch.device("cuda", 0)
    A1, B1, _ = inputs(W, M, N, Kpr, "int", seeds=(1, 2, 3))
    A2, B2, _ = inputs(W, M, N, Kpr, "int", seeds=(4, 5, 6))
    op = b.GemmRS(M, N, W * Kpr, W, 1.0, 0.0, "fp32", device=dev)
    b.gemm_rs_set_reduce_mode(op.handle, mode)
    Ad, Bd = A1.to(dev), B1.to(dev)
    srcs = [(A1.to(dev), B1.to(dev)), (A2.to(dev), B2.to(dev))]
    Ys = [op.new_output() for _ in range(3)]
    op.run(Ad, Bd, None, Ys[0])           # encodes the tensor maps before the capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream(dev)
    s.wait_stream(torch.cuda.current_stream(dev))
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            for i in range(3):
                Ad.copy_(srcs[i % 2][0])
                Bd.copy_(srcs[i % 2][1])
                op.run(Ad, Bd, None, Ys[i], stream=s)
    torch.cuda.synchronize()
    refs = [oracle_y(A1, B1, None, 1.0, 0.0, "fp32"), oracle_y(A2, B2, None, 1.0, 0.0, "fp32")]
    for _ in range(5):
        for Y in Ys:
            Y.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert op.status() == b.GEMM_RS_OK
        for i, Y in enumerate(Ys):
            np.testing.assert_array_equal(to_np_y(Y), refs[i % 2])
        assert int(op.flags_view().abs().sum()) == 0


def test_two_handles_on_two_streams_at_once():
    from tensor_gemm_reduce_tcgen05_gb300 import binding as b
    dev = torch.device("cuda", 0)
    cases = [(8, 2048, 2048, 256, (1, 2, 3)), (4, 1024, 3072, 192, (7, 8, 9))]
    ops, args, refs = [], [], []
    for (W, M, N, Kpr, seeds) in cases:
        A, B, _ = inputs(W, M, N, Kpr, "int", seeds=seeds)
        ops.append(b.GemmRS(M, N, W * Kpr, W, 1.0, 0.0, "fp32", device=dev))
        args.append((A.to(dev), B.to(dev)))
        refs.append(oracle_y(A, B, None, 1.0, 0.0, "fp32"))
    streams = [torch.cuda.Stream(dev) for _ in cases]
    torch.cuda.synchronize()
    outs = [[], []]
    for _ in range(4):                     # interleaved launches on both streams
        for k in range(2):
            with torch.cuda.stream(streams[k]):
                outs[k].append(ops[k].run(*args[k], stream=streams[k]))
    torch.cuda.synchronize()
    for k in range(2):
        assert ops[k].status(streams[k]) == b.GEMM_RS_OK
        for Y in outs[k]:
            np.testing.assert_array_equal(to_np_y(Y), refs[k])


def test_device_given_without_an_index():
    """device="cuda" (no index) means the current device: tensors on cuda:0 are
    accepted, as in the usage example."""
    from tensor_gemm_reduce_tcgen05_gb300 import binding as b
    W, M, N, Kpr = 2, 256, 256, 64
    A, B, _ = inputs(W, M, N, Kpr, "int")
    op = b.GemmRS(M, N, W * Kpr, W, alpha=1.0, beta=0.0, y_dtype="fp32", device="cuda")
    Y = op.run(A.cuda(), B.cuda())
    assert op.status() == b.GEMM_RS_OK
    np.testing.assert_array_equal(to_np_y(Y), oracle_y(A, B, None, 1.0, 0.0, "fp32"))
    ag = b.AgGemm(512, 64, 64, 2, 1.0, "fp32", device="cuda")
    X = torch.zeros(512, 64, dtype=torch.bfloat16, device="cuda")
    B1 = torch.zeros(2, 64, 64, dtype=torch.bfloat16, device="cuda")
    H = ag.run(X, B1)
    assert ag.status() == b.GEMM_RS_OK
    assert not H.float().abs().sum().item()
