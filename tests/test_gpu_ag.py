"""Parity of the fused AG+GEMM CUDA path with its oracle, through the C ABI.

Integer-valued inputs make every sum exact, so those runs must match bit for
bit; normal inputs must meet the fp32 / bf16 tolerances; the device tile order
must equal the library's schedule and follow the pages' consumption order
(checked against the oracle's chunk order); repeated calls must be
bit-identical; a wait for a chunk that never arrives must time out cleanly.
"""
import numpy as np
import pytest
import torch

import oracle
from helpers import assert_close, to_np_y
from schedule_props import check_ag_schedule
from tensor_gemm_reduce_tcgen05_gb300.inputs import (AG_WORKLOADS, bf16_bits, make_ag_inputs,
                                                     sample_rows)

pytestmark = pytest.mark.gpu

SHAPES = [
    # W, M, N, K                     what it covers
    (2, 512, 256, 256),            # two ranks, one tile column
    (3, 768, 264, 200),            # ragged N (tail of 8 columns) and ragged K (200 = 3*64 + 8)
    (1, 256, 72, 64),              # W = 1: a plain GEMM, no copies
    (8, 2048, 512, 128),           # eight ranks, one 256-row tile per chunk
    (16, 16 * 256, 64, 64),        # W = 16
    (4, 2048, 1000, 136),          # two 256-row tiles per chunk, ragged N
    (2, 512, 8, 8),                # N = 8 and K = 8: TMA boxes larger than the tensors
    (4, 1024, 16, 24),             # small N and K, four ranks
    (2, 512, 320, 64),             # N % 64 == 0, not % 256: the 4D B box runs past N (zeros)
]


def run_ag(X, B1, W, M, N, K, alpha, y_dtype, calls=1, record=None):
    from tensor_gemm_reduce_tcgen05_gb300 import binding as b
    dev = torch.device("cuda", 0)
    op = b.AgGemm(M, N, K, W, alpha, y_dtype, device=dev)
    if record is not None:
        b.ag_gemm_set_debug(op.handle, record.data_ptr(), 0)
    Xd, Bd = X.to(dev), B1.to(dev)
    H = op.new_output()
    H.view(torch.uint8).fill_(0xFF)  # NaN everywhere: every element must be written
    for _ in range(calls):
        op.run(Xd, Bd, H)
    torch.cuda.synchronize()
    assert op.status() == 0, "device status reports a timeout"
    return to_np_y(H), op


def oracle_h(X, B1, alpha, y_dtype, rows=None):
    return oracle.ag_gemm(bf16_bits(X), bf16_bits(B1), alpha, y_dtype, rows=rows)


@pytest.mark.parametrize("y_dtype", ["fp32", "bf16"])
@pytest.mark.parametrize("W,M,N,K", SHAPES)
def test_integer_inputs_bit_exact(W, M, N, K, y_dtype):
    X, B1 = make_ag_inputs(W, M, N, K, "int", "int")
    h, _ = run_ag(X, B1, W, M, N, K, 1.0, y_dtype)
    np.testing.assert_array_equal(h, oracle_h(X, B1, 1.0, y_dtype))


@pytest.mark.parametrize("y_dtype", ["fp32", "bf16"])
@pytest.mark.parametrize("W,M,N,K", SHAPES[:4])
def test_normal_inputs_within_tolerance(W, M, N, K, y_dtype):
    X, B1 = make_ag_inputs(W, M, N, K, "normal", "normal")
    h, _ = run_ag(X, B1, W, M, N, K, 0.5, y_dtype)
    ref = oracle_h(X, B1, 0.5, y_dtype)
    for r in range(W):
        assert_close(h[r], ref[r], y_dtype, f"rank {r} of {(W, M, N, K)}")


def test_repeated_calls_identical_and_signals_counted():
    """Five calls on one workspace are bit-identical; every remote (rank, chunk)
    signal ends at calls * slices and a rank's own chunk is never signalled."""
    W, M, N, K = 4, 1024, 512, 256
    X, B1 = make_ag_inputs(W, M, N, K, "normal", "normal")
    h1, op1 = run_ag(X, B1, W, M, N, K, 1.0, "fp32", calls=1)
    h5, op5 = run_ag(X, B1, W, M, N, K, 1.0, "fp32", calls=5)
    np.testing.assert_array_equal(h1, h5)
    sig = op5.signals_view().cpu().numpy().reshape(W, W)
    slices = op5.plan["slices"]
    expect = np.full((W, W), 5 * slices)
    np.fill_diagonal(expect, 0)
    np.testing.assert_array_equal(sig, expect)


def test_device_tile_order_matches_schedule():
    from tensor_gemm_reduce_tcgen05_gb300 import binding as b
    for (W, M, N, K) in [(8, 2048, 768, 64), (3, 1536, 264, 64)]:
        X, B1 = make_ag_inputs(W, M, N, K, "int", "int")
        n = W * (M // 256) * -(-N // 256)
        rec = torch.full((n, 4), -1, dtype=torch.int32, device="cuda:0")
        h, op = run_ag(X, B1, W, M, N, K, 1.0, "fp32", record=rec)
        rec = rec.cpu().numpy()
        np.testing.assert_array_equal(rec[:, :3], b.ag_gemm_schedule(M, N, W))
        check_ag_schedule(rec[:, :3], W, M, N, 256, 256)
        workers = op.plan["grid"] // 2
        np.testing.assert_array_equal(rec[:, 3], np.arange(n) % workers)
        np.testing.assert_array_equal(h, oracle_h(X, B1, 1.0, "fp32"))


def test_missing_chunk_times_out_and_recovers():
    """With the copies switched off, the wait for a remote chunk runs out: the
    kernel records a timeout and exits, the context stays usable, and after a
    reset the next call is exact."""
    from tensor_gemm_reduce_tcgen05_gb300 import binding as b
    W, M, N, K = 2, 512, 256, 128
    X, B1 = make_ag_inputs(W, M, N, K, "int", "int")
    dev = torch.device("cuda", 0)
    op = b.AgGemm(M, N, K, W, 1.0, "fp32", device=dev)
    Xd, Bd = X.to(dev), B1.to(dev)
    b.ag_gemm_set_timeout_cycles(op.handle, 1 << 22)
    b.ag_gemm_set_debug(op.handle, 0, b.AG_GEMM_DEBUG_SKIP_COPIES)
    op.run(Xd, Bd)
    torch.cuda.synchronize()
    assert op.status() == b.GEMM_RS_ERR_TIMEOUT
    op.reset()
    b.ag_gemm_set_debug(op.handle, 0, 0)
    b.ag_gemm_set_timeout_cycles(op.handle, 1 << 32)
    H = op.run(Xd, Bd)
    torch.cuda.synchronize()
    assert op.status() == 0
    np.testing.assert_array_equal(to_np_y(H), oracle_h(X, B1, 1.0, "fp32"))


@pytest.mark.parametrize("name", sorted(AG_WORKLOADS))
def test_full_size_workload_on_row_sample(name):
    """The full-size workload in the launch configuration the benchmark times,
    on a row sample of every rank's output."""
    w = AG_WORKLOADS[name]
    X, B1 = make_ag_inputs(w.W, w.M, w.N, w.K, w.x_dist, w.b_dist)
    h, _ = run_ag(X, B1, w.W, w.M, w.N, w.K, w.alpha, w.y_dtype, calls=2)
    rows = sample_rows(w.M, w.W, BM=256, n_random=8, n_boundaries=4)
    ref = oracle_h(X, B1, w.alpha, w.y_dtype, rows=rows)
    for r in range(w.W):
        assert_close(h[r][rows], ref[r], w.y_dtype, f"{name} rank {r}")
