"""Parity of the fused CUDA path with the oracle, through the C ABI.

Small cases are compared element by element.  They span several tiles and
ragged tails in M, N and K, chunks that do not align with tiles, and all
three tile widths.  The full-size workloads are compared on a row sample the
oracle computes one row at a time.  Integer-valued inputs make every sum exact,
so those runs must match bit for bit.
"""
import numpy as np
import pytest
import torch

import oracle
from helpers import assert_close, inputs, oracle_y, run_gpu, to_np_y
from schedule_props import check_rs_schedule
from tensor_gemm_reduce_tcgen05_gb300.inputs import (WORKLOADS, bf16_bits, sample_rows,
                                                     workload_inputs)

pytestmark = pytest.mark.gpu

SHAPES = [
    # W, M, N, Kpr                                      what it covers
    (2, 256, 256, 256),    # the tiny workload: 2x1 tiles, 4 k-blocks
    (3, 300, 520, 200),    # ragged M, N and K; chunks of 100 rows straddle tiles
    (8, 64, 512, 192),     # 8-row chunks: one row tile holds every chunk
    (1, 200, 72, 64),      # W = 1 is a plain GEMM; N below one tile
    (16, 16 * 9, 136, 72), # W = 16, 9-row chunks, ragged K
    (4, 512, 768, 128),    # several row tiles per chunk
    (4, 512, 320, 128),    # N % 64 == 0 but not % 256: the last tile's B box runs past N (zeros)
]


TILES = [(128, 256), (128, 128), (128, 64), (256, 256)]  # (256, 256): the CTA-pair kernel


MODES = [0, 1, 2]  # GEMM_RS_REDUCE_CHAIN, _LAST_ARRIVER, _TWO_LEVEL


ORDERS = [1, 2]  # GEMM_RS_RANKS_SEQUENTIAL (the default), GEMM_RS_RANKS_INTERLEAVED


@pytest.mark.parametrize("order", ORDERS)
@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("tile", TILES)
@pytest.mark.parametrize("W,M,N,Kpr", SHAPES)
def test_integer_inputs_bit_exact(W, M, N, Kpr, tile, mode, order):
    A, B, _ = inputs(W, M, N, Kpr, "int")
    y, plan, op = run_gpu(A, B, None, W, M, N, Kpr, 1.0, 0.0, "fp32", tile_m=tile[0],
                          tile_n=tile[1], reduce_mode=mode, rank_order=order)
    assert (plan["bm"], plan["bn"], plan["reduce_mode"], plan["rank_order"]) == \
        (tile[0], tile[1], mode, order)
    assert int(op.flags_view().abs().sum()) == 0
    ref = oracle_y(A, B, None, 1.0, 0.0, "fp32")
    np.testing.assert_array_equal(y, ref)


@pytest.mark.parametrize("tile", [(128, 256), (256, 256)])
@pytest.mark.parametrize("W,M,N,Kpr", SHAPES[:3])
def test_integer_inputs_with_c_bit_exact(W, M, N, Kpr, tile):
    A, B, C = inputs(W, M, N, Kpr, "int", c_dist="int")
    for y_dtype in ("fp32", "bf16"):
        y, _, _ = run_gpu(A, B, C, W, M, N, Kpr, 0.5, 1.0, y_dtype, tile_m=tile[0],
                          tile_n=tile[1])
        ref = oracle_y(A, B, C, 0.5, 1.0, y_dtype)
        np.testing.assert_array_equal(y, ref)


@pytest.mark.parametrize("order", ORDERS)
@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("W,M,N,Kpr", SHAPES)
@pytest.mark.parametrize("y_dtype", ["fp32", "bf16"])
def test_normal_inputs_within_tolerance(W, M, N, Kpr, y_dtype, mode, order):
    A, B, C = inputs(W, M, N, Kpr, "normal", c_dist="normal1")
    y, _, _ = run_gpu(A, B, C, W, M, N, Kpr, 0.5, 1.0, y_dtype, reduce_mode=mode,
                      rank_order=order)
    assert_close(y, oracle_y(A, B, C, 0.5, 1.0, y_dtype), y_dtype, f"{(W, M, N, Kpr)}")


def test_tiny_workload_full_compare():
    w = WORKLOADS["tiny_w2"]
    A, B, C = workload_inputs(w)
    y, _, _ = run_gpu(A, B, C, w.W, w.M, w.N, w.Kpr, w.alpha, w.beta, w.y_dtype)
    assert_close(y, oracle_y(A, B, C, w.alpha, w.beta, w.y_dtype), w.y_dtype, w.name)


def test_nan_poisoned_workspace_and_output():
    """Every partial slot that is read is written in the same call, and every
    output element is written."""
    W, M, N, Kpr = 3, 300, 520, 200
    A, B, _ = inputs(W, M, N, Kpr, "int")
    for tile in ((128, 256), (128, 64), (256, 256)):
        for mode in MODES:
            for order in ORDERS:
                y, _, _ = run_gpu(A, B, None, W, M, N, Kpr, 1.0, 0.0, "fp32", tile_m=tile[0],
                                  tile_n=tile[1], poison=True, reduce_mode=mode,
                                  rank_order=order)
                np.testing.assert_array_equal(y, oracle_y(A, B, None, 1.0, 0.0, "fp32"))


def test_beta_zero_ignores_nan_c():
    W, M, N, Kpr = 2, 256, 256, 64
    A, B, _ = inputs(W, M, N, Kpr, "int")
    from tensor_gemm_reduce_tcgen05_gb300.binding import GemmRS
    op = GemmRS(M, N, W * Kpr, W, 1.0, 0.0, "fp32", device="cuda:0")
    Cnan = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda:0")
    Y = op.run(A.cuda(), B.cuda(), Cnan)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(to_np_y(Y), oracle_y(A, B, None, 1.0, 0.0, "fp32"))


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("tile_m", [None, 256])
def test_k_zero_gives_w_beta_c(tile_m, mode):
    """K = 0: no MMA runs, so the MMA thread hands each accumulator over by a
    plain arrival (on both CTAs' barriers in the CTA-pair kernel, tile_m = 256)
    and the epilogue reads zeros instead of TMEM; Y = W * beta * C exactly."""
    W, M, N = 4, 256, 264
    _, _, C = inputs(W, M, N, 8, "int", c_dist="normal1")
    A = torch.zeros((W, M, 0), dtype=torch.bfloat16)
    B = torch.zeros((W, 0, N), dtype=torch.bfloat16)
    y, plan, _ = run_gpu(A, B, C, W, M, N, 0, 1.0, 1.0, "fp32", tile_m=tile_m, reduce_mode=mode,
                         poison=True, calls=2)
    if tile_m is not None:
        assert plan["bm"] == tile_m
    np.testing.assert_array_equal(y, W * C.float().numpy())


def test_empty_problem_is_a_no_op():
    from tensor_gemm_reduce_tcgen05_gb300.binding import GemmRS
    op = GemmRS(0, 64, 128, 2, 1.0, 0.0, "fp32", device="cuda:0")
    A = torch.zeros((2, 0, 64), dtype=torch.bfloat16, device="cuda:0")
    B = torch.zeros((2, 64, 64), dtype=torch.bfloat16, device="cuda:0")
    op.run(A, B)
    torch.cuda.synchronize()
    assert op.status() == 0


@pytest.mark.parametrize("mode", MODES)
def test_twenty_calls_bit_identical_and_counters_reset(mode):
    """Workspace reused across back-to-back calls with no memset: identical
    results every call, and every tile counter is 0 afterwards."""
    W, M, N, Kpr = 4, 1024, 640, 256
    A, B, _ = inputs(W, M, N, Kpr, "uniform")
    from tensor_gemm_reduce_tcgen05_gb300 import binding as b
    op = b.GemmRS(M, N, W * Kpr, W, 1.0, 0.0, "fp32", device="cuda:0")
    b.gemm_rs_set_reduce_mode(op.handle, mode)
    Ad, Bd = A.cuda(), B.cuda()
    outs = [op.run(Ad, Bd) for _ in range(20)]
    torch.cuda.synchronize()
    assert op.status() == 0
    first = outs[0].cpu()
    for o in outs[1:]:
        assert torch.equal(o.cpu().view(torch.int32), first.view(torch.int32))
    assert int(op.flags_view().abs().sum()) == 0
    assert_close(first.numpy(), oracle_y(A, B, None, 1.0, 0.0, "fp32"), "fp32", "20 calls")


def test_device_schedule_record_follows_the_swizzle():
    """The order the kernel really walked (its device record) equals the
    library's host schedule, and follows the pages' swizzle: each rank-tile
    once, each rank's chunks in the oracle's chunk order in every column, W
    distinct chunks per step with the ranks side by side.  Plans with column
    groups, row groups and both rank orders, for both kernels."""
    from tensor_gemm_reduce_tcgen05_gb300 import binding as b
    for (W, M, N, Kpr, bm, bn, G, RG, ro) in [(8, 1024, 1024, 64, 128, 256, 0, 0, 0),
                                              (8, 1024, 1024, 64, 128, 256, 0, 0, 2),
                                              (3, 300, 520, 64, 128, 128, 2, 1, 2),
                                              (3, 300, 520, 64, 128, 128, 2, 1, 1),
                                              (8, 64, 8192, 64, 128, 64, 0, 0, 0),
                                              (8, 4096, 1024, 64, 256, 256, 0, 0, 2),
                                              (8, 4096, 1024, 64, 256, 256, 0, 0, 1),
                                              (8, 4096, 2048, 64, 256, 256, 3, 1, 2),
                                              (8, 4096, 2048, 64, 256, 256, 2, 0, 1),
                                              (4, 4096, 2048, 64, 256, 256, 0, 3, 0),
                                              (3, 300, 520, 64, 256, 256, 1, 0, 2)]:
        A, B, _ = inputs(W, M, N, Kpr, "int")
        op = b.GemmRS(M, N, W * Kpr, W, 1.0, 0.0, "fp32", device="cuda:0", tile_m=bm, tile_n=bn)
        b.gemm_rs_set_schedule(op.handle, G, RG, ro)
        nM, nN = -(-M // bm), -(-N // bn)
        rec = torch.full((W * nM * nN, 4), -1, dtype=torch.int32, device="cuda:0")
        b.gemm_rs_set_debug(op.handle, rec.data_ptr(), 0)
        Y = op.run(A.cuda(), B.cuda())
        torch.cuda.synchronize()
        rec = rec.cpu().numpy()
        plan = op.plan
        inter = ro == 2
        assert plan["rank_order"] == (b.GEMM_RS_RANKS_INTERLEAVED if inter
                                      else b.GEMM_RS_RANKS_SEQUENTIAL)
        lib_sched = b.gemm_rs_schedule(M, N, W, bm, bn, plan["colgroup"], plan["rowgroup"],
                                       plan["rank_order"])
        np.testing.assert_array_equal(rec[:, :3], lib_sched)
        check_rs_schedule(rec[:, :3], W, M, N, bm, bn, inter)
        grid = op.plan["grid"]
        workers = grid // 2 if bm == 256 else grid  # CTA pairs process one entry each
        np.testing.assert_array_equal(rec[:, 3], np.arange(rec.shape[0]) % workers)
        np.testing.assert_array_equal(to_np_y(Y), oracle_y(A, B, None, 1.0, 0.0, "fp32"))


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("tile", [(128, 256), (256, 256)])
def test_timeout_path_reports_and_recovers(tile, mode):
    """A stalled producer makes the MMA warp's bounded wait run out.  The
    kernel records the timeout, exits, and the context stays usable, in every
    reduce mode."""
    from tensor_gemm_reduce_tcgen05_gb300 import binding as b
    W, M, N, Kpr = 4, 512, 256, 128
    A, B, _ = inputs(W, M, N, Kpr, "int")
    op = b.GemmRS(M, N, W * Kpr, W, 1.0, 0.0, "fp32", device="cuda:0", tile_m=tile[0],
                  tile_n=tile[1])
    b.gemm_rs_set_reduce_mode(op.handle, mode)
    Ad, Bd = A.cuda(), B.cuda()
    b.gemm_rs_set_timeout_cycles(op.handle, 1 << 22)
    b.gemm_rs_set_debug(op.handle, 0, b.GEMM_RS_DEBUG_STALL_PRODUCER)
    op.run(Ad, Bd)
    assert op.status() == b.GEMM_RS_ERR_TIMEOUT
    assert "timed out" in b.gemm_rs_last_error()
    assert op.status() == b.GEMM_RS_OK        # the status word was cleared
    b.gemm_rs_set_debug(op.handle, 0, 0)
    b.gemm_rs_set_timeout_cycles(op.handle, 1 << 32)
    op.reset()
    Y = op.run(Ad, Bd)
    torch.cuda.synchronize()
    assert op.status() == 0
    np.testing.assert_array_equal(to_np_y(Y), oracle_y(A, B, None, 1.0, 0.0, "fp32"))


def test_reduce_modes_agree_and_each_is_deterministic():
    """All reductions and both rank orders on one shape with many tiles per
    chunk: each is bit-identical across calls, and all agree within the fp32
    tolerance (they differ only in summation order).  With the ranks one after
    another, the chain folds in rank order, the last arriver's order."""
    W, M, N, Kpr = 8, 2048, 1536, 512
    A, B, _ = inputs(W, M, N, Kpr, "normal")
    outs = {}
    for mode in MODES:
        for order in ORDERS:
            y1, _, op = run_gpu(A, B, None, W, M, N, Kpr, 1.0, 0.0, "fp32", reduce_mode=mode,
                                calls=3, rank_order=order)
            y2, _, _ = run_gpu(A, B, None, W, M, N, Kpr, 1.0, 0.0, "fp32", reduce_mode=mode,
                               rank_order=order)
            np.testing.assert_array_equal(y1, y2)
            outs[mode, order] = y1
    ref = oracle_y(A, B, None, 1.0, 0.0, "fp32")
    for key, y in outs.items():
        assert_close(y, outs[1, 1], "fp32", f"{key} vs last arriver")
        assert_close(y, ref, "fp32", f"{key} vs oracle")


def test_baseline_reduce_kernel_matches_oracle():
    """The unfused baseline's separate reduce step, given exact per-rank
    partials, reproduces the oracle's fold."""
    from tensor_gemm_reduce_tcgen05_gb300 import binding as b
    W, M, N, Kpr = 4, 256, 264, 64
    A, B, C = inputs(W, M, N, Kpr, "int", c_dist="int")
    P = torch.stack([A[r].float() @ B[r].float() for r in range(W)]).cuda().contiguous()
    for y_dtype in ("fp32", "bf16"):
        Y = torch.empty((M, N), dtype=torch.float32 if y_dtype == "fp32" else torch.bfloat16,
                        device="cuda:0")
        b.gemm_rs_reduce_partials(P.data_ptr(), b.GEMM_RS_FP32, C.cuda().data_ptr(), Y.data_ptr(),
                                  M, N, W, 0.5, 1.0,
                                  b.GEMM_RS_FP32 if y_dtype == "fp32" else b.GEMM_RS_BF16)
        torch.cuda.synchronize()
        np.testing.assert_array_equal(to_np_y(Y), oracle_y(A, B, C, 0.5, 1.0, y_dtype))


@pytest.mark.parametrize("order", ORDERS)
@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("name", ["ffn_w8_m4096", "ffn_w8_m8192_bias", "decode_w8_m64",
                                  "ffn_w4_m16384_x20"])
def test_full_size_workloads_on_row_sample(name, mode, order):
    """The full-size workloads in the launch configuration the benchmark
    times, checked on a row sample: every chunk's first and last row, four
    row-tile boundaries (both rows at each), and 8 seeded random rows.  The
    oracle streams all of B once per row, so the sample stays small."""
    w = WORKLOADS[name]
    A, B, C = workload_inputs(w)
    y, plan, op = run_gpu(A, B, C, w.W, w.M, w.N, w.Kpr, w.alpha, w.beta, w.y_dtype,
                          calls=w.calls, reduce_mode=mode, rank_order=order)
    rows = sample_rows(w.M, w.W, n_random=8, n_boundaries=4)
    ref = oracle_y(A, B, C, w.alpha, w.beta, w.y_dtype, rows=rows)
    assert_close(y[rows], ref, w.y_dtype, name)
    assert int(op.flags_view().abs().sum()) == 0


def test_chunked_two_stream_baseline_matches_oracle():
    """The benchmark's chunked two-stream comparator (per-chunk cuBLAS GEMMs on
    one stream, the reduce of the previous chunk on another) computes the same
    Y: exact for integer-valued inputs."""
    import bench
    from tensor_gemm_reduce_tcgen05_gb300 import binding as b
    W, M, N, Kpr = 4, 512, 264, 64
    A, B, C = inputs(W, M, N, Kpr, "int", c_dist="int")
    dev = torch.device("cuda", 0)
    Ad, Bd, Cd = A.to(dev), B.to(dev), C.to(dev)
    stream = torch.cuda.current_stream(dev)
    for y_dtype in ("fp32", "bf16"):
        Y = torch.empty((M, N), dtype=torch.float32 if y_dtype == "fp32" else torch.bfloat16,
                        device=dev)
        y_code = b.GEMM_RS_FP32 if y_dtype == "fp32" else b.GEMM_RS_BF16
        run = bench.chunked_baseline(W, M, N, 0.5, 1.0, y_code, Ad, Bd, Cd, Y, stream, dev)
        run()
        run()
        torch.cuda.synchronize()
        np.testing.assert_array_equal(to_np_y(Y), oracle_y(A, B, C, 0.5, 1.0, y_dtype))


DEGENERATE = [
    # W, M, N, Kpr          what it covers
    (4, 4, 8, 8),         # one row per chunk, N = 8 (one 16-byte column group), K/W = 8
    (2, 256, 8, 16),      # N = 8 with full row tiles, K/W = 16 (a quarter of a k-block)
    (8, 1024, 24, 8),     # K/W = 8 on the CTA-pair tile, N of three 8-column groups
    (16, 16, 264, 8),     # W = 16, one row per chunk, ragged N
]


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("tile", TILES)
@pytest.mark.parametrize("W,M,N,Kpr", DEGENERATE)
def test_degenerate_shapes_bit_exact(W, M, N, Kpr, tile, mode):
    """Sizes at the edges of the layout rules: the smallest K per rank and N
    (TMA boxes larger than the tensor, zero fill), one row per chunk, W = 16."""
    A, B, C = inputs(W, M, N, Kpr, "int", c_dist="int")
    y, _, op = run_gpu(A, B, C, W, M, N, Kpr, 0.5, 1.0, "fp32", tile_m=tile[0], tile_n=tile[1],
                       reduce_mode=mode, poison=True, calls=2)
    np.testing.assert_array_equal(y, oracle_y(A, B, C, 0.5, 1.0, "fp32"))
    assert int(op.flags_view().abs().sum()) == 0


def test_output_beyond_2_to_the_31_elements():
    """M*N = 2^31 (Y 8.6 GB in fp32, partial workspace 17 GB): the epilogue's
    and the folds' 64-bit index arithmetic, checked bit-exact on rows up to
    the last one, with small K so the call is short."""
    from tensor_gemm_reduce_tcgen05_gb300 import binding as b
    from tensor_gemm_reduce_tcgen05_gb300.inputs import sample_rows
    W, M, N, Kpr = 2, 65536, 32768, 64
    A, B, _ = inputs(W, M, N, Kpr, "int")
    dev = torch.device("cuda", 0)
    op = b.GemmRS(M, N, W * Kpr, W, 1.0, 0.0, "fp32", device=dev)
    Y = op.run(A.to(dev), B.to(dev))
    torch.cuda.synchronize()
    assert op.status() == b.GEMM_RS_OK
    rows = np.unique(np.concatenate([sample_rows(M, W, n_random=4, n_boundaries=2),
                                     [M - 1, M - 2, M // 2 + 1]]))
    y = Y[torch.from_numpy(rows).to(dev)].cpu().numpy()
    np.testing.assert_array_equal(y, oracle_y(A, B, None, 1.0, 0.0, "fp32", rows=rows))
    assert int(op.flags_view().abs().sum()) == 0
    del Y, op
    torch.cuda.empty_cache()
