"""Seeded random shapes, bit-exact against the oracle.

The fixed grid of test_gpu_parity.py picks shapes by what they cover.  This
sweep draws them: W from 1 to 16, chunk heights from 1 row up, ragged N and
K, every tile, reduce mode and rank order, with and without the C term, both
output types.  Inputs are integers in {-2..2}, so every sum is exact and the
GPU result must equal the oracle's bit for bit, with a NaN-poisoned workspace
and Y and two calls in a row (every slot read is written in the same call,
every output element is written, and the state words end at zero).  Larger
random shapes run the library's default plan (mostly the CTA-pair kernel) and
are checked on sampled rows; normal inputs must give the same bits from two
handles and repeated calls.
"""
import numpy as np
import pytest

from helpers import inputs, oracle_y, run_gpu

pytestmark = pytest.mark.gpu

TILES = [(128, 256), (128, 128), (128, 64), (256, 256)]


def _cases(n=24, seed=20261203):
    rng = np.random.default_rng(seed)
    out = []
    for _ in range(n):
        W = int(rng.integers(1, 17))
        R = int(rng.integers(1, max(2, 1024 // W)))
        M = W * R
        N = 8 * int(rng.integers(1, 97))
        Kpr = 8 * int(rng.integers(1, max(2, 2048 // (8 * W))))
        tile = TILES[int(rng.integers(0, len(TILES)))]
        mode = int(rng.integers(0, 3))
        order = int(rng.integers(1, 3))
        beta = float(rng.choice([0.0, 0.5]))
        y_dtype = str(rng.choice(["fp32", "bf16"]))
        out.append((W, M, N, Kpr, tile, mode, order, beta, y_dtype))
    return out


@pytest.mark.parametrize("W,M,N,Kpr,tile,mode,order,beta,y_dtype", _cases())
def test_random_shapes_bit_exact(W, M, N, Kpr, tile, mode, order, beta, y_dtype):
    A, B, C = inputs(W, M, N, Kpr, "int", c_dist="int" if beta != 0 else None, seeds=(M, N, Kpr))
    y, plan, op = run_gpu(A, B, C, W, M, N, Kpr, 1.0, beta, y_dtype, tile_m=tile[0],
                          tile_n=tile[1], reduce_mode=mode, rank_order=order, poison=True,
                          calls=2)
    assert (plan["bm"], plan["bn"], plan["reduce_mode"]) == (tile[0], tile[1], mode)
    np.testing.assert_array_equal(y, oracle_y(A, B, C, 1.0, beta, y_dtype))
    assert int(op.flags_view().abs().sum()) == 0


def _large_cases(n=16, seed=20261204):
    """Larger shapes (up to M = 4096, N = 2048, K = 4096), where the default
    plan picks the CTA-pair kernel and a rank's pass spans several waves."""
    rng = np.random.default_rng(seed)
    out = []
    for _ in range(n):
        W = int(rng.integers(1, 17))
        R = int(rng.integers(1, max(2, 4096 // W)))
        M = W * R
        N = 8 * int(rng.integers(1, 257))
        Kpr = 8 * int(rng.integers(1, max(2, 4096 // (8 * W))))
        mode = int(rng.integers(0, 3))
        order = int(rng.integers(1, 3))
        beta = float(rng.choice([0.0, 1.0]))
        y_dtype = str(rng.choice(["fp32", "bf16"]))
        out.append((W, M, N, Kpr, mode, order, beta, y_dtype))
    return out


@pytest.mark.parametrize("W,M,N,Kpr,mode,order,beta,y_dtype", _large_cases())
def test_random_large_shapes_bit_exact_on_sampled_rows(W, M, N, Kpr, mode, order, beta, y_dtype):
    """The default plan (tile and schedule chosen by the library), integer
    inputs, three calls on a NaN-poisoned workspace and Y: every chunk's first
    and last rows and seeded random rows equal the oracle's bit for bit."""
    A, B, C = inputs(W, M, N, Kpr, "int", c_dist="int" if beta != 0 else None, seeds=(M, N, Kpr))
    y, plan, op = run_gpu(A, B, C, W, M, N, Kpr, 1.0, beta, y_dtype, reduce_mode=mode,
                          rank_order=order, poison=True, calls=3)
    R = M // W
    rng = np.random.default_rng(M * 31 + N)
    rows = np.unique(np.concatenate([np.arange(0, M, R), np.arange(R - 1, M, R),
                                     rng.integers(0, M, 16)]))
    np.testing.assert_array_equal(y[rows], oracle_y(A, B, C, 1.0, beta, y_dtype, rows=rows))
    assert int(op.flags_view().abs().sum()) == 0


@pytest.mark.parametrize("case", range(6))
def test_normal_inputs_identical_across_handles_and_calls(case):
    """Normal inputs, alpha 0.5 and beta 1 with a N(0,1) C: two handles (the
    second calling once, the first twice) give the same bits, in every reduce
    mode and rank order."""
    rng = np.random.default_rng(900 + case)
    W = int(rng.integers(2, 17))
    R = int(rng.integers(8, 512))
    M, N, Kpr = W * R, 8 * int(rng.integers(8, 129)), 8 * int(rng.integers(8, 257))
    mode, order = case % 3, 1 + case % 2
    A, B, C = inputs(W, M, N, Kpr, "normal", c_dist="normal1", seeds=(case, 5, 6))
    y1, _, _ = run_gpu(A, B, C, W, M, N, Kpr, 0.5, 1.0, "fp32", reduce_mode=mode,
                       rank_order=order, calls=2)
    y2, _, _ = run_gpu(A, B, C, W, M, N, Kpr, 0.5, 1.0, "fp32", reduce_mode=mode,
                       rank_order=order, calls=1)
    np.testing.assert_array_equal(y1, y2)
