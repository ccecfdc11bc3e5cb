"""Seeded random shapes, bit-exact against the oracle.

The fixed grid of test_gpu_parity.py picks shapes by what they cover.  This
sweep draws them: W from 1 to 16, chunk heights from 1 row up, ragged N and
K, every tile, reduce mode and rank order, with and without the C term, both
output types.  Inputs are integers in {-2..2}, so every sum is exact and the
GPU result must equal the oracle's bit for bit, with a NaN-poisoned workspace
and Y and two calls in a row (every slot read is written in the same call,
every output element is written, and the state words end at zero).
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
