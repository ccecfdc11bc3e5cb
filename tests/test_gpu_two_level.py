"""The two-level reduction (GEMM_RS_REDUCE_TWO_LEVEL) against the oracle's
two-level fold ("flux实现：sm80 gemm+rs", section "2D Ring优化": the ranks of a
node meet first, then the nodes' sums).

The inputs make every partial exact and every fold order-sensitive: each rank's
partial is v * s with v drawn from {+-2^25, +-2^24, +-2^23, +-3, +-1} per row
and s = +-1 per column (one nonzero column of A_r, so the GEMM adds nothing but
zeros to the product).  fp32 sums of such terms round differently under
different groupings, so a fold that groups the ranks differently from
y = (p_0 + ... + p_{h-1}) + (p_h + ... + p_{W-1}), h = ceil(W/2), fails a
bit-exact comparison.
"""
import numpy as np
import pytest
import torch

import oracle
from helpers import run_gpu
from tensor_gemm_reduce_tcgen05_gb300.inputs import bf16_bits

VALUES = np.array([2.0 ** 25, 2.0 ** 24, 2.0 ** 23, 3.0, 1.0])


def order_sensitive_inputs(W, M, N, Kpr, seed):
    """A [W, M, Kpr] and B [W, Kpr, N] (bf16) whose partials are exact."""
    rng = np.random.default_rng(seed)
    v = rng.choice(VALUES, size=(W, M)) * rng.choice([-1.0, 1.0], size=(W, M))
    s = rng.choice([-1.0, 1.0], size=(W, N))
    A = np.zeros((W, M, Kpr), dtype=np.float32)
    B = np.zeros((W, Kpr, N), dtype=np.float32)
    A[:, :, 0] = v
    B[:, 0, :] = s
    return torch.from_numpy(A).to(torch.bfloat16), torch.from_numpy(B).to(torch.bfloat16)


def _fold(parts):
    y = parts[0].astype(np.float32)
    for p in parts[1:]:
        y = (y + p.astype(np.float32)).astype(np.float32)
    return y


@pytest.mark.parametrize("W", [2, 3, 4, 5, 8])
def test_inputs_separate_the_two_folds(W):
    """CPU: on these inputs the oracle's two-level fold is the two groups'
    rank-order folds added (worked out here with numpy), and it differs from the
    one-level rank-order fold on many elements once the groups have two ranks."""
    M, N, Kpr = 16 * W, 48, 8
    A, B = order_sensitive_inputs(W, M, N, Kpr, seed=W)
    Af, Bf = A.float().numpy(), B.float().numpy()
    parts = [Af[r] @ Bf[r] for r in range(W)]           # exact: one nonzero term
    h = (W + 1) // 2
    two = oracle.gemm_rs(bf16_bits(A), bf16_bits(B), None, 1.0, 0.0, "fp32", split=h)
    one = oracle.gemm_rs(bf16_bits(A), bf16_bits(B), None, 1.0, 0.0, "fp32")
    np.testing.assert_array_equal(two, (_fold(parts[:h]) + _fold(parts[h:])).astype(np.float32))
    np.testing.assert_array_equal(one, _fold(parts))
    if W >= 4:
        assert (two != one).mean() > 0.05


SHAPES = [
    # W, M, N, Kpr
    (2, 256, 256, 64),
    (3, 300, 520, 64),     # ragged; a group of one rank
    (4, 512, 768, 64),     # several row tiles per chunk
    (5, 640, 264, 64),     # groups of 3 and 2
    (8, 2048, 1536, 64),   # many tiles, groups of 4
    (16, 16 * 9, 136, 64), # W = 16, 9-row chunks
]


@pytest.mark.gpu
@pytest.mark.parametrize("order", [1, 2])
@pytest.mark.parametrize("tile", [(128, 256), (128, 64), (256, 256)])
@pytest.mark.parametrize("W,M,N,Kpr", SHAPES)
def test_two_level_fold_order_bit_exact(W, M, N, Kpr, tile, order):
    """Bit-exact against the oracle's two-level fold, with the ranks one after
    another and side by side, and every state word back at 0 afterwards."""
    A, B = order_sensitive_inputs(W, M, N, Kpr, seed=100 + W)
    y, plan, op = run_gpu(A, B, None, W, M, N, Kpr, 1.0, 0.0, "fp32", tile_m=tile[0],
                          tile_n=tile[1], reduce_mode=2, rank_order=order, calls=2)
    assert plan["reduce_mode"] == 2
    ref = oracle.gemm_rs(bf16_bits(A), bf16_bits(B), None, 1.0, 0.0, "fp32",
                         split=(W + 1) // 2)
    np.testing.assert_array_equal(y, ref)
    assert int(op.flags_view().abs().sum()) == 0


@pytest.mark.gpu
@pytest.mark.parametrize("mode", [0, 1])
def test_one_level_folds_are_rank_order(mode):
    """The same inputs through the one-level reductions with the ranks one
    after another: bit-exact against the rank-order fold (and so different from
    the two-level result)."""
    W, M, N, Kpr = 8, 2048, 1536, 64
    A, B = order_sensitive_inputs(W, M, N, Kpr, seed=7)
    y, _, _ = run_gpu(A, B, None, W, M, N, Kpr, 1.0, 0.0, "fp32", reduce_mode=mode,
                      rank_order=1)
    np.testing.assert_array_equal(
        y, oracle.gemm_rs(bf16_bits(A), bf16_bits(B), None, 1.0, 0.0, "fp32"))


@pytest.mark.gpu
def test_reduce_mode_may_change_between_calls():
    """Every call leaves the tile state words at 0 in every mode, so one handle
    may switch modes between calls: each call equals a fresh handle's result in
    that mode, bit for bit, and the state words end at 0."""
    from tensor_gemm_reduce_tcgen05_gb300 import binding as b
    W, M, N, Kpr = 8, 2048, 1536, 64
    A, B = order_sensitive_inputs(W, M, N, Kpr, seed=11)
    fresh = {m: run_gpu(A, B, None, W, M, N, Kpr, 1.0, 0.0, "fp32", reduce_mode=m)[0]
             for m in (0, 1, 2)}
    dev = torch.device("cuda", 0)
    op = b.GemmRS(M, N, W * Kpr, W, 1.0, 0.0, "fp32", device=dev)
    Ad, Bd = A.to(dev), B.to(dev)
    for m in (2, 0, 1, 2, 1, 0, 2):
        b.gemm_rs_set_reduce_mode(op.handle, m)
        Y = op.run(Ad, Bd)
        torch.cuda.synchronize()
        assert op.status() == 0
        np.testing.assert_array_equal(Y.cpu().numpy(), fresh[m])
        assert int(op.flags_view().abs().sum()) == 0
