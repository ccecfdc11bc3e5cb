"""Pins for the AG+GEMM oracle (no GPU needed).

The AG+GEMM output of rank r is alpha * X @ B1_r over the all-gathered rows X.
The oracle is checked against exact rational arithmetic, int64 and float64
matrix products, closed forms, the bf16 rounding of a library cast, and the
rank-offset order printed on the pages (tests/golden/swizzle_rank_offset_w8.txt:
each rank starts at its own chunk, the order an all-gather delivers chunks in).
"""
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "swizzle_rank_offset_w8.txt")


def _bits(a: np.ndarray) -> np.ndarray:
    """bf16 bit patterns of float32 values that are exact in bf16."""
    return (np.ascontiguousarray(a, dtype=np.float32).view(np.uint32) >> 16).astype(np.uint16)


def _to_bf16_bits(t: torch.Tensor) -> np.ndarray:
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def _bf16_value(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << 16).view(np.float32)


@pytest.mark.parametrize("W,M,N,K,alpha,seed", [(1, 3, 4, 5, 1.0, 0), (2, 4, 3, 7, 0.5, 1),
                                                  (3, 3, 5, 9, -1.25, 2)])
def test_exact_rational_tiny(W, M, N, K, alpha, seed):
    """fp32 output = the exact sum alpha * X B1_r rounded once to fp32."""
    g = torch.Generator().manual_seed(seed)
    X = _to_bf16_bits(torch.randn(M, K, generator=g))
    B1 = _to_bf16_bits(torch.randn(W, K, N, generator=g))
    H = oracle.ag_gemm(X, B1, alpha, "fp32")
    Xf, Bf = _bf16_value(X), _bf16_value(B1)
    for r in range(W):
        for m in range(M):
            for n in range(N):
                exact = Fraction(alpha) * sum((Fraction(float(Xf[m, k])) * Fraction(float(Bf[r, k, n]))
                                               for k in range(K)), Fraction(0))
                # the double accumulation is exact here (bf16 products of few terms),
                # so the one rounding to fp32 is the nearest float32 of the exact value
                assert H[r, m, n] == np.float32(float(exact))


def test_integer_inputs_match_int64_matmul():
    rng = np.random.default_rng(3)
    W, M, N, K = 4, 64, 40, 96
    X = rng.integers(-2, 3, (M, K))
    B1 = rng.integers(-2, 3, (W, K, N))
    H = oracle.ag_gemm(_bits(X), _bits(B1), 1.0, "fp32")
    ref = np.stack([X @ B1[r] for r in range(W)]).astype(np.float32)
    np.testing.assert_array_equal(H, ref)


def test_normal_inputs_match_float64_matmul():
    g = torch.Generator().manual_seed(4)
    W, M, N, K = 3, 48, 32, 256
    X = _to_bf16_bits(torch.randn(M, K, generator=g) * 0.02)
    B1 = _to_bf16_bits(torch.randn(W, K, N, generator=g) * 0.02)
    H = oracle.ag_gemm(X, B1, 0.75, "fp32")
    Xf, Bf = _bf16_value(X).astype(np.float64), _bf16_value(B1).astype(np.float64)
    ref = np.stack([0.75 * (Xf @ Bf[r]) for r in range(W)])
    np.testing.assert_allclose(H, ref.astype(np.float32), rtol=1e-6, atol=1e-9)


def test_closed_forms_and_w1():
    rng = np.random.default_rng(5)
    X = rng.integers(-2, 3, (16, 24))
    B1 = rng.integers(-2, 3, (2, 24, 8))
    assert not oracle.ag_gemm(_bits(X), _bits(B1), 0.0, "fp32").any()       # alpha = 0
    H1 = oracle.ag_gemm(_bits(X), _bits(B1[:1]), 2.0, "fp32")               # W = 1: plain GEMM
    np.testing.assert_array_equal(H1[0], (2 * X @ B1[0]).astype(np.float32))


def test_bf16_output_is_rne_of_fp32():
    g = torch.Generator().manual_seed(6)
    X = _to_bf16_bits(torch.randn(32, 128, generator=g))
    B1 = _to_bf16_bits(torch.randn(2, 128, 24, generator=g))
    h32 = oracle.ag_gemm(X, B1, 1.0, "fp32")
    h16 = oracle.ag_gemm(X, B1, 1.0, "bf16")
    np.testing.assert_array_equal(h16, _to_bf16_bits(torch.from_numpy(h32)))


def test_row_sample_matches_full():
    rng = np.random.default_rng(7)
    X = rng.integers(-2, 3, (40, 16))
    B1 = rng.integers(-2, 3, (3, 16, 12))
    full = oracle.ag_gemm(_bits(X), _bits(B1), 1.0, "fp32")
    rows = np.array([0, 7, 39, 20])
    np.testing.assert_array_equal(oracle.ag_gemm(_bits(X), _bits(B1), 1.0, "fp32", rows=rows),
                                  full[:, rows])


def test_ffn_chain_identity_with_the_gemm_rs_oracle():
    """The two halves of a tensor-parallel FFN, each by its own oracle: the
    AG+GEMM output H_r is the A_r of the GEMM+RS, and the result is
    X @ (sum_r B1_r B2_r), checked in int64."""
    rng = np.random.default_rng(8)
    W, M, K, Nr, N2 = 4, 32, 24, 8, 16
    X = rng.integers(-2, 3, (M, K))
    B1 = rng.integers(-1, 2, (W, K, Nr))
    B2 = rng.integers(-1, 2, (W, Nr, N2))
    H = oracle.ag_gemm(_bits(X), _bits(B1), 1.0, "fp32")          # [W][M][Nr], exact
    Y = oracle.gemm_rs(_bits(H), _bits(B2), None, 1.0, 0.0, "fp32")
    ref = sum(X @ B1[r] @ B2[r] for r in range(W)).astype(np.float32)
    np.testing.assert_array_equal(Y, ref)


def _printed_orders():
    orders = {}
    with open(GOLDEN) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rank, seq = line.split(":")
                orders[int(rank)] = [int(x) for x in seq.split()]
    return orders


def test_ag_chunk_order_is_the_printed_rank_offset_order():
    """Each rank takes its chunks starting at its own, as printed for ranks 0
    and 1 of eight ("flux精读" §4.1).  The other ranks and sizes are pinned by
    the properties in test_oracle_schedule.py (every chunk once per rank, own
    chunk first, W distinct chunks per step)."""
    order = oracle.ag_chunk_order(8)
    for r, seq in _printed_orders().items():
        assert order[r].tolist() == seq
