"""Pins for the CPU oracle (no GPU needed).

Each test compares the oracle with something other than itself:
  * exact rational arithmetic (Python fractions) on tiny inputs, within the
    fp32 rounding bound;
  * numpy float64 matmul of the full-K GEMM (the library routine) for beta=0
    and for W=1;
  * integer-valued inputs, where every sum is exact and the result is unique;
  * closed forms: alpha=0, beta=0, alpha=beta=0, beta=0 with NaN in C;
  * a crafted case where only the rank-order fp32 fold gives the printed value;
  * torch's bf16 rounding for the output conversion.
Each plausible mistake (a dropped rank, k or C term, a wrong sign, a
transposed operand, C applied once instead of per rank, a different fold
order, truncation instead of round-to-nearest-even) fails at least one test.
"""
import math
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from tensor_gemm_reduce_tcgen05_gb300.inputs import bf16_bits, make_inputs

U = 2.0 ** -24  # unit roundoff of fp32


def _f(bits):
    return oracle.float_from_bf16(bits).astype(np.float64)


def _exact(A, B, C, alpha, beta):
    """Exact sum over ranks of alpha*A_r*B_r + beta*C, as Fractions, plus the
    sum of magnitudes of the terms (for the rounding bound)."""
    W, M, Kpr = A.shape
    N = B.shape[2]
    Af, Bf = _f(A), _f(B)
    Cf = None if C is None else _f(C)
    al, be = Fraction(alpha), Fraction(beta)
    ex = [[Fraction(0)] * N for _ in range(M)]
    mag = np.zeros((M, N))
    for r in range(W):
        for m in range(M):
            for n in range(N):
                s = sum((Fraction(Af[r, m, k]) * Fraction(Bf[r, k, n]) for k in range(Kpr)),
                        Fraction(0))
                t = al * s
                tm = abs(float(alpha)) * float(sum(abs(Af[r, m, k] * Bf[r, k, n])
                                                   for k in range(Kpr)))
                if beta != 0:
                    t += be * Fraction(Cf[m, n])
                    tm += abs(beta * Cf[m, n])
                ex[m][n] += t
                mag[m, n] += tm
    return ex, mag


@pytest.mark.parametrize("W,M,N,Kpr,alpha,beta,seed", [
    (1, 3, 5, 4, 1.0, 0.0, 11),
    (2, 4, 3, 5, 1.0, 0.0, 12),
    (3, 6, 4, 2, 0.5, 1.0, 13),
    (4, 4, 7, 3, -1.25, 0.75, 14),
    (2, 2, 8, 16, 2.0, -1.0, 15),
])
def test_exact_rational_tiny(W, M, N, Kpr, alpha, beta, seed):
    A, B, C = make_inputs(W, M, N, Kpr, "uniform", "uniform",
                          "normal1" if beta != 0 else None, seeds=(seed, seed + 1, seed + 2))
    A, B = bf16_bits(A), bf16_bits(B)
    C = None if C is None else bf16_bits(C)
    y = oracle.gemm_rs(A, B, C, alpha, beta, "fp32").astype(np.float64)
    ex, mag = _exact(A, B, C, alpha, beta)
    for m in range(M):
        for n in range(N):
            bound = (W + 1) * U * mag[m, n] * 1.01 + 1e-30
            assert abs(y[m, n] - float(ex[m][n])) <= bound, (m, n, y[m, n], float(ex[m][n]))


@pytest.mark.parametrize("W,M,N,Kpr", [(1, 64, 48, 96), (4, 96, 40, 64), (8, 64, 24, 32)])
def test_matches_numpy_full_k_gemm(W, M, N, Kpr):
    """beta = 0: the sum over ranks equals the full-K GEMM of the concatenated
    shards (W = 1 is a plain GEMM)."""
    A, B, _ = make_inputs(W, M, N, Kpr, "normal", "normal")
    Ab, Bb = bf16_bits(A), bf16_bits(B)
    alpha = 1.5
    y = oracle.gemm_rs(Ab, Bb, None, alpha, 0.0, "fp32").astype(np.float64)
    A_full = np.concatenate([_f(Ab)[r] for r in range(W)], axis=1)   # [M, K]
    B_full = np.concatenate([_f(Bb)[r] for r in range(W)], axis=0)   # [K, N]
    ref = alpha * (A_full @ B_full)
    mag = abs(alpha) * (np.abs(A_full) @ np.abs(B_full))
    assert np.all(np.abs(y - ref) <= (W + 1) * U * mag * 1.01 + 1e-30)
    # The operand orientation is pinned too: the transposed product differs.
    if M == N:
        assert not np.allclose(y, alpha * (A_full @ B_full).T, atol=1e-3)


@pytest.mark.parametrize("W,M,N,Kpr,alpha,beta", [
    (2, 8, 8, 16, 1.0, 0.0), (4, 12, 16, 8, 0.5, 1.0), (8, 16, 8, 24, 1.0, 1.0),
    (3, 9, 24, 40, -2.0, 0.5),
])
def test_integer_inputs_exact(W, M, N, Kpr, alpha, beta):
    """Integer inputs: every partial sum is exact in fp32, so the result is
    unique and equals the integer computation bit for bit."""
    A, B, C = make_inputs(W, M, N, Kpr, "int", "int", "int" if beta != 0 else None)
    Ai = A.to(torch.int64).numpy()
    Bi = B.to(torch.int64).numpy()
    S = sum(Ai[r] @ Bi[r] for r in range(W)).astype(np.float64)
    ref = alpha * S
    if beta != 0:
        ref = ref + W * beta * C.to(torch.int64).numpy().astype(np.float64)
    y = oracle.gemm_rs(bf16_bits(A), bf16_bits(B), None if C is None else bf16_bits(C),
                       alpha, beta, "fp32")
    np.testing.assert_array_equal(y.astype(np.float64), ref)


def test_closed_form_alpha_zero_is_w_times_beta_c():
    """alpha = 0: Y = W * beta * C exactly.  C is applied by every rank
    (the literal reading of the per-rank epilogue)."""
    W, M, N, Kpr = 4, 8, 16, 8
    A, B, C = make_inputs(W, M, N, Kpr, "uniform", "uniform", "normal1")
    y = oracle.gemm_rs(bf16_bits(A), bf16_bits(B), bf16_bits(C), 0.0, 1.0, "fp32")
    np.testing.assert_array_equal(y, (W * C.to(torch.float32)).numpy())
    y2 = oracle.gemm_rs(bf16_bits(A), bf16_bits(B), bf16_bits(C), 0.0, -0.5, "fp32")
    np.testing.assert_array_equal(y2, (-0.5 * W * C.to(torch.float32)).numpy())


def test_closed_form_zero_and_nan_c_ignored_when_beta_zero():
    W, M, N, Kpr = 2, 4, 8, 8
    A, B, _ = make_inputs(W, M, N, Kpr, "uniform", "uniform")
    Cnan = np.full((M, N), 0x7fc0, dtype=np.uint16)  # bf16 NaN
    y = oracle.gemm_rs(bf16_bits(A), bf16_bits(B), None, 0.0, 0.0, "fp32")
    assert np.all(y == 0.0)
    y1 = oracle.gemm_rs(bf16_bits(A), bf16_bits(B), None, 1.0, 0.0, "fp32")
    y2 = oracle.gemm_rs(bf16_bits(A), bf16_bits(B), Cnan, 1.0, 0.0, "fp32")
    assert np.all(np.isfinite(y2))
    np.testing.assert_array_equal(y1, y2)
    y3 = oracle.gemm_rs(bf16_bits(A), bf16_bits(B), Cnan, 1.0, 1.0, "fp32")
    assert np.all(np.isnan(y3))


def test_fold_is_in_rank_order():
    """p_0 = 2^27, p_1 = -2^27, p_2 = 1.  The rank-order fold gives
    (p_0 + p_1) + p_2 = 1.  Folding in any other order gives 0, because
    2^27 + 1 rounds back to 2^27 in fp32."""
    W, M, N, Kpr = 3, 3, 1, 1
    a = np.array([2.0 ** 14, -(2.0 ** 14), 1.0], dtype=np.float32)
    b = np.array([2.0 ** 13, 2.0 ** 13, 1.0], dtype=np.float32)
    A = np.zeros((W, M, Kpr), dtype=np.float32)
    B = np.zeros((W, Kpr, N), dtype=np.float32)
    for r in range(W):
        A[r, :, 0] = a[r]
        B[r, 0, 0] = b[r]
    y = oracle.gemm_rs(oracle.bf16_from_float(A), oracle.bf16_from_float(B), None, 1.0, 0.0,
                       "fp32")
    assert np.all(y == 1.0)
    # Reversing the rank order gives the other answer: the fold order matters.
    yr = oracle.gemm_rs(oracle.bf16_from_float(A[::-1].copy()),
                        oracle.bf16_from_float(B[::-1].copy()), None, 1.0, 0.0, "fp32")
    assert np.all(yr == 0.0)


def test_two_level_fold_associates_by_group():
    """p = (2^27, 1, -2^27, 1).  One level: ((2^27 + 1) + -2^27) + 1 = 1, since
    2^27 + 1 rounds to 2^27.  Two levels of two ranks: (2^27 + 1) + (-2^27 + 1)
    = 2^27 + -2^27 = 0.  The group sums are formed first, then added."""
    W, M, N, Kpr = 4, 4, 1, 1
    a = np.array([2.0 ** 14, 1.0, -(2.0 ** 14), 1.0], dtype=np.float32)
    b = np.array([2.0 ** 13, 1.0, 2.0 ** 13, 1.0], dtype=np.float32)
    A = np.zeros((W, M, Kpr), dtype=np.float32)
    B = np.zeros((W, Kpr, N), dtype=np.float32)
    for r in range(W):
        A[r, :, 0] = a[r]
        B[r, 0, 0] = b[r]
    Ab, Bb = oracle.bf16_from_float(A), oracle.bf16_from_float(B)
    assert np.all(oracle.gemm_rs(Ab, Bb, None, 1.0, 0.0, "fp32") == 1.0)
    assert np.all(oracle.gemm_rs(Ab, Bb, None, 1.0, 0.0, "fp32", split=2) == 0.0)
    # split 0 and out-of-range splits are the one-level fold
    assert np.all(oracle.gemm_rs(Ab, Bb, None, 1.0, 0.0, "fp32", split=4) == 1.0)


def test_two_level_fold_is_exact_on_integer_inputs():
    """Integer-valued inputs make every partial sum exact, so any association
    gives the one-level result bit for bit (here: int64 products)."""
    rng = np.random.default_rng(9)
    W, M, N, Kpr = 6, 12, 16, 24
    A = rng.integers(-2, 3, (W, M, Kpr)).astype(np.float32)
    B = rng.integers(-2, 3, (W, Kpr, N)).astype(np.float32)
    ref = sum(A[r].astype(np.int64) @ B[r].astype(np.int64) for r in range(W)).astype(np.float32)
    Ab, Bb = oracle.bf16_from_float(A), oracle.bf16_from_float(B)
    for split in (0, 1, 3, 5):
        np.testing.assert_array_equal(oracle.gemm_rs(Ab, Bb, None, 1.0, 0.0, "fp32", split=split),
                                      ref)


def test_bf16_conversion_matches_torch_rne():
    g = torch.Generator().manual_seed(5)
    x = torch.randn(200000, generator=g) * 1000
    specials = torch.tensor([0.0, -0.0, float("inf"), -float("inf"), 3.3895314e38, 3.4e38,
                             1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, 1.0 + 2 ** -9, 1e-40, -1e-40],
                            dtype=torch.float32)
    # exact ties: the low 16 bits are 0x8000
    ties = (torch.randint(0, 2 ** 12, (1000,), generator=g, dtype=torch.int32) * 65536
            + 32768 + 0x3f800000).view(torch.float32)
    assert torch.all(torch.isfinite(ties))
    x = torch.cat([x, specials, ties])
    ours = oracle.bf16_from_float(x.numpy())
    ref = x.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(ours, ref)
    nan = oracle.bf16_from_float(np.array([float("nan")], dtype=np.float32))
    assert oracle.float_from_bf16(nan)[0] != oracle.float_from_bf16(nan)[0]


def test_bf16_output_is_rne_of_fp32_output():
    W, M, N, Kpr = 4, 16, 24, 32
    A, B, C = make_inputs(W, M, N, Kpr, "normal", "normal", "normal1")
    args = (bf16_bits(A), bf16_bits(B), bf16_bits(C), 0.5, 1.0)
    y32 = oracle.gemm_rs(*args, y_dtype="fp32")
    y16 = oracle.gemm_rs(*args, y_dtype="bf16")
    ref = torch.from_numpy(y32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(y16, ref)


def test_row_sample_equals_full_rows():
    W, M, N, Kpr = 4, 40, 16, 24
    A, B, C = make_inputs(W, M, N, Kpr, "normal", "normal", "normal1")
    args = (bf16_bits(A), bf16_bits(B), bf16_bits(C), 0.5, 1.0)
    full = oracle.gemm_rs(*args, y_dtype="fp32")
    rows = [39, 0, 17, 10, 10]
    part = oracle.gemm_rs(*args, y_dtype="fp32", rows=rows)
    np.testing.assert_array_equal(part, full[rows])


def test_row_chunk_partition():
    """Chunk c is the R = M/W contiguous rows [c*R, (c+1)*R): W chunks of
    equal size that tile the output in order."""
    for W, M in [(1, 5), (2, 256), (8, 64), (3, 300), (8, 4096)]:
        c, i = oracle.row_chunk(W, M)
        R = M // W
        counts = np.bincount(c, minlength=W)
        assert counts.tolist() == [R] * W
        assert np.all(np.diff(c) >= 0)
        assert np.all(i[c == c] < R)
        starts = np.nonzero(i == 0)[0]
        assert starts.tolist() == [k * R for k in range(W)]
    with pytest.raises(ValueError):
        oracle.row_chunk(3, 10)


def test_rejects_bad_arguments():
    A = np.zeros((2, 3, 4), dtype=np.uint16)
    B = np.zeros((2, 4, 8), dtype=np.uint16)
    with pytest.raises(ValueError):
        oracle.gemm_rs(A, B, None, 1.0, 0.0)  # M = 3 is not a multiple of W = 2
    A = np.zeros((2, 4, 4), dtype=np.uint16)
    with pytest.raises(ValueError):
        oracle.gemm_rs(A, B, None, 1.0, 1.0)  # beta != 0 needs C


def test_empty_shapes():
    for (W, M, N, Kpr) in [(2, 0, 8, 4), (2, 4, 0, 4), (2, 4, 8, 0)]:
        A = np.zeros((W, M, Kpr), dtype=np.uint16)
        B = np.zeros((W, Kpr, N), dtype=np.uint16)
        y = oracle.gemm_rs(A, B, None, 1.0, 0.0, "fp32")
        assert y.shape == (M, N)
        assert np.all(y == 0)
    # K = 0 with beta != 0 leaves Y = W * beta * C
    C = bf16_bits(make_inputs(1, 4, 8, 1, "uniform", "uniform", "normal1")[2])
    y = oracle.gemm_rs(np.zeros((2, 4, 0), np.uint16), np.zeros((2, 0, 8), np.uint16), C,
                       1.0, 1.0, "fp32")
    np.testing.assert_array_equal(y, 2 * oracle.float_from_bf16(C))
