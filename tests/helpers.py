"""Shared test helpers: run the CUDA path through the C ABI and compare it
with the oracle on the same seeded inputs."""
from __future__ import annotations

import numpy as np
import torch

import oracle
from tensor_gemm_reduce_tcgen05_gb300.inputs import bf16_bits, make_inputs

# Tolerances of the path (fp32 partials, fp32 fold, bf16 or fp32 output):
#   fp32 Y: relative Frobenius error <= 1e-4, and per element |d| <= 1e-3 + 1e-3*|ref|
#   bf16 Y: per element |d| <= 1e-2 + 1e-2*|ref|
FP32_FROB = 1e-4
FP32_ATOL = 1e-3
FP32_RTOL = 1e-3
BF16_ATOL = 1e-2
BF16_RTOL = 1e-2


def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    return oracle.float_from_bf16(bits)


def to_np_y(Y: torch.Tensor) -> np.ndarray:
    """A device Y as numpy: float32 for fp32, uint16 bit patterns for bf16."""
    Yc = Y.detach().cpu()
    if Yc.dtype == torch.bfloat16:
        return bf16_bits(Yc)
    return Yc.numpy()


def assert_close(y_gpu: np.ndarray, y_ref: np.ndarray, y_dtype: str, what: str = ""):
    """Tolerances of the path, element by element."""
    if y_dtype == "bf16":
        g, r = bf16_to_f32(y_gpu).astype(np.float64), bf16_to_f32(y_ref).astype(np.float64)
        bad = np.abs(g - r) > BF16_ATOL + BF16_RTOL * np.abs(r)
        assert not bad.any(), f"{what}: {bad.sum()} elements outside bf16 tolerance; first at " \
                              f"{np.argwhere(bad)[:5].tolist()} gpu={g[bad][:5]} ref={r[bad][:5]}"
    else:
        g, r = y_gpu.astype(np.float64), y_ref.astype(np.float64)
        bad = np.abs(g - r) > FP32_ATOL + FP32_RTOL * np.abs(r)
        assert not bad.any(), f"{what}: {bad.sum()} elements outside fp32 tolerance; first at " \
                              f"{np.argwhere(bad)[:5].tolist()} gpu={g[bad][:5]} ref={r[bad][:5]}"
        den = np.linalg.norm(r)
        if den > 0:
            frob = np.linalg.norm(g - r) / den
            assert frob <= FP32_FROB, f"{what}: relative Frobenius error {frob:.3e}"
    assert np.all(np.isfinite(g)) == np.all(np.isfinite(r)), f"{what}: non-finite mismatch"


def run_gpu(A, B, C, W, M, N, Kpr, alpha, beta, y_dtype, tile_n=None, calls=1, poison=False,
            tile_m=None, reduce_mode=None, rank_order=None):
    """Run the fused path through the C ABI.  Returns (Y as numpy, plan, op)."""
    from tensor_gemm_reduce_tcgen05_gb300 import binding as b
    dev = torch.device("cuda", 0)
    op = b.GemmRS(M, N, W * Kpr, W, alpha, beta, y_dtype, device=dev, tile_n=tile_n,
                  tile_m=tile_m)
    if reduce_mode is not None:
        b.gemm_rs_set_reduce_mode(op.handle, reduce_mode)
    if rank_order is not None:
        b.gemm_rs_set_schedule(op.handle, 0, 0, rank_order)
    Ad, Bd = A.to(dev), B.to(dev)
    Cd = None if C is None else C.to(dev)
    Y = op.new_output()
    if poison:
        Y.view(torch.uint8).fill_(0xFF)                      # NaN in both dtypes
        op.workspace[256 + op.flags_view().numel() * 4:].fill_(0xFF)
    for _ in range(calls):
        op.run(Ad, Bd, Cd, Y)
    torch.cuda.synchronize()
    assert op.status() == 0, "device status reports a timeout"
    return to_np_y(Y), op.plan, op


def oracle_y(A, B, C, alpha, beta, y_dtype, rows=None):
    return oracle.gemm_rs(bf16_bits(A), bf16_bits(B), None if C is None else bf16_bits(C),
                          alpha, beta, y_dtype, rows=rows)


def inputs(W, M, N, Kpr, dist="normal", c_dist=None, seeds=(1, 2, 3)):
    return make_inputs(W, M, N, Kpr, dist, dist, c_dist, seeds=seeds)
