"""The tensor-parallel FFN chain on one GPU (AG+GEMM, then GEMM+RS on its
output) through ffn_tp_run, against the two oracles composed."""
import numpy as np
import pytest
import torch

import oracle
from helpers import assert_close, to_np_y
from tensor_gemm_reduce_tcgen05_gb300.inputs import _draw, bf16_bits, make_ag_inputs

pytestmark = pytest.mark.gpu


def run_chain(W, M, K, Nr, N2, dist, alpha1, alpha2, beta, y_dtype):
    from tensor_gemm_reduce_tcgen05_gb300 import binding as b
    dev = torch.device("cuda", 0)
    X, B1 = make_ag_inputs(W, M, Nr, K, dist, dist)
    B2 = _draw((W, Nr, N2), dist, 13)
    C = _draw((M, N2), dist, 14) if beta != 0 else None
    ag = b.AgGemm(M, Nr, K, W, alpha1, "bf16", device=dev)
    rs = b.GemmRS(M, N2, W * Nr, W, alpha2, beta, y_dtype, device=dev)
    Xd, B1d, B2d = X.to(dev), B1.to(dev), B2.to(dev)
    Cd = None if C is None else C.to(dev)
    H = ag.new_output()
    Y = rs.new_output()
    for _ in range(2):
        b.ffn_tp_run(ag.handle, rs.handle, Xd.data_ptr(), B1d.data_ptr(), H.data_ptr(),
                     B2d.data_ptr(), 0 if Cd is None else Cd.data_ptr(), Y.data_ptr(),
                     torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    assert ag.status() == 0 and rs.status() == 0
    # oracle chain on the oracle's own bf16 H
    h_ref = oracle.ag_gemm(bf16_bits(X), bf16_bits(B1), alpha1, "bf16")
    y_ref = oracle.gemm_rs(h_ref, bf16_bits(B2), None if C is None else bf16_bits(C), alpha2, beta,
                           y_dtype)
    return to_np_y(H), h_ref, to_np_y(Y), y_ref


@pytest.mark.parametrize("y_dtype", ["fp32", "bf16"])
def test_chain_integer_inputs_bit_exact(y_dtype):
    """K = 64 keeps every |H| <= 256, exact in bf16, so both stages are exact."""
    h, h_ref, y, y_ref = run_chain(4, 1024, 64, 64, 256, "int", 1.0, 1.0, 1.0, y_dtype)
    np.testing.assert_array_equal(h, h_ref)
    np.testing.assert_array_equal(y, y_ref)


@pytest.mark.parametrize("y_dtype", ["fp32", "bf16"])
def test_chain_normal_inputs_within_tolerance(y_dtype):
    h, h_ref, y, y_ref = run_chain(8, 2048, 512, 256, 512, "normal", 1.0, 0.5, 0.0, y_dtype)
    for r in range(8):
        assert_close(h[r], h_ref[r], "bf16", f"H rank {r}")
    assert_close(y, y_ref, y_dtype, "Y")


def test_chain_rejects_mismatched_handles():
    from tensor_gemm_reduce_tcgen05_gb300 import binding as b
    dev = torch.device("cuda", 0)
    ag = b.AgGemm(1024, 64, 64, 4, 1.0, "bf16", device=dev)
    rs = b.GemmRS(1024, 256, 4 * 128, 4, 1.0, 0.0, "fp32", device=dev)  # K/W = 128 != 64
    with pytest.raises(b.GemmRSError):
        b.ffn_tp_run(ag.handle, rs.handle, 0, 0, 0, 0, 0, 0, 0)
