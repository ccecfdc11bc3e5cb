"""The bounds-checked build (libgemm_rs_checked.so, compiled with
GEMM_RS_CHECKED) runs the parity cases in a process of its own: every global
access of the GEMM+RS epilogue and folds, and of the AG+GEMM copies, signals
and H stores, is tested against its buffer, and one outside it would be
skipped and reported as GEMM_RS_ERR_BOUNDS.  The runs must
report none and stay bit-exact.  (A memory checker is not available on this
pool; this and the NaN-poison tests stand in for it.)

Also fault injection on the host side of the state words: a workspace whose
tile state words hold garbage gives a wrong result but no hang and no fault
(every wait is bounded and every slot index comes from the schedule), and
gemm_rs_reset restores exact results."""
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

from helpers import inputs, oracle_y, run_gpu, to_np_y

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CHECKED = os.path.join(ROOT, "tensor_gemm_reduce_tcgen05_gb300", "libgemm_rs_checked.so")

SCRIPT = r"""
import sys
sys.path.insert(0, {root!r}); sys.path.insert(0, {tests!r})
import numpy as np
from tensor_gemm_reduce_tcgen05_gb300 import binding as b
from helpers import inputs, oracle_y, run_gpu
assert "checked" in b.gemm_rs_version(), b.gemm_rs_version()
cases = 0
shapes = [(2, 256, 256, 256), (3, 300, 520, 200), (8, 64, 512, 192), (1, 200, 72, 64),
          (16, 16 * 9, 136, 72), (4, 512, 768, 128), (4, 512, 320, 128)]
for (W, M, N, Kpr) in shapes:
    A, B, C = inputs(W, M, N, Kpr, "int", c_dist="int")
    ref = oracle_y(A, B, C, 0.5, 1.0, "fp32")
    for tile in ((128, 256), (128, 128), (128, 64), (256, 256)):
        for mode in (0, 1, 2):
            for order in (1, 2):
                y, plan, op = run_gpu(A, B, C, W, M, N, Kpr, 0.5, 1.0, "fp32", tile_m=tile[0],
                                      tile_n=tile[1], reduce_mode=mode, rank_order=order,
                                      poison=True, calls=2)
                np.testing.assert_array_equal(y, ref)
                cases += 1
print("checked cases", cases)
from tensor_gemm_reduce_tcgen05_gb300.inputs import make_ag_inputs
from helpers import to_np_y
import oracle, torch
ag_cases = 0
for (W, M, N, K) in [(2, 512, 256, 256), (3, 768, 264, 200), (1, 256, 72, 64),
                     (8, 2048, 512, 128), (16, 16 * 256, 64, 64), (4, 2048, 1000, 136)]:
    X, B1 = make_ag_inputs(W, M, N, K, "int", "int")
    for y_dtype in ("fp32", "bf16"):
        op = b.AgGemm(M, N, K, W, 1.0, y_dtype, device="cuda:0")
        H = op.new_output()
        H.view(torch.uint8).fill_(0xFF)
        for _ in range(2):
            op.run(X.cuda(), B1.cuda(), H)
        torch.cuda.synchronize()
        assert op.status() == 0
        np.testing.assert_array_equal(to_np_y(H), oracle.ag_gemm(
            oracle.bf16_from_float(X.float().numpy()), oracle.bf16_from_float(B1.float().numpy()),
            1.0, y_dtype))
        ag_cases += 1
print("checked ag cases", ag_cases)
# M*N = 2^31 output elements: the 64-bit index arithmetic of the epilogue and folds
W, M, N, Kpr = 2, 65536, 32768, 64
A, B, _ = inputs(W, M, N, Kpr, "int")
rows = np.array([0, 1, M // 2, M - 2, M - 1])
ref = oracle_y(A, B, None, 1.0, 0.0, "fp32", rows=rows)
for mode in (0, 1, 2):
    op = b.GemmRS(M, N, W * Kpr, W, 1.0, 0.0, "fp32", device="cuda:0")
    b.gemm_rs_set_reduce_mode(op.handle, mode)
    Y = op.run(A.cuda(), B.cuda())
    torch.cuda.synchronize()
    assert op.status() == 0
    np.testing.assert_array_equal(Y[torch.from_numpy(rows).cuda()].cpu().numpy(), ref)
    del Y, op
    torch.cuda.empty_cache()
print("checked big ok")
# the entry point that allocates nothing: its static scratch, every access checked
na_cases = 0
for (W, M, N, Kpr, beta, y_dtype) in [(4, 512, 520, 200, 1.0, "bf16"), (8, 64, 1024, 192, 0.0, "fp32"),
                                     (3, 300, 520, 64, 0.5, "fp32")]:
    A, B, C = inputs(W, M, N, Kpr, "int", c_dist="int" if beta != 0 else None)
    ref = oracle_y(A, B, C if beta != 0 else None, 1.0, beta, y_dtype)
    code = b.GEMM_RS_BF16 if y_dtype == "bf16" else b.GEMM_RS_FP32
    Ad, Bd = A.cuda(), B.cuda()
    Cd = C.cuda() if beta != 0 else None
    for _ in range(2):
        Y = torch.empty((M, N), dtype=torch.bfloat16 if y_dtype == "bf16" else torch.float32,
                        device="cuda:0")
        Y.view(torch.uint8).fill_(0xFF)
        b.gemm_rs_run_noalloc(M, N, W * Kpr, W, 1.0, beta, code, Ad.data_ptr(), Bd.data_ptr(),
                              0 if Cd is None else Cd.data_ptr(), Y.data_ptr(), 0)
        torch.cuda.synchronize()
        assert b.gemm_rs_noalloc_status(0) == 0
        np.testing.assert_array_equal(to_np_y(Y), ref)
    na_cases += 1
print("checked noalloc cases", na_cases)
"""


def test_checked_build_finds_no_access_out_of_bounds():
    assert os.path.exists(CHECKED), "build() makes the checked library too"
    env = dict(os.environ, GEMM_RS_LIBRARY=CHECKED)
    r = subprocess.run([sys.executable, "-c", SCRIPT.format(root=ROOT, tests=HERE)], env=env,
                       capture_output=True, text=True, timeout=1200)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-3000:]
    assert "checked cases 168" in r.stdout
    assert "checked ag cases 12" in r.stdout
    assert "checked big ok" in r.stdout
    assert "checked noalloc cases 3" in r.stdout


@pytest.mark.parametrize("mode", [0, 1, 2])
def test_garbage_state_words_then_reset(mode):
    from tensor_gemm_reduce_tcgen05_gb300 import binding as b
    W, M, N, Kpr = 4, 512, 768, 128
    A, B, _ = inputs(W, M, N, Kpr, "int")
    dev = torch.device("cuda", 0)
    op = b.GemmRS(M, N, W * Kpr, W, 1.0, 0.0, "fp32", device=dev)
    b.gemm_rs_set_reduce_mode(op.handle, mode)
    b.gemm_rs_set_timeout_cycles(op.handle, 1 << 26)
    Ad, Bd = A.to(dev), B.to(dev)
    flags = op.flags_view()
    g = torch.Generator(device="cpu").manual_seed(mode)
    flags.copy_(torch.randint(0, 1 << 30, flags.shape, generator=g, dtype=torch.int32))
    op.run(Ad, Bd)
    torch.cuda.synchronize()
    assert op.status() in (b.GEMM_RS_OK, b.GEMM_RS_ERR_TIMEOUT)
    op.reset()
    b.gemm_rs_set_timeout_cycles(op.handle, 1 << 32)
    for _ in range(2):
        Y = op.run(Ad, Bd)
        torch.cuda.synchronize()
        assert op.status() == b.GEMM_RS_OK
        np.testing.assert_array_equal(to_np_y(Y), oracle_y(A, B, None, 1.0, 0.0, "fp32"))
        assert int(op.flags_view().abs().sum()) == 0
