"""C-ABI checks that need no GPU: the library loads, exports every symbol
include/gemm_rs.h and include/ag_gemm.h declare, validates arguments before
touching the device, and its host-side tile schedules equal the oracle's bit
for bit."""
import os
import re

import numpy as np
import pytest

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "gemm_rs.h")
HEADERS = [HEADER, os.path.join(ROOT, "include", "ag_gemm.h")]


@pytest.fixture(scope="module")
def b():
    from tensor_gemm_reduce_tcgen05_gb300 import build, binding
    build.build()
    binding.lib()
    return binding


def _declared():
    names = set()
    for h in HEADERS:
        text = re.sub(r"/\*.*?\*/", "", open(h).read(), flags=re.S)
        names |= set(re.findall(r"\b((?:gemm_rs|ag_gemm|ffn_tp)_[a-z_]+)\s*\(", text))
    return sorted(names)


def test_exports_every_declared_symbol(b):
    names = _declared()
    assert "gemm_rs_create" in names and "gemm_rs_run" in names and "gemm_rs_destroy" in names
    assert "ag_gemm_create" in names and "ag_gemm_run" in names and "ag_gemm_destroy" in names
    assert "ffn_tp_run" in names
    L = b.lib()
    missing = [n for n in names if not hasattr(L, n)]
    assert not missing, missing


def test_checked_build_exports_the_same_symbols():
    """The bounds-checked build is the same ABI: every declared symbol is there,
    and its version string names the flavour."""
    import ctypes
    from tensor_gemm_reduce_tcgen05_gb300 import build
    path = build.build(checked=True)
    L = ctypes.CDLL(path)
    missing = [n for n in _declared() if not hasattr(L, n)]
    assert not missing, missing
    L.gemm_rs_version.restype = ctypes.c_char_p
    assert b"checked" in L.gemm_rs_version()


@pytest.mark.parametrize("path", ["gemm_rs.h", "ag_gemm.h"])
def test_no_torch_types_in_header(path):
    text = open(os.path.join(ROOT, "include", path)).read()
    assert "torch" not in text.lower().replace("pytorch", "")
    assert "at::" not in text and "c10" not in text


def test_version(b):
    assert "sm_103a" in b.gemm_rs_version()


@pytest.mark.parametrize("W,M,N,bn", [
    (2, 256, 256, 256), (8, 4096, 4096, 256), (8, 8192, 8192, 256), (8, 64, 8192, 64),
    (4, 16384, 5120, 256), (3, 300, 520, 128), (1, 200, 72, 64), (5, 640, 1000, 256),
    (16, 16 * 7, 64, 64), (7, 7 * 129, 264, 128),
])
def test_schedule_matches_oracle(b, W, M, N, bn):
    orders = ((b.GEMM_RS_RANKS_INTERLEAVED, "interleaved"), (b.GEMM_RS_RANKS_SEQUENTIAL, "sequential"),
              (b.GEMM_RS_RANKS_DEFAULT, "sequential"))
    for G, RG in ((0, 0), (1, 0), (2, 3), (5, 1), (0, 2), (3, 5)):
        for code, order in orders:
            ours = b.gemm_rs_schedule(M, N, W, 128, bn, G, RG, code)
            ref = oracle.schedule(W, M, N, 128, bn, G, RG, order)
            np.testing.assert_array_equal(ours, ref)
            # the CTA-pair kernel walks 256-row tiles
            np.testing.assert_array_equal(b.gemm_rs_schedule(M, N, W, 256, 256, G, RG, code),
                                          oracle.schedule(W, M, N, 256, 256, G, RG, order))


def test_workspace_bytes(b):
    assert b.gemm_rs_workspace_bytes(256, 256, 512, 2) == 256 + 256 + 2 * 256 * 256 * 4
    # invalid shapes give 0
    assert b.gemm_rs_workspace_bytes(255, 256, 512, 2) == 0
    assert b.gemm_rs_workspace_bytes(256, 250, 512, 2) == 0
    assert b.gemm_rs_workspace_bytes(256, 256, 511, 2) == 0
    assert b.gemm_rs_workspace_bytes(256, 256, 2 * 12, 2) == 0   # K/W = 12 is not a multiple of 8
    assert b.gemm_rs_workspace_bytes(256, 256, 512, 0) == 0
    assert b.gemm_rs_workspace_bytes(256, 256, 512, 17) == 0
    # covers every tile width: padded to 128 rows and 256 columns
    ws = b.gemm_rs_workspace_bytes(300, 520, 3 * 200, 3)
    assert ws >= 3 * 384 * 768 * 4


@pytest.mark.parametrize("M,N,K,W,code", [
    (255, 256, 512, 2, -2), (256, 250, 512, 2, -2), (256, 256, 511, 2, -2), (256, 256, 24, 2, -2),
    (-8, 256, 512, 2, -2), (256, 256, 512, 0, -1), (256, 256, 512, 17, -1),
])
def test_create_rejects_bad_shapes_before_touching_the_device(b, M, N, K, W, code):
    with pytest.raises(b.GemmRSError) as e:
        b.gemm_rs_create(M, N, K, W, 1.0, 0.0, 0, 0, 0, 1 << 20, 1 << 30, 0)
    assert e.value.code == code
    assert b.gemm_rs_last_error() != ""


def test_create_rejects_bad_dtypes_and_workspace(b):
    with pytest.raises(b.GemmRSError) as e:
        b.gemm_rs_create(256, 256, 512, 2, 1.0, 0.0, 1, 0, 0, 1 << 20, 1 << 30, 0)
    assert e.value.code == b.GEMM_RS_ERR_UNSUPPORTED
    with pytest.raises(b.GemmRSError) as e:
        b.gemm_rs_create(256, 256, 512, 2, 1.0, 0.0, 0, 0, 0, 0, 1 << 30, 0)
    assert e.value.code == b.GEMM_RS_ERR_ARG
    with pytest.raises(b.GemmRSError) as e:
        b.gemm_rs_create(256, 256, 512, 2, 1.0, 0.0, 0, 0, 0, (1 << 20) + 16, 1 << 30, 0)
    assert e.value.code == b.GEMM_RS_ERR_ALIGN
    with pytest.raises(b.GemmRSError) as e:
        b.gemm_rs_create(256, 256, 512, 2, 1.0, 0.0, 0, 0, 0, 1 << 20, 1000, 0)
    assert e.value.code == b.GEMM_RS_ERR_WORKSPACE
    with pytest.raises(b.GemmRSError) as e:
        b.gemm_rs_create(256, 256, 512, 2, float("nan"), 0.0, 0, 0, 0, 1 << 20, 1 << 30, 0)
    assert e.value.code == b.GEMM_RS_ERR_ARG


def test_null_handle_calls_fail_cleanly(b):
    for fn in (b.lib().gemm_rs_status, b.lib().gemm_rs_reset):
        assert fn(None, None) == b.GEMM_RS_ERR_ARG
    assert b.lib().gemm_rs_run(None, None, None, None, None, None) == b.GEMM_RS_ERR_ARG
    assert b.lib().gemm_rs_destroy(None) == 0
    with pytest.raises(b.GemmRSError):
        b.gemm_rs_schedule(255, 256, 2, 128, 256)
    with pytest.raises(b.GemmRSError):
        b.gemm_rs_schedule(256, 256, 2, 64, 256)
    with pytest.raises(b.GemmRSError):
        b.gemm_rs_schedule(256, 256, 2, 128, 256, 0, 0, 3)  # unknown rank order


def test_reduce_partials_validates(b):
    L = b.lib()
    assert L.gemm_rs_reduce_partials(None, 1, None, None, 4, 12, 2, 1.0, 0.0, 1, None) == \
        b.GEMM_RS_ERR_SHAPE
    assert L.gemm_rs_reduce_partials(None, 1, None, None, 4, 16, 0, 1.0, 0.0, 1, None) == \
        b.GEMM_RS_ERR_ARG
    assert L.gemm_rs_reduce_partials(None, 1, None, None, 0, 16, 2, 1.0, 0.0, 1, None) == 0


@pytest.mark.parametrize("W,M,N", [(1, 256, 72), (2, 512, 256), (8, 2048, 768), (8, 4096, 1792),
                                   (3, 1536, 1000), (16, 16 * 256, 64)])
def test_ag_schedule_matches_oracle(b, W, M, N):
    np.testing.assert_array_equal(b.ag_gemm_schedule(M, N, W), oracle.ag_schedule(W, M, N, 256, 256))


def test_ag_shape_checks(b):
    assert b.ag_gemm_workspace_bytes(4096, 1792, 4096, 8) == 256 + 256 + 8 * 4096 * 4096 * 2
    assert b.ag_gemm_workspace_bytes(4096 - 256, 1792, 4096, 8) == 0   # 256-row tiles straddle chunks
    assert b.ag_gemm_workspace_bytes(4096, 1790, 4096, 8) == 0         # N not a multiple of 8
    assert b.ag_gemm_workspace_bytes(4096, 1792, 4092, 8) == 0         # K not a multiple of 8
    assert b.ag_gemm_workspace_bytes(4096, 1792, 4096, 17) == 0
    with pytest.raises(b.GemmRSError):
        b.ag_gemm_schedule(300, 256, 2)
