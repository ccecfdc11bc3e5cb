"""C-ABI checks that need no GPU: the library loads, exports every symbol
include/gemm_rs.h and include/ag_gemm.h declare, validates arguments before
touching the device, and its host-side tile schedules follow the pages'
swizzle (checked against the oracle's chunk order, schedule_props.py) and
keep the arrival order its chain reduction relies on."""
import os
import re

import numpy as np
import pytest

import oracle
from schedule_props import check_ag_schedule, check_rs_schedule

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


def test_noalloc_scratch_size_is_the_headers(b):
    """The static scratch's size comes from the library and equals the header's
    GEMM_RS_NOALLOC_SCRATCH_BYTES (read without touching a device)."""
    text = open(HEADER).read()
    m = re.search(r"#define GEMM_RS_NOALLOC_SCRATCH_BYTES \((\d+)u \* (\d+)u \* (\d+)u\)", text)
    assert m, "the header defines the scratch size"
    want = int(m.group(1)) * int(m.group(2)) * int(m.group(3))
    assert b.gemm_rs_noalloc_scratch_bytes() == want


def test_version(b):
    assert "sm_103a" in b.gemm_rs_version()


SCHEDULE_SHAPES = [
    (2, 256, 256, 256), (8, 4096, 4096, 256), (8, 8192, 8192, 256), (8, 64, 8192, 64),
    (4, 16384, 5120, 256), (3, 300, 520, 128), (1, 200, 72, 64), (5, 640, 1000, 256),
    (16, 16 * 7, 64, 64), (7, 7 * 129, 264, 128),
]
SCHEDULE_GROUPS = ((0, 0), (1, 0), (2, 3), (5, 1), (0, 2), (3, 5), (4, 0), (8, 0))


@pytest.mark.parametrize("W,M,N,bn", SCHEDULE_SHAPES)
def test_schedule_follows_the_swizzle(b, W, M, N, bn):
    """Every plan of the library, both tile heights and both rank orders: each
    rank-tile once, each rank's chunks in the pages' order in every column,
    and (ranks side by side) W different chunks at every step."""
    for G, RG in SCHEDULE_GROUPS:
        for code in (b.GEMM_RS_RANKS_INTERLEAVED, b.GEMM_RS_RANKS_SEQUENTIAL,
                     b.GEMM_RS_RANKS_DEFAULT):
            inter = code == b.GEMM_RS_RANKS_INTERLEAVED
            for bm, tbn in ((128, bn), (256, 256)):
                check_rs_schedule(b.gemm_rs_schedule(M, N, W, bm, tbn, G, RG, code), W, M, N,
                                  bm, tbn, inter)


@pytest.mark.parametrize("W,M,N,bn", SCHEDULE_SHAPES)
def test_rank_orders_keep_each_ranks_own_order(b, W, M, N, bn):
    """The two rank orders differ only in how the ranks share the device: each
    rank's own sequence of tiles is the same, and with the ranks one after
    another each column group is one block per rank, in rank order."""
    for G, RG in SCHEDULE_GROUPS:
        side = b.gemm_rs_schedule(M, N, W, 128, bn, G, RG, b.GEMM_RS_RANKS_INTERLEAVED)
        seq = b.gemm_rs_schedule(M, N, W, 128, bn, G, RG, b.GEMM_RS_RANKS_SEQUENTIAL)
        np.testing.assert_array_equal(b.gemm_rs_schedule(M, N, W, 128, bn, G, RG,
                                                         b.GEMM_RS_RANKS_DEFAULT), seq)
        nM, nN = -(-M // 128), -(-N // bn)
        assert np.array_equal(side[:, 0], np.tile(np.arange(W), nM * nN))
        for r in range(W):
            assert np.array_equal(seq[seq[:, 0] == r], side[side[:, 0] == r])
        group = nN if G <= 0 or G >= nN else G
        start = 0
        for g0 in range(0, nN, group):
            gn = min(group, nN - g0)
            block = seq[start:start + W * nM * gn]
            assert np.array_equal(block[:, 0], np.repeat(np.arange(W), nM * gn))
            assert set(block[:, 2].tolist()) == set(range(g0, g0 + gn))
            start += W * nM * gn


@pytest.mark.parametrize("W,M,N,BM,BN,G", [
    (8, 4096, 4096, 256, 256, 0), (4, 16384, 5120, 256, 256, 0), (8, 8192, 8192, 256, 256, 0),
    (2, 1024, 2048, 128, 256, 0), (8, 4096, 4096, 256, 256, 8), (8, 8192, 8192, 256, 256, 16),
    (4, 16384, 5120, 256, 256, 8)])
def test_interleaved_contributions_arrive_in_step_order(b, W, M, N, BM, BN, G):
    """Ranks side by side: every output tile's W contributions come in step
    order (the order the chain reduction folds them in), each at least about
    (1 - 1/W) of a step after the previous one, also with column groups."""
    sched = b.gemm_rs_schedule(M, N, W, BM, BN, G, 0, b.GEMM_RS_RANKS_INTERLEAVED)
    nM, nN = -(-M // BM), -(-N // BN)
    group = nN if G <= 0 or G >= nN else G
    key = oracle.tile_chunk(W, M, BM)
    order = oracle.chunk_order(W)
    seen = {}
    for g, (r, mt, nt) in enumerate(sched.tolist()):
        seen.setdefault((mt, nt), []).append((g, r))
    for (mt, nt), lst in seen.items():
        steps = [order[r].tolist().index(key[mt]) for (_, r) in lst]
        assert steps == list(range(W))
        g0 = (nt // group) * group
        per_step = nM * min(group, nN - g0)
        gaps = [lst[i + 1][0] - lst[i][0] for i in range(W - 1)]
        assert min(gaps) >= per_step * (W - 1) // W - W


@pytest.mark.parametrize("W,M,N,BM,BN,G", [
    (8, 4096, 4096, 256, 256, 0), (4, 16384, 5120, 256, 256, 0), (8, 8192, 8192, 256, 256, 0),
    (8, 4096, 4096, 256, 256, 8), (8, 8192, 8192, 256, 256, 4), (3, 300, 520, 128, 128, 0),
    (5, 5 * 256, 1000, 128, 256, 2)])
def test_sequential_contributions_arrive_in_rank_order(b, W, M, N, BM, BN, G):
    """Ranks one after another: every output tile's contributions come in rank
    order, at least T*(W-2)/W entries apart (T = a rank's tiles in the tile's
    column group): the chain reduction then folds in rank order."""
    sched = b.gemm_rs_schedule(M, N, W, BM, BN, G, 0, b.GEMM_RS_RANKS_SEQUENTIAL)
    nM, nN = -(-M // BM), -(-N // BN)
    group = nN if G <= 0 or G >= nN else G
    seen = {}
    for g, (r, mt, nt) in enumerate(sched.tolist()):
        seen.setdefault((mt, nt), []).append((g, r))
    for (mt, nt), lst in seen.items():
        assert [r for _, r in lst] == list(range(W))
        T = nM * min(group, nN - (nt // group) * group)
        gaps = [lst[i + 1][0] - lst[i][0] for i in range(W - 1)]
        assert min(gaps) >= T * (W - 2) // W


def test_ranks_start_on_different_columns_when_one_row_tile_holds_every_chunk(b):
    """M = 64, W = 8: one row tile (keyed to chunk 0).  The library starts
    rank r's sweep at column ((W-r) mod W)*nN/W, so the ranks side by side
    begin on W different column tiles."""
    W, M, N, BM, BN = 8, 64, 8192, 128, 64
    sched = b.gemm_rs_schedule(M, N, W, BM, BN, 0, 0, b.GEMM_RS_RANKS_INTERLEAVED)
    nN = N // BN
    assert sched[:W, 2].tolist() == [(((W - r) % W) * nN) // W for r in range(W)]
    assert len(set(sched[:W, 2].tolist())) == W


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
    assert b.lib().gemm_rs_run_streamed(None, None, None, None, None, None, None, None, None,
                                        None, None) == b.GEMM_RS_ERR_ARG
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
def test_ag_schedule_follows_the_consumption_order(b, W, M, N):
    check_ag_schedule(b.ag_gemm_schedule(M, N, W), W, M, N, 256, 256)


def test_ag_shape_checks(b):
    assert b.ag_gemm_workspace_bytes(4096, 1792, 4096, 8) == 256 + 256 + 8 * 4096 * 4096 * 2
    assert b.ag_gemm_workspace_bytes(4096 - 256, 1792, 4096, 8) == 0   # 256-row tiles straddle chunks
    assert b.ag_gemm_workspace_bytes(4096, 1790, 4096, 8) == 0         # N not a multiple of 8
    assert b.ag_gemm_workspace_bytes(4096, 1792, 4092, 8) == 0         # K not a multiple of 8
    assert b.ag_gemm_workspace_bytes(4096, 1792, 4096, 17) == 0
    with pytest.raises(b.GemmRSError):
        b.ag_gemm_schedule(300, 256, 2)
