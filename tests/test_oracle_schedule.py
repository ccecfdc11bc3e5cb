"""Pins for the oracle's swizzle and for the schedule checks (no GPU needed).

The oracle states what the pages fix of the tile order: each rank's chunk
order (remote chunks first, the local chunk last, each rank offset by its
rank) and the chunk each row tile goes to.  It is pinned here by the order
printed on the pages (tests/golden/swizzle_rank_offset_w8.txt), by the
properties the pages state (W distinct chunks at every step), and by the
row-to-chunk partition.  The checks in schedule_props.py, which compare the
library's schedules with the oracle, are pinned by planting mistakes in a
correct schedule and seeing each one caught.
"""
import os

import numpy as np
import pytest

import oracle
from schedule_props import (ScheduleError, check_ag_schedule, check_chunk_orders,
                            check_distinct_chunks_per_step, check_rs_schedule)

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "swizzle_rank_offset_w8.txt")


def _printed_orders():
    orders = {}
    with open(GOLDEN) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            rank, seq = line.split(":")
            orders[int(rank)] = [int(x) for x in seq.split()]
    return orders


def test_chunk_order_matches_printed_rank_offset_order():
    """"flux精读" §4.1 prints ranks 0 and 1 of eight starting at their own
    chunk; "flux实现" moves the local chunk to the end.  So the oracle's
    order with its last entry moved to the front is the printed one."""
    order = oracle.chunk_order(8)
    printed = _printed_orders()
    assert set(printed) == {0, 1}
    for r, seq in printed.items():
        mine = order[r].tolist()
        assert mine[-1] == r
        assert [mine[-1]] + mine[:-1] == seq


def test_ag_chunk_order_is_the_printed_order():
    """The all-gather side takes its own rows first: exactly the printed order."""
    order = oracle.ag_chunk_order(8)
    for r, seq in _printed_orders().items():
        assert order[r].tolist() == seq


@pytest.mark.parametrize("W", list(range(1, 17)))
def test_chunk_order_properties(W):
    """Each rank writes every chunk once, its own last; at every step the W
    ranks write W different chunks (the point of the offset, §4.1); the
    all-gather order is the same cycle with the local chunk moved to the
    front."""
    order = oracle.chunk_order(W)
    ag = oracle.ag_chunk_order(W)
    assert order.shape == (W, W)
    for r in range(W):
        assert sorted(order[r].tolist()) == list(range(W))
        assert order[r, -1] == r
        assert ag[r].tolist() == [r] + order[r, :-1].tolist()
    for s in range(W):
        assert sorted(order[:, s].tolist()) == list(range(W))
        assert sorted(ag[:, s].tolist()) == list(range(W))


def test_chunk_order_rejects_bad_w():
    with pytest.raises(ValueError):
        oracle.chunk_order(0)


@pytest.mark.parametrize("W,M,BM", [(2, 256, 128), (8, 4096, 256), (8, 64, 128), (4, 400, 128),
                                    (3, 300, 128), (16, 16 * 7, 128), (7, 7 * 129, 128),
                                    (8, 8192, 256), (1, 200, 128)])
def test_tile_chunk_is_the_chunk_of_the_first_row(W, M, BM):
    """Each row tile goes with the chunk of its first row (the row-to-chunk
    partition, pinned on its own); keys never decrease; when a chunk is a
    whole number of tiles, each chunk gets exactly R/BM consecutive tiles."""
    key = oracle.tile_chunk(W, M, BM)
    chunk, _ = oracle.row_chunk(W, M)
    nM = -(-M // BM)
    assert key.shape == (nM,)
    for mt in range(nM):
        assert key[mt] == chunk[mt * BM]
    assert np.all(np.diff(key) >= 0)
    R = M // W
    if R % BM == 0:
        assert key.tolist() == [c for c in range(W) for _ in range(R // BM)]


def test_tile_chunk_rejects_bad_arguments():
    with pytest.raises(ValueError):
        oracle.tile_chunk(3, 100, 128)  # M is not a multiple of W


def _plain_rs_schedule(W, M, N, BM, BN, interleaved):
    """A schedule built straight from the oracle's order: for each rank, for
    each step, the chunk's row tiles, each swept over all columns."""
    order = oracle.chunk_order(W)
    key = oracle.tile_chunk(W, M, BM)
    nN = -(-N // BN)
    per_rank = []
    for r in range(W):
        lst = []
        for c in order[r]:
            for nt in range(nN):
                for mt in np.nonzero(key == c)[0]:
                    lst.append((r, int(mt), nt))
        per_rank.append(lst)
    if interleaved:
        return np.array([per_rank[r][p] for p in range(len(per_rank[0])) for r in range(W)],
                        dtype=np.int32)
    return np.array([e for lst in per_rank for e in lst], dtype=np.int32)


@pytest.mark.parametrize("interleaved", [True, False])
def test_checks_accept_a_plain_schedule(interleaved):
    W, M, N, BM, BN = 8, 8 * 256, 768, 128, 256
    check_rs_schedule(_plain_rs_schedule(W, M, N, BM, BN, interleaved), W, M, N, BM, BN,
                      interleaved)


def _mutations(s, W, BM, M):
    """Plausible mistakes in a tile order, each planted in a copy."""
    R = M // W
    out = {}
    m = s.copy()
    m[[0, 1]] = m[[1, 0]]                      # two entries of different ranks swapped
    out["swap across ranks"] = m
    m = s.copy()
    m[5] = m[6]                                # a tile computed twice, another dropped
    out["duplicate"] = m
    r0 = np.nonzero(s[:, 0] == 0)[0]
    m = s.copy()
    last = r0[-1]
    first = r0[0]
    m[[first, last]] = m[[last, first]]        # rank 0's own chunk tile moved to the front
    out["local chunk first"] = m
    m = s.copy()
    m[:, 1] = (m[:, 1] + R // BM) % (M // BM)  # every tile keyed one chunk further on
    out["chunk shifted"] = m
    m = s.copy()
    m[:, 0] = (m[:, 0] + 1) % W                # ranks relabelled
    out["rank relabelled"] = m
    return out


@pytest.mark.parametrize("interleaved", [True, False])
def test_checks_catch_planted_mistakes(interleaved):
    W, M, N, BM, BN = 8, 8 * 256, 768, 128, 256
    good = _plain_rs_schedule(W, M, N, BM, BN, interleaved)
    for name, bad in _mutations(good, W, BM, M).items():
        if name == "swap across ranks" and not interleaved:
            bad = good.copy()
            i, j = 0, W * 2 * 3  # rank 0 and rank 1 blocks exchange an entry
            bad[[i, j]] = bad[[j, i]]
        with pytest.raises(ScheduleError):
            check_rs_schedule(bad, W, M, N, BM, BN, interleaved)


def test_step_check_catches_two_ranks_on_one_chunk():
    W, M, N, BM, BN = 4, 4 * 128, 512, 128, 256
    good = _plain_rs_schedule(W, M, N, BM, BN, True)
    key = oracle.tile_chunk(W, M, BM)
    check_distinct_chunks_per_step(good, W, key)
    bad = good.copy()
    bad[1, 1] = bad[0, 1]
    with pytest.raises(ScheduleError):
        check_distinct_chunks_per_step(bad, W, key)


def test_ag_check_catches_the_reduce_scatter_order():
    """An AG order with the local chunk last (the reduce-scatter's) is caught."""
    W, M, N, BM, BN = 4, 4 * 256, 512, 256, 256
    rs = _plain_rs_schedule(W, M, N, BM, BN, False)
    with pytest.raises(ScheduleError):
        check_ag_schedule(rs, W, M, N, BM, BN)
    key = oracle.tile_chunk(W, M, BM)
    check_chunk_orders(rs, W, M, N, BM, BN, oracle.chunk_order(W), key)
