"""Pins for the oracle's tile schedule (no GPU needed).

The schedule is checked against the order printed on the pages
(tests/golden/swizzle_rank_offset_w8.txt) and against the properties that
the pages state: remote chunks first and the local chunk last; each rank
offset by its rank, so that the W ranks target W different chunks at every
step; and every rank-tile visited exactly once.
"""
import os

import numpy as np
import pytest

import oracle

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


def _chunk_sequence(sched, W, M, BM, r):
    """Chunk order of rank r, read off its tiles' chunk keys."""
    R = M // W
    seq = []
    for (rr, mt, nt) in sched:
        if rr != r:
            continue
        c = (mt * BM) // R
        if not seq or seq[-1] != c:
            seq.append(c)
    return seq


def test_matches_printed_rank_offset_order():
    W, M, N, BM, BN = 8, 8 * 256, 512, 128, 256
    sched = oracle.schedule(W, M, N, BM, BN)
    printed = _printed_orders()
    assert set(printed) == {0, 1}
    for r, order in printed.items():
        seq = _chunk_sequence(sched, W, M, BM, r)
        assert seq[-1] == r                      # local chunk last
        assert [seq[-1]] + seq[:-1] == order      # = printed order, local moved to the front


@pytest.mark.parametrize("W,M,N,BM,BN", [
    (2, 256, 256, 128, 256), (8, 4096, 4096, 128, 256), (4, 16384, 5120, 128, 256),
    (8, 64, 8192, 128, 64), (3, 300, 520, 128, 128), (1, 200, 72, 128, 64),
    (5, 5 * 128, 1000, 128, 256),
])
def test_schedule_properties(W, M, N, BM, BN):
    sched = oracle.schedule(W, M, N, BM, BN)
    nM, nN = -(-M // BM), -(-N // BN)
    assert sched.shape == (W * nM * nN, 3)
    # every rank-tile exactly once
    keys = set(map(tuple, sched.tolist()))
    assert len(keys) == W * nM * nN
    assert keys == {(r, m, n) for r in range(W) for m in range(nM) for n in range(nN)}
    # ranks run side by side
    assert np.array_equal(sched[:, 0], np.tile(np.arange(W), nM * nN))
    R = M // W
    for r in range(W):
        seq = _chunk_sequence(sched, W, M, BM, r)
        expect = [(r + 1 + s) % W for s in range(W)]
        present = {(mt * BM) // R for mt in range(nM)}
        assert seq == [c for c in expect if c in present]
    if R % BM == 0:
        # every position p: the W ranks target W distinct chunks
        per_p = sched.reshape(nM * nN, W, 3)
        for p in range(nM * nN):
            chunks = {(int(mt) * BM) // R for (_, mt, _) in per_p[p]}
            assert len(chunks) == W


def test_rank_column_offset_when_one_chunk_holds_all_tiles():
    """M = 64, W = 8: chunks of 8 rows, one row tile.  The ranks then start
    on different column tiles."""
    W, M, N, BM, BN = 8, 64, 8192, 128, 64
    sched = oracle.schedule(W, M, N, BM, BN)
    nN = N // BN
    first = sched[:W]
    assert first[:, 2].tolist() == [(r * nN) // W for r in range(W)]
