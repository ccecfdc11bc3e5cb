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


@pytest.mark.parametrize("order", ["interleaved", "sequential"])
@pytest.mark.parametrize("G,RG", [(0, 0), (1, 0), (3, 0), (0, 1), (2, 3)])
@pytest.mark.parametrize("W,M,N,BM,BN", [
    (2, 256, 256, 128, 256), (8, 4096, 4096, 128, 256), (4, 16384, 5120, 128, 256),
    (8, 64, 8192, 128, 64), (3, 300, 520, 128, 128), (1, 200, 72, 128, 64),
    (5, 5 * 128, 1000, 128, 256), (8, 4096, 4096, 256, 256),
])
def test_schedule_properties(W, M, N, BM, BN, G, RG, order):
    sched = oracle.schedule(W, M, N, BM, BN, G, RG, order)
    nM, nN = -(-M // BM), -(-N // BN)
    assert sched.shape == (W * nM * nN, 3)
    # every rank-tile exactly once
    keys = set(map(tuple, sched.tolist()))
    assert len(keys) == W * nM * nN
    assert keys == {(r, m, n) for r in range(W) for m in range(nM) for n in range(nN)}
    if order == "interleaved":
        # ranks run side by side
        assert np.array_equal(sched[:, 0], np.tile(np.arange(W), nM * nN))
    else:
        # per column group, one rank after another; each rank's own order unchanged
        group = nN if G <= 0 or G >= nN else G
        start = 0
        for g0 in range(0, nN, group):
            gn = min(group, nN - g0)
            block = sched[start:start + W * nM * gn]
            assert np.array_equal(block[:, 0], np.repeat(np.arange(W), nM * gn))
            assert set(block[:, 2].tolist()) == set(range(g0, g0 + gn))
            start += W * nM * gn
        side = oracle.schedule(W, M, N, BM, BN, G, RG, "interleaved")
        for r in range(W):
            assert np.array_equal(sched[sched[:, 0] == r], side[side[:, 0] == r])
    R = M // W
    groups = 1 if G <= 0 or G >= nN else -(-nN // G)
    for r in range(W):
        seq = _chunk_sequence(sched, W, M, BM, r)
        present = {(mt * BM) // R for mt in range(nM)}
        expect = [c for c in [(r + 1 + s) % W for s in range(W)] if c in present]
        if len(expect) == 1:
            assert seq == expect
        else:
            assert seq == expect * groups  # remote chunks first, local last, in every group
    if R % BM == 0 and order == "interleaved":
        # every position p: the W ranks target W distinct chunks
        per_p = sched.reshape(nM * nN, W, 3)
        for p in range(nM * nN):
            chunks = {(int(mt) * BM) // R for (_, mt, _) in per_p[p]}
            assert len(chunks) == W


def test_every_sweep_runs_forward_from_the_rank_offset():
    """Each step sweeps a rank's column tiles forward from ((W-r) mod W)*nN/W
    (one column group)."""
    W, M, N, BM, BN = 4, 4 * 128, 2048, 128, 256
    sched = oracle.schedule(W, M, N, BM, BN)
    nN = N // BN
    for r in range(W):
        cols = [int(nt) for (rr, mt, nt) in sched if rr == r]
        rot = (((W - r) % W) * nN) // W
        for s in range(W):
            assert cols[s * nN:(s + 1) * nN] == [(j + rot) % nN for j in range(nN)]


def test_row_groups_sweep_all_columns_per_group():
    """With row groups of 2 row tiles, a step of a 6-tile chunk makes three
    forward sweeps over the column tiles, each covering its two row tiles for
    every column."""
    W, M, N, BM, BN, RG = 2, 2 * 6 * 128, 1024, 128, 256, 2
    sched = oracle.schedule(W, M, N, BM, BN, 0, RG)
    nN = N // BN
    mine = [(int(mt), int(nt)) for (rr, mt, nt) in sched if rr == 0]
    step0 = mine[:6 * nN]              # rank 0, step 0: chunk 1 (row tiles 6..11)
    rot = (W * nN // W) % nN  # rank 0: offset ((W-0) mod W)*nN/W = 0
    for k in range(3):
        sweep = step0[k * 2 * nN:(k + 1) * 2 * nN]
        cols = [sweep[2 * i][1] for i in range(nN)]
        assert cols == [(j + rot) % nN for j in range(nN)]
        for i in range(nN):
            assert [sweep[2 * i][0], sweep[2 * i + 1][0]] == [6 + 2 * k, 7 + 2 * k]


@pytest.mark.parametrize("W,M,N,BM,BN,G", [
    (8, 4096, 4096, 256, 256, 0), (4, 16384, 5120, 256, 256, 0), (8, 8192, 8192, 256, 256, 0),
    (2, 1024, 2048, 128, 256, 0), (8, 4096, 4096, 256, 256, 8), (8, 8192, 8192, 256, 256, 16),
    (4, 16384, 5120, 256, 256, 8)])
def test_tile_contributions_arrive_in_step_order(W, M, N, BM, BN, G):
    """For every output tile, the global order visits its W rank contributions
    in step order, each at least (1 - 1/W) of a step after the previous one,
    also with column groups (a step then covers one group's columns).  The
    chain reduction folds them in that order."""
    sched = oracle.schedule(W, M, N, BM, BN, G)
    nM, nN = -(-M // BM), -(-N // BN)
    group = nN if G <= 0 or G >= nN else G
    R = M // W
    seen = {}
    for g, (r, mt, nt) in enumerate(sched.tolist()):
        seen.setdefault((mt, nt), []).append((g, r))
    for (mt, nt), lst in seen.items():
        c = (mt * BM) // R
        steps = [((c - r - 1) % W) for (_, r) in lst]
        assert steps == list(range(W))               # arrival order = step order
        g0 = (nt // group) * group
        per_step = nM * min(group, nN - g0)          # global entries per step of this group
        gaps = [lst[i + 1][0] - lst[i][0] for i in range(W - 1)]
        assert min(gaps) >= per_step * (W - 1) // W - W  # ranks interleave: -1 per rank


@pytest.mark.parametrize("W,M,N,BM,BN,G", [
    (8, 4096, 4096, 256, 256, 0), (4, 16384, 5120, 256, 256, 0), (8, 8192, 8192, 256, 256, 0),
    (8, 4096, 4096, 256, 256, 8), (3, 300, 520, 128, 128, 0), (5, 5 * 256, 1000, 128, 256, 2)])
def test_sequential_ranks_arrive_in_rank_order(W, M, N, BM, BN, G):
    """With the ranks one after another (per column group), every output tile
    sees its W rank contributions in rank order 0 .. W-1 (the order the chain
    reduction folds in, the same as the last arriver's).  Rank r+1 reaches a
    tile at most one of its steps (T/W entries) earlier in its own pass over
    the group than rank r, give or take the column offset, so consecutive
    contributions lie at least T*(W-2)/W entries apart (T = a rank's tiles in
    the tile's column group)."""
    sched = oracle.schedule(W, M, N, BM, BN, G, 0, "sequential")
    nM, nN = -(-M // BM), -(-N // BN)
    group = nN if G <= 0 or G >= nN else G
    seen = {}
    for g, (r, mt, nt) in enumerate(sched.tolist()):
        seen.setdefault((mt, nt), []).append((g, r))
    for (mt, nt), lst in seen.items():
        assert [r for _, r in lst] == list(range(W))
        g0 = (nt // group) * group
        T = nM * min(group, nN - g0)
        gaps = [lst[i + 1][0] - lst[i][0] for i in range(W - 1)]
        assert min(gaps) >= T * (W - 2) // W


def test_rank_column_offset_when_one_chunk_holds_all_tiles():
    """M = 64, W = 8: chunks of 8 rows, one row tile (keyed to chunk 0).  Rank
    r reaches chunk 0 at step s = W-1-r and sweeps forward from column
    ((W-r) mod W)*nN/W, so the ranks start on different column tiles."""
    W, M, N, BM, BN = 8, 64, 8192, 128, 64
    sched = oracle.schedule(W, M, N, BM, BN)
    nN = N // BN
    first = sched[:W]
    expect = []
    for r in range(W):
        expect.append((((W - r) % W) * nN) // W)  # one sweep per rank, forward
    assert first[:, 2].tolist() == expect
    assert len(set(expect)) == W
