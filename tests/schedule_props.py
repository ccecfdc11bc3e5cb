"""Checks of a tile order against what the pages fix of it (test helpers).

The pages fix each rank's chunk order and the chunk each row tile goes to
(the oracle's ``chunk_order``, ``ag_chunk_order`` and ``tile_chunk``), and
state two properties of the swizzle: every rank-tile is computed once, and at
every step the ranks write different chunks ("flux精读" §4.1).  Everything
finer (column groups, row groups, the rank offset of the column sweep, how
the W ranks share one device) is the library's choice.  So a schedule from
the library, or the device's record of one, is checked here against those
page-defined facts only:

  * every (r, mt, nt) appears exactly once;
  * for every rank and every column tile, the chunks of the rank's tiles in
    that column come in the rank's chunk order (a chunk's tiles together,
    the local chunk last for the reduce-scatter, first for the all-gather);
  * with the ranks side by side (entry p*W + r is rank r's p-th tile) and
    chunks a whole number of row tiles, the W entries of every step go to W
    different chunks.
"""
from __future__ import annotations

import numpy as np

import oracle


class ScheduleError(AssertionError):
    pass


def _expect(cond, msg):
    if not cond:
        raise ScheduleError(msg)


def _collapse(seq):
    out = []
    for c in seq:
        if not out or out[-1] != c:
            out.append(c)
    return out


def check_chunk_orders(sched, W, M, N, BM, BN, order, key):
    """Coverage and per-(rank, column) chunk order of an (r, mt, nt) array."""
    sched = np.asarray(sched)
    nM, nN = len(key), -(-N // BN)
    _expect(sched.shape == (W * nM * nN, 3), f"shape {sched.shape} != {(W * nM * nN, 3)}")
    flat = (sched[:, 0].astype(np.int64) * nM + sched[:, 1]) * nN + sched[:, 2]
    _expect(bool(np.all((sched[:, 0] >= 0) & (sched[:, 0] < W) & (sched[:, 1] >= 0)
                        & (sched[:, 1] < nM) & (sched[:, 2] >= 0) & (sched[:, 2] < nN))),
            "an entry lies outside the rank-tile grid")
    _expect(np.array_equal(np.sort(flat), np.arange(W * nM * nN)),
            "some rank-tile is missing or repeated")
    present = set(int(c) for c in key)
    for r in range(W):
        expect = [int(c) for c in order[r] if int(c) in present]
        mine = sched[sched[:, 0] == r]
        for nt in range(nN):
            col = mine[mine[:, 2] == nt]
            got = _collapse([int(key[mt]) for mt in col[:, 1]])
            _expect(got == expect, f"rank {r}, column tile {nt}: chunks {got}, expected {expect}")


def check_distinct_chunks_per_step(sched, W, key):
    """Ranks side by side: entry p*W + r is rank r's, and each step's W
    entries go to W different chunks."""
    sched = np.asarray(sched)
    per = sched.reshape(-1, W, 3)
    _expect(bool(np.all(per[:, :, 0] == np.arange(W))), "entries are not rank-interleaved")
    chunks = key[per[:, :, 1]]
    srt = np.sort(chunks, axis=1)
    _expect(bool(np.all(srt[:, 1:] != srt[:, :-1])), "two ranks write one chunk in the same step")


def check_rs_schedule(sched, W, M, N, BM, BN, interleaved: bool):
    """A GEMM+RS tile order against the pages' swizzle."""
    key = oracle.tile_chunk(W, M, BM)
    check_chunk_orders(sched, W, M, N, BM, BN, oracle.chunk_order(W), key)
    if interleaved and (M // W) % BM == 0:
        check_distinct_chunks_per_step(sched, W, key)


def check_ag_schedule(sched, W, M, N, BM, BN):
    """An AG+GEMM tile order against the pages' consumption order."""
    key = oracle.tile_chunk(W, M, BM)
    check_chunk_orders(sched, W, M, N, BM, BN, oracle.ag_chunk_order(W), key)
