"""The multi-GPU form's exchange plan on the host (no GPU): the copies every rank's pack and unpack
stages make, checked against one another over seeded random parameter lists.

* What rank p packs into block q of its all-to-all buffer is exactly what rank q unpacks from block p
  of its receive buffer: same offsets, same lengths, same worker row and word range at both ends.
* The same holds for the all-gather: rank q's block is unpacked by every other rank as it was packed.
* Coverage: for every segment, the sign words of the shards the ranks serve partition the segment's
  words, and every rank ends the step holding every server word and scale exactly once (its own
  plus the unpacked ones); every worker's scales reach every rank.
* Bounds: every copy stays inside its block and its region row.
* Sizes: block sizes are the same on every rank, and a rank's workspace shrinks with the world size
  (it keeps c for its own workers only).
"""
import numpy as np
import pytest

import communication_compressed_optimizer_compress_gb300 as ob
import oracle
from communication_compressed_optimizer_compress_gb300 import dist as D


def _configs(count, seed):
    rng = np.random.default_rng(seed)
    out = []
    for _ in range(count):
        T = int(rng.integers(1, 7))
        numel = [int(rng.choice([0, 1, 31, 33, 100, 777, 4096, int(rng.integers(1, 30000))])) for _ in range(T)]
        if sum(numel) == 0:
            numel[0] = 5
        world = int(rng.choice([1, 2, 3, 4, 8]))
        n = world * int(rng.integers(1, 4))
        block = int(rng.choice([0, 0, 32, 96, 4096]))
        out.append((numel, n, world, block))
    return out


CONFIGS = _configs(40, 5) + [([340_000_000 // 1000], 16, 16, 0), ([100, 33, 0, 700], 4, 2, 0)]


@pytest.mark.parametrize("numel,n,world,block", CONFIGS)
def test_exchange_plan_pairs_and_covers(numel, n, world, block):
    cfg = ob.make_config(numel, n, 1, scale_block=block)
    segs = oracle.scale_blocks(numel, block)
    T = len(segs)
    woff = np.concatenate([[0], np.cumsum([(L + 31) // 32 for L in segs])]).astype(np.int64)
    Wd = int(woff[-1])
    nl = n // world
    plans = [D.plan_exchange(cfg, r, world) for r in range(world)]
    sb, bb = plans[0][1], plans[0][2]
    assert all(p[1] == sb and p[2] == bb for p in plans)
    rows_of = [{st: [row for row in p[0] if row[0] == st] for st in range(4)} for p in plans]
    row_len = {0: Wd, 1: T, 2: Wd, 3: n}
    n_rows = {0: n, 1: n, 2: 1, 3: T}
    for r in range(world):
        for st, regs in rows_of[r].items():
            block = sb if st < 2 else bb
            for (_, sreg, srow, soff, dreg, drow, doff, ln) in regs:
                assert ln > 0
                for reg, row, off in ((sreg, srow, soff), (dreg, drow, doff)):
                    if reg == 4:
                        assert 0 <= row < world and 0 <= off and off + ln <= block
                        assert row != r or st == 2  # no rank copies its own block (stage 2 writes the one it sends)
                    else:
                        assert 0 <= row < n_rows[reg] and 0 <= off and off + ln <= row_len[reg]
    # all-to-all: rank p's pack into block q == rank q's unpack from block p
    for p in range(world):
        for q in range(world):
            if p == q:
                continue
            packed = sorted((doff, ln, sreg, srow, soff) for (_, sreg, srow, soff, _, drow, doff, ln) in rows_of[p][0]
                            if drow == q)
            unpacked = sorted((soff, ln, dreg, drow, doff) for (_, _, srow, soff, dreg, drow, doff, ln) in rows_of[q][1]
                              if srow == p)
            assert packed == unpacked, (p, q)
    # all-gather: rank q's block, as packed by q, is unpacked identically by every other rank
    for q in range(world):
        packed = sorted((doff, ln, sreg, srow, soff) for (_, sreg, srow, soff, _, _, doff, ln) in rows_of[q][2])
        for p in range(world):
            if p == q:
                continue
            unpacked = sorted((soff, ln, dreg, drow, doff) for (_, _, srow, soff, dreg, drow, doff, ln) in rows_of[p][3]
                              if srow == q)
            assert packed == unpacked, (p, q)
    # coverage of the server words and scales on every rank, and of the worker scales
    for r in range(world):
        words = np.zeros(Wd, int)
        scales = np.zeros((T, n), int)
        for k, L in enumerate(segs):
            for j in range(r * nl, (r + 1) * nl):  # this rank's own shards
                lo, hi = oracle.shard(L, n, j)
                scales[k, j] += 1
                if hi > lo:
                    words[woff[k] + lo // 32: woff[k] + (hi + 31) // 32] += 1
        for (_, _, _, _, dreg, drow, doff, ln) in rows_of[r][3]:
            if dreg == 2:
                words[doff: doff + ln] += 1
            else:
                scales[drow, doff: doff + ln] += 1
        assert np.all(words == 1) and np.all(scales == 1), r
        wsc = np.zeros((n, T), int)
        wsc[r * nl:(r + 1) * nl] += 1
        for (_, _, _, _, dreg, drow, doff, ln) in rows_of[r][1]:
            if dreg == 1:
                wsc[drow, doff: doff + ln] += 1
        assert np.all(wsc == 1), r
    if world > 1:  # (tiny lists: the 256-byte alignment of the pieces hides the difference)
        ws_rank, ws_one = D.workspace_size_rank(cfg, 0, world), ob.workspace_size(cfg)
        assert ws_rank <= ws_one and (ws_rank < ws_one or sum(numel) < 10_000)


def test_rank_arguments_are_checked():
    cfg = ob.make_config([1000], 4, 1)
    for rank, world in ((0, 3), (2, 2), (-1, 2), (0, 0)):
        with pytest.raises(ob.OneBitError) as e:
            D.plan_exchange(cfg, rank, world)
        assert e.value.status == ob.ERR_INVALID_ARG
    rows, sb, bb = D.plan_exchange(cfg, 0, 1)
    assert rows == []  # one rank moves nothing
