"""Pins of the schedule oracle's stream-K tail (no GPU): the partition of the tail's k-blocks,
the owners, the walking order that keeps every wait pointing at a lower-numbered worker, and
the whole tiles before the tail."""

import itertools

import pytest

from oracle import schedule as s

CASES = [(16, 16, 76, 16, 32), (32, 16, 76, 12, 128), (4, 25, 76, 8, 16), (3, 7, 5, 2, 9),
         (1, 1, 4, 1, 3), (5, 3, 7, 1, 1), (9, 4, 11, 3, 5), (2, 3, 4, 8, 64)]


@pytest.mark.parametrize("m,n,P,g,KB", CASES)
@pytest.mark.parametrize("column_major", [False, True])
def test_every_tile_and_k_block_once(m, n, P, g, KB, column_major):
    rows = s.enumerate_units_streamk(m, n, P, g, KB, column_major)
    cover = {}
    for (c, w, bx, by, part, k_lo, k_hi, unit) in rows:
        assert 0 <= k_lo < k_hi <= KB
        for k in range(k_lo, k_hi):
            assert (bx, by, k) not in cover, (bx, by, k)
            cover[(bx, by, k)] = c
    assert set(cover) == set(itertools.product(range(m), range(n), range(KB)))


@pytest.mark.parametrize("m,n,P,g,KB", CASES)
def test_owners_walk_last_and_wait_only_on_lower_workers(m, n, P, g, KB):
    rows = s.enumerate_units_streamk(m, n, P, g, KB)
    R = (m * n) % P
    tail = [r for r in rows if r[4] >= 2]
    owners = {}
    for c in range(P):
        mine = [r for r in rows if r[0] == c]
        assert [r[1] for r in mine] == list(range(len(mine)))       # w counts the worker's units
        parts = [r[4] for r in mine if r[4] >= 2]
        assert parts in ([], [2], [3], [2, 3])                      # one each at most, owned last
        assert all(r[4] == -1 for r in mine[:len(mine) - len(parts)])  # whole tiles come first
    for (c, w, bx, by, part, k_lo, k_hi, unit) in tail:
        if part == 3:
            assert k_hi == KB and (bx, by) not in owners
            owners[(bx, by)] = c
    assert len(owners) == R
    for t in range(R):
        owner, contributors = s.streamk_contributors(t, P, R, KB)
        assert all(j < owner for j in contributors)
        segs = [r for r in tail if r[0] == owner and r[4] == 3]
        assert len(segs) == 1
        for j in contributors:   # a contributor's single contribution is to this tile
            contrib = [r for r in tail if r[0] == j and r[4] == 2]
            assert len(contrib) == 1 and (contrib[0][2], contrib[0][3]) == (segs[0][2], segs[0][3])


def test_whole_tiles_are_the_grid_stride_without_the_tail():
    m, n, P, g, KB = 16, 16, 76, 16, 32
    rows = s.enumerate_units_streamk(m, n, P, g, KB)
    whole = [(c, w, bx, by) for (c, w, bx, by, part, *_r) in rows if part == -1]
    ref = [r for r in s.enumerate_schedule(m, n, P, g) if r[0] + r[1] * P < m * n - (m * n) % P]
    assert sorted(whole) == sorted(ref)


def test_worked_partition_4096_cube_pair_tiles():
    # 256 tiles of 256 x 256 over 76 CTA pairs, 32 k-blocks of 128: 28 tail tiles, 896 k-blocks,
    # worker c takes [896c/76, 896(c+1)/76): 11 or 12 k-blocks
    assert s.streamk_range(0, 76, 28, 32) == (0, 11)
    assert s.streamk_range(1, 76, 28, 32) == (11, 23)
    assert s.streamk_range(2, 76, 28, 32) == (23, 35)
    assert s.streamk_segments(2, 76, 28, 32) == [(1, 0, 3, False), (0, 23, 32, True)]
    assert s.streamk_contributors(0, 76, 28, 32) == (2, [0, 1])
    assert s.streamk_range(75, 76, 28, 32)[1] == 896
