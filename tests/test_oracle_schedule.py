"""Pins for oracle.schedule: the persistent grouped tile order.

Tied to things other than the decode formula itself:
* every tile of the grid is visited exactly once, for every grid up to 24 x 24 and
  several group widths and worker counts (a wrong tail panel skips or repeats tiles);
* group width 1 is plain column-major order of the tile grid and a single panel
  (group >= n_blocks) is plain row-major order -- textbook orders;
* panels are visited left to right and, inside a panel, M-tiles top to bottom;
* worker c owns exactly the ids c, c+P, ... and its clock w counts 0, 1, 2, ...;
* a few values evaluated by hand from the page's decode at the workloads' grids.
"""

import itertools

import pytest

from oracle import schedule


GRIDS = [(m, n) for m in range(1, 25) for n in range(1, 25)]


@pytest.mark.parametrize("group", [1, 2, 3, 8, 16])
def test_every_tile_exactly_once(group):
    for m, n in GRIDS:
        seen = [schedule.tile_coord(t, m, n, group) for t in range(m * n)]
        assert sorted(seen) == [(bx, by) for bx in range(m) for by in range(n)], (m, n, group)


def test_group_one_is_column_major():
    for m, n in GRIDS:
        for t in range(m * n):
            assert schedule.tile_coord(t, m, n, 1) == (t % m, t // m)


def test_single_panel_is_row_major():
    for m, n in GRIDS:
        for g in (n, n + 1, 64):
            for t in range(m * n):
                assert schedule.tile_coord(t, m, n, g) == (t // n, t % n)


@pytest.mark.parametrize("group", [2, 3, 8])
def test_panels_left_to_right_and_rows_top_to_bottom(group):
    for m, n in GRIDS:
        coords = [schedule.tile_coord(t, m, n, group) for t in range(m * n)]
        panels = [by // group for _, by in coords]
        assert panels == sorted(panels)
        for p in set(panels):
            rows = [bx for (bx, by) in coords if by // group == p]
            assert rows == sorted(rows)
            # every row of the panel holds the panel's full width, consecutively
            width = min(group, n - p * group)
            for r in range(m):
                ids = [t for t, (bx, by) in enumerate(coords) if bx == r and by // group == p]
                assert ids == list(range(ids[0], ids[0] + width))


@pytest.mark.parametrize("workers", [1, 7, 148, 160])
def test_worker_partition_and_clock(workers):
    for m, n, g in itertools.product([1, 3, 8, 13], [1, 4, 9, 28], [1, 8]):
        rows = schedule.enumerate_schedule(m, n, workers, g)
        assert len(rows) == m * n
        for c in range(workers):
            mine = [r for r in rows if r[0] == c]
            expect = max(0, -(-(m * n - c) // workers))
            assert len(mine) == expect
            assert [r[1] for r in mine] == list(range(expect))
        assert rows == sorted(rows, key=lambda r: (r[0], r[1]))
        assert sorted((r[2], r[3]) for r in rows) == [(x, y) for x in range(m) for y in range(n)]


def test_worked_values_at_workload_grids():
    # 8192^3 with 128x256 tiles: 64 x 32 tiles, group 8 (all panels full).
    # t=153 (worker 5 at w=1 with 148 workers): 153 // 8 = 19 -> bx = 19 % 64 = 19,
    # by = 153 % 8 + (19 // 64) * 8 = 1
    assert schedule.tile_coord(0, 64, 32, 8) == (0, 0)
    assert schedule.tile_coord(7, 64, 32, 8) == (0, 7)
    assert schedule.tile_coord(8, 64, 32, 8) == (1, 0)
    assert schedule.tile_coord(153, 64, 32, 8) == (19, 1)
    assert schedule.tile_coord(512, 64, 32, 8) == (0, 8)    # first id of panel 1
    assert schedule.tile_coord(2047, 64, 32, 8) == (63, 31)
    # 1024^3: 8 x 4 tiles; one panel of width 4 (< group 8): row-major
    assert schedule.tile_coord(7, 8, 4, 8) == (1, 3)
    assert schedule.tile_coord(8, 8, 4, 8) == (2, 0)
    assert schedule.tile_coord(31, 8, 4, 8) == (7, 3)
    # 4000 x 7000: 32 x 28 tiles; three full panels (ids 0..767), then a panel of width 4
    assert schedule.tile_coord(767, 32, 28, 8) == (31, 23)
    assert schedule.tile_coord(768, 32, 28, 8) == (0, 24)
    assert schedule.tile_coord(771, 32, 28, 8) == (0, 27)
    assert schedule.tile_coord(772, 32, 28, 8) == (1, 24)
    assert schedule.tile_coord(895, 32, 28, 8) == (31, 27)
    # 256^3: 2 x 1 tiles, 148 workers: workers 0 and 1 take one tile each, the rest none
    assert schedule.enumerate_schedule(2, 1, 148, 8) == [(0, 0, 0, 0), (1, 0, 1, 0)]


def test_bad_arguments():
    with pytest.raises(ValueError):
        schedule.tile_coord(6, 2, 3, 8)
    with pytest.raises(ValueError):
        schedule.enumerate_schedule(0, 3, 4, 8)
