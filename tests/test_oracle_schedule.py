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


@pytest.mark.parametrize("workers", [1, 3, 7, 76, 148, 152])
def test_units_cover_every_tile_exactly_once(workers):
    # whole tiles plus half tiles: each tile is covered either once whole or by both halves
    for m, n, g in itertools.product([1, 2, 5, 8, 13, 32], [1, 3, 4, 9, 28, 32], [1, 8]):
        rows = schedule.enumerate_units(m, n, workers, g)
        cover = {}
        for (_, _, bx, by, part) in rows:
            cover.setdefault((bx, by), []).append(part)
        assert sorted(cover) == [(x, y) for x in range(m) for y in range(n)]
        for parts in cover.values():
            assert sorted(parts) in ([-1], [0, 1])


def test_tail_split_only_when_the_last_wave_is_at_most_half_full():
    # 8192^3 single tiles: 2048 = 13 * 152 + 72, 2 * 72 <= 152 -> split the last 72 tiles
    assert schedule.tail_split_point(64, 32, 152) == (1976, 1976 + 144)
    # 8192^3 pair tiles: 1024 = 13 * 76 + 36
    assert schedule.tail_split_point(32, 32, 76) == (988, 988 + 72)
    # 4000 x 7000 single: 896 = 5 * 152 + 136 and 2 * 136 > 152: no split
    assert schedule.tail_split_point(32, 28, 152) == (896, 896)
    # fewer tiles than workers: every tile is split when 2T <= P
    assert schedule.tail_split_point(8, 4, 152) == (0, 64)
    assert schedule.tail_split_point(8, 4, 76) == (0, 64)
    assert schedule.tail_split_point(8, 8, 76) == (64, 64)
    # exact waves: nothing to split
    assert schedule.tail_split_point(8, 19, 152) == (152, 152)


def test_units_without_split_are_the_page_schedule():
    for m, n, p, g in [(64, 32, 152, 8), (32, 28, 148, 8), (8, 4, 148, 8), (5, 9, 7, 3)]:
        plain = schedule.enumerate_units(m, n, p, g, split_tail=False)
        assert plain == [r + (-1,) for r in schedule.enumerate_schedule(m, n, p, g)]


def test_split_units_follow_the_grid_stride_and_the_grouped_order():
    m, n, p, g = 64, 32, 152, 8
    first, units = schedule.tail_split_point(m, n, p)
    rows = schedule.enumerate_units(m, n, p, g)
    for (c, w, bx, by, part) in rows:
        u = c + w * p
        if u < first:
            assert part == -1 and (bx, by) == schedule.tile_coord(u, m, n, g)
        else:
            assert (bx, by) == schedule.tile_coord(first + (u - first) // 2, m, n, g)
            assert part == (u - first) % 2
    # workers' unit counts differ by at most one
    counts = [sum(1 for r in rows if r[0] == c) for c in range(p)]
    assert max(counts) - min(counts) <= 1


@pytest.mark.parametrize("group", [1, 2, 3, 8, 16])
def test_column_major_every_tile_exactly_once(group):
    for m, n in GRIDS:
        seen = [schedule.tile_coord_column_major(t, m, n, group) for t in range(m * n)]
        assert sorted(seen) == [(bx, by) for bx in range(m) for by in range(n)], (m, n, group)


def test_column_major_textbook_orders():
    for m, n in GRIDS:
        for t in range(m * n):
            # group 1: row-major walk of the tile grid; one panel (group >= m): column-major
            assert schedule.tile_coord_column_major(t, m, n, 1) == (t // n, t % n)
            assert schedule.tile_coord_column_major(t, m, n, m) == (t % m, t // m)


def test_column_major_panels_top_to_bottom():
    m, n, g = 13, 9, 4
    coords = [schedule.tile_coord_column_major(t, m, n, g) for t in range(m * n)]
    panels = [bx // g for bx, _ in coords]
    assert panels == sorted(panels)
    # inside a panel, ids run down M first: g consecutive ids share by
    assert coords[:4] == [(0, 0), (1, 0), (2, 0), (3, 0)]
    assert coords[4] == (0, 1)


def test_column_major_units_cover_every_tile():
    for m, n, p in [(32, 28, 76), (5, 9, 7), (64, 32, 152)]:
        rows = schedule.enumerate_units(m, n, p, 8, split_tail=True, column_major=True)
        cover = {}
        for (_, _, bx, by, part) in rows:
            cover.setdefault((bx, by), []).append(part)
        assert sorted(cover) == [(x, y) for x in range(m) for y in range(n)]
        assert all(sorted(v) in ([-1], [0, 1]) for v in cover.values())
