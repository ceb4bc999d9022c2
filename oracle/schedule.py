"""Brute-force persistent tile schedule (oracle; test infrastructure only).

Output tiles form an m_blocks x n_blocks grid; ``bx`` indexes M-tiles (rows) and ``by``
N-tiles (columns), as in ``A[bx * block_M : ...]`` and ``B[..., by * block_N : ...]`` of
``gemm_persistent`` ("[Feature] Introduce tile scheduler #2441", examples/gemm_sm100/
gemm_tcgen5mma_ws_persistent.py).

Persistent traversal: worker ``c`` of ``P`` workers visits linear tile ids
``t = c + w * P`` for w = 0, 1, ... while ``t < m_blocks * n_blocks``; ``w`` is the
worker's single iteration clock (``sched.current_iter[0]``), and before the scheduler
the same loop was ``tile_id = sm_num * w + block_id``.

Grouped decode of a linear id: tiles are walked in panels of ``group`` N-tiles; inside
a panel ids run along N first, then down all M-tiles:

    bx = (t // g) % m_blocks
    by = t % g + (t // g) // m_blocks * g

The page asserts ``n_blocks % (2 * group_size) == 0`` so it never meets a partial
panel.  Reading taken for the last panel when ``n_blocks % g != 0``: it is the same
walk on a panel narrowed to its real width ``n_blocks % g``, so every id in
[0, m_blocks * n_blocks) names a distinct tile and no id is skipped.
"""


def tile_coord(t, m_blocks, n_blocks, group):
    """Linear tile id -> (bx, by) under the grouped order with a narrowed last panel."""
    if not (0 <= t < m_blocks * n_blocks):
        raise ValueError(f"tile id {t} outside [0, {m_blocks * n_blocks})")
    full_panels = n_blocks // group
    first_tail_id = full_panels * group * m_blocks
    if t < first_tail_id:
        g = group
        bx = (t // g) % m_blocks
        by = t % g + (t // g) // m_blocks * g
        return bx, by
    # last panel: the same decode with g := its width, offset to its first column
    g = n_blocks - full_panels * group
    u = t - first_tail_id
    bx = (u // g) % m_blocks
    by = full_panels * group + u % g + (u // g) // m_blocks * g
    return bx, by


def enumerate_schedule(m_blocks, n_blocks, num_workers, group):
    """Rows (worker, w, bx, by), ordered by worker, then by w."""
    if min(m_blocks, n_blocks, num_workers, group) < 1:
        raise ValueError("m_blocks, n_blocks, num_workers and group must be >= 1")
    total = m_blocks * n_blocks
    rows = []
    for c in range(num_workers):
        w = 0
        while c + w * num_workers < total:
            t = c + w * num_workers
            bx, by = tile_coord(t, m_blocks, n_blocks, group)
            rows.append((c, w, bx, by))
            w += 1
    return rows


def tile_coord_column_major(t, m_blocks, n_blocks, group):
    """The ``column_major`` order of the scheduler: panels of ``group`` M-tiles, ids running
    along M first, then across N -- the grouped decode with the roles of M and N exchanged."""
    by, bx = tile_coord(t, n_blocks, m_blocks, group)
    return bx, by


def tail_split_point(m_blocks, n_blocks, num_workers):
    """(F, units): tiles 0..F-1 stay whole; when the last partial wave holds R = T - F tiles
    with 0 < 2R <= P, each of those R tiles becomes two half-width units, else F = T."""
    total = m_blocks * n_blocks
    rem = total % num_workers
    if rem == 0 or 2 * rem > num_workers:
        return total, total
    first = total - rem
    return first, first + 2 * rem


def unit_tile(u, m_blocks, n_blocks, group, first_split, column_major=False):
    """Unit id -> (bx, by, part): part -1 is a whole tile, 0 / 1 the left / right half (in N)
    of tile first_split + (u - first_split) // 2."""
    decode = tile_coord_column_major if column_major else tile_coord
    if u < first_split:
        bx, by = decode(u, m_blocks, n_blocks, group)
        return bx, by, -1
    t = first_split + (u - first_split) // 2
    bx, by = decode(t, m_blocks, n_blocks, group)
    return bx, by, (u - first_split) % 2


def enumerate_units(m_blocks, n_blocks, num_workers, group, split_tail=True, column_major=False):
    """Rows (worker, w, bx, by, part) of the persistent traversal over work units, ordered
    by worker, then w.  Without the split (or when it does not apply) every unit is a whole
    tile and the rows are those of enumerate_schedule with part = -1.

    Reading beyond the pages (the grouped traversal itself is the page's): the last partial
    wave, if at most half the workers would be busy in it, is cut into half-width units so
    that it takes half a tile's time; unit ids keep the grid stride c, c + P, ...
    """
    if min(m_blocks, n_blocks, num_workers, group) < 1:
        raise ValueError("m_blocks, n_blocks, num_workers and group must be >= 1")
    if split_tail:
        first, units = tail_split_point(m_blocks, n_blocks, num_workers)
    else:
        first = units = m_blocks * n_blocks
    rows = []
    for c in range(num_workers):
        w = 0
        while c + w * num_workers < units:
            bx, by, part = unit_tile(c + w * num_workers, m_blocks, n_blocks, group, first,
                                     column_major)
            rows.append((c, w, bx, by, part))
            w += 1
    return rows


# ---------------------------------------------------------------- stream-K tail
# Reading beyond the pages (their scheduler walks whole tiles): the library can instead split
# the last partial wave along K (on request; it never does by itself).  With T tiles and P workers, the R = T mod P tiles that come
# last in the traversal form the tail; their k-blocks, numbered tile-major (tile i of the tail
# owns numbers i*KB .. i*KB + KB - 1), are cut into P contiguous ranges, worker c taking
# [floor(c*R*KB/P), floor((c+1)*R*KB/P)).  The whole tiles before the tail keep the grid stride.
# A worker's range is shorter than KB (R < P), so it meets at most two tail tiles.  The worker
# whose range holds a tail tile's last k-block owns that tile: it adds the other workers' partial
# sums of the tile to its own and stores the tile.  A worker walks its part of the later tile
# (a contribution) before its part of the earlier one (which it owns), so every owner waits only
# for lower-numbered workers' contributions, each made first in its worker's range.


def streamk_range(c, workers, sk_tiles, k_blocks):
    """Worker c's k-blocks [lo, hi) of the tail, tile-major."""
    total = sk_tiles * k_blocks
    return total * c // workers, total * (c + 1) // workers


def streamk_segments(c, workers, sk_tiles, k_blocks):
    """Worker c's tail segments in the order it walks them: (tail tile index, k_lo, k_hi, owns).
    Brute force over the range's k-blocks, grouped by tile."""
    lo, hi = streamk_range(c, workers, sk_tiles, k_blocks)
    by_tile = {}
    for g in range(lo, hi):
        by_tile.setdefault(g // k_blocks, []).append(g % k_blocks)
    segs = []
    for t, ks in by_tile.items():
        assert ks == list(range(ks[0], ks[-1] + 1))
        segs.append((t, ks[0], ks[-1] + 1, ks[-1] == k_blocks - 1))
    segs.sort(key=lambda s: s[3])            # contributions first, the owned tile last
    return segs


def streamk_contributors(t, workers, sk_tiles, k_blocks):
    """(owner, [contributing workers]) of tail tile t: every worker whose range meets the tile,
    the owner being the one holding its last k-block."""
    meets = []
    for c in range(workers):
        lo, hi = streamk_range(c, workers, sk_tiles, k_blocks)
        if lo < hi and lo < (t + 1) * k_blocks and hi > t * k_blocks:
            meets.append(c)
    owner = [c for c in meets
             if streamk_range(c, workers, sk_tiles, k_blocks)[0] <= (t + 1) * k_blocks - 1
             < streamk_range(c, workers, sk_tiles, k_blocks)[1]]
    assert len(owner) == 1
    return owner[0], [c for c in meets if c != owner[0]]


def enumerate_units_streamk(m_blocks, n_blocks, num_workers, group, k_blocks,
                            column_major=False):
    """Rows (worker, w, bx, by, part, k_lo, k_hi, unit) of the traversal with the stream-K
    tail: whole tiles (part -1, k 0..KB, unit = their linear id) on the grid stride, then each
    worker's tail segments in walking order (part 2 = a contribution, 3 = the owned tile; unit =
    D + 2c + part - 2, D = the number of whole tiles).  Ordered by worker, then w."""
    if min(m_blocks, n_blocks, num_workers, group, k_blocks) < 1:
        raise ValueError("m_blocks, n_blocks, num_workers, group and k_blocks must be >= 1")
    decode = tile_coord_column_major if column_major else tile_coord
    total = m_blocks * n_blocks
    sk = total % num_workers
    whole = total - sk
    rows = []
    for c in range(num_workers):
        w = 0
        while c + w * num_workers < whole:
            bx, by = decode(c + w * num_workers, m_blocks, n_blocks, group)
            rows.append((c, w, bx, by, -1, 0, k_blocks, c + w * num_workers))
            w += 1
        if sk:
            for (t, k_lo, k_hi, owns) in streamk_segments(c, num_workers, sk, k_blocks):
                bx, by = decode(whole + t, m_blocks, n_blocks, group)
                part = 3 if owns else 2
                rows.append((c, w, bx, by, part, k_lo, k_hi, whole + 2 * c + part - 2))
                w += 1
    return rows
