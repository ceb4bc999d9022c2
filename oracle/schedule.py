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
