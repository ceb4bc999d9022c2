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
