"""Writes the tile-schedule fixtures in this folder from the CPU oracle alone.

    python tests/golden/make_golden.py

Each fixture is the persistent schedule of one workload's tile grid (128 x 256 output
tiles) over 148 workers with group width 8: one row ``worker w bx by`` per tile, ordered
by worker, then by w.  The schedule is the grouped persistent traversal of
"[Feature] Introduce tile scheduler #2441" (examples/gemm_sm100/
gemm_tcgen5mma_ws_persistent.py, ``gemm_persistent``), with the narrowed last panel
read for grids whose N-tile count is not a multiple of the group width.
"""

import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

from oracle import schedule  # noqa: E402

BLOCK_M, BLOCK_N = 128, 256
WORKERS, GROUP = 148, 8
CASES = {
    "schedule_256x256.txt": (256, 256),
    "schedule_1024x1024.txt": (1024, 1024),
    "schedule_4000x7000.txt": (4000, 7000),
    "schedule_8192x8192.txt": (8192, 8192),
}


def grid(M, N):
    return -(-M // BLOCK_M), -(-N // BLOCK_N)


def main():
    for name, (M, N) in CASES.items():
        m, n = grid(M, N)
        rows = schedule.enumerate_schedule(m, n, WORKERS, GROUP)
        with open(os.path.join(HERE, name), "w") as f:
            f.write(f"# M={M} N={N} tiles {BLOCK_M}x{BLOCK_N}: m_blocks={m} n_blocks={n} "
                    f"workers={WORKERS} group={GROUP}\n")
            f.write("# written by tests/golden/make_golden.py from oracle.schedule\n")
            for r in rows:
                f.write("%d %d %d %d\n" % r)


if __name__ == "__main__":
    main()
