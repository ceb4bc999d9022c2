"""The schedule entry point that allocates no device memory, tg_tile_schedule_noalloc.

tg_tile_schedule_ex stages its rows in a device buffer it allocates and frees inside the call.
Callers whose device memory is all owned by their own pool allocator, or that must not stall
on cudaFree (which waits for the whole device), use tg_tile_schedule_noalloc instead: it
stages the rows in a fixed array in the library's device image.  Its rows must equal the
oracle's enumeration of the same traversal (and therefore the allocating call's).  The file is
named so that pytest collects it last.
"""

import pytest

import persistent_warp_specialized_gb300 as tg
from oracle import schedule

from gpu_helpers import ensure_library


@pytest.mark.gpu
def test_noalloc_schedule_equals_the_allocating_one_on_consecutive_calls():
    ensure_library()
    # a large schedule, then smaller ones: the array keeps the previous call's rows, so a
    # second call that copied back anything it did not write would differ here
    cases = [
        (256, 128, 152, 8, True, False),    # 32768 tiles, tail split on 152 workers
        (32, 32, 76, 8, True, False),       # the pair kernel's 8192^3 schedule
        (5, 7, 152, 8, True, True),         # fewer tiles than workers, column-major
        (16, 28, 76, 8, False, False),      # 4096 x 7168 in pair tiles, no split
    ]
    for m, n, sms, group, split, cm in cases:
        want = schedule.enumerate_units(m, n, sms, group, split_tail=split, column_major=cm)
        for _ in range(2):
            got = tg.tg_tile_schedule_noalloc(m, n, sms, group, split_tail=split,
                                              column_major=cm)
            assert got == want, (m, n, sms, group, split, cm)
            assert got == tg.tg_tile_schedule_ex(m, n, sms, group, split_tail=split,
                                                 column_major=cm)


@pytest.mark.gpu
def test_noalloc_schedule_at_its_maximum_size():
    ensure_library()
    m, n = 256, 256                         # exactly TG_SCHEDULE_NOALLOC_MAX_UNITS tiles
    assert m * n == tg.TG_SCHEDULE_NOALLOC_MAX_UNITS
    got = tg.tg_tile_schedule_noalloc(m, n, 152, 8, split_tail=False)
    assert len(got) == m * n
    assert got == schedule.enumerate_units(m, n, 152, 8, split_tail=False)


def test_noalloc_schedule_rejects_sizes_beyond_its_scratch():
    # the size check returns before any CUDA call, so this runs without a GPU
    ensure_library()
    with pytest.raises(tg.TgError) as e:
        tg.tg_tile_schedule_noalloc(257, 256, 152, 8, split_tail=False)
    assert e.value.code == tg.TG_ERR_ARG
    assert "scratch" in str(e.value)
    with pytest.raises(tg.TgError) as e:              # the tail split adds units
        tg.tg_tile_schedule_noalloc(256, 256, 151, 8, split_tail=True)
    assert e.value.code == tg.TG_ERR_ARG
