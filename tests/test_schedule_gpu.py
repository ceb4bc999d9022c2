"""GPU: the device tile scheduler against the oracle's brute-force enumeration (bit-exact),
the GEMM kernel's own trace against the same enumeration, and the watchdog.
"""

import itertools
import os

import numpy as np
import pytest
import torch

import persistent_warp_specialized_gb300 as tg
from persistent_warp_specialized_gb300 import workloads as wl
from oracle import schedule

from gpu_helpers import VARIANTS, assert_within_tolerance, ensure_library, oracle_bits

pytestmark = pytest.mark.gpu

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ensure_library()


def test_schedule_brute_force_grids():
    for m, n, g, p in itertools.product([1, 2, 5, 8, 13, 32], [1, 3, 4, 9, 16, 28],
                                        [1, 3, 8], [1, 7, 148, 160]):
        assert tg.tg_tile_schedule(m, n, p, g) == schedule.enumerate_schedule(m, n, p, g), (m, n, g, p)


@pytest.mark.parametrize("name", sorted(f for f in os.listdir(GOLDEN) if f.startswith("schedule_")))
def test_schedule_matches_stored_fixture(name):
    meta = {}
    rows = []
    for line in open(os.path.join(GOLDEN, name)):
        if line.startswith("#"):
            meta.update(dict(t.split("=") for t in line[1:].split() if "=" in t))
            continue
        rows.append(tuple(int(x) for x in line.split()))
    got = tg.tg_tile_schedule(int(meta["m_blocks"]), int(meta["n_blocks"]), int(meta["workers"]),
                              int(meta["group"]))
    assert got == rows


def test_unit_schedule_brute_force_grids():
    for m, n, g, p in itertools.product([1, 2, 5, 8, 13, 32, 64], [1, 3, 4, 9, 16, 28, 32],
                                        [1, 8], [1, 7, 76, 148, 152]):
        for split, cm in itertools.product((False, True), (False, True)):
            got = tg.tg_tile_schedule_ex(m, n, p, g, split, cm)
            want = schedule.enumerate_units(m, n, p, g, split, cm)
            assert got == want, (m, n, g, p, split, cm)


def test_config1_schedule_148_workers():
    # the 256^3 workload: 2 x 1 tiles over 148 workers, group 8
    assert tg.tg_tile_schedule(2, 1, wl.SCHEDULE_CHECK_WORKERS, wl.SCHEDULE_CHECK_GROUP) == [
        (0, 0, 0, 0), (1, 0, 1, 0)]


@pytest.mark.parametrize("plain,column_major", [(False, False), (True, False), (False, True)])
@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("M,N,K", [(4000, 7000, 256), (8192, 8192, 64), (1024, 1024, 1024),
                                   (256, 256, 256), (4000, 2048, 128), (2560, 2560, 128)])
def test_kernel_followed_the_schedule(M, N, K, variant, plain, column_major):
    # the epilogue of the real GEMM records (worker, w, bx, by, part) for every unit it stored
    shape = tg.tg_gemm_launch_shape(M, N, K, variant, plain)
    m_tiles, n_tiles, workers = shape["m_tiles"], shape["n_tiles"], shape["workers"]
    units = shape["units"]
    a, b = wl.make_inputs(M, N, K, "bf16", "uniform", seed=M)
    a_d, b_d = a.cuda(), b.cuda()
    c = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    trace = torch.full((units, 5), -7, dtype=torch.int32, device="cuda")
    assert tg.tg_gemm_persistent_debug(a_d, b_d, c, M, N, K, "bf16", variant=variant,
                                       trace=trace, plain=plain, column_major=column_major) == 0
    want = schedule.enumerate_units(m_tiles, n_tiles, workers, tg.tg_gemm_config()["group"],
                                    split_tail=not plain, column_major=column_major)
    assert len(want) == units
    by_unit = {}
    for (worker, w, bx, by, part) in want:
        by_unit[worker + w * workers] = (worker, w, bx, by, part)
    got = trace.cpu().numpy()
    for u in range(units):
        assert tuple(int(v) for v in got[u]) == by_unit[u], u
    # the debug build computes the same product
    assert_within_tolerance(wl.bits(c.cpu()), oracle_bits(a, b, "bf16"), "bf16", "debug build")


@pytest.mark.parametrize("variant", VARIANTS)
def test_watchdog_fires_and_context_survives(variant):
    # CTA 0's producer never fills pipeline phase 5: the MMA role's wait on it cannot
    # complete, the 20 ms watchdog must end every role and report TG_ERR_TIMEOUT
    M, N, K = 512, 512, 1024
    a, b = wl.make_inputs(M, N, K, "bf16", "uniform", seed=1)
    a_d, b_d = a.cuda(), b.cuda()
    c = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(tg.TgError) as e:
        tg.tg_gemm_persistent_debug(a_d, b_d, c, M, N, K, "bf16", variant=variant,
                                    watchdog_ns=20_000_000, inject_skip_phase=5)
    assert e.value.code == tg.TG_ERR_TIMEOUT
    assert "watchdog" in str(e.value)
    # the context is intact: the status word was cleared and the next GEMM is correct
    assert tg.tg_device_status() == 0
    tg.tg_gemm_persistent_ex(a_d, b_d, c, M, N, K, "bf16", variant=variant)
    torch.cuda.synchronize()
    assert tg.tg_device_status() == 0
    assert_within_tolerance(wl.bits(c.cpu()), oracle_bits(a, b, "bf16"), "bf16", "after watchdog")
