"""GPU: the device tile scheduler against the oracle's brute-force enumeration (bit-exact),
the GEMM kernel's own trace against the same enumeration, and the watchdog.
"""

import itertools
import math
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


@pytest.mark.parametrize("variant,cta,plain", [(v, 0, False) for v in VARIANTS] +
                         [("pair", 1, False), ("wide", 1, False), ("pair", 0, True),
                          ("pair", 1, True)])
def test_watchdog_fires_and_context_survives(variant, cta, plain):
    # the producer of CTA ``cta`` never fills pipeline phase 1: the MMA role's wait on it cannot
    # complete, the 20 ms watchdog must end every role and report TG_ERR_TIMEOUT.  In a CTA
    # pair, CTA 0 (even) skipping leaves a phase that only the odd CTA filled, CTA 1 (odd) one
    # that only the even CTA armed: the abort path must see both kinds of copies land.  With
    # ``plain`` the pair kernel runs the 2 x 2 tiles whole instead of as half-width units.
    M, N, K = 512, 512, 1024
    a, b = wl.make_inputs(M, N, K, "bf16", "uniform", seed=1)
    a_d, b_d = a.cuda(), b.cuda()
    c = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(tg.TgError) as e:
        tg.tg_gemm_persistent_debug(a_d, b_d, c, M, N, K, "bf16", variant=variant,
                                    watchdog_ns=20_000_000, inject_skip_phase=(cta << 32) + 1,
                                    plain=plain)
    assert e.value.code == tg.TG_ERR_TIMEOUT
    assert "watchdog" in str(e.value)
    # the context is intact: the status word was cleared and the next GEMM is correct
    assert tg.tg_device_status() == 0
    tg.tg_gemm_persistent_ex(a_d, b_d, c, M, N, K, "bf16", variant=variant)
    torch.cuda.synchronize()
    assert tg.tg_device_status() == 0
    assert_within_tolerance(wl.bits(c.cpu()), oracle_bits(a, b, "bf16"), "bf16", "after watchdog")


@pytest.mark.parametrize("M,N,K", [(256, 512, 128), (2560, 2560, 256), (4096, 4096, 192),
                                   (8192, 8192, 128), (4000, 7000, 128)])
def test_dynamic_persistence_runs_every_unit_once(M, N, K):
    # cluster launch control: one CTA per unit; a running CTA takes over the units of CTAs
    # not launched yet.  Which CTA runs which unit is up to the hardware; what is fixed is
    # the set of units and the decode of each (the oracle's, with the tail split of a
    # launch over all SMs), and that a CTA starts with the unit of its own index.
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    shape = tg.tg_gemm_launch_shape(M, N, K, "single", dynamic=True)
    units = shape["units"]
    assert shape["ctas"] == units
    want = schedule.enumerate_units(shape["m_tiles"], shape["n_tiles"], sms,
                                    tg.tg_gemm_config()["group"], split_tail=True)
    assert len(want) == units
    decode = {worker + w * sms: (bx, by, part) for (worker, w, bx, by, part) in want}
    a, b = wl.small_int_inputs(M, N, K, "bf16", seed=K)
    c = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    trace = torch.full((units, 5), -7, dtype=torch.int32, device="cuda")
    assert tg.tg_gemm_persistent_debug(a.cuda(), b.cuda(), c, M, N, K, "bf16", variant="single",
                                       trace=trace, dynamic=True,
                                       watchdog_ns=1_000_000_000) == 0
    got = trace.cpu().numpy()
    per_cta = {}
    for u in range(units):
        cta, w, bx, by, part = (int(v) for v in got[u])
        assert (bx, by, part) == decode[u], u
        assert 0 <= cta < units
        if w == 0:
            assert cta == u, (u, cta)
        per_cta.setdefault(cta, []).append(w)
    for cta, ws in per_cta.items():
        assert sorted(ws) == list(range(len(ws))), cta
    assert sum(len(ws) for ws in per_cta.values()) == units
    # integer inputs: every partial sum is exact, so the product is bit-exact
    assert np.array_equal(wl.bits(c.cpu()), oracle_bits(a, b, "bf16"))


def test_dynamic_persistence_matches_oracle_on_uniform_inputs():
    M, N, K = 4000, 7000, 2048
    a, b = wl.make_inputs(M, N, K, "bf16", "uniform", seed=5)
    c = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    tg.tg_gemm_persistent_ex(a.cuda(), b.cuda(), c, M, N, K, "bf16", variant="single",
                             dynamic=True)
    torch.cuda.synchronize()
    assert tg.tg_device_status() == 0
    assert_within_tolerance(wl.bits(c.cpu()), oracle_bits(a, b, "bf16"), "bf16", "dynamic")


def test_dynamic_persistence_watchdog():
    M, N, K = 512, 512, 1024
    a, b = wl.make_inputs(M, N, K, "bf16", "uniform", seed=1)
    a_d, b_d = a.cuda(), b.cuda()
    c = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(tg.TgError) as e:
        tg.tg_gemm_persistent_debug(a_d, b_d, c, M, N, K, "bf16", variant="single", dynamic=True,
                                    watchdog_ns=20_000_000, inject_skip_phase=5)
    assert e.value.code == tg.TG_ERR_TIMEOUT
    assert tg.tg_device_status() == 0
    tg.tg_gemm_persistent_ex(a_d, b_d, c, M, N, K, "bf16", variant="single", dynamic=True)
    torch.cuda.synchronize()
    assert tg.tg_device_status() == 0
    assert_within_tolerance(wl.bits(c.cpu()), oracle_bits(a, b, "bf16"), "bf16", "after watchdog")


def test_dynamic_needs_single_variant():
    a = torch.zeros((256, 256), dtype=torch.bfloat16, device="cuda")
    c = torch.empty_like(a)
    with pytest.raises(tg.TgError) as e:
        tg.tg_gemm_persistent_ex(a, a, c, 256, 256, 256, "bf16", variant="pair", dynamic=True)
    assert e.value.code == tg.TG_ERR_ARG


@pytest.mark.parametrize("group", [1, 3, 12])
@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("M,N,K", [(4096, 4096, 64), (4000, 7000, 128)])
def test_group_width_option_followed(M, N, K, variant, group):
    # TG_SCHEDULE_GROUP(g): the kernel walks the grouped order of width g, as the oracle does
    shape = tg.tg_gemm_launch_shape(M, N, K, variant)
    units = shape["units"]
    a, b = wl.small_int_inputs(M, N, K, "bf16", seed=group)
    c = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    trace = torch.full((units, 5), -7, dtype=torch.int32, device="cuda")
    assert tg.tg_gemm_persistent_debug(a.cuda(), b.cuda(), c, M, N, K, "bf16", variant=variant,
                                       trace=trace, group=group) == 0
    want = schedule.enumerate_units(shape["m_tiles"], shape["n_tiles"], shape["workers"], group,
                                    split_tail=True)
    by_unit = {worker + w * shape["workers"]: (worker, w, bx, by, part)
               for (worker, w, bx, by, part) in want}
    got = trace.cpu().numpy()
    for u in range(units):
        assert tuple(int(v) for v in got[u]) == by_unit[u], u
    assert np.array_equal(wl.bits(c.cpu()), oracle_bits(a, b, "bf16"))


@pytest.mark.parametrize("M,N,K,rows", [(4096, 4096, 64, "rows"), (2048, 40960, 1024, "columns"),
                                        (8192, 8192, 4104, "groups")])
def test_auto_traversal_is_reported_and_followed(M, N, K, rows):
    # TG_VARIANT_AUTO picks the traversal too: whole rows of tiles when B fits in half of the
    # L2 (64 MiB), whole columns when only A does, else balanced groups; tg_gemm_launch_shape
    # reports it and the kernel's trace follows the oracle's enumeration of it
    shape = tg.tg_gemm_launch_shape(M, N, K)
    # "groups": neither operand fits; the wide kernel's 256 x 512 tiles take groups of
    # round(sqrt(2 P)) M-tiles in column order, square tiles the page's 8 in row order
    wide = shape["tile_n"] > shape["tile_m"]
    groups = (int(math.sqrt(2 * shape["workers"]) + 0.5), 1) if wide else (8, 0)
    want_order = {"rows": (shape["n_tiles"], 0), "columns": (shape["m_tiles"], 1),
                  "groups": groups}[rows]
    assert (shape["group"], shape["column_major"]) == want_order
    units = shape["units"]
    a, b = wl.small_int_inputs(M, N, K, "bf16", lo=-1, hi=1, seed=K)
    c = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    trace = torch.full((units, 5), -7, dtype=torch.int32, device="cuda")
    assert tg.tg_gemm_persistent_debug(a.cuda(), b.cuda(), c, M, N, K, "bf16", trace=trace) == 0
    want = schedule.enumerate_units(shape["m_tiles"], shape["n_tiles"], shape["workers"],
                                    shape["group"], split_tail=True,
                                    column_major=bool(shape["column_major"]))
    by_unit = {worker + w * shape["workers"]: (worker, w, bx, by, part)
               for (worker, w, bx, by, part) in want}
    got = trace.cpu().numpy()
    for u in range(units):
        assert tuple(int(v) for v in got[u]) == by_unit[u], u
    assert np.array_equal(wl.bits(c.cpu()), oracle_bits(a, b, "bf16"))


@pytest.mark.parametrize("M,N,K,want", [(1024, 1024, 4096, 2), (512, 512, 8192, 2),
                                        (1024, 1024, 1024, 1), (1024, 1024, 2048, 1),
                                        (128, 1024, 8192, 1), (2048, 1024, 4096, 2)])
def test_auto_takes_the_pair_kernel_for_long_k_below_a_wave(M, N, K, want):
    # below one wave of pair tiles, TG_VARIANT_AUTO still takes the CTA-pair kernel once
    # K >= 4096 and M fills its 256 rows (measured faster there), else the single-CTA kernel,
    # for the dense and the MXFP8 GEMM alike; the product is exact on integer inputs either way
    shape = tg.tg_gemm_launch_shape(M, N, K)
    pair_tiles = ((M + 255) // 256) * ((N + 255) // 256)
    assert pair_tiles < torch.cuda.get_device_properties(0).multi_processor_count // 2
    assert shape["variant"] == want
    assert tg.tg_gemm_launch_shape(M, N, K, mxfp8=True)["variant"] == want
    a, b = wl.small_int_inputs(M, N, K, "bf16", lo=-1, hi=1, seed=K + M)
    c = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    tg.tg_gemm_persistent(a.cuda(), b.cuda(), c, M, N, K, "bf16")
    torch.cuda.synchronize()
    assert tg.tg_device_status() == 0
    assert np.array_equal(wl.bits(c.cpu()), oracle_bits(a, b, "bf16"))
