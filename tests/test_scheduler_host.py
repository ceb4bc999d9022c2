"""The kernels' tile scheduler (tg_tile_scheduler.cuh) built for the host with g++ and run
against the schedule oracle: whole tiles, the tail split and the stream-K tail (no GPU)."""

import os
import shutil
import subprocess

import pytest

from oracle import schedule as s

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "persistent_warp_specialized_gb300", "csrc")


@pytest.fixture(scope="module")
def driver(tmp_path_factory):
    cxx = shutil.which("g++")
    if cxx is None:
        pytest.skip("g++ not found")
    out = str(tmp_path_factory.mktemp("sched") / "scheduler_driver")
    subprocess.run([cxx, "-O1", "-std=c++17", "-D__host__=", "-D__device__=", "-I", CSRC,
                    os.path.join(ROOT, "tests", "scheduler_driver.cpp"), "-o", out], check=True)
    return out


def run(driver, m, n, P, g, kb, col, split, tail):
    text = subprocess.run([driver] + [str(x) for x in (m, n, P, g, kb, int(col), int(split), tail)],
                          check=True, capture_output=True, text=True).stdout
    return [tuple(int(x) for x in line.split()) for line in text.splitlines()]


CASES = [(16, 16, 76, 16, 32), (32, 16, 76, 12, 128), (4, 25, 76, 8, 16), (3, 7, 5, 2, 9),
         (1, 1, 4, 1, 3), (5, 3, 7, 1, 1), (9, 4, 11, 3, 5), (2, 3, 4, 8, 64), (8, 4, 152, 8, 16)]


@pytest.mark.parametrize("m,n,P,g,kb", CASES)
@pytest.mark.parametrize("col", [False, True])
def test_stream_k_tail_matches_the_oracle(driver, m, n, P, g, kb, col):
    tail = (m * n) % P
    got = run(driver, m, n, P, g, kb, col, False, tail)
    assert got == s.enumerate_units_streamk(m, n, P, g, kb, col)


@pytest.mark.parametrize("m,n,P,g,kb", CASES)
@pytest.mark.parametrize("col", [False, True])
@pytest.mark.parametrize("split", [False, True])
def test_whole_and_half_units_match_the_oracle(driver, m, n, P, g, kb, col, split):
    got = run(driver, m, n, P, g, kb, col, split, 0)
    ref = s.enumerate_units(m, n, P, g, split_tail=split, column_major=col)
    assert [r[:5] for r in got] == ref
    assert all(r[5:7] == (0, kb) for r in got)
