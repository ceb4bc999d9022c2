"""Host-side logic of bench.py, on the CPU: max over ranks with two gloo ranks, the clock
summary, and the reference arm (the CPU oracle) end to end on the smallest workload."""

import json
import os
import socket
import subprocess
import sys
import time

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    import torch.distributed as dist

    bench.init_dist(world, "gloo")
    bench.barrier()
    got = bench.max_over_ranks(1.5 + rank * 2.0)
    out.put((rank, got))
    dist.destroy_process_group()


def test_max_over_ranks_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    results = sorted(q.get(timeout=10) for _ in range(2))
    assert results == [(0, 3.5), (1, 3.5)]


def test_max_over_ranks_single_process_is_identity():
    sys.path.insert(0, ROOT)
    import bench

    assert bench.max_over_ranks(2.25) == 2.25


def test_clock_summary_keeps_only_the_timed_window():
    sys.path.insert(0, ROOT)
    import bench

    def row(t, mhz, power_cap="Not Active"):
        stamp = time.strftime("%Y/%m/%d %H:%M:%S", time.localtime(int(t))) + ".%03d" % int((t % 1) * 1000)
        return (f"{stamp}, 0, {mhz}, 2070, 1200.0, 0x0000000000000004, Not Active, Not Active, "
                f"Not Active, {power_cap}")

    t0 = 1_800_000_000.0
    lines = [row(t0 - 5, 300), row(t0 + 0.2, 1500), row(t0 + 0.4, 1400, "Active"),
             row(t0 + 0.6, 1600), row(t0 + 9, 200)]
    c = bench.parse_clock_csv(lines, t0, t0 + 1.0)
    assert c["samples"] == 3
    assert c["sm_mhz"] == 1500
    assert c["sm_max_mhz"] == 2070
    assert c["reasons"] == ["sw_power_cap"]
    empty = bench.parse_clock_csv(lines, t0 + 100, t0 + 101)
    assert empty["samples"] == 0 and empty["sm_mhz"] is None


def test_reference_arm_prints_one_json_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--workload", "gemm_256_f16", "--steps", "3", "--warmup", "1"],
                       capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference"
    assert d["unit"] == "TFLOP/s" and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0
    assert d["config"]["workload"] == "gemm_256_f16"


def test_reference_arm_nonzero_rank_does_no_work():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--workload", "gemm_256_f16", "--steps", "1", "--warmup", "0"],
                       capture_output=True, text=True, timeout=300, cwd=ROOT, env=env)
    assert r.returncode == 0
    assert r.stdout.strip() == ""


def test_mxfp8_reference_arm_prints_one_json_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--workload", "mxfp8_512", "--steps", "2", "--warmup", "1"],
                       capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["value"] > 0
    assert d["config"]["workload"] == "mxfp8_512" and d["config"]["in_dtype"] == "e4m3"
    assert d["cpu_baseline"]["kind"] == "oracle"


def test_oracle_sample_grows_past_the_fixed_cost_of_a_call():
    sys.path.insert(0, ROOT)
    import bench

    # every call costs 30 ms plus 0.1 ms per row: a 32-row probe would predict ~1 ms per row
    calls = []

    def run(rows):
        calls.append(rows)
        time.sleep(0.03 + 1e-4 * rows)
        return rows

    rows, dt, out = bench.timed_oracle_sample(run, 100000, 0.4)
    assert out == rows == calls[-1]
    assert dt >= 0.2
    assert rows > 32 * 0.4 / (0.03 + 32e-4)    # more than the one-probe estimate
    rows, dt, out = bench.timed_oracle_sample(run, 200, 10.0)
    assert rows == 200                        # never beyond M


def test_reference_block_side_bounds_one_step():
    sys.path.insert(0, ROOT)
    import bench

    # a call costs 1 ms per unit of r (the operand decode) plus r^2 / 4e6 s (the product)
    def run(r):
        time.sleep(1e-6 * r + r * r / 4e6)

    r = bench.block_side(run, 8192, 0.2)
    t0 = time.perf_counter()
    run(r)
    dt = time.perf_counter() - t0
    assert 0.1 <= dt <= 0.9
    assert bench.block_side(run, 100, 5.0) == 100     # never beyond the matrix


def test_mxfp8_workload_rejects_the_dense_only_variant():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--workload", "mxfp8_512",
                        "--variant", "wide", "--steps", "1", "--warmup", "0"],
                       capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert r.returncode == 2 and r.stdout.strip() == ""
    assert "dense" in r.stderr
