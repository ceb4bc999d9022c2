#!/usr/bin/env python3
"""Throughput of the persistent warp-specialized GEMM on GB300: one JSON line.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl tg|reference]
                    [--workload gemm_8192_bf16 | mxfp8_8192]

A step is one pass of the whole hot path: one tg_gemm_persistent call (one kernel launch)
on the workload's seeded synthetic inputs, already resident in HBM.  ``value`` is
2MNK / (device time per step) in TFLOP/s, timed with CUDA events on the launching stream
over K back-to-back steps after W warm-up steps.  The 8192^3 bf16 inputs (A + B = 256 MiB)
are larger than the 129 MB L2, so no flush runs between steps.

Also reported: ``e2e`` (the same metric through tg_gemm_persistent_host: pinned host A, B
copied in and C copied out every step; consecutive steps alternate between two streams with
their own device buffers, so one step's copies overlap the other's GEMM), ``roofline`` (tensor-bound: achieved TFLOP/s over
the measured cuBLAS bf16 peak of this GPU type), ``clocks`` (nvidia-smi sampled during the
timed region) and ``cpu_baseline`` (the CPU oracle timed on a bounded row slab of the same
workload, which also checks the GPU's rows of that slab).  ``pct_of_dense_peak`` quotes the
value against the one stated dense bf16 peak (``dense_peak``: 2.5 PFLOP/s, with its source).

With the 8192^3 workload two more records follow the headline:
* ``sustained``: back-to-back launches for ``--sustained-seconds`` (3 s) with clocks sampled,
  the rate the kernel holds at the GPU's power limit;
* ``per_config``: every workload of the metric (256^3 and 1024^3 fp16, 4096^3 and 8192^3
  bf16, 4000 x 7000 x 2048 bf16) and the block-scaled MXFP8 GEMM at 8192^3, each timed as the
  pages' benchmark times the kernel (50 warm-up and 50 timed launches), here with L2 flushed
  before every timed launch and CUDA events around each; with the kernel the library picked,
  compulsory DRAM GB/s, the CPU oracle's rate over the whole C on the host cores, and the gate
  checked on every output.

``--impl reference`` times the CPU oracle instead (there is no other implementation of this
path to run); under torchrun only rank 0 runs it.

With N > 1 ranks (torchrun), every rank runs the whole workload on its own GPU (replicas:
the path needs no exchange between GPUs); time is the max over ranks, value the sum.
"""

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "GEMM TFLOP/s (2MNK/t) at 4096³/8192³ bf16 on 1 GB300; % of dense tensor peak"
UNIT = "TFLOP/s"
# The one dense bf16/fp16 tensor peak "% of dense tensor peak" is quoted against: NVIDIA's GB300
# NVL72 datasheet gives 360 PFLOP/s FP16/BF16 for 72 GPUs with 2:4 sparsity, i.e. 2.5 PFLOP/s
# dense per GPU (152 SMs x 8192 flop/clk reach it at 2.0 GHz).
DENSE_PEAK_TFLOPS = 2500.0
DENSE_PEAK_SOURCE = ("NVIDIA GB300 NVL72 datasheet: FP16/BF16 tensor 360 PFLOP/s per 72 GPUs "
                     "with 2:4 sparsity = 2.5 PFLOP/s dense per GPU")
DENSE_FLOP_PER_CLK_PER_SM = 8192         # derived: one 128x256x16 MMA per 128 cycles
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
PROFILES = os.path.join(ROOT, "profiles")
KERNEL_NAMES = {1: "gemm_persistent_ws", 2: "gemm_pair_ws", 3: "gemm_pair_wide_ws"}   # by tg variant


def parse_args(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["tg", "reference"], default="tg")
    ap.add_argument("--workload", default="gemm_8192_bf16")
    ap.add_argument("--variant", choices=["auto", "single", "pair", "wide"], default="auto",
                    help="kernel variant (auto: the library's choice, as tg_gemm_persistent)")
    ap.add_argument("--e2e-steps", type=int, default=20,
                    help="end-to-end steps through the host-buffer entry point (0: leave out)")
    ap.add_argument("--cpu-seconds", type=float, default=12.0,
                    help="target CPU time of the oracle sample (cpu_baseline)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-per-config", action="store_true",
                    help="skip the per-workload records (every workload of the metric, each timed "
                         "with L2 flushed before every launch and checked against the oracle)")
    ap.add_argument("--sustained-seconds", type=float, default=3.0,
                    help="length of the sustained back-to-back run of the headline workload "
                         "(0: skip)")
    return ap.parse_args(argv)


# ----------------------------------------------------------------------------- ranks
def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def init_dist(world, backend):
    import torch.distributed as dist

    if world > 1 and not dist.is_initialized():
        dist.init_process_group(backend=backend)


def barrier():
    import torch.distributed as dist

    if dist.is_available() and dist.is_initialized():
        dist.barrier()


def max_over_ranks(x, device=None):
    """Max of a float over all ranks (the value itself when not distributed)."""
    import torch
    import torch.distributed as dist

    if not (dist.is_available() and dist.is_initialized()):
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device or "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ----------------------------------------------------------------------------- helpers
def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return json.load(f), "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


def blas_threads():
    """Threads numpy's BLAS uses (the oracle's matrix product), best effort."""
    try:
        from threadpoolctl import threadpool_info

        n = [i["num_threads"] for i in threadpool_info() if i.get("user_api") == "blas"]
        if n:
            return int(n[0])
    except Exception:
        pass
    import ctypes

    try:
        with open("/proc/self/maps") as f:
            libs = sorted({l.split()[-1] for l in f if "openblas" in l.lower() and ".so" in l})
        for path in libs:
            lib = ctypes.CDLL(path)
            for sym in ("scipy_openblas_get_num_threads64_", "openblas_get_num_threads64_",
                        "openblas_get_num_threads"):
                if hasattr(lib, sym):
                    return int(getattr(lib, sym)())
    except Exception:
        pass
    return len(os.sched_getaffinity(0))


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled every 20 ms in a child process (several
    samples fall inside even a ~10 ms timed region)."""

    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.out = None

    def start(self):
        self.out = tempfile.NamedTemporaryFile(mode="w+", suffix=".csv", delete=False)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=self.out, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.5)

    def stop(self, t0, t1):
        if self.proc is None:
            return None
        time.sleep(0.2)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.out.flush()
        self.out.seek(0)
        lines = self.out.read().strip().splitlines()
        self.out.close()
        os.unlink(self.out.name)
        return parse_clock_csv(lines, t0, t1)


CLOCK_REASONS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")


def parse_clock_csv(lines, t0, t1):
    """Summarise nvidia-smi rows (ClockSampler.FIELDS, csv, no header, no units) whose
    timestamp lies in [t0, t1] (host epoch seconds): median and max SM clock, and every
    throttle reason seen active."""
    rows = []
    for line in lines:
        parts = [p.strip() for p in line.split(",")]
        if len(parts) < 10:
            continue
        try:
            stamp, frac = (parts[0].split(".") + ["0"])[:2]
            ts = time.mktime(time.strptime(stamp, "%Y/%m/%d %H:%M:%S")) + float("0." + frac)
            rows.append((ts, float(parts[2]), float(parts[3]), parts[6:10]))
        except ValueError:
            continue
    inside = [r for r in rows if t0 - 0.05 <= r[0] <= t1 + 0.05]
    if not inside:
        return {"sm_mhz": None, "sm_max_mhz": max((r[2] for r in rows), default=None),
                "reasons": [], "samples": 0}
    reasons = sorted({CLOCK_REASONS[i] for r in inside for i, v in enumerate(r[3])
                      if v.lower() == "active"})
    return {"sm_mhz": statistics.median(r[1] for r in inside),
            "sm_max_mhz": max(r[2] for r in inside), "reasons": reasons,
            "samples": len(inside)}


def profile_traffic(kernel, workload):
    """DRAM bytes per launch of ``kernel`` on ``workload`` from its committed ncu summary
    (profiles/<kernel>_<size>_<dtype>.md), or None if there is none or the kernel's sources
    changed since that capture."""
    from persistent_warp_specialized_gb300 import _build

    tag = workload.replace("gemm_", "")
    try:
        text = open(os.path.join(PROFILES, f"{kernel}_{tag}.md")).read()
    except OSError:
        return None
    vals = {}
    for line in text.splitlines():
        line = line.strip().strip("-* ")
        if ":" in line:
            k, v = line.split(":", 1)
            vals[k.strip().strip("`")] = v.strip().strip("`")
    if vals.get("source_stamp") != _build.kernel_stamp(kernel):
        return None
    try:
        return float(vals["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


def oracle_slab(a_bits, b_bits, fmt, rows):
    from oracle import gemm as ogemm

    return ogemm.gemm_ref(a_bits[:rows], b_bits, fmt)


def timed_oracle_sample(run, M, seconds):
    """Run ``run(rows)`` (the oracle on rows [0, rows) of C) on growing samples until one takes
    at least half of ``seconds`` or covers all M rows; return (rows, seconds taken, result) of
    that last run.  Each oracle call has a fixed part (decoding all of B) that a small probe
    would wrongly count per row."""
    rows = min(M, 32)
    while True:
        t0 = time.perf_counter()
        out = run(rows)
        dt = time.perf_counter() - t0
        if dt >= 0.5 * seconds or rows >= M:
            return rows, dt, out
        rows = min(M, int(rows * min(8.0, max(2.0, seconds / max(dt, 1e-6)))))


def block_side(run, limit, seconds):
    """Side r of the square block C[:r, :r] that ``run(r)`` (the oracle on that block: r rows
    of A, r columns of B) computes in about ``seconds``; r doubles from 64 until one run takes
    at least half of that, so calibrating costs about one step."""
    r = min(limit, 64)
    while True:
        t0 = time.perf_counter()
        run(r)
        if time.perf_counter() - t0 >= 0.5 * seconds or r >= limit:
            return r
        r = min(limit, 2 * r)


# ----------------------------------------------------------------------------- reference arm
def run_reference(args):
    world, rank, _ = dist_env()
    if rank != 0:
        return 0
    from persistent_warp_specialized_gb300 import workloads as wl

    w = wl.WORKLOADS[args.workload]
    a, b = wl.workload_inputs(w)
    a_bits, b_bits = wl.bits(a), wl.bits(b)
    steps, warm = max(1, args.steps), max(0, args.warmup)
    per_step = max(0.05, min(2.0, 150.0 / (steps + warm)))

    def block(r):
        from oracle import gemm as ogemm

        return ogemm.gemm_ref(a_bits[:r], b_bits[:, :r], w.dtype)

    r = block_side(block, min(w.M, w.N), per_step)
    for _ in range(warm):
        block(r)
    t0 = time.perf_counter()
    for _ in range(steps):
        block(r)
    dt = time.perf_counter() - t0
    value = 2.0 * r * r * w.K * steps / dt / 1e12
    sample = (f"block C[:{r}, :{r}] of C = A.B for {w.name} ({r} x {r} outputs, K={w.K}) per "
              f"step: decode, binary64 product, round to {w.dtype}")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
        "n_gpus": world, "steps": steps, "warmup": warm, "ms_per_step": dt / steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": workload_config(w),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": blas_threads(), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def workload_config(w):
    return {"workload": w.name, "M": w.M, "N": w.N, "K": w.K, "in_out_dtype": w.dtype,
            "accumulate": "fp32", "inputs": f"{w.dist}, seed {w.seed}",
            "l2": "inputs larger than L2 (no flush)" if 2 * (w.M * w.K + w.K * w.N) > 129e6
                  else "inputs fit in L2 (no flush; warm L2)",
            "tile": "single 128x256 (block_K 64, 4 stages), pair 256x256 (block_K 128, 3 stages) or "
                    "wide pair 256x512 (block_K 64, 4 stages), as config.launch says; persistent: one "
                    "scheduler worker per SM (single) or SM pair (pair, wide pair)"}


# ----------------------------------------------------------------------------- GPU arm
def timed_region(step, steps, warm, dev, stream, world):
    """W untimed steps, then K steps between CUDA events on ``stream`` with a barrier and a
    device synchronisation on both sides and nvidia-smi clocks sampled meanwhile.  Returns
    (this rank's ms per step, max over ranks, clocks)."""
    import torch

    import persistent_warp_specialized_gb300 as tg

    for _ in range(warm):
        step()
    torch.cuda.synchronize(dev)
    tg.tg_device_status(stream)
    sampler = ClockSampler(dev.index)
    sampler.start()
    barrier()
    torch.cuda.synchronize(dev)
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    t0 = time.time()
    ev0.record(stream)
    for _ in range(steps):
        step()
    ev1.record(stream)
    torch.cuda.synchronize(dev)
    t1 = time.time()
    barrier()
    clocks = sampler.stop(t0, t1)
    ms_local = ev0.elapsed_time(ev1) / steps
    tg.tg_device_status(stream)
    return ms_local, max_over_ranks(ms_local, dev if world > 1 else None), clocks


def time_e2e(make_step, e_steps, dev, world, lanes=2):
    """ms per step of end-to-end steps issued round-robin on ``lanes`` streams, each with its
    own buffers (make_step(j, stream) -> step function), so one step's copies overlap another's
    kernels.  Every step copies its own inputs in and its result out."""
    import torch

    streams = [torch.cuda.Stream(dev) for _ in range(lanes)]
    steps = [make_step(j, streams[j]) for j in range(lanes)]
    for i in range(2 * lanes):
        steps[i % lanes]()
    torch.cuda.synchronize(dev)
    barrier()
    cur = torch.cuda.current_stream(dev)
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    start.record(cur)
    for st in streams:
        st.wait_event(start)
    for i in range(e_steps):
        steps[i % lanes]()
    for st in streams:
        done = torch.cuda.Event()
        done.record(st)
        cur.wait_event(done)
    end.record(cur)
    torch.cuda.synchronize(dev)
    return max_over_ranks(start.elapsed_time(end) / e_steps, dev if world > 1 else None)


L2_FLUSH_BYTES = 256 << 20     # written before every per-config launch: twice the 129 MB L2
PER_CONFIG_WARMUP = 50         # the pages' benchmark: do_bench(..., _n_warmup=50, _n_repeat=50)
PER_CONFIG_REPEAT = 50


def time_flushed(step, dev, flush, warmup=PER_CONFIG_WARMUP, repeat=PER_CONFIG_REPEAT):
    """Device milliseconds of ``step`` per launch: ``warmup`` untimed launches, then ``repeat``
    launches, each after a write of a buffer twice the size of L2 and between its own pair of
    CUDA events on the launching stream.  Returns (median, best, mean of the back-to-back
    launches of the warm-up's second half, which run with a warm L2)."""
    import torch

    stream = torch.cuda.current_stream(dev)
    half = max(1, warmup // 2)
    for _ in range(warmup - half):
        step()
    b0 = torch.cuda.Event(enable_timing=True)
    b1 = torch.cuda.Event(enable_timing=True)
    b0.record(stream)
    for _ in range(half):
        step()
    b1.record(stream)
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(repeat)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(repeat)]
    for i in range(repeat):
        flush.zero_()
        starts[i].record(stream)
        step()
        ends[i].record(stream)
    torch.cuda.synchronize(dev)
    ms = sorted(a.elapsed_time(b) for a, b in zip(starts, ends))
    return statistics.median(ms), ms[0], b0.elapsed_time(b1) / half


def oracle_full(w, a_cpu, b_cpu):
    """The oracle's whole C for ``w`` on the host cores: (bits, seconds)."""
    from oracle import gemm as ogemm
    from persistent_warp_specialized_gb300 import workloads as wl

    a_bits, b_bits = wl.bits(a_cpu), wl.bits(b_cpu)
    t0 = time.perf_counter()
    ref = ogemm.gemm_ref(a_bits, b_bits, w.dtype)
    return ref, time.perf_counter() - t0


def gate(got_bits, ref_bits, fmt):
    """(within |C - C_ref| <= 5e-3 + 1e-2 |C_ref| everywhere and finite, max |C - C_ref|)."""
    import numpy as np

    from oracle import formats

    got = formats.decode(got_bits, fmt)
    want = formats.decode(ref_bits, fmt)
    err = np.abs(got - want)
    ok = bool(np.isfinite(got).all() and (err <= 5e-3 + 1e-2 * np.abs(want)).all())
    return ok, float(err.max())


def per_config_records(dev, peaks, headline, cores):
    """One record per workload of the metric: device TFLOP/s (median and best of 50 launches
    after 50 warm-up, L2 flushed before each), the kernel the library picked, compulsory DRAM
    GB/s, the CPU oracle's TFLOP/s on the host cores over the whole C, and whether every
    output is within the gate.  ``headline``: (workload, a_cpu, b_cpu, a, b, c, ref, secs) of
    the workload already on the device and checked, so it is neither drawn nor computed twice."""
    import torch

    import persistent_warp_specialized_gb300 as tg
    from persistent_warp_specialized_gb300 import workloads as wl

    hbm = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    records = []
    for w in wl.WORKLOADS.values():
        if headline is not None and w.name == headline[0].name:
            _, a_cpu, b_cpu, a, b, c, ref, secs = headline
        else:
            a_cpu, b_cpu = wl.workload_inputs(w)
            a, b = a_cpu.to(dev), b_cpu.to(dev)
            c = torch.empty((w.M, w.N), dtype=wl.TORCH_DTYPES[w.dtype], device=dev)
            ref = secs = None

        def step(a=a, b=b, c=c, w=w):
            tg.tg_gemm_persistent(a, b, c, w.M, w.N, w.K, w.dtype)

        med, best, warm = time_flushed(step, dev, flush)
        tg.tg_device_status()
        if ref is None:
            ref, secs = oracle_full(w, a_cpu, b_cpu)
        ok, max_err = gate(wl.bits(c.cpu()), ref, w.dtype)
        launch = tg.tg_gemm_launch_shape(w.M, w.N, w.K)
        compulsory = 2 * (w.M * w.K + w.K * w.N + w.M * w.N)
        tflops = w.flops / (med * 1e-3) / 1e12
        records.append({
            "workload": w.name, "M": w.M, "N": w.N, "K": w.K, "dtype": w.dtype,
            "inputs": f"{w.dist}, seed {w.seed}",
            "kernel": KERNEL_NAMES[launch["variant"]], "launch": launch,
            "tflops": tflops, "tflops_best": w.flops / (best * 1e-3) / 1e12,
            "ms_median": med, "ms_best": best,
            "frac_of_dense_peak": tflops / DENSE_PEAK_TFLOPS,
            "tflops_back_to_back_warm_l2": w.flops / (warm * 1e-3) / 1e12,
            "compulsory_bytes": compulsory,
            "hbm_gbs": compulsory / (med * 1e-3) / 1e9,
            "hbm_frac": compulsory / (med * 1e-3) / 1e9 / hbm,
            "cpu_oracle_tflops": w.flops / secs / 1e12, "cpu_oracle_s": secs,
            "cpu_oracle_cores": cores,
            "within_tolerance": ok, "max_abs_err": max_err,
            "timing": f"{PER_CONFIG_WARMUP} warm-up + {PER_CONFIG_REPEAT} timed launches, each "
                      f"after a {L2_FLUSH_BYTES >> 20} MiB write (L2 flushed), CUDA events per "
                      f"launch; median",
        })
        del a, b, c
    del flush
    torch.cuda.empty_cache()
    return records


def mx_per_config_record(dev, peaks, cores, rows=1024):
    """The block-scaled MXFP8 workload at 8192^3: the GEMM kernel alone and the whole step
    (both scale packs + the GEMM), each timed like the dense records, plus the oracle on
    ``rows`` rows of C (its time scaled to TFLOP/s) and the gate on those rows."""
    import torch

    import persistent_warp_specialized_gb300 as tg
    from oracle import mx
    from persistent_warp_specialized_gb300 import workloads as wl

    M, N, K, seed = wl.MX_WORKLOADS["mxfp8_8192"]
    host = wl.make_mx_inputs(M, N, K, seed)
    a, sa, b, sb = (t.to(dev) for t in host)
    c = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    sa_p = torch.empty(tg.tg_mxfp8_scale_bytes(M, K), dtype=torch.uint8, device=dev)
    sb_p = torch.empty(tg.tg_mxfp8_scale_bytes(N, K), dtype=torch.uint8, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    flops = 2.0 * M * N * K

    def gemm():
        tg.tg_gemm_mxfp8(a, sa_p, b, sb_p, c, M, N, K, "bf16")

    def step():
        tg.tg_mxfp8_pack_scales(sa, sa_p, M, K)
        tg.tg_mxfp8_pack_scales(sb, sb_p, N, K)
        gemm()

    step_med, _, _ = time_flushed(step, dev, flush)
    med, best, warm = time_flushed(gemm, dev, flush)
    tg.tg_device_status()
    an, san, bn, sbn = (t.numpy() for t in host)
    t0 = time.perf_counter()
    ref = mx.gemm_mxfp8_ref(an[:rows], san[:rows], bn, sbn, "bf16")
    secs = time.perf_counter() - t0
    ok, max_err = gate(wl.bits(c[:rows].cpu()), ref, "bf16")
    launch = tg.tg_gemm_launch_shape(M, N, K, mxfp8=True)
    tflops = flops / (med * 1e-3) / 1e12
    compulsory = M * K + N * K + (M * K + N * K) // 32 + 2 * M * N   # GEMM: A, B, scales, C
    rec = {
        "workload": "mxfp8_8192", "M": M, "N": N, "K": K, "dtype": "e4m3 (e8m0 scales per 32), bf16 out",
        "inputs": f"MX-quantized N(0,1) / N(0,1/K) draws, seed {seed}",
        "kernel": "gemm_mxfp8_pair_ws", "launch": launch,
        "tflops": tflops, "tflops_best": flops / (best * 1e-3) / 1e12, "ms_median": med,
        "tflops_step_with_packs": flops / (step_med * 1e-3) / 1e12,
        "frac_of_dense_peak": tflops / (2 * DENSE_PEAK_TFLOPS),
        "tflops_back_to_back_warm_l2": flops / (warm * 1e-3) / 1e12,
        "compulsory_bytes": compulsory, "hbm_gbs": compulsory / (med * 1e-3) / 1e9,
        "hbm_frac": compulsory / (med * 1e-3) / 1e9 / float(peaks.get("hbm_gbs", 6800.0)),
        "cpu_oracle_tflops": 2.0 * rows * N * K / secs / 1e12, "cpu_oracle_s": secs,
        "cpu_oracle_cores": cores, "cpu_oracle_sample": f"rows [0, {rows}) of C",
        "within_tolerance": ok, "max_abs_err": max_err, "checked_rows": rows,
        "timing": "as the dense records; tflops is the GEMM kernel alone",
    }
    del a, sa, b, sb, c, sa_p, sb_p, flush
    torch.cuda.empty_cache()
    return rec


def sustained_record(step, flops, ms_estimate, seconds, dev, stream, world):
    """Back-to-back launches of the headline step for about ``seconds`` with clocks sampled:
    what the kernel holds once the GPU sits at its power limit."""
    n = max(10, int(seconds / max(ms_estimate * 1e-3, 1e-6)))
    ms_local, ms, clocks = timed_region(step, n, 3, dev, stream, world)
    tflops = flops / (ms * 1e-3) / 1e12
    return {"launches": n, "seconds": n * ms * 1e-3, "ms_per_launch": ms, "tflops": tflops,
            "frac_of_dense_peak": tflops / DENSE_PEAK_TFLOPS, "clocks": clocks}


def run_tg(args):
    import torch

    world, rank, local = dist_env()
    if world > 1:
        torch.cuda.set_device(local)
        init_dist(world, "nccl")
    else:
        torch.cuda.set_device(0)
    dev = torch.device("cuda", torch.cuda.current_device())

    import persistent_warp_specialized_gb300 as tg
    from persistent_warp_specialized_gb300 import _build
    from persistent_warp_specialized_gb300 import workloads as wl

    _build.build()
    tg.load_library()
    w = {**wl.WORKLOADS, **wl.PROFILE_WORKLOADS}[args.workload]
    a_cpu, b_cpu = wl.workload_inputs(w)
    a = a_cpu.to(dev)
    b = b_cpu.to(dev)
    c = torch.empty((w.M, w.N), dtype=wl.TORCH_DTYPES[w.dtype], device=dev)
    stream = torch.cuda.current_stream(dev)
    sms = torch.cuda.get_device_properties(dev).multi_processor_count

    if args.variant == "auto":
        def step():
            tg.tg_gemm_persistent(a, b, c, w.M, w.N, w.K, w.dtype, stream)
    else:
        def step():
            tg.tg_gemm_persistent_ex(a, b, c, w.M, w.N, w.K, w.dtype, stream, args.variant)

    steps, warm = max(1, args.steps), max(3, args.warmup)
    ms_local, ms, clocks = timed_region(step, steps, warm, dev, stream, world)
    value = world * w.flops / (ms * 1e-3) / 1e12

    # end to end through the host-buffer entry point: H2D A, B + kernel + D2H C per step
    a_h, b_h = a_cpu.pin_memory(), b_cpu.pin_memory()

    def make_e2e_step(j, st):
        c_h = torch.empty((w.M, w.N), dtype=wl.TORCH_DTYPES[w.dtype]).pin_memory()
        a2, b2, c2 = torch.empty_like(a), torch.empty_like(b), torch.empty_like(c)

        def e2e_step():
            tg.tg_gemm_persistent_host(a_h, b_h, c_h, a2, b2, c2, w.M, w.N, w.K, w.dtype, st)
        return e2e_step

    e2e = None                       # --e2e-steps 0: profiling runs leave the e2e leg out
    if args.e2e_steps > 0:
        e_ms = time_e2e(make_e2e_step, args.e2e_steps, dev, world)
        tg.tg_device_status(stream)
        h2d = 2 * (w.M * w.K + w.K * w.N)
        d2h = 2 * w.M * w.N
        e2e = {"value": world * w.flops / (e_ms * 1e-3) / 1e12, "unit": UNIT,
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e_ms,
               "streams": 2, "api": "tg_gemm_persistent_host"}

    launch = tg.tg_gemm_launch_shape(w.M, w.N, w.K, args.variant)
    kernel = KERNEL_NAMES[launch["variant"]]
    peaks, peak_src = measured_peaks()
    achieved = w.flops / (ms_local * 1e-3) / 1e12
    peak = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    if w.dtype == "f16":
        peak_note = "bf16 peak x 1 (fp16 and bf16 share the dense tensor rate)"
    else:
        peak_note = "bf16 burst peak"
    roofline = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": UNIT,
                "frac": achieved / peak, "kernel": kernel,
                "traffic": profile_traffic(kernel, w.name),
                "peak_source": f"{peak_src} ({peak_note}, cuBLAS torch.matmul)",
                "frac_of_sustained": achieved / float(peaks.get("bf16_tflops_sustained", peak)),
                "frac_of_dense_peak": achieved / DENSE_PEAK_TFLOPS,
                "dense_peak_tflops": DENSE_PEAK_TFLOPS}
    if clocks and clocks.get("sm_mhz"):
        clk_peak = sms * DENSE_FLOP_PER_CLK_PER_SM * clocks["sm_mhz"] * 1e6 / 1e12
        roofline["frac_of_clock_peak"] = achieved / clk_peak
        roofline["clock_peak_tflops"] = clk_peak

    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": steps,
        "warmup": warm, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": w.dtype, "data": "synthetic (seeded; see config.inputs)",
        "config": dict(workload_config(w), sms=sms,
                       launch=launch),
        "gpu_launches": steps, "e2e": e2e, "roofline": roofline, "clocks": clocks,
        "pct_of_dense_peak": 100.0 * value / world / DENSE_PEAK_TFLOPS,
        "dense_peak": {"tflops": DENSE_PEAK_TFLOPS, "source": DENSE_PEAK_SOURCE},
    }

    headline = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        a_bits, b_bits = wl.bits(a_cpu), wl.bits(b_cpu)
        rows, dt, ref = timed_oracle_sample(lambda r: oracle_slab(a_bits, b_bits, w.dtype, r),
                                            w.M, args.cpu_seconds)
        ok, max_err = gate(wl.bits(c[:rows].cpu()), ref, w.dtype)
        cores = blas_threads()
        line["cpu_baseline"] = {
            "value": 2.0 * rows * w.N * w.K / dt / 1e12, "unit": UNIT, "cores": cores,
            "kind": "oracle",
            "sample": f"rows [0, {rows}) of C ({rows} x {w.N} outputs, K={w.K}): decode, "
                      f"binary64 product (numpy/OpenBLAS), round to {w.dtype}; {dt:.1f} s"}
        line["parity_sample"] = {"rows": rows, "cols": w.N, "within_tolerance": ok,
                                 "max_abs_err": max_err}
        if rows == w.M and args.variant == "auto":
            headline = (w, a_cpu, b_cpu, a, b, c, ref, dt)

    if args.sustained_seconds > 0 and w.name == "gemm_8192_bf16":
        line["sustained"] = sustained_record(step, w.flops, ms, args.sustained_seconds, dev,
                                             stream, world)
        line["sustained"]["tflops"] *= world

    if rank == 0 and world == 1 and not args.no_per_config and not args.no_cpu_baseline:
        cores = blas_threads()
        del a_h, b_h
        line["per_config"] = per_config_records(dev, peaks, headline, cores)
        headline = None
        del a, b, c
        torch.cuda.empty_cache()
        line["per_config"].append(mx_per_config_record(dev, peaks, cores))
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()
    return 0


# ----------------------------------------------------------------------------- MXFP8 workload
MX_METRIC = "block-scaled MXFP8 GEMM TFLOP/s (2MNK/t) at 8192³ on 1 GB300; % of dense fp8 tensor peak"


def mx_oracle_slab(a, sa, b, sb, rows):
    from oracle import mx

    return mx.gemm_mxfp8_ref(a[:rows], sa[:rows], b, sb, "bf16")


def mx_config(name, M, N, K, seed):
    return {"workload": name, "M": M, "N": N, "K": K, "in_dtype": "e4m3",
            "scale": "e8m0 per 32 K-elements of each A row and B column", "out_dtype": "bf16",
            "accumulate": "fp32", "inputs": f"MX-quantized N(0,1) / N(0,1/K) draws, seed {seed}",
            "l2": "inputs larger than L2 (no flush)",
            "tile": "CTA pair: 256 x 256 x 128 bytes, 6 stages (single CTA: 128 x 256, 4 stages); "
                    "persistent",
            "step": "pack both operands' scales (2 launches) + the GEMM (1 launch)"}


def run_reference_mx(args):
    world, rank, _ = dist_env()
    if rank != 0:
        return 0
    from persistent_warp_specialized_gb300 import workloads as wl

    M, N, K, seed = wl.MX_WORKLOADS[args.workload]
    a, sa, b, sb = (t.numpy() for t in wl.make_mx_inputs(M, N, K, seed))
    steps, warm = max(1, args.steps), max(0, args.warmup)
    per_step = max(0.05, min(2.0, 150.0 / (steps + warm)))

    def block(r):
        from oracle import mx

        return mx.gemm_mxfp8_ref(a[:r], sa[:r], b[:r], sb[:r], "bf16")

    r = block_side(block, min(M, N), per_step)
    for _ in range(warm):
        block(r)
    t0 = time.perf_counter()
    for _ in range(steps):
        block(r)
    dt = time.perf_counter() - t0
    value = 2.0 * r * r * K * steps / dt / 1e12
    sample = (f"block C[:{r}, :{r}] of the MXFP8 product ({r} x {r} outputs, K={K}) per step: "
              f"decode, scale, binary64 product, round to bf16")
    print(json.dumps({
        "impl": "reference", "metric": MX_METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": steps, "warmup": warm, "ms_per_step": dt / steps * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": mx_config(args.workload, M, N, K, seed),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": blas_threads(), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)
    return 0


def run_tg_mx(args):
    import torch

    world, rank, local = dist_env()
    if world > 1:
        torch.cuda.set_device(local)
        init_dist(world, "nccl")
    else:
        torch.cuda.set_device(0)
    dev = torch.device("cuda", torch.cuda.current_device())

    import persistent_warp_specialized_gb300 as tg
    from persistent_warp_specialized_gb300 import _build
    from persistent_warp_specialized_gb300 import workloads as wl

    _build.build()
    tg.load_library()
    M, N, K, seed = wl.MX_WORKLOADS[args.workload]
    host = wl.make_mx_inputs(M, N, K, seed)
    a, sa, b, sb = (t.to(dev) for t in host)
    c = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    sa_p = torch.empty(tg.tg_mxfp8_scale_bytes(M, K), dtype=torch.uint8, device=dev)
    sb_p = torch.empty(tg.tg_mxfp8_scale_bytes(N, K), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    flops = 2.0 * M * N * K

    # a step: both operands' row-major scales packed, then the GEMM (three launches)
    def gemm_only():
        tg.tg_gemm_mxfp8_ex(a, sa_p, b, sb_p, c, M, N, K, "bf16", stream, args.variant)

    def step():
        tg.tg_mxfp8_pack_scales(sa, sa_p, M, K, stream)
        tg.tg_mxfp8_pack_scales(sb, sb_p, N, K, stream)
        gemm_only()

    launch = tg.tg_gemm_launch_shape(M, N, K, args.variant, mxfp8=True)   # the GEMM's launch
    kernel = "gemm_mxfp8_pair_ws" if launch["variant"] == tg.TG_VARIANT_PAIR else "gemm_mxfp8_ws"

    steps, warm = max(1, args.steps), max(3, args.warmup)
    ms_local, ms, clocks = timed_region(step, steps, warm, dev, stream, world)
    value = world * flops / (ms * 1e-3) / 1e12
    gemm_ms, _, _ = timed_region(gemm_only, steps, 3, dev, stream, world)

    # end to end: pinned host inputs copied in, scales packed, the GEMM, C copied out
    pinned = [t.pin_memory() for t in host]

    def make_e2e_step(j, st):
        dev2 = [torch.empty_like(t, device=dev) for t in host]
        sa2, sb2, c2 = torch.empty_like(sa_p), torch.empty_like(sb_p), torch.empty_like(c)
        c_h = torch.empty((M, N), dtype=torch.bfloat16).pin_memory()

        def e2e_step():
            with torch.cuda.stream(st):
                for d, h in zip(dev2, pinned):
                    d.copy_(h, non_blocking=True)
            tg.tg_mxfp8_pack_scales(dev2[1], sa2, M, K, st)
            tg.tg_mxfp8_pack_scales(dev2[3], sb2, N, K, st)
            tg.tg_gemm_mxfp8_ex(dev2[0], sa2, dev2[2], sb2, c2, M, N, K, "bf16", st, args.variant)
            with torch.cuda.stream(st):
                c_h.copy_(c2, non_blocking=True)
        return e2e_step

    e_ms = time_e2e(make_e2e_step, max(1, args.e2e_steps), dev, world)
    tg.tg_device_status(stream)
    e2e = {"value": world * flops / (e_ms * 1e-3) / 1e12, "unit": UNIT,
           "h2d_bytes_per_step": sum(t.numel() for t in host), "d2h_bytes_per_step": 2 * M * N,
           "ms_per_step": e_ms, "streams": 2}

    peaks, peak_src = measured_peaks()
    achieved = flops / (gemm_ms * 1e-3) / 1e12    # the GEMM kernel alone
    peak = 2.0 * float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    roofline = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": UNIT,
                "frac": achieved / peak, "kernel": kernel,
                "kernel_ms": gemm_ms,
                "traffic": profile_traffic(kernel, f"{M}_mxfp8"),
                "peak_source": f"{peak_src}: bf16 burst peak x 2 (the nominal dense fp8 / bf16 "
                               f"ratio, 2)",
                "frac_of_dense_peak": achieved / (2 * DENSE_PEAK_TFLOPS),
                "dense_peak_tflops": 2 * DENSE_PEAK_TFLOPS}
    line = {
        "metric": MX_METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": steps,
        "warmup": warm, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "e4m3", "data": "synthetic (seeded; see config.inputs)",
        "config": dict(mx_config(args.workload, M, N, K, seed), sms=sms, launch=launch),
        "gpu_launches": 3 * steps, "e2e": e2e, "roofline": roofline, "clocks": clocks,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        import numpy as np

        from oracle import formats

        an, san, bn, sbn = (t.numpy() for t in host)
        rows, dt, ref = timed_oracle_sample(lambda r: mx_oracle_slab(an, san, bn, sbn, r), M,
                                            args.cpu_seconds)
        got = formats.decode(wl.bits(c[:rows].cpu()), "bf16")
        want = formats.decode(ref, "bf16")
        err = np.abs(got - want)
        ok = bool(np.isfinite(got).all() and (err <= 5e-3 + 1e-2 * np.abs(want)).all())
        line["cpu_baseline"] = {
            "value": 2.0 * rows * N * K / dt / 1e12, "unit": UNIT, "cores": blas_threads(),
            "kind": "oracle",
            "sample": f"rows [0, {rows}) of C ({rows} x {N} outputs, K={K}): decode, scale, "
                      f"binary64 product (numpy/OpenBLAS), round to bf16; {dt:.1f} s"}
        line["parity_sample"] = {"rows": rows, "cols": N, "within_tolerance": ok,
                                 "max_abs_err": float(err.max())}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()
    return 0


def main(argv=None):
    args = parse_args(argv)
    from persistent_warp_specialized_gb300 import workloads as wl

    if args.workload in wl.MX_WORKLOADS:
        if args.variant == "wide":
            print("--variant wide is a dense-GEMM kernel; the MXFP8 GEMM has single and pair",
                  file=sys.stderr)
            return 2
        return run_reference_mx(args) if args.impl == "reference" else run_tg_mx(args)
    if args.impl == "reference":
        return run_reference(args)
    return run_tg(args)


if __name__ == "__main__":
    sys.exit(main())
