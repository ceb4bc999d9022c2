"""GPU parity of the stream-K tail (tg_gemm_persistent_ws): the last partial wave of the CTA-pair
kernels split along K, partial sums exchanged through the workspace.  Integer inputs must be
bit-exact (every fp32 partial sum is exact, so any split gives the same bits: a lost, doubled
or misplaced k-range shows), the debug trace must follow the schedule oracle's stream-K
enumeration, and the workspace rules and the watchdog must hold."""

import numpy as np
import pytest
import torch

import persistent_warp_specialized_gb300 as tg
from persistent_warp_specialized_gb300 import workloads as wl
from oracle import schedule

from gpu_helpers import assert_within_tolerance, ensure_library, nan_filled, oracle_bits

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ensure_library()


def workspace_for(M, N, K, variant, streamk=True):
    n = tg.tg_gemm_workspace_bytes(M, N, K, variant, streamk=streamk)
    return torch.empty(max(n, 256), dtype=torch.uint8, device="cuda")


def run_ws(a_cpu, b_cpu, dtype, variant, streamk=True, ws=None):
    M, K = a_cpu.shape
    N = b_cpu.shape[1]
    c = nan_filled(M, N, dtype)
    if ws is None:
        ws = workspace_for(M, N, K, variant, streamk)
    tg.tg_gemm_persistent_ws(a_cpu.cuda(), b_cpu.cuda(), c, M, N, K, dtype, ws, variant=variant,
                             streamk=streamk)
    torch.cuda.synchronize()
    assert tg.tg_device_status() == 0
    return wl.bits(c.cpu())


# (M, N, K): several tail sizes against the 76-or-so resident pairs, ragged M / N / K, tails
# with more workers than k-blocks (empty ranges, many contributors per tile) and a single k-block
SHAPES = {
    "pair": [(1024, 6400, 512), (512, 1024, 512), (1000, 6000, 504), (256, 256, 64),
             (768, 768, 512), (2304, 2304, 384)],
    "wide": [(1024, 12800, 512), (512, 2048, 512), (1000, 6000, 504), (256, 512, 64),
             (768, 1536, 512), (2304, 4608, 256)],
}
CASES = [(v, s) for v, shapes in SHAPES.items() for s in shapes]


@pytest.mark.parametrize("variant,shape", CASES)
def test_integer_inputs_are_bit_exact(variant, shape):
    # entries in [-2, 2], K <= 512: |C| <= 2048, exact in fp16 whatever the split
    M, N, K = shape
    launch = tg.tg_gemm_launch_shape(M, N, K, variant, workspace=True, streamk=True)
    assert launch["sk_tiles"] == (launch["m_tiles"] * launch["n_tiles"]) % launch["workers"]
    a, b = wl.small_int_inputs(M, N, K, "f16", seed=M + N + K)
    assert np.array_equal(run_ws(a, b, "f16", variant), oracle_bits(a, b, "f16"))


@pytest.mark.parametrize("variant,shape", [("pair", (1024, 6400, 4096)), ("wide", (1024, 12800, 2048)),
                                           ("pair", (1000, 6000, 1000)), ("wide", (2000, 4000, 3000))])
def test_normal_inputs_within_tolerance(variant, shape):
    M, N, K = shape
    a, b = wl.make_inputs(M, N, K, "bf16", "normal", seed=K)
    assert_within_tolerance(run_ws(a, b, "bf16", variant), oracle_bits(a, b, "bf16"), "bf16",
                            f"{shape} {variant}")


@pytest.mark.parametrize("variant,shape", CASES[:3] + CASES[6:9])
def test_kernel_followed_the_stream_k_schedule(variant, shape):
    M, N, K = shape
    launch = tg.tg_gemm_launch_shape(M, N, K, variant, workspace=True, streamk=True)
    workers, units = launch["workers"], launch["units"]
    block_k = 128 if variant == "pair" else 64
    want = schedule.enumerate_units_streamk(launch["m_tiles"], launch["n_tiles"], workers,
                                            launch["group"], -(-K // block_k),
                                            bool(launch["column_major"]))
    assert units == launch["split_from"] + 2 * workers
    a, b = wl.make_inputs(M, N, K, "bf16", "uniform", seed=M)
    c = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    trace = torch.full((units, 5), -7, dtype=torch.int32, device="cuda")
    ws = workspace_for(M, N, K, variant)
    assert tg.tg_gemm_persistent_debug(a.cuda(), b.cuda(), c, M, N, K, "bf16", variant=variant,
                                       trace=trace, workspace=ws, streamk=True) == 0
    got = trace.cpu().numpy()
    seen = set()
    for (worker, w, bx, by, part, k_lo, k_hi, unit) in want:
        assert tuple(int(x) for x in got[unit]) == (worker, w, bx, by, part), unit
        seen.add(unit)
    assert all(tuple(got[u]) == (-7,) * 5 for u in range(units) if u not in seen)
    assert_within_tolerance(wl.bits(c.cpu()), oracle_bits(a, b, "bf16"), "bf16", "debug build")


def test_the_tail_is_taken_only_when_asked():
    # 4096^3: 256 pair tiles over the resident pairs leave a partial wave; with a workspace but
    # no TG_SCHEDULE_STREAMK the library keeps the half-width units (and needs no workspace)
    M = N = K = 4096
    plain = tg.tg_gemm_launch_shape(M, N, K, workspace=True)
    assert plain["sk_tiles"] == 0 and plain["workspace_bytes"] == 0
    assert tg.tg_gemm_workspace_bytes(M, N, K) == 0
    forced = tg.tg_gemm_launch_shape(M, N, K, "pair", workspace=True, streamk=True)
    tiles = forced["m_tiles"] * forced["n_tiles"]
    assert forced["sk_tiles"] == tiles % forced["workers"]
    assert forced["workspace_bytes"] == tg.tg_gemm_workspace_bytes(M, N, K, "pair", streamk=True)
    # full size, forced: sampled rows against the oracle
    a, b = wl.make_inputs(M, N, K, "bf16", "normal", seed=3)
    c = nan_filled(M, N, "bf16")
    ws = workspace_for(M, N, K, "pair")
    tg.tg_gemm_persistent_ws(a.cuda(), b.cuda(), c, M, N, K, "bf16", ws, variant="pair",
                             streamk=True)
    torch.cuda.synchronize()
    assert tg.tg_device_status() == 0
    rows = np.random.default_rng(0).choice(M, 64, replace=False)
    assert_within_tolerance(wl.bits(c.cpu())[rows], oracle_bits(a[rows], b, "bf16"), "bf16",
                            "4096^3 rows")


def test_one_workspace_across_launches():
    # a later launch must not take an earlier launch's flags for its own
    M, N, K = 1024, 6400, 512
    ws = workspace_for(M, N, K, "pair")
    for seed in range(3):
        a, b = wl.small_int_inputs(M, N, K, "f16", seed=seed)
        assert np.array_equal(run_ws(a, b, "f16", "pair", ws=ws), oracle_bits(a, b, "f16"))


def test_workspace_rules():
    M, N, K = 1024, 6400, 512
    a = torch.zeros((M, K), dtype=torch.float16, device="cuda")
    b = torch.zeros((K, N), dtype=torch.float16, device="cuda")
    c = torch.empty((M, N), dtype=torch.float16, device="cuda")
    need = tg.tg_gemm_workspace_bytes(M, N, K, "pair", streamk=True)
    assert need > 0
    ws = torch.empty(need + 512, dtype=torch.uint8, device="cuda")
    with pytest.raises(tg.TgError) as e:      # forced, no workspace
        tg.tg_gemm_persistent_ws(a, b, c, M, N, K, "f16", None, variant="pair", streamk=True)
    assert e.value.code == tg.TG_ERR_ARG
    with pytest.raises(tg.TgError) as e:      # forced, too small
        tg.tg_gemm_persistent_ws(a, b, c, M, N, K, "f16", ws, variant="pair", streamk=True,
                                 workspace_bytes=need - 1)
    assert e.value.code == tg.TG_ERR_ARG
    with pytest.raises(tg.TgError) as e:      # not 256-byte aligned
        tg.tg_gemm_persistent_ws(a, b, c, M, N, K, "f16", ws.data_ptr() + 16, variant="pair",
                                 streamk=True, workspace_bytes=need)
    assert e.value.code == tg.TG_ERR_ALIGN
    with pytest.raises(tg.TgError) as e:      # the flag without a workspace entry point
        tg.tg_gemm_persistent_ex(a, b, c, M, N, K, "f16", variant=tg.TG_VARIANT_PAIR | tg.TG_SCHEDULE_STREAMK)
    assert e.value.code == tg.TG_ERR_ARG
    # without the flag the workspace is not used (none, or any size)
    tg.tg_gemm_persistent_ws(a, b, c, M, N, K, "f16", None, variant="pair")
    tg.tg_gemm_persistent_ws(a, b, c, M, N, K, "f16", ws, variant="pair", workspace_bytes=16)
    torch.cuda.synchronize()
    assert tg.tg_device_status() == 0
    assert int(torch.count_nonzero(c)) == 0


@pytest.mark.parametrize("variant,cta", [("pair", 0), ("pair", 1), ("wide", 1)])
def test_watchdog_with_the_tail(variant, cta):
    # a skipped fill stops the pairs; owners waiting for contributions must stop too
    M, N, K = 1024, 6400 if variant == "pair" else 12800, 512
    a, b = wl.small_int_inputs(M, N, K, "f16", seed=1)
    a_d, b_d = a.cuda(), b.cuda()
    c = torch.empty((M, N), dtype=torch.float16, device="cuda")
    ws = workspace_for(M, N, K, variant)
    with pytest.raises(tg.TgError) as e:
        tg.tg_gemm_persistent_debug(a_d, b_d, c, M, N, K, "f16", variant=variant,
                                    watchdog_ns=20_000_000, inject_skip_phase=(cta << 32) + 1,
                                    workspace=ws, streamk=True)
    assert e.value.code == tg.TG_ERR_TIMEOUT
    assert tg.tg_device_status() == 0
    assert np.array_equal(run_ws(a, b, "f16", variant, ws=ws), oracle_bits(a, b, "f16"))
