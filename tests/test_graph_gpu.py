"""GPU: GEMMs captured in a CUDA graph and replayed.

A launch-bound loop of GEMMs can be captured once and replayed (torch.cuda.graph captures the
calls made on its stream).  The library's entry points only query pointer attributes and
launch kernels (with programmatic dependent launch) on the caller's stream, so they can be
captured.  Here a chain of dense GEMMs (each reading the previous one's output, one per dense
kernel) and an MXFP8 GEMM with its two scale packs are captured, the inputs are rewritten in
place between replays, and every replay must give the oracle's product of the current inputs
bit for bit.
"""

import numpy as np
import pytest
import torch

import persistent_warp_specialized_gb300 as tg
from persistent_warp_specialized_gb300 import workloads as wl
from oracle import mx

from gpu_helpers import ensure_library, oracle_bits

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ensure_library()


def test_captured_gemms_follow_their_inputs_on_every_replay():
    M = N = K = 512
    dt = torch.bfloat16
    eye = torch.eye(K, dtype=dt, device="cuda")
    a = torch.empty((M, K), dtype=dt, device="cuda")
    b = torch.empty((K, N), dtype=dt, device="cuda")
    c1, c2, c3 = (torch.empty((M, N), dtype=dt, device="cuda") for _ in range(3))
    Mm, Nm, Km = 256, 512, 256
    am = torch.empty((Mm, Km), dtype=torch.uint8, device="cuda")
    bm = torch.empty((Nm, Km), dtype=torch.uint8, device="cuda")
    sam = torch.empty((Mm, Km // 32), dtype=torch.uint8, device="cuda")
    sbm = torch.empty((Nm, Km // 32), dtype=torch.uint8, device="cuda")
    pa = torch.empty(tg.tg_mxfp8_scale_bytes(Mm, Km), dtype=torch.uint8, device="cuda")
    pb = torch.empty(tg.tg_mxfp8_scale_bytes(Nm, Km), dtype=torch.uint8, device="cuda")
    cm = torch.empty((Mm, Nm), dtype=dt, device="cuda")

    def step(s=None):
        tg.tg_gemm_persistent_ex(a, b, c1, M, N, K, "bf16", stream=s, variant="single")
        tg.tg_gemm_persistent_ex(c1, eye, c2, M, N, N, "bf16", stream=s, variant="pair")
        tg.tg_gemm_persistent_ex(c2, eye, c3, M, N, N, "bf16", stream=s, variant="wide")
        tg.tg_mxfp8_pack_scales(sam, pa, Mm, Km, s)
        tg.tg_mxfp8_pack_scales(sbm, pb, Nm, Km, s)
        tg.tg_gemm_mxfp8(am, pa, bm, pb, cm, Mm, Nm, Km, "bf16", stream=s)

    def load(seed):
        a_h, b_h = wl.small_int_inputs(M, N, K, "bf16", lo=-1, hi=1, seed=seed)
        a.copy_(a_h)
        b.copy_(b_h)
        m = wl.mx_int_inputs(Mm, Nm, Km, seed=seed)
        for dst, src in zip((am, sam, bm, sbm), m):
            dst.copy_(src)
        return a_h, b_h, m

    # warm-up outside the capture (the library sets up the device on its first call)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        load(0)
        step(side)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()

    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()                          # the capture stream is the current stream
    for seed in (1, 2, 3):
        a_h, b_h, (am_h, sam_h, bm_h, sbm_h) = load(seed)
        for t in (c1, c2, c3, cm):
            t.view(torch.int16).fill_(-1)
        graph.replay()
        torch.cuda.synchronize()
        assert tg.tg_device_status() == 0
        want = oracle_bits(a_h, b_h, "bf16")
        for t in (c1, c2, c3):
            assert np.array_equal(wl.bits(t.cpu()), want), seed
        want_mx = mx.gemm_mxfp8_ref(am_h.numpy(), sam_h.numpy(), bm_h.numpy(), sbm_h.numpy(),
                                    "bf16")
        assert np.array_equal(wl.bits(cm.cpu()), want_mx), seed
