"""GPU: launches queued back to back on one stream keep the stream's order of memory effects.

Every GEMM and scale-pack launch may begin while the previous kernel in the stream is still
finishing (programmatic dependent launch); each kernel waits for that kernel before its first
global memory access.  These chains are queued without any synchronisation between launches
and fail if a kernel read an operand before the previous launch had finished writing it (read
after write), or wrote its output while the previous launch still read that buffer (write after
read).
"""

import numpy as np
import pytest
import torch

import persistent_warp_specialized_gb300 as tg
from persistent_warp_specialized_gb300 import workloads as wl
from oracle import mx

from gpu_helpers import VARIANTS, assert_within_tolerance, ensure_library, oracle_bits

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ensure_library()


@pytest.mark.parametrize("variant", VARIANTS)
def test_each_launch_reads_the_previous_launch_output(variant):
    M = N = K = 4096
    a, b = wl.make_inputs(M, N, K, "bf16", dist="normal", seed=21)
    eye = torch.eye(N, dtype=torch.bfloat16).cuda()
    a_dev, b_dev = a.cuda(), b.cuda()
    outs = [torch.empty((M, N), dtype=torch.bfloat16, device="cuda") for _ in range(6)]
    torch.cuda.synchronize()
    # C_0 = A B, then C_i = C_(i-1) I: each launch reads what the one before it wrote
    tg.tg_gemm_persistent_ex(a_dev, b_dev, outs[0], M, N, K, "bf16", variant=variant)
    for i in range(1, len(outs)):
        tg.tg_gemm_persistent_ex(outs[i - 1], eye, outs[i], M, N, N, "bf16", variant=variant)
    torch.cuda.synchronize()
    assert tg.tg_device_status() == 0
    first = wl.bits(outs[0].cpu())
    assert_within_tolerance(first, oracle_bits(a, b, "bf16"), "bf16", f"first GEMM ({variant})")
    for i in range(1, len(outs)):
        # one non-zero product per output: C_(i-1) I is C_(i-1) exactly
        assert np.array_equal(wl.bits(outs[i].cpu()), first), f"launch {i} ({variant})"


@pytest.mark.parametrize("variant", VARIANTS)
def test_a_launch_does_not_overwrite_what_the_previous_launch_reads(variant):
    M = N = K = 4096
    a, b = wl.make_inputs(M, N, K, "bf16", dist="normal", seed=22)
    x, _ = wl.make_inputs(M, K, K, "bf16", dist="normal", seed=23)
    eye = torch.eye(K, dtype=torch.bfloat16).cuda()
    a_dev, b_dev, x_dev = a.cuda(), b.cuda(), x.cuda()
    c = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    torch.cuda.synchronize()
    tg.tg_gemm_persistent_ex(a_dev, b_dev, c, M, N, K, "bf16", variant=variant)     # reads A
    tg.tg_gemm_persistent_ex(x_dev, eye, a_dev, M, K, K, "bf16", variant=variant)   # A := X I
    torch.cuda.synchronize()
    assert tg.tg_device_status() == 0
    assert_within_tolerance(wl.bits(c.cpu()), oracle_bits(a, b, "bf16"), "bf16",
                            f"GEMM whose A was overwritten next ({variant})")
    assert np.array_equal(wl.bits(a_dev.cpu()), wl.bits(x))


def test_scale_pack_waits_for_the_gemm_reading_the_old_scales():
    M = N = K = 4096
    a, sa, b, sb = wl.mx_int_inputs(M, N, K, seed=31)
    _, sa2, _, sb2 = wl.mx_int_inputs(M, N, K, seed=32)
    a_dev, b_dev = a.cuda(), b.cuda()
    sa_dev, sb_dev, sa2_dev, sb2_dev = sa.cuda(), sb.cuda(), sa2.cuda(), sb2.cuda()
    pa = tg.mxfp8_pack(sa_dev, K)
    pb = tg.mxfp8_pack(sb_dev, K)
    c = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    torch.cuda.synchronize()
    tg.tg_gemm_mxfp8(a_dev, pa, b_dev, pb, c, M, N, K, "bf16")    # reads the packed scales
    tg.tg_mxfp8_pack_scales(sa2_dev, pa, M, K)                     # then overwrites them
    tg.tg_mxfp8_pack_scales(sb2_dev, pb, N, K)
    c2 = torch.empty_like(c)
    tg.tg_gemm_mxfp8(a_dev, pa, b_dev, pb, c2, M, N, K, "bf16")   # reads the new ones
    torch.cuda.synchronize()
    assert tg.tg_device_status() == 0
    an, bn = a.numpy(), b.numpy()
    assert np.array_equal(wl.bits(c.cpu()), mx.gemm_mxfp8_ref(an, sa.numpy(), bn, sb.numpy(), "bf16"))
    assert np.array_equal(wl.bits(c2.cpu()),
                          mx.gemm_mxfp8_ref(an, sa2.numpy(), bn, sb2.numpy(), "bf16"))
