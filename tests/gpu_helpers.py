"""Shared helpers of the GPU parity tests: run the CUDA path, compare with the oracle."""

import numpy as np
import torch

import persistent_warp_specialized_gb300 as tg
from persistent_warp_specialized_gb300 import _build
from persistent_warp_specialized_gb300 import workloads as wl
from oracle import formats
from oracle import gemm as ogemm

# The acceptance bound of the GEMM (elementwise, C_ref rounded to the output type):
#     |C - C_ref| <= ATOL + RTOL * |C_ref|
ATOL = 5e-3
RTOL = 1e-2


def ensure_library():
    _build.build()
    tg.load_library()


def nan_filled(M, N, dtype):
    c = torch.empty((M, N), dtype=wl.TORCH_DTYPES[dtype], device="cuda")
    c.view(torch.int16).fill_(-1)          # 0xFFFF: a NaN in both formats
    return c


# the kernel variants every parity test runs; "auto" is what tg_gemm_persistent (and the
# benchmark) runs
VARIANTS = ["single", "pair", "wide"]


def run_gpu(a_cpu, b_cpu, dtype, stream=None, variant=None):
    """C bits (numpy uint16) from the GEMM on device copies of a_cpu, b_cpu: through
    tg_gemm_persistent when ``variant`` is None, else tg_gemm_persistent_ex(variant)."""
    M, K = a_cpu.shape
    N = b_cpu.shape[1]
    a = a_cpu.cuda()
    b = b_cpu.cuda()
    c = nan_filled(M, N, dtype)
    if variant is None:
        tg.tg_gemm_persistent(a, b, c, M, N, K, dtype, stream)
    else:
        tg.tg_gemm_persistent_ex(a, b, c, M, N, K, dtype, stream, variant)
    torch.cuda.synchronize()
    assert tg.tg_device_status() == 0
    return wl.bits(c.cpu())


def oracle_bits(a_cpu, b_cpu, dtype):
    return ogemm.gemm_ref(wl.bits(a_cpu), wl.bits(b_cpu), dtype)


def assert_within_tolerance(c_bits, ref_bits, dtype, what=""):
    c = formats.decode(c_bits, dtype)
    r = formats.decode(ref_bits, dtype)
    assert c.shape == r.shape
    nonfinite = ~np.isfinite(c)
    assert not nonfinite.any(), f"{what}: {nonfinite.sum()} non-finite outputs, first at {np.argwhere(nonfinite)[:4].tolist()}"
    err = np.abs(c - r)
    bad = err > ATOL + RTOL * np.abs(r)
    if bad.any():
        idx = np.argwhere(bad)[:6].tolist()
        raise AssertionError(
            f"{what}: {int(bad.sum())} of {bad.size} outside |C-C_ref| <= {ATOL} + {RTOL}|C_ref|; "
            f"first at {idx}; max err {err.max():.4g}")
    return float(err.max())


def ulp_diff_stats(c_bits, ref_bits, dtype):
    """(count of elements more than one output ulp from C_ref, max |C - C_ref| / ulp)."""
    c = formats.decode(c_bits, dtype)
    r = formats.decode(ref_bits, dtype)
    u = formats.ulp(ref_bits, dtype)
    d = np.abs(c - r) / u
    return int((d > 1.0).sum()), float(d.max())


def assert_within_accumulation_bound(c_bits, ref_bits, a_cpu, b_cpu, dtype, what=""):
    """A bound tighter than the acceptance gate, from the arithmetic of the kernel.

    The kernel sums K exact products in fp32 and rounds once to the output type; the oracle
    rounds the exact sum once.  With S = |A|.|B| (binary64) and the fp32 summation bound
    gamma_K = K u / (1 - K u), u = 2^-23 (one unit of fp32 roundoff, allowing the tensor
    core to truncate rather than round), every element must satisfy
        |C - C_ref| <= 2 ulp(C_ref) + gamma_K S.
    Near-zero outputs with heavy cancellation may be many output ulps off and still inside it.
    """
    a = formats.decode(wl.bits(a_cpu), dtype)
    b = formats.decode(wl.bits(b_cpu), dtype)
    s = np.abs(a) @ np.abs(b)
    K = a.shape[1]
    u = 2.0 ** -23
    gamma = K * u / (1 - K * u)
    c = formats.decode(c_bits, dtype)
    r = formats.decode(ref_bits, dtype)
    bound = 2.0 * formats.ulp(ref_bits, dtype) + gamma * s
    bad = np.abs(c - r) > bound
    assert not bad.any(), (f"{what}: {int(bad.sum())} elements outside the fp32 accumulation "
                           f"bound; first at {np.argwhere(bad)[:4].tolist()}")
