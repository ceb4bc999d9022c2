"""Seeded synthetic GEMM workloads: shapes, dtypes, value distributions and seeds.

This module only draws random numbers (torch's CPU generator) and casts them to the
input dtype; it holds none of the GEMM's arithmetic.  Both the CUDA path and the CPU
oracle take their inputs from here, so both see the same bits.

The five workloads are the square fp16 problems at 256^3 and 1024^3, the square bf16
problems at 4096^3 and 8192^3 (entries N(0, 1/sqrt(K)), so that the entries of C are
O(1)), and a ragged bf16 problem 4000 x 7000 x 2048 whose edge tiles are partial in
both M and N.  No public dataset is involved.
"""

from dataclasses import dataclass

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    M: int
    N: int
    K: int
    dtype: str          # "f16" or "bf16": input and output type; accumulation is fp32
    dist: str           # "uniform" (U[-1, 1]) or "normal" (N(0, 1/sqrt(K)))
    seed: int

    @property
    def flops(self):
        return 2 * self.M * self.N * self.K


WORKLOADS = {
    w.name: w
    for w in (
        Workload("gemm_256_f16", 256, 256, 256, "f16", "uniform", 1),
        Workload("gemm_1024_f16", 1024, 1024, 1024, "f16", "uniform", 2),
        Workload("gemm_4096_bf16", 4096, 4096, 4096, "bf16", "normal", 3),
        Workload("gemm_8192_bf16", 8192, 8192, 8192, "bf16", "normal", 4),
        Workload("gemm_4000x7000x2048_bf16", 4000, 7000, 2048, "bf16", "uniform", 5),
    )
}

# A smaller case of the 8192^3 kernel for detailed profiles (inputs still larger than L2).
PROFILE_WORKLOADS = {
    w.name: w for w in (Workload("gemm_6144_bf16", 6144, 6144, 6144, "bf16", "normal", 7),)
}

# number of workers and group width the tile schedule of the 256^3 workload is checked with
SCHEDULE_CHECK_WORKERS = 148
SCHEDULE_CHECK_GROUP = 8

TORCH_DTYPES = {"f16": torch.float16, "bf16": torch.bfloat16}


def _draw(shape, dist, k, gen):
    if dist == "uniform":
        return torch.rand(shape, generator=gen, dtype=torch.float32) * 2.0 - 1.0
    if dist == "normal":
        return torch.randn(shape, generator=gen, dtype=torch.float32) * (1.0 / float(k) ** 0.5)
    raise ValueError(f"unknown distribution {dist!r}")


def make_inputs(M, N, K, dtype, dist="uniform", seed=0):
    """A [M, K] and B [K, N] row-major CPU tensors of ``dtype`` ("f16"/"bf16")."""
    gen = torch.Generator().manual_seed(int(seed))
    tdt = TORCH_DTYPES[dtype]
    a = _draw((M, K), dist, K, gen).to(tdt).contiguous()
    b = _draw((K, N), dist, K, gen).to(tdt).contiguous()
    return a, b


def workload_inputs(w):
    return make_inputs(w.M, w.N, w.K, w.dtype, w.dist, w.seed)


def small_int_inputs(M, N, K, dtype, lo=-2, hi=2, seed=0):
    """Integer-valued entries in [lo, hi]: every partial sum is exact in fp32."""
    gen = torch.Generator().manual_seed(int(seed))
    tdt = TORCH_DTYPES[dtype]
    a = torch.randint(lo, hi + 1, (M, K), generator=gen).to(tdt).contiguous()
    b = torch.randint(lo, hi + 1, (K, N), generator=gen).to(tdt).contiguous()
    return a, b


def bits(t):
    """The 16-bit patterns of a CPU fp16/bf16 tensor as a numpy uint16 array (no copy)."""
    import numpy as np

    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


# ---------------------------------------------------------------- block-scaled MXFP8 inputs
# The MXFP8 workload runs at the size of the dense headline (8192^3, bf16 output); the tests
# add small, ragged and integer-valued cases.
MX_WORKLOADS = {
    "mxfp8_8192": (8192, 8192, 8192, 6),   # M, N, K, seed
    "mxfp8_6144": (6144, 6144, 6144, 8),   # a smaller case for detailed profiles
    "mxfp8_512": (512, 512, 512, 9),       # a small case the oracle finishes at once
}
MX_BLOCK = 32


def _mx_quantize(x):
    """x [R, K] float32 -> (E4M3 bytes [R, K], E8M0 bytes [R, K/32]) by the OCP Microscaling
    recipe: per block of 32 along K, shared exponent floor(log2(max |x|)) - 8 (8 = the largest
    E4M3 exponent), elements x / 2^e saturated to +-448 and cast by torch (round to nearest
    even); all-zero blocks take the exponent -127."""
    R, K = x.shape
    blocks = x.reshape(R, K // MX_BLOCK, MX_BLOCK)
    amax = blocks.abs().amax(dim=2)
    e = torch.where(amax > 0, torch.floor(torch.log2(torch.where(amax > 0, amax, 1.0))) - 8,
                    torch.full_like(amax, -127.0)).clamp(-127, 127)
    scaled = (blocks / torch.exp2(e)[:, :, None]).clamp(-448.0, 448.0)
    q = scaled.reshape(R, K).to(torch.float8_e4m3fn).view(torch.uint8).contiguous()
    s = (e + 127).to(torch.uint8).contiguous()
    return q, s


def make_mx_inputs(M, N, K, seed=0):
    """(A [M, K], SFA [M, K/32], B [N, K], SFB [N, K/32]) as CPU uint8 tensors: A and B are
    N(0, 1) and N(0, 1/K) draws quantized to MXFP8 (so entries of C are O(1))."""
    gen = torch.Generator().manual_seed(int(seed))
    a = torch.randn((M, K), generator=gen, dtype=torch.float32)
    b = torch.randn((N, K), generator=gen, dtype=torch.float32) * (1.0 / float(K) ** 0.5)
    qa, sa = _mx_quantize(a)
    qb, sb = _mx_quantize(b)
    return qa, sa, qb, sb


# E4M3 byte patterns of the integers -4 .. 4
_E4M3_INT = {-4: 0xC8, -3: 0xC4, -2: 0xC0, -1: 0xB8, 0: 0x00, 1: 0x38, 2: 0x40, 3: 0x44, 4: 0x48}


def mx_int_inputs(M, N, K, seed=0, scale_lo=126, scale_hi=128):
    """Integer elements in [-4, 4] with scales 2^(s - 127), s in [scale_lo, scale_hi]: every
    partial sum of the product is exact in fp32 for K up to 2^13."""
    gen = torch.Generator().manual_seed(int(seed))
    lut = torch.tensor([_E4M3_INT[v] for v in range(-4, 5)], dtype=torch.uint8)
    a = lut[torch.randint(0, 9, (M, K), generator=gen)].contiguous()
    b = lut[torch.randint(0, 9, (N, K), generator=gen)].contiguous()
    sa = torch.randint(scale_lo, scale_hi + 1, (M, K // MX_BLOCK), generator=gen).to(torch.uint8)
    sb = torch.randint(scale_lo, scale_hi + 1, (N, K // MX_BLOCK), generator=gen).to(torch.uint8)
    return a, sa.contiguous(), b, sb.contiguous()
