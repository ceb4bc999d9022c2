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
