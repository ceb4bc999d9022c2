"""GPU: seeded random shapes, integer-valued inputs, every kernel bit-exact against the oracle.

Shapes are drawn to hit the edges the fixed cases may miss: M and N from 1 row/column (N a
multiple of 8) up to several tiles with ragged remainders, K tails that are not a multiple of
the k-block, problems smaller than one tile and problems whose tile count leaves a partial
last wave (so the tail split applies).  Integer inputs make every partial sum exact in fp32,
so the kernels must equal the oracle bit for bit.
"""

import numpy as np
import pytest
import torch

import persistent_warp_specialized_gb300 as tg
from persistent_warp_specialized_gb300 import workloads as wl
from oracle import mx

from gpu_helpers import VARIANTS, ensure_library, nan_filled, oracle_bits

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ensure_library()


def _shapes(seed, count, k_step):
    rng = np.random.default_rng(seed)
    out = []
    for _ in range(count):
        M = int(rng.choice([1, 7, 127, 128, 129, 255, 257, 640, 1000, 1531, 2049]))
        N = int(8 * rng.integers(1, 320))
        K = int(k_step * rng.integers(1, 24))
        out.append((M, N, K))
    return out


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("M,N,K", _shapes(2024, 16, 8))
def test_dense_random_shapes_bit_exact(M, N, K, variant):
    a, b = wl.small_int_inputs(M, N, K, "bf16", seed=M * 7 + N + K)
    c = nan_filled(M, N, "bf16")
    tg.tg_gemm_persistent_ex(a.cuda(), b.cuda(), c, M, N, K, "bf16", variant=variant)
    torch.cuda.synchronize()
    assert tg.tg_device_status() == 0
    assert np.array_equal(wl.bits(c.cpu()), oracle_bits(a, b, "bf16")), (M, N, K, variant)


@pytest.mark.parametrize("variant", ["single", "pair"])
@pytest.mark.parametrize("M,N,K", _shapes(2025, 12, 128))
def test_mxfp8_random_shapes_bit_exact(M, N, K, variant):
    a, sa, b, sb = wl.mx_int_inputs(M, N, K, seed=M + 3 * N + K)
    c = nan_filled(M, N, "bf16")
    tg.tg_gemm_mxfp8_ex(a.cuda(), tg.mxfp8_pack(sa.cuda(), K), b.cuda(), tg.mxfp8_pack(sb.cuda(), K),
                        c, M, N, K, "bf16", variant=variant)
    torch.cuda.synchronize()
    assert tg.tg_device_status() == 0
    want = mx.gemm_mxfp8_ref(a.numpy(), sa.numpy(), b.numpy(), sb.numpy(), "bf16")
    assert np.array_equal(wl.bits(c.cpu()), want), (M, N, K, variant)
