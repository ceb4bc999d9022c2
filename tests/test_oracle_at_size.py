"""Pins for the oracle's fast contraction at the sizes where it actually runs.

``oracle.gemm.gemm_f64`` and ``oracle.mx.gemm_mxfp8_f64`` sum in binary64 through numpy's
float64 matrix product, a BLAS routine with its own blocking, threading and order.  The pins in
``test_oracle_gemm.py`` and ``test_oracle_mx.py`` use shapes small enough for a BLAS to take a
different, unblocked path, so these repeat the closed forms at sizes past any BLAS block and
compare the BLAS with answers that come from no BLAS:

* integer-valued operands: every partial sum is an integer far below 2^53, so any binary64
  order gives the exact result, which numpy's integer matrix product (its own loops, not
  BLAS) or an int64 rank-1-update loop computes independently;
* all-ones operands with K = 8192 (C = 8192 exactly) and identity factors (C = the other
  operand, bit for bit) at 2048 x 2048;
* non-integer operands: the BLAS sum against the oracle's loop-over-k statement of the same
  sum, within the binary64 error bound of two orders, and the rounded outputs equal wherever
  that bound does not straddle a rounding boundary of the output type.

A dropped or repeated block, a wrong leading dimension, a transposed operand or a thread
writing the wrong panel in the library path fails these.
"""

import numpy as np
import pytest
import torch

from oracle import formats, gemm, mx


def _bits_of(values, fmt):
    return formats.round_rne(np.asarray(values, dtype=np.float64), fmt)


@pytest.fixture(scope="module")
def int_operands_1024():
    rng = np.random.default_rng(1024)
    ai = rng.integers(-2, 3, (1024, 1024)).astype(np.int64)
    bi = rng.integers(-2, 3, (1024, 1024)).astype(np.int64)
    return ai, bi, ai @ bi                   # numpy's integer product: no BLAS


@pytest.mark.parametrize("fmt", ["f16", "bf16"])
def test_blas_sum_is_exact_on_integers_at_1024_cubed(int_operands_1024, fmt):
    ai, bi, exact = int_operands_1024
    a, b = _bits_of(ai, fmt), _bits_of(bi, fmt)
    c64 = gemm.gemm_f64(a, b, fmt)
    assert np.array_equal(c64, exact.astype(np.float64))
    assert np.array_equal(gemm.gemm_ref(a, b, fmt), _bits_of(exact, fmt))


def test_blas_sum_is_exact_on_integers_at_2048x2048x512():
    rng = np.random.default_rng(2048)
    M, N, K = 2048, 2048, 512
    ai = rng.integers(-2, 3, (M, K)).astype(np.int64)
    bi = rng.integers(-2, 3, (K, N)).astype(np.int64)
    exact = np.zeros((M, N), dtype=np.int64)
    for k in range(K):                       # int64 rank-1 updates: no BLAS, no rounding
        exact += np.multiply.outer(ai[:, k], bi[k, :])
    a, b = _bits_of(ai, "bf16"), _bits_of(bi, "bf16")
    assert np.array_equal(gemm.gemm_f64(a, b, "bf16"), exact.astype(np.float64))
    assert np.array_equal(gemm.gemm_ref(a, b, "bf16"), _bits_of(exact, "bf16"))


@pytest.mark.parametrize("fmt", ["f16", "bf16"])
def test_all_ones_with_k_8192_gives_8192(fmt):
    a = _bits_of(np.ones((512, 8192)), fmt)
    b = _bits_of(np.ones((8192, 512)), fmt)
    c = formats.decode(gemm.gemm_ref(a, b, fmt), fmt)
    assert np.array_equal(c, np.full((512, 512), 8192.0))


def test_identity_factors_at_2048():
    rng = np.random.default_rng(11)
    n = 2048
    x = _bits_of(rng.standard_normal((n, n)), "bf16")
    eye = _bits_of(np.eye(n), "bf16")
    assert np.array_equal(gemm.gemm_ref(eye, x, "bf16"), x)     # I . X = X (not X^T)
    assert np.array_equal(gemm.gemm_ref(x, eye, "bf16"), x)     # X . I = X


def _agree_within_two_orders(c_blas, c_loop, absum, K, fmt):
    """|c_blas - c_loop| <= 2 gamma_K sum|ab|, and equal rounded outputs wherever the interval
    of that width around c_loop rounds to a single value of ``fmt``."""
    gamma = K * 2.0 ** -53 / (1 - K * 2.0 ** -53)
    bound = 2 * gamma * absum
    assert (np.abs(c_blas - c_loop) <= bound + 2.0 ** -1074).all()
    lo = formats.round_rne(c_loop - bound, fmt)
    hi = formats.round_rne(c_loop + bound, fmt)
    sure = lo == hi
    assert sure.mean() > 0.999
    assert np.array_equal(formats.round_rne(c_blas, fmt)[sure], lo[sure])


@pytest.mark.parametrize("fmt", ["f16", "bf16"])
def test_blas_sum_equals_the_loop_over_k_on_ragged_random_operands(fmt):
    rng = np.random.default_rng(600 if fmt == "f16" else 601)
    M, N, K = 600, 700, 1100
    a = _bits_of(rng.uniform(-1, 1, (M, K)), fmt)
    b = _bits_of(rng.uniform(-1, 1, (K, N)), fmt)
    c_loop = gemm.gemm_f64_by_k(a, b, fmt)
    absum = gemm.gemm_f64_by_k(_bits_of(np.abs(formats.decode(a, fmt)), fmt),
                               _bits_of(np.abs(formats.decode(b, fmt)), fmt), fmt)
    _agree_within_two_orders(gemm.gemm_f64(a, b, fmt), c_loop, absum, K, fmt)


def _e4m3_bits(values):
    t = torch.tensor(np.asarray(values, dtype=np.float32)).to(torch.float8_e4m3fn)
    return t.view(torch.uint8).numpy()


def test_mx_blas_sum_is_exact_on_integers_at_1024_cubed():
    rng = np.random.default_rng(4096)
    M = N = K = 1024
    ai = rng.integers(-4, 5, (M, K)).astype(np.int64)
    bi = rng.integers(-4, 5, (N, K)).astype(np.int64)     # B given as [N, K]
    unit = np.full((M, K // mx.BLOCK), 127, np.uint8)    # E8M0 127 = 2^0
    c64 = mx.gemm_mxfp8_f64(_e4m3_bits(ai), unit, _e4m3_bits(bi), unit)
    assert np.array_equal(c64, (ai @ bi.T).astype(np.float64))


def test_mx_blas_sum_equals_the_loop_over_k_with_spread_scales():
    rng = np.random.default_rng(77)
    M, N, K = 300, 520, 1024
    a = _e4m3_bits(rng.standard_normal((M, K)))
    b = _e4m3_bits(rng.standard_normal((N, K)))
    sa = rng.integers(117, 138, (M, K // mx.BLOCK)).astype(np.uint8)   # 2^-10 .. 2^10
    sb = rng.integers(117, 138, (N, K // mx.BLOCK)).astype(np.uint8)
    c_loop = mx.gemm_mxfp8_f64_by_k(a, sa, b, sb)
    absum = np.zeros_like(c_loop)
    xa, xb = np.abs(mx.scaled(a, sa)), np.abs(mx.scaled(b, sb))
    for k in range(K):
        absum += np.multiply.outer(xa[:, k], xb[:, k])
    _agree_within_two_orders(mx.gemm_mxfp8_f64(a, sa, b, sb), c_loop, absum, K, "bf16")
