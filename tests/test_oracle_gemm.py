"""Pins for oracle.gemm: closed forms, exact rational brute force and integer arithmetic.

A plausible mistake in the oracle -- a transposed operand, a dropped or repeated term,
a wrong decode or rounding -- fails at least one of these:
* all-ones matrices give C = K exactly;
* an identity factor reproduces the other operand bit for bit (A = I gives B, B = I gives A);
* on tiny non-square shapes every entry of both binary64 statements of the sum (the library
  product and the loop over k) equals the exact rational sum computed with Python's
  ``fractions`` (products and sums done without rounding), to within the binary64
  summation error bound, and the rounded result equals the correctly rounded
  exact sum whenever the exact sum is not within that bound of a rounding boundary;
* integer-valued inputs give exactly Python's integer matrix product.
"""

from fractions import Fraction

import numpy as np
import pytest

from oracle import formats, gemm


def _bits_of(values, fmt):
    return formats.round_rne(np.asarray(values, dtype=np.float64), fmt)


@pytest.mark.parametrize("fmt", ["f16", "bf16"])
@pytest.mark.parametrize("K", [1, 7, 256, 1024, 2048, 8192])
def test_all_ones_gives_k(fmt, K):
    M, N = 3, 5
    a = _bits_of(np.ones((M, K)), fmt)
    b = _bits_of(np.ones((K, N)), fmt)
    c = gemm.gemm_ref(a, b, fmt)
    assert np.array_equal(formats.decode(c, fmt), np.full((M, N), float(K)))


@pytest.mark.parametrize("fmt", ["f16", "bf16"])
def test_identity_factors_reproduce_operand(fmt):
    rng = np.random.default_rng(3)
    n = 40
    x = _bits_of(rng.uniform(-4, 4, (n, 24)), fmt)        # [n, 24]
    eye = _bits_of(np.eye(n), fmt)
    assert np.array_equal(gemm.gemm_ref(eye, x, fmt), x)  # I . X = X
    y = _bits_of(rng.uniform(-4, 4, (24, n)), fmt)        # [24, n]
    assert np.array_equal(gemm.gemm_ref(y, eye, fmt), y)  # Y . I = Y


def _exact(a_bits, b_bits, fmt):
    a = formats.decode(a_bits, fmt)
    b = formats.decode(b_bits, fmt)
    M, K = a.shape
    N = b.shape[1]
    out = [[Fraction(0)] * N for _ in range(M)]
    absum = np.zeros((M, N))
    for i in range(M):
        for j in range(N):
            s = Fraction(0)
            for k in range(K):
                s += Fraction(float(a[i, k])) * Fraction(float(b[k, j]))
                absum[i, j] += abs(float(a[i, k]) * float(b[k, j]))
            out[i][j] = s
    return out, absum


@pytest.mark.parametrize("fmt", ["f16", "bf16"])
@pytest.mark.parametrize("shape", [(3, 5, 7), (4, 1, 9), (1, 6, 2), (5, 3, 33)])
def test_tiny_shapes_against_exact_rationals(fmt, shape):
    M, N, K = shape
    rng = np.random.default_rng(M * 100 + N * 10 + K)
    a = _bits_of(rng.uniform(-1, 1, (M, K)), fmt)
    b = _bits_of(rng.uniform(-1, 1, (K, N)), fmt)
    c64 = gemm.gemm_f64(a, b, fmt)
    c64_by_k = gemm.gemm_f64_by_k(a, b, fmt)
    assert c64.shape == (M, N) and c64_by_k.shape == (M, N)
    exact, absum = _exact(a, b, fmt)
    gamma = K * 2.0 ** -53 / (1 - K * 2.0 ** -53)
    cref = gemm.gemm_ref(a, b, fmt)
    for i in range(M):
        for j in range(N):
            for c in (c64, c64_by_k):        # the library sum and the loop over k
                err = abs(Fraction(float(c[i, j])) - exact[i][j])
                assert err <= Fraction(gamma * absum[i, j]) + Fraction(1, 1 << 1074)
            # the rounded result: round the (binary64-nearest) exact value once
            nearest = float(exact[i][j])
            want = formats.round_rne(np.array([nearest]), fmt)[0]
            # skip only if a rounding boundary of fmt lies within the error bound
            lo = formats.round_rne(np.array([nearest - 2 * gamma * absum[i, j]]), fmt)[0]
            hi = formats.round_rne(np.array([nearest + 2 * gamma * absum[i, j]]), fmt)[0]
            if lo == hi:
                assert cref[i, j] == want


@pytest.mark.parametrize("fmt,lim", [("f16", 2), ("bf16", 2)])
def test_integer_inputs_match_python_integers(fmt, lim):
    rng = np.random.default_rng(7)
    M, N, K = 17, 33, 65
    ai = rng.integers(-lim, lim + 1, (M, K))
    bi = rng.integers(-lim, lim + 1, (K, N))
    a = _bits_of(ai, fmt)
    b = _bits_of(bi, fmt)
    c = formats.decode(gemm.gemm_ref(a, b, fmt), fmt)
    want = [[sum(int(ai[i, k]) * int(bi[k, j]) for k in range(K)) for j in range(N)] for i in range(M)]
    # |C| <= 65 * 4 = 260: exact in f16 (< 2048); in bf16 only up to 256 is exact, so
    # compare the correctly rounded integer
    want_bits = formats.round_rne(np.array(want, dtype=np.float64), fmt)
    assert np.array_equal(formats.round_rne(c, fmt), want_bits)


def test_entries_equal_rows_and_columns_of_full_product():
    rng = np.random.default_rng(5)
    a = _bits_of(rng.uniform(-1, 1, (50, 40)), "bf16")
    b = _bits_of(rng.uniform(-1, 1, (40, 30)), "bf16")
    full = gemm.gemm_ref(a, b, "bf16")
    rows = np.array([0, 7, 49])
    cols = np.array([29, 3, 0, 11])
    assert np.array_equal(gemm.gemm_ref_entries(a, b, rows, cols, "bf16"), full[np.ix_(rows, cols)])


def test_shape_mismatch_is_rejected():
    a = np.zeros((3, 4), np.uint16)
    b = np.zeros((5, 2), np.uint16)
    with pytest.raises(ValueError):
        gemm.gemm_f64(a, b, "f16")
    with pytest.raises(ValueError):
        gemm.gemm_f64_by_k(a, b, "f16")
