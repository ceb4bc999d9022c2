"""Pins for oracle.mx: E4M3 / E8M0 decoding and the block-scaled MXFP8 product.

Tied to things other than the oracle itself: torch's own float8_e4m3fn and float8_e8m0fnu
conversions (every byte pattern), values fixed by the format definitions, an exact
rational brute force written as a different formulation (a per-element loop that looks
the scale of each k up by its block), and invariants of the scaling (a scale step of one
doubles exactly one block's contribution) that catch a wrong block index, a scale applied
to the wrong operand or a transposed B.
"""

from fractions import Fraction

import numpy as np
import pytest
import torch

from oracle import formats, mx

ALL8 = np.arange(256, dtype=np.uint8)


def test_e4m3_decode_matches_torch_for_every_pattern():
    ours = mx.decode_e4m3(ALL8)
    ref = torch.from_numpy(ALL8.copy()).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])
    assert np.array_equal(np.signbit(ours[~nan]), np.signbit(ref[~nan]))


def test_e4m3_values_fixed_by_the_format():
    v = mx.decode_e4m3(np.array([0x38, 0x7E, 0x01, 0x08, 0x07, 0x80, 0xB8, 0x3C, 0x7F, 0xFF],
                                np.uint8))
    assert list(v[:8]) == [1.0, 448.0, 2.0 ** -9, 2.0 ** -6, 7 * 2.0 ** -9, -0.0, -1.0, 1.5]
    assert np.signbit(v[5])
    assert np.isnan(v[8]) and np.isnan(v[9])
    # no infinities: S.1111.110 is the largest finite magnitude
    assert np.isfinite(mx.decode_e4m3(ALL8)[(ALL8 & 0x7F) != 0x7F]).all()


@pytest.mark.skipif(not hasattr(torch, "float8_e8m0fnu"), reason="torch without float8_e8m0fnu")
def test_e8m0_decode_matches_torch_for_every_pattern():
    ours = mx.decode_e8m0(ALL8)
    ref = torch.from_numpy(ALL8.copy()).view(torch.float8_e8m0fnu).to(torch.float64).numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])


def test_e8m0_values_fixed_by_the_format():
    v = mx.decode_e8m0(np.array([127, 128, 126, 0, 254, 255], np.uint8))
    assert list(v[:5]) == [1.0, 2.0, 0.5, 2.0 ** -127, 2.0 ** 127]
    assert np.isnan(v[5])


def _rand_e4m3(shape, rng, emin=4, emax=10):
    """E4M3 patterns with exponent field in [emin, emax] (|x| in [2^-3, 2^3] by default)."""
    s = rng.integers(0, 2, shape) << 7
    e = rng.integers(emin, emax + 1, shape) << 3
    f = rng.integers(0, 8, shape)
    return (s | e | f).astype(np.uint8)


def _rand_scales(shape, rng, lo=125, hi=129):
    return rng.integers(lo, hi + 1, shape).astype(np.uint8)


def _exact(a, sa, b, sb):
    """Per-element loop in exact rationals; the scale of k is that of block k // 32."""
    M, K = a.shape
    N = b.shape[0]
    av = mx.decode_e4m3(a)
    bv = mx.decode_e4m3(b)
    out = [[Fraction(0)] * N for _ in range(M)]
    for i in range(M):
        for j in range(N):
            acc = Fraction(0)
            for k in range(K):
                blk = k // 32
                acc += (Fraction(float(av[i, k])) * Fraction(2) ** (int(sa[i, blk]) - 127)
                        * Fraction(float(bv[j, k])) * Fraction(2) ** (int(sb[j, blk]) - 127))
            out[i][j] = acc
    return out


@pytest.mark.parametrize("M,N,K", [(3, 5, 32), (4, 2, 96), (1, 7, 64), (6, 1, 128)])
def test_tiny_shapes_against_exact_rationals(M, N, K):
    # element exponents in [-3, 3] and scales in 2^[-2, 2]: every partial sum spans fewer
    # than 53 bits, so the binary64 result must equal the exact sum
    rng = np.random.default_rng(M * 1000 + N * 10 + K)
    a = _rand_e4m3((M, K), rng)
    b = _rand_e4m3((N, K), rng)
    sa = _rand_scales((M, K // 32), rng)
    sb = _rand_scales((N, K // 32), rng)
    c64 = mx.gemm_mxfp8_f64(a, sa, b, sb)
    assert c64.shape == (M, N)
    exact = _exact(a, sa, b, sb)
    for i in range(M):
        for j in range(N):
            assert Fraction(float(c64[i, j])) == exact[i][j]
    cref = mx.gemm_mxfp8_ref(a, sa, b, sb, "bf16")
    want = formats.round_rne(np.array([[float(x) for x in row] for row in exact]), "bf16")
    assert np.array_equal(cref, want)


def test_one_scale_step_doubles_exactly_one_block():
    rng = np.random.default_rng(9)
    M, N, K = 8, 6, 128
    a = _rand_e4m3((M, K), rng)
    b = _rand_e4m3((N, K), rng)
    sa = _rand_scales((M, K // 32), rng)
    sb = _rand_scales((N, K // 32), rng)
    base = mx.gemm_mxfp8_f64(a, sa, b, sb)
    for blk in range(K // 32):
        # the contribution of block blk alone (others zeroed in A)
        a_blk = np.zeros_like(a)
        a_blk[:, blk * 32:(blk + 1) * 32] = a[:, blk * 32:(blk + 1) * 32]
        part = mx.gemm_mxfp8_f64(a_blk, sa, b, sb)
        sa2 = sa.copy()
        sa2[2, blk] += 1                       # row 2 of A, block blk
        got = mx.gemm_mxfp8_f64(a, sa2, b, sb)
        want = base.copy()
        want[2] += part[2]
        assert np.allclose(got, want, rtol=0, atol=1e-12 * np.abs(base).max())
        assert np.array_equal(np.delete(got, 2, 0), np.delete(base, 2, 0))
        sb2 = sb.copy()
        sb2[4, blk] += 1                       # column 4 of C (row 4 of B), block blk
        got = mx.gemm_mxfp8_f64(a, sa, b, sb2)
        want = base.copy()
        want[:, 4] += part[:, 4]
        assert np.allclose(got, want, rtol=0, atol=1e-12 * np.abs(base).max())
        assert np.array_equal(np.delete(got, 4, 1), np.delete(base, 4, 1))


def test_identity_a_returns_scaled_b_transposed():
    # A = I (32 x 32, unit scales): C[i, j] = b[j, i] * 2^(sb[j, 0] - 127)
    rng = np.random.default_rng(4)
    N = 20
    a = np.zeros((32, 32), np.uint8)
    a[np.arange(32), np.arange(32)] = 0x38
    sa = np.full((32, 1), 127, np.uint8)
    b = _rand_e4m3((N, 32), rng)
    sb = _rand_scales((N, 1), rng)
    c = mx.gemm_mxfp8_f64(a, sa, b, sb)
    want = (mx.decode_e4m3(b) * np.ldexp(1.0, sb.astype(np.int64) - 127)).T
    assert np.array_equal(c, want)


def test_integer_inputs_match_python_integers():
    # E4M3 holds every integer in [-16, 16]; unit scales give Python's integer product
    rng = np.random.default_rng(21)
    M, N, K = 9, 11, 64
    ai = rng.integers(-4, 5, (M, K))
    bi = rng.integers(-4, 5, (N, K))
    lut = {int(v): int(p) for p, v in zip(ALL8, mx.decode_e4m3(ALL8))
           if np.isfinite(v) and float(v).is_integer() and not (v == 0 and np.signbit(v))}
    a = np.vectorize(lut.get)(ai).astype(np.uint8)
    b = np.vectorize(lut.get)(bi).astype(np.uint8)
    ones = np.full((M, K // 32), 127, np.uint8)
    c = mx.gemm_mxfp8_f64(a, ones, b, np.full((N, K // 32), 127, np.uint8))
    want = [[sum(int(ai[i, k]) * int(bi[j, k]) for k in range(K)) for j in range(N)]
            for i in range(M)]
    assert np.array_equal(c, np.array(want, dtype=np.float64))


def test_entries_equal_the_full_product():
    rng = np.random.default_rng(5)
    a = _rand_e4m3((40, 64), rng)
    b = _rand_e4m3((30, 64), rng)
    sa = _rand_scales((40, 2), rng)
    sb = _rand_scales((30, 2), rng)
    full = mx.gemm_mxfp8_ref(a, sa, b, sb, "bf16")
    rows, cols = np.array([0, 17, 39]), np.array([29, 2, 0])
    assert np.array_equal(mx.gemm_mxfp8_ref_entries(a, sa, b, sb, rows, cols, "bf16"),
                          full[np.ix_(rows, cols)])


def test_shape_mismatches_are_rejected():
    a = np.zeros((4, 64), np.uint8)
    with pytest.raises(ValueError):
        mx.gemm_mxfp8_f64(a, np.zeros((4, 1), np.uint8), a, np.zeros((4, 2), np.uint8))
    with pytest.raises(ValueError):
        mx.gemm_mxfp8_f64(a, np.zeros((4, 2), np.uint8), np.zeros((4, 32), np.uint8),
                          np.zeros((4, 1), np.uint8))
