"""Block-scaled MXFP8 GEMM with binary64 accumulation (oracle; test infrastructure only).

The second workload of "[Feature] Introduce tile scheduler #2441" is a block-scaled MXFP8
GEMM on the same persistent scheduler (examples/blockscaled_gemm_sm100/
gemm_mxfp8_blockscaled_1d1d.py: TMA load, MMA, scale-factor and epilogue roles, each
driven by its own ``PersistentTileScheduler``; the PR overview and the review comments
on that file).  The pages name the roles but not the number formats, so the plain
reading of "MXFP8" is taken: the OCP Microscaling format, where a block of 32 consecutive
elements shares one scale.  "1d1d": both operands are scaled along K only, A per row and
B per column, one scale per 32 K-elements of each.

Element type E4M3 (1 sign, 4 exponent bits with bias 7, 3 fraction bits; no infinities;
S.1111.111 is NaN; largest finite 448).  Scale type E8M0 (8 exponent bits, no sign, no
fraction: 2^(e - 127); 0xFF is NaN).

    C[i, j] = round_out( sum_k  a[i, k] * 2^(sa[i, k // 32] - 127)
                              *  b[j, k] * 2^(sb[j, k // 32] - 127) )

Layouts: ``a`` [M, K] and ``b`` [N, K] hold E4M3 byte patterns, both K-contiguous (B is
given as N rows of K, so that each of its columns' 32-element blocks is contiguous like
A's); ``sa`` [M, K/32] and ``sb`` [N, K/32] hold E8M0 byte patterns.  Every product of two
E4M3 values has at most 8 significant bits and the scales are powers of two within
2^+-254, so every scaled product is exact in binary64; the sum is binary64 (numpy's
float64 matrix product, a library step); the result is rounded once to the output type.
``gemm_mxfp8_f64_by_k`` states the same sum without a library contraction (K rank-1
updates in k order); the pins compare the two, and the library product with exact integer
arithmetic, at sizes where the library blocks and threads.
"""

import numpy as np

from . import formats

BLOCK = 32


def decode_e4m3(bits):
    """E4M3 byte patterns -> exact binary64 values, from the field definition."""
    b = np.asarray(bits).astype(np.int64)
    sign = np.where(b & 0x80, -1.0, 1.0)
    e = (b >> 3) & 0xF
    f = (b & 0x7).astype(np.float64)
    normal = sign * np.ldexp(1.0 + f / 8.0, e - 7)
    subnormal = sign * np.ldexp(f / 8.0, -6)
    out = np.where(e == 0, subnormal, normal)
    return np.where((b & 0x7F) == 0x7F, np.nan, out)


def decode_e8m0(bits):
    """E8M0 byte patterns -> 2^(e - 127) in binary64 (0xFF is NaN)."""
    e = np.asarray(bits).astype(np.int64)
    return np.where(e == 0xFF, np.nan, np.ldexp(1.0, e - 127))


def scaled(x_bits, s_bits):
    """The real values of one operand: element [r, k] times its block scale [r, k // 32]."""
    x = decode_e4m3(x_bits)
    s = decode_e8m0(s_bits)
    if x.ndim != 2 or s.ndim != 2 or x.shape[0] != s.shape[0] or x.shape[1] != BLOCK * s.shape[1]:
        raise ValueError(f"operand {x.shape} and scales {s.shape} do not match (block {BLOCK})")
    return x * np.repeat(s, BLOCK, axis=1)


def gemm_mxfp8_f64(a_bits, sa_bits, b_bits, sb_bits):
    """Exact scaled products, binary64 sums: the [M, N] float64 matrix A . B^T."""
    a = scaled(a_bits, sa_bits)
    b = scaled(b_bits, sb_bits)
    if a.shape[1] != b.shape[1]:
        raise ValueError(f"K of A ({a.shape[1]}) and B ({b.shape[1]}) differ")
    return a @ b.T


def gemm_mxfp8_f64_by_k(a_bits, sa_bits, b_bits, sb_bits):
    """The same sum as K rank-1 updates of the scaled operands in k order, binary64."""
    a = scaled(a_bits, sa_bits)
    b = scaled(b_bits, sb_bits)
    if a.shape[1] != b.shape[1]:
        raise ValueError(f"K of A ({a.shape[1]}) and B ({b.shape[1]}) differ")
    c = np.zeros((a.shape[0], b.shape[0]), dtype=np.float64)
    for k in range(a.shape[1]):
        c += np.multiply.outer(a[:, k], b[:, k])
    return c


def gemm_mxfp8_ref(a_bits, sa_bits, b_bits, sb_bits, out_fmt="bf16"):
    """C_ref bits: the binary64 result rounded (ties to even) to ``out_fmt``."""
    return formats.round_rne(gemm_mxfp8_f64(a_bits, sa_bits, b_bits, sb_bits), out_fmt)


def gemm_mxfp8_ref_entries(a_bits, sa_bits, b_bits, sb_bits, rows, cols, out_fmt="bf16"):
    """C_ref restricted to rows x cols (index arrays)."""
    rows = np.asarray(rows)
    cols = np.asarray(cols)
    return gemm_mxfp8_ref(np.asarray(a_bits)[rows], np.asarray(sa_bits)[rows],
                          np.asarray(b_bits)[cols], np.asarray(sb_bits)[cols], out_fmt)
