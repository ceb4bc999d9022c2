"""Plain dense GEMM with binary64 accumulation (oracle; test infrastructure only).

C[i, j] = round_out( sum_k A[i, k] * B[k, j] )

A is [M, K] and B is [K, N], both row-major, given as 16-bit patterns of ``in_fmt``;
C is [M, N] in ``out_fmt``.  This is the contraction that ``gemm_persistent`` in
"[Feature] Introduce tile scheduler #2441" (examples/gemm_sm100/
gemm_tcgen5mma_ws_persistent.py) computes tile by tile: ``T.tcgen05_gemm(A_shared,
B_shared, C_tmem_*, clear_accum=k == 0)`` over the k-blocks, then the epilogue casts
``C_local`` to ``out_dtype``.  The method reaches the plain result up to the order of
its fp32 additions, so the oracle is the plain definition: every product of two
binary16/bfloat16 values is exact in binary64 (at most 22 significant bits), the sum is
accumulated in binary64 by numpy's float64 matrix product (a library step), and the
result is rounded once to the output type.

Two statements of the same binary64 sum are kept:
* ``gemm_f64_by_k`` is the definition written out: K rank-1 updates C += A[:, k] B[k, :],
  taken in k order with elementwise binary64 multiplies and adds (the i and j loops of the
  triple loop are numpy's elementwise loops; no library contraction).  It is slow (K passes
  over C) and serves as the reference the fast form is pinned against.
* ``gemm_f64`` is the same sum by numpy's float64 matrix product (BLAS): blocked, threaded
  and in its own order.  Every binary64 sum of the same terms lies within
  gamma_K * sum_k |A[i,k] B[k,j]| of the exact sum (gamma_K = K u / (1 - K u), u = 2^-53),
  so the two differ by at most twice that, far below half an ulp of the 16-bit output for
  all but outputs within that distance of a rounding boundary.  The pins compare them at
  sizes where the BLAS takes its blocked, multithreaded path, and compare the BLAS with
  exact integer arithmetic there.
"""

import numpy as np

from . import formats


def gemm_f64(a_bits, b_bits, in_fmt):
    """Exact products, binary64 sums: returns the [M, N] float64 matrix A.B."""
    a = formats.decode(a_bits, in_fmt)
    b = formats.decode(b_bits, in_fmt)
    if a.ndim != 2 or b.ndim != 2 or a.shape[1] != b.shape[0]:
        raise ValueError(f"shapes {a.shape} x {b.shape} do not contract")
    return a @ b


def gemm_f64_by_k(a_bits, b_bits, in_fmt):
    """The same sum without a library contraction: K rank-1 updates in k order, binary64."""
    a = formats.decode(a_bits, in_fmt)
    b = formats.decode(b_bits, in_fmt)
    if a.ndim != 2 or b.ndim != 2 or a.shape[1] != b.shape[0]:
        raise ValueError(f"shapes {a.shape} x {b.shape} do not contract")
    c = np.zeros((a.shape[0], b.shape[1]), dtype=np.float64)
    for k in range(a.shape[1]):
        c += np.multiply.outer(a[:, k], b[k, :])
    return c


def gemm_ref(a_bits, b_bits, in_fmt, out_fmt=None):
    """C_ref bits: the binary64 product rounded (ties to even) to ``out_fmt``."""
    return formats.round_rne(gemm_f64(a_bits, b_bits, in_fmt), out_fmt or in_fmt)


def gemm_ref_entries(a_bits, b_bits, rows, cols, in_fmt, out_fmt=None):
    """C_ref restricted to rows x cols (index arrays): A[rows, :] . B[:, cols]."""
    rows = np.asarray(rows)
    cols = np.asarray(cols)
    sub_a = np.asarray(a_bits)[rows, :]
    sub_b = np.asarray(b_bits)[:, cols]
    return gemm_ref(sub_a, sub_b, in_fmt, out_fmt)
