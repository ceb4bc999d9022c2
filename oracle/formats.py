"""IEEE-754 binary16 and bfloat16 from their field definitions (oracle; test infrastructure).

Both formats are 16-bit: 1 sign bit, ``ebits`` exponent bits with bias ``2^(ebits-1)-1``,
and ``mbits`` stored fraction bits.  binary16: ebits=5, mbits=10.  bfloat16 is the upper
half of binary32: ebits=8, mbits=7.  The GEMM's ``in_dtype``/``out_dtype`` are one of the
two ("[Feature] Introduce tile scheduler #2441", examples/gemm_sm100/
gemm_tcgen5mma_ws_persistent.py, ``main``: ``in_dtype, out_dtype, accum_dtype``).

``decode`` maps bit patterns to exact binary64 values; ``round_rne`` rounds binary64
values to the nearest representable value, ties to even (IEEE-754 roundTiesToEven),
with gradual underflow and overflow to infinity.  Neither uses a library conversion:
the tests compare them with numpy's float16 and with binary32 truncation, which is how
they are pinned.
"""

import numpy as np

# name -> (exponent bits, stored fraction bits)
FIELDS = {
    "f16": (5, 10),
    "bf16": (8, 7),
}


def _params(fmt):
    ebits, mbits = FIELDS[fmt]
    bias = (1 << (ebits - 1)) - 1
    emin = 1 - bias            # exponent of the smallest normal number
    emax = bias                # exponent of the largest finite number
    return ebits, mbits, bias, emin, emax


def decode(bits, fmt):
    """16-bit patterns (uint16 array) -> exact binary64 values.

    normal   (0 < e < 2^ebits-1): (-1)^s * 2^(e-bias) * (1 + f/2^mbits)
    subnormal (e == 0):           (-1)^s * 2^emin     * (f/2^mbits)
    e == 2^ebits-1:               +-inf if f == 0, else NaN
    """
    ebits, mbits, bias, emin, _ = _params(fmt)
    b = np.asarray(bits).astype(np.uint16).astype(np.int64)
    s = (b >> 15) & 1
    e = (b >> mbits) & ((1 << ebits) - 1)
    f = b & ((1 << mbits) - 1)
    frac = f.astype(np.float64) / float(1 << mbits)
    normal = np.ldexp(1.0 + frac, (e - bias).astype(np.int64))
    sub = np.ldexp(frac, emin)
    mag = np.where(e == 0, sub, normal)
    special = e == (1 << ebits) - 1
    mag = np.where(special & (f == 0), np.inf, mag)
    mag = np.where(special & (f != 0), np.nan, mag)
    return np.where(s == 1, -mag, mag)


def round_rne(x, fmt):
    """binary64 values -> 16-bit patterns of the nearest value of ``fmt`` (ties to even).

    For finite |x| let E = floor(log2|x|), raised to emin below the normal range (the
    spacing of the subnormals is that of the smallest binade).  The spacing of ``fmt``
    at |x| is 2^(E-mbits); |x| / 2^(E-mbits) is rounded to an integer n, ties to even.
    If rounding carried into the next binade (n == 2^(mbits+1)) the exponent grows by
    one.  A result whose exponent exceeds emax is infinity.  NaN maps to the quiet NaN
    with the sign bit clear.
    """
    ebits, mbits, bias, emin, emax = _params(fmt)
    x = np.asarray(x, dtype=np.float64)
    sign = np.signbit(x).astype(np.int64)
    a = np.abs(x)
    finite = np.isfinite(a)
    positive = finite & (a > 0)
    # frexp: a = m * 2^e with m in [0.5, 1)  =>  floor(log2 a) = e - 1
    _, e2 = np.frexp(np.where(positive, a, 1.0))
    E = np.maximum(e2.astype(np.int64) - 1, emin)
    q = E - mbits                                  # exponent of the spacing at a
    n = np.rint(np.ldexp(np.where(finite, a, 0.0), -q))   # np.rint: ties to even
    carry = n >= float(1 << (mbits + 1))
    n = np.where(carry, n / 2.0, n)
    E = np.where(carry, E + 1, E)
    n = n.astype(np.int64)
    normal = n >= (1 << mbits)
    exp_field = np.where(normal, E + bias, 0)
    frac_field = np.where(normal, n - (1 << mbits), n)
    bits = (exp_field << mbits) | frac_field
    inf_bits = ((1 << ebits) - 1) << mbits
    nan_bits = inf_bits | (1 << (mbits - 1))
    bits = np.where(finite & (E > emax), inf_bits, bits)
    bits = np.where(np.isinf(x), inf_bits, bits)
    bits = bits | (sign << 15)
    bits = np.where(np.isnan(x), nan_bits, bits)
    return bits.astype(np.uint16)


def ulp(bits, fmt):
    """Spacing of ``fmt`` at the (finite) values encoded by ``bits``: 2^(E-mbits)."""
    ebits, mbits, bias, emin, _ = _params(fmt)
    b = np.asarray(bits).astype(np.uint16).astype(np.int64)
    e = (b >> mbits) & ((1 << ebits) - 1)
    E = np.where(e == 0, emin, e - bias)
    return np.ldexp(1.0, (E - mbits).astype(np.int64))
