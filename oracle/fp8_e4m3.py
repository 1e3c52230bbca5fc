"""OCP FP8 E4M3 ("e4m3fn") codec, float64 reference (test infrastructure only).

The FP8 KV cache is named as a way to halve KV memory, with per-channel or
per-token scaling granularity ([LLM-INF] section 5.3, FP8 KV cache).  The
pages do not define the format; this module follows the OCP 8-bit floating
point specification for E4M3:

* 1 sign bit, 4 exponent bits (bias 7), 3 mantissa bits;
* exponent field 0 encodes subnormals  (-1)^s * 2^-6 * (m / 8);
* other fields encode normals         (-1)^s * 2^(e-7) * (1 + m / 8);
* no infinities; S.1111.111 is NaN; the largest finite magnitude is
  S.1111.110 = 448.

The encoder rounds to nearest, ties to even, and saturates finite values
whose magnitude exceeds 448 to +-448 ("satfinite").  NaN maps to the NaN code
0x7F (sign kept).  It works on exact float64 arithmetic (every float32 and
every E4M3 value is exact in float64, and the grid steps are powers of two),
so its result does not depend on any rounding mode.
"""
import numpy as np

E4M3_MAX = 448.0
_MIN_NORMAL_EXP = -6          # 2^-6 is the smallest normal magnitude
_SUBNORMAL_STEP = 2.0 ** -9   # 2^-6 * 1/8


def e4m3_decode(codes):
    """Decode uint8 E4M3 codes to float64 (NaN for the two NaN codes)."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = (c & 0x7).astype(np.float64)
    sub = sign * (2.0 ** _MIN_NORMAL_EXP) * (m / 8.0)
    norm = sign * np.ldexp(1.0 + m / 8.0, (e - 7).astype(np.int64))
    out = np.where(e == 0, sub, norm)
    out = np.where((c & 0x7F) == 0x7F, np.nan, out)
    return out.astype(np.float64)


def _round_half_even(x):
    """Round non-negative float64 values to the nearest integer, ties to even."""
    return np.rint(x)  # IEEE rint: round-half-to-even in the default mode


def e4m3_encode(x):
    """Encode float values (float32 or float64) to uint8 E4M3 codes.

    Round to nearest even on the E4M3 grid, saturate finite overflow to
    +-448, keep the sign of zero, NaN -> 0x7F | sign.
    """
    xf = np.asarray(x, dtype=np.float64)
    sign_bit = np.signbit(xf).astype(np.int64) << 7
    a = np.abs(xf)
    nan = np.isnan(xf)
    a = np.where(nan, 0.0, a)
    a = np.minimum(a, E4M3_MAX)            # satfinite (inf included)

    # Grid step for the binade of a: 2^(floor(log2 a) - 3), never below the
    # subnormal step 2^-9.
    with np.errstate(divide="ignore"):
        ex = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    # log2 of an exact power of two is exact; guard against log2 rounding
    # just below an integer for values a hair under a power of two.
    ex = np.where(np.ldexp(1.0, ex.astype(np.int64)) > a, ex - 1, ex)
    ex = np.where(np.ldexp(1.0, (ex + 1).astype(np.int64)) <= a, ex + 1, ex)
    ex = np.maximum(ex, _MIN_NORMAL_EXP)
    step = np.ldexp(1.0, (ex - 3).astype(np.int64))
    q = _round_half_even(a / step) * step   # exact: step is a power of two
    q = np.minimum(q, E4M3_MAX)

    # Bit pattern of the rounded magnitude q.
    is_sub = q < 2.0 ** _MIN_NORMAL_EXP
    sub_code = np.rint(q / _SUBNORMAL_STEP).astype(np.int64)      # 0..8
    with np.errstate(divide="ignore"):
        qe = np.floor(np.log2(np.where(q > 0, q, 1.0))).astype(np.int64)
    qe = np.where(np.ldexp(1.0, qe) > q, qe - 1, qe)
    mant = np.rint((q / np.ldexp(1.0, qe) - 1.0) * 8.0).astype(np.int64)
    norm_code = ((qe + 7) << 3) | mant
    mag = np.where(is_sub, sub_code, norm_code)
    mag = np.where(nan, 0x7F, mag)
    return (sign_bit | mag).astype(np.uint8)
