"""FP8 (E4M3) drafter weights: per-row quantization and its exact inverse.

Test infrastructure only (see the package docstring).

Source: the product doc "Speculative decoding" (introduction) and the model
card "Beam-1.0-501B-A23B-DFlash2" (section "Serve") serve the models in bf16,
FP8 and NVFP4.  The pages do not say which FP8 format or how it is scaled.
Reading taken here:
  * format: the E4M3 encoding with no infinities (1 sign bit, 4 exponent
    bits with bias 7, 3 mantissa bits; exponent field 0 holds subnormals
    m/8 * 2^-6; the code with all exponent and mantissa bits set is NaN, so
    the largest finite magnitude is 1.75 * 2^8 = 448);
  * scaling: one float32 scale per output row (per output channel of a
    Linear layer), s_r = max_j |w_rj| / 448 computed in float32, or 1 for a
    row of zeros;
  * rounding: x = w / s_r rounded to float32, then to the nearest E4M3
    value, ties to the value whose mantissa's last bit is 0, magnitudes above
    448 saturating to 448, the sign bit kept also where x rounds to zero;
  * only the weights are quantized; the dequantized weight is code value *
    s_r exactly (float64 here).
"""

import numpy as np

E4M3_MAX = 448.0


def e4m3_value(code):
    """Real value of E4M3 codes (uint8 array); NaN for the two NaN codes."""
    c = np.asarray(code, dtype=np.uint8).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = c & 0x7
    mag = np.where(e == 0, m / 8.0 * 2.0 ** -6, (1.0 + m / 8.0) * 2.0 ** (e - 7.0))
    mag = np.where((e == 15) & (m == 7), np.nan, mag)
    return sign * mag


def e4m3_round(x):
    """Codes (uint8) of float32 values x: nearest E4M3 value, ties to an even
    mantissa, magnitudes beyond 448 saturate.  x must not be NaN.

    Below 2^-6 the E4M3 values are the multiples of 2^-9; in the binade
    [2^e, 2^(e+1)) they are the multiples of 2^(e-3).  Rounding |x| to that
    grid with round-half-even gives the mantissa count m (the scaling by a
    power of two is exact in float32, so only the rounding to an integer
    rounds); the codes 0x00 .. 0x7E enumerate the
    non-negative values in increasing order, so the code is m for the
    subnormal grid (m = 8 is 2^-6, code 0x08) and 8 (e + 7) + (m - 8) in
    binade e (m = 16 is the next binade's first value, same formula)."""
    x = np.asarray(x, dtype=np.float32)
    a = np.minimum(np.abs(x), np.float32(E4M3_MAX))
    _, k = np.frexp(a)                                  # a = f 2^k, f in [0.5, 1)
    e = np.maximum(k - 1, -6).astype(np.int32)          # binade; subnormals share -6's grid
    m = np.rint(np.ldexp(a, 3 - e)).astype(np.int32)    # round half to even
    code = np.where(a < np.float32(2.0 ** -6), m, 8 * (e + 7) + (m - 8)).astype(np.uint8)
    # the sign bit follows x, also where it rounds to zero
    return np.where(np.signbit(x), code | np.uint8(0x80), code).astype(np.uint8)


def quantize_rows(w):
    """(codes uint8 [rows, cols], scales float32 [rows]) of a weight matrix
    (any float array, widened to float32 first)."""
    w = np.asarray(w, dtype=np.float32)
    amax = np.abs(w).max(axis=1)
    scale = np.where(amax > 0, amax / np.float32(E4M3_MAX), np.float32(1.0)).astype(np.float32)
    x = (w / scale[:, None]).astype(np.float32)
    return e4m3_round(x), scale


# value of every code (the formula of e4m3_value, tabulated once)
_VALUE = e4m3_value(np.arange(256, dtype=np.uint8))


def dequantize_rows(codes, scales):
    """float64 weights code value * s_r."""
    return _VALUE[np.asarray(codes, dtype=np.uint8)] * np.asarray(scales, dtype=np.float64)[:, None]
