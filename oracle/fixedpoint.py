"""Exact integer inverse-CDF sampling.

Test infrastructure only (see the package docstring).

Every draw of the method (the drafter's y ~ q, the resample from the residual
[p - q]+ after a rejection, and the bonus token from the target's next
distribution; "DFlash vs DFlash 2" blog, section "The problem: one expensive
token at a time") is an inverse-CDF draw.  To make the draw reproducible
bit for bit on any machine, the weights are moved to a fixed-point grid and
the cumulative sum is taken in integers, which is associative:

    R_v = floor(r_v * 2^45)           r_v a float32 weight in [0, 1]
    Z   = sum_v R_v                   exact; < 2^63 for V <= 2^18
    T   = floor(u64 * Z / 2^64)       u64 uniform on [0, 2^64)
    v*  = min { v : R_0 + ... + R_v > T }

so that P(v* = v) = R_v / Z up to 2^-64.  Because T < Z, v* always exists
when Z > 0.  The scaling by 2^45 is exact in float arithmetic (a power of
two) and the conversion truncates, i.e. floors, non-negative values.
"""

import numpy as np

SCALE_BITS = 45
_MASK32 = np.uint64(0xFFFFFFFF)


def to_fixed(r):
    """float32 weights (>= 0) -> uint64 fixed-point weights R_v."""
    r = np.asarray(r, dtype=np.float32).astype(np.float64)
    if np.any(r < 0) or np.any(r > 1):
        raise ValueError("fixed-point weights must lie in [0, 1]")
    return np.floor(r * float(2 ** SCALE_BITS)).astype(np.uint64)


def mulhi64(a, b):
    """floor(a * b / 2^64) for uint64 arrays, via 32-bit halves."""
    a = np.asarray(a, dtype=np.uint64)
    b = np.asarray(b, dtype=np.uint64)
    s32 = np.uint64(32)
    a_lo, a_hi = a & _MASK32, a >> s32
    b_lo, b_hi = b & _MASK32, b >> s32
    ll = a_lo * b_lo
    lh = a_lo * b_hi
    hl = a_hi * b_lo
    hh = a_hi * b_hi
    # middle column: (ll >> 32) + lo(lh) + lo(hl) < 3 * 2^32, no overflow
    mid = (ll >> s32) + (lh & _MASK32) + (hl & _MASK32)
    return hh + (lh >> s32) + (hl >> s32) + (mid >> s32)


def sample_rows(R, u64):
    """Inverse-CDF draw for each row.

    R:   uint64 [..., V] fixed-point weights (row sums must be > 0)
    u64: uint64 [...]    uniforms
    Returns int64 [...] indices.
    """
    R = np.asarray(R, dtype=np.uint64)
    u64 = np.asarray(u64, dtype=np.uint64)
    cdf = np.cumsum(R, axis=-1, dtype=np.uint64)
    Z = cdf[..., -1]
    if np.any(Z == 0):
        raise ValueError("a row with zero mass cannot be sampled")
    T = mulhi64(u64, Z)
    # smallest v with cdf[v] > T
    return np.argmax(cdf > T[..., None], axis=-1).astype(np.int64)


def sample_row_exact(weights, u64):
    """Scalar reference draw in Python integers (used to pin sample_rows)."""
    R = [int(x) for x in to_fixed(weights)]
    Z = sum(R)
    T = (int(u64) * Z) >> 64
    acc = 0
    for v, r in enumerate(R):
        acc += r
        if acc > T:
            return v
    raise ValueError("a row with zero mass cannot be sampled")
