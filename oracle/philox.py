"""Philox-4x32-10, written from its published definition.

Test infrastructure only (see the package docstring).

Definition (Salmon et al., SC'11, "Parallel random numbers: as easy as
1, 2, 3", section on the Philox family): a 128-bit counter (c0, c1, c2, c3)
and a 64-bit key (k0, k1).  One round computes the two 32x32->64 products
M0*c0 and M1*c2 and sets

    (c0, c1, c2, c3) <- (hi(M1*c2) ^ c1 ^ k0,  lo(M1*c2),
                          hi(M0*c0) ^ c3 ^ k1,  lo(M0*c0)),

after which the key is bumped by the Weyl constants (W0, W1).  Ten rounds.

How the uniforms are taken from one output block (w0..w3) is a
convention of this library and its oracle; the pages name no generator:

    counter = (step_lo, step_hi, position, purpose), key = (seed_lo, seed_hi)
    purpose 0: the drafter's draw y ~ q;  1: the accept test;  2: the
    residual / bonus draw.
    u24 = w0 >> 8                 (accept test: u = u24 * 2^-24)
    u64 = (w1 << 32) | w2         (inverse-CDF draws)
"""

import numpy as np

M0 = 0xD2511F53
M1 = 0xCD9E8D57
W0 = 0x9E3779B9
W1 = 0xBB67AE85
MASK32 = np.uint64(0xFFFFFFFF)

PURPOSE_DRAFT = 0
PURPOSE_ACCEPT = 1
PURPOSE_RESIDUAL = 2


def philox4x32_10(ctr, key):
    """Vectorised Philox-4x32-10.

    ctr: integer array [..., 4] (each entry < 2^32); key: integer array [..., 2].
    Returns a uint64 array [..., 4] whose entries are the 32-bit outputs.
    """
    ctr = np.asarray(ctr, dtype=np.uint64)
    key = np.asarray(key, dtype=np.uint64)
    c0, c1, c2, c3 = (ctr[..., i] & MASK32 for i in range(4))
    k0 = key[..., 0] & MASK32
    k1 = key[..., 1] & MASK32
    m0 = np.uint64(M0)
    m1 = np.uint64(M1)
    for _ in range(10):
        p0 = m0 * c0          # < 2^64: exact in uint64
        p1 = m1 * c2
        hi0, lo0 = p0 >> np.uint64(32), p0 & MASK32
        hi1, lo1 = p1 >> np.uint64(32), p1 & MASK32
        c0, c1, c2, c3 = hi1 ^ c1 ^ k0, lo1, hi0 ^ c3 ^ k1, lo0
        k0 = (k0 + np.uint64(W0)) & MASK32
        k1 = (k1 + np.uint64(W1)) & MASK32
    return np.stack([c0, c1, c2, c3], axis=-1)


def block(seed, step, position, purpose):
    """Philox output for (seed, step, position, purpose); broadcasts."""
    seed = np.asarray(seed, dtype=np.uint64)
    step = np.asarray(step, dtype=np.uint64)
    position = np.asarray(position, dtype=np.uint64)
    purpose = np.asarray(purpose, dtype=np.uint64)
    seed, step, position, purpose = np.broadcast_arrays(seed, step, position, purpose)
    ctr = np.stack([step & MASK32, step >> np.uint64(32), position, purpose], axis=-1)
    key = np.stack([seed & MASK32, seed >> np.uint64(32)], axis=-1)
    return philox4x32_10(ctr, key)


def uniform24(seed, step, position, purpose):
    """24-bit integer u24 in [0, 2^24); the uniform is u24 * 2^-24."""
    w = block(seed, step, position, purpose)
    return w[..., 0] >> np.uint64(8)


def uniform64(seed, step, position, purpose):
    """64-bit integer uniform (w1 << 32) | w2 in [0, 2^64)."""
    w = block(seed, step, position, purpose)
    return (w[..., 1] << np.uint64(32)) | w[..., 2]
