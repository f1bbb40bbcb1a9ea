"""Philox4x32-10 and the uniforms the verify step draws (oracle; test infrastructure only).

Definition: Salmon, Moraes, Dror and Shaw, "Parallel Random Numbers: As Easy as 1, 2, 3"
(SC'11), section 3.3. One round maps a 4-word counter with a 2-word key:

    (hi0, lo0) = M0 * x0          (full 64-bit product split into 32-bit halves)
    (hi1, lo1) = M1 * x2
    x' = (hi1 ^ x1 ^ k0,  lo1,  hi0 ^ x3 ^ k1,  lo0)

with multipliers M0 = 0xD2511F53, M1 = 0xCD9E8D57 (Table 2) and, between rounds, the Weyl key
schedule k0 += 0x9E3779B9, k1 += 0xBB67AE85 (mod 2^32). Philox4x32-10 runs ten rounds.

How the verify step uses it (the pages ask for "deterministic seeded sampling", DS4Server issue
#98, *Verification*; the layout below is this project's own choice):

    key     = (seed mod 2^32, seed >> 32)
    counter = (pos mod 2^32, pos >> 32, 0, purpose)
    u       = (word0 >> 8) * 2^-24          -- 24-bit uniform on [0, 1 - 2^-24]

``pos`` is the absolute sequence position the draw decides, ``purpose`` separates the draws
made for one position (draft sample, ratio test, residual sample, bonus sample). A 24-bit
uniform is exactly representable in float32 and float64, so both sides see the same number.

Pinned by the Random123 known-answer vectors (tests/golden/philox4x32_10_kat.txt) and by a
chi-square uniformity test of the 24-bit uniforms.
"""

import numpy as np

MASK32 = 0xFFFFFFFF
PHILOX_M0 = 0xD2511F53
PHILOX_M1 = 0xCD9E8D57
PHILOX_W0 = 0x9E3779B9
PHILOX_W1 = 0xBB67AE85
ROUNDS = 10

PURPOSE_DRAFT = 1
PURPOSE_ACCEPT = 2
PURPOSE_RESIDUAL = 3
PURPOSE_BONUS = 4


def philox4x32_10(counter, key):
    """One Philox4x32-10 block: 4 counter words, 2 key words -> 4 output words (Python ints)."""
    x0, x1, x2, x3 = (int(c) & MASK32 for c in counter)
    k0, k1 = (int(k) & MASK32 for k in key)
    for rnd in range(ROUNDS):
        if rnd > 0:
            k0 = (k0 + PHILOX_W0) & MASK32
            k1 = (k1 + PHILOX_W1) & MASK32
        p0 = PHILOX_M0 * x0
        p1 = PHILOX_M1 * x2
        hi0, lo0 = p0 >> 32, p0 & MASK32
        hi1, lo1 = p1 >> 32, p1 & MASK32
        x0, x1, x2, x3 = hi1 ^ x1 ^ k0, lo1, hi0 ^ x3 ^ k1, lo0
    return x0, x1, x2, x3


def philox4x32_10_np(c0, c1, c2, c3, k0, k1):
    """Vectorised Philox4x32-10 over numpy arrays (broadcast); same rounds as ``philox4x32_10``."""
    x = [np.asarray(c, dtype=np.uint64) & MASK32 for c in (c0, c1, c2, c3)]
    k0 = np.asarray(k0, dtype=np.uint64) & MASK32
    k1 = np.asarray(k1, dtype=np.uint64) & MASK32
    x0, x1, x2, x3 = np.broadcast_arrays(*x)
    x0, x1, x2, x3 = (a.copy() for a in (x0, x1, x2, x3))
    m0 = np.uint64(PHILOX_M0)
    m1 = np.uint64(PHILOX_M1)
    mask = np.uint64(MASK32)
    sh = np.uint64(32)
    for rnd in range(ROUNDS):
        if rnd > 0:
            k0 = (k0 + np.uint64(PHILOX_W0)) & mask
            k1 = (k1 + np.uint64(PHILOX_W1)) & mask
        p0 = m0 * x0  # < 2^64, exact in uint64
        p1 = m1 * x2
        hi0, lo0 = p0 >> sh, p0 & mask
        hi1, lo1 = p1 >> sh, p1 & mask
        x0, x1, x2, x3 = hi1 ^ x1 ^ k0, lo1, hi0 ^ x3 ^ k1, lo0
    return x0, x1, x2, x3


def uniform(seed, pos, purpose):
    """The 24-bit uniform for (seed, absolute position, purpose), as a Python float."""
    seed = int(seed)
    pos = int(pos)
    w0, _, _, _ = philox4x32_10(
        (pos & MASK32, (pos >> 32) & MASK32, 0, int(purpose)),
        (seed & MASK32, (seed >> 32) & MASK32),
    )
    return (w0 >> 8) * 2.0 ** -24


def uniform_np(seed, pos, purpose):
    """Vectorised ``uniform`` (seed, pos, purpose broadcast); returns float64 array."""
    seed = np.asarray(seed, dtype=np.uint64)
    pos = np.asarray(pos, dtype=np.uint64)
    purpose = np.asarray(purpose, dtype=np.uint64)
    w0, _, _, _ = philox4x32_10_np(
        pos & np.uint64(MASK32), pos >> np.uint64(32), np.zeros_like(pos), purpose,
        seed & np.uint64(MASK32), seed >> np.uint64(32),
    )
    return (w0 >> np.uint64(8)).astype(np.float64) * 2.0 ** -24


def make_uniform_source(seed):
    """A callable (pos, purpose) -> u bound to one request's seed (what ``accept`` consumes)."""
    return lambda pos, purpose: uniform(seed, pos, purpose)
