"""Philox4x64-10, written from its published definition.

TEST INFRASTRUCTURE ONLY (see oracle/__init__.py).

Definition: J. K. Salmon, M. A. Moraes, R. O. Dror, D. E. Shaw, "Parallel
random numbers: as easy as 1, 2, 3", SC'11, section 4 (the Philox S-box:
two 64x64->128 multiplies per round, the high halves xored with the other two
counter words and the round key, the key bumped by Weyl constants between
rounds), 10 rounds.

Role in the verify step: "Speculative decoding on RDNA" §03 ("how hipfire
does it"): all of a request's random draws come from a single stream fixed by
the request's seed, so replaying a seed reproduces its tokens.  The pages do
not name the generator; the
reading taken here is a counter-based Philox, keyed by the request seed and
addressed by (position, row, purpose), so each draw is a pure function of
where it is used:

    key     = (seed, 0)
    counter = (position, row, purpose, 0)
    u       = (first output word >> 40) * 2**-24      in [0, 1), a float32

(24 random bits, exactly representable in float32, the precision in which
the policy decides draws and accept tests).

purpose 0 = a draft draw (used by the tests to draw drafts from q),
purpose 1 = the accept uniform of a row, purpose 2 = the emit draw of a row
(residual, bonus or tree-descent draw).
"""
import numpy as np

MASK64 = (1 << 64) - 1
# multipliers and Weyl increments of Philox4x64 (SC'11, table of constants)
PHILOX_M0 = 0xD2E7470EE14C6C93
PHILOX_M1 = 0xCA5A826395121157
PHILOX_W0 = 0x9E3779B97F4A7C15
PHILOX_W1 = 0xBB67AE8584CAA73B
ROUNDS = 10

PURPOSE_DRAFT = 0
PURPOSE_ACCEPT = 1
PURPOSE_EMIT = 2


def philox4x64_10(counter, key):
    """One Philox4x64-10 block: 4 x 64-bit counter words, 2 x 64-bit key words
    -> 4 x 64-bit output words (Python ints)."""
    x0, x1, x2, x3 = (int(c) & MASK64 for c in counter)
    k0, k1 = (int(k) & MASK64 for k in key)
    for rnd in range(ROUNDS):
        if rnd:
            k0 = (k0 + PHILOX_W0) & MASK64
            k1 = (k1 + PHILOX_W1) & MASK64
        p0 = PHILOX_M0 * x0
        p1 = PHILOX_M1 * x2
        hi0, lo0 = p0 >> 64, p0 & MASK64
        hi1, lo1 = p1 >> 64, p1 & MASK64
        x0, x1, x2, x3 = hi1 ^ x1 ^ k0, lo1, hi0 ^ x3 ^ k1, lo0
    return x0, x1, x2, x3


def uniform(seed, position, row, purpose):
    """The float32 uniform in [0, 1) that the window draws at (row, purpose)."""
    w0 = philox4x64_10((position, row, purpose, 0), (seed, 0))[0]
    return np.float32(w0 >> 40) * np.float32(2.0 ** -24)


# ---------------------------------------------------------------------------
# vectorised form (same arithmetic on numpy uint64 arrays), used to draw the
# uniforms of many windows at once in the statistical tests.

_LO32 = np.uint64(0xFFFFFFFF)
_S32 = np.uint64(32)


def _mulhilo64(a, b):
    """Full 64x64 -> 128-bit product of uint64 arrays, as (hi, lo)."""
    a = np.asarray(a, dtype=np.uint64)
    b = np.asarray(b, dtype=np.uint64)
    a_lo, a_hi = a & _LO32, a >> _S32
    b_lo, b_hi = b & _LO32, b >> _S32
    ll = a_lo * b_lo
    lh = a_lo * b_hi
    hl = a_hi * b_lo
    hh = a_hi * b_hi
    mid = (ll >> _S32) + (lh & _LO32) + (hl & _LO32)
    lo = (ll & _LO32) | ((mid & _LO32) << _S32)
    hi = hh + (lh >> _S32) + (hl >> _S32) + (mid >> _S32)
    return hi, lo


def philox4x64_10_array(c0, c1, c2, c3, k0, k1):
    """Philox4x64-10 over broadcastable uint64 arrays."""
    with np.errstate(over="ignore"):
        x0, x1, x2, x3 = (np.asarray(c, dtype=np.uint64) for c in (c0, c1, c2, c3))
        k0 = np.asarray(k0, dtype=np.uint64)
        k1 = np.asarray(k1, dtype=np.uint64)
        m0, m1 = np.uint64(PHILOX_M0), np.uint64(PHILOX_M1)
        w0, w1 = np.uint64(PHILOX_W0), np.uint64(PHILOX_W1)
        for rnd in range(ROUNDS):
            if rnd:
                k0 = k0 + w0
                k1 = k1 + w1
            hi0, lo0 = _mulhilo64(m0, x0)
            hi1, lo1 = _mulhilo64(m1, x2)
            x0, x1, x2, x3 = hi1 ^ x1 ^ k0, lo1, hi0 ^ x3 ^ k1, lo0
    return x0, x1, x2, x3


def uniform_array(seeds, position, row, purpose):
    """uniform() for an array of seeds (same position/row/purpose)."""
    seeds = np.asarray(seeds, dtype=np.uint64)
    z = np.zeros_like(seeds)
    w0 = philox4x64_10_array(z + np.uint64(position), z + np.uint64(row),
                             z + np.uint64(purpose), z, seeds, z)[0]
    return (w0 >> np.uint64(40)).astype(np.float32) * np.float32(2.0 ** -24)
