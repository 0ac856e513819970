"""vexp: the exponential that the sampler policy uses on both sides.

TEST INFRASTRUCTURE ONLY (see oracle/__init__.py).

"Speculative decoding on RDNA" §03 ("how hipfire does it") fixes that p is
the AR sampler's distribution with the same pool, tie order and summation.
For the GPU and this oracle to produce the same kept set and the same draw
bit for bit, both must evaluate the softmax weights with the same double
operations, so neither side may call its platform's exp.  The pages name no
exp; the reading taken here is a textbook one:

  * argument reduction of Cody & Waite ("Software Manual for the Elementary
    Functions", 1980): n = nearest integer (ties to even) to z / ln 2, and
    r = (z - n*C1) - n*C2, where C1 is ln 2 with the low 32 bits of its
    significand cleared (so n*C1 is exact for |n| < 2**32) and C2 is the
    double nearest to ln 2 - C1;
  * e**r by its Taylor series to degree 13 (|r| <= ln2/2, truncation error
    below 5e-18), in Horner form, coefficients 1/j! rounded to nearest;
  * multiplication by 2**n built exactly from the exponent bits.

Only IEEE-754 double +, -, x (round to nearest) are used, in the order
written here; Python evaluates each one separately (no fused multiply-add).
Valid for z in [-708, 709]; below -708 the result is 0 (the policy only ever
calls it with z <= 0).
"""
import struct

# C1 = ln 2 with the low 32 significand bits cleared; C2 = nearest(ln 2 - C1).
LN2_C1 = float.fromhex("0x1.62e4200000000p-1")
LN2_C2 = float.fromhex("0x1.fdf473de6af28p-22")
INV_LN2 = float.fromhex("0x1.71547652b82fep+0")   # nearest double to 1/ln 2
# 1/j! for j = 0..13, each rounded to the nearest double
TAYLOR = [float.fromhex(h) for h in (
    "0x1.0000000000000p+0", "0x1.0000000000000p+0", "0x1.0000000000000p-1",
    "0x1.5555555555555p-3", "0x1.5555555555555p-5", "0x1.1111111111111p-7",
    "0x1.6c16c16c16c17p-10", "0x1.a01a01a01a01ap-13", "0x1.a01a01a01a01ap-16",
    "0x1.71de3a556c734p-19", "0x1.27e4fb7789f5cp-22", "0x1.ae64567f544e4p-26",
    "0x1.1eed8eff8d898p-29", "0x1.6124613a86d09p-33")]
Z_MIN = -708.0
Z_MAX = 709.0


def pow2(n):
    """2**n as a double, from its bit pattern (normal range only)."""
    return struct.unpack("<d", struct.pack("<Q", (n + 1023) << 52))[0]


def vexp(z):
    z = float(z)
    if not (z >= Z_MIN):          # also catches NaN
        return 0.0
    if z > Z_MAX:
        return float("inf")
    n = round(z * INV_LN2)        # Python rounds half to even
    nf = float(n)
    r = (z - nf * LN2_C1) - nf * LN2_C2
    p = TAYLOR[13]
    for j in range(12, -1, -1):
        p = p * r + TAYLOR[j]
    return p * pow2(n)
