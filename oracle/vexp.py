"""vexp: the exponential that the sampler policy uses on both sides.

TEST INFRASTRUCTURE ONLY (see oracle/__init__.py).

"Speculative decoding on RDNA" §03 ("how hipfire does it") fixes p as the
AR sampler's distribution, computed on that sampler's pool with its
tie-breaking and summation.
For the GPU and this oracle to produce the same kept set and the same draw
bit for bit, both must evaluate the softmax weights with the same float
operations, so neither side may call its platform's exp.  The pages fix
neither the exp nor the precision of the sampler; the readings taken here:

  * precision: IEEE-754 binary32, rounded to nearest (the kernel's precision;
    every integer the policy decides -- kept counts, draws, accept tests --
    is decided in it on both sides);
  * argument reduction of Cody & Waite ("Software Manual for the Elementary
    Functions", 1980): n = nearest integer (ties to even) to z / ln 2, and
    r = (z - n*C1) - n*C2, where C1 is ln 2 rounded to float32 with its low
    8 significand bits cleared (16 significant bits, so n*C1 is exact for
    |n| < 256) and C2 is the float32 nearest to ln 2 - C1;
  * e**r by its Taylor series to degree 7 (|r| <= ln2/2, truncation error
    below 6e-9, a tenth of a float32 ulp), in Horner form, coefficients the
    float32 values nearest to 1/j!;
  * multiplication by 2**n built exactly from the exponent bits.

Only float32 +, -, x (round to nearest) are used, in the order written
here, each rounded separately (no fused multiply-add).  Valid for z in
[-87, 88]; below -87 the result is 0, so every result is a normal float32.
The policy only calls it with z <= 0.
"""
import numpy as np

F = np.float32

LN2_C1 = np.float32(float.fromhex("0x1.62e4000000000p-1"))    # bits 0x3f317200
LN2_C2 = np.float32(float.fromhex("0x1.7f7d1c0000000p-20"))   # bits 0x35bfbe8e
INV_LN2 = np.float32(float.fromhex("0x1.7154760000000p+0"))   # bits 0x3fb8aa3b
# float32 nearest to 1/j!, j = 0..7
TAYLOR = [np.float32(float.fromhex(h)) for h in (
    "0x1.0000000000000p+0", "0x1.0000000000000p+0", "0x1.0000000000000p-1",
    "0x1.5555560000000p-3", "0x1.5555560000000p-5", "0x1.1111120000000p-7",
    "0x1.6c16c20000000p-10", "0x1.a01a020000000p-13")]
Z_MIN = np.float32(-87.0)
Z_MAX = np.float32(88.0)


def pow2(n):
    """2**n as a float32, from its bit pattern (normal range only)."""
    return np.uint32((int(n) + 127) << 23).view(np.float32)


def vexp(z):
    z = np.float32(z)
    if not (z >= Z_MIN):          # also catches NaN
        return F(0.0)
    if z > Z_MAX:
        return F(np.inf)
    with np.errstate(all="ignore"):
        nf = np.rint(F(z * INV_LN2))          # nearest, ties to even
        r = F(F(z - F(nf * LN2_C1)) - F(nf * LN2_C2))
        p = TAYLOR[7]
        for j in range(6, -1, -1):
            p = F(F(p * r) + TAYLOR[j])
        return F(p * pow2(int(nf)))
