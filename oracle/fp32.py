"""Single-precision steps the pages fix, written out exactly (oracle; test infrastructure only).

The sampled-drafting and verification commits of openvino.genai PR #4847 ("Add DSpark
and DFlash v2 drafts and sampled drafting to DFlash speculative decoding") compute
softmax weights with a single-precision exponential of float logits, flush exponents
below -64 to zero (commit on the thresholded TopPFilter), and sum the weights in double
(commit on double-precision multinomial sums). A drawn token is an integer decided by
those float weights, so the oracle and the kernels must evaluate the very same
single-precision function. It is defined here, not borrowed from a libm:

    weight(d) = 0                                   if d < -64
              = 2^n * P(f)                          otherwise, where
    t = fl32(d * LOG2E),  n = rint(t),  f = t - n   (exact),
    P(f) = Horner form of sum_{k<=7} (ln 2)^k f^k / k!  with correctly rounded fp32 FMAs.

This is the Taylor expansion of 2^f = e^(f ln 2) after the usual reduction to
|f| <= 1/2; the coefficients are (ln 2)^k / k! rounded to float32. Every operation
is one IEEE-754 correctly rounded float32 operation, so any conforming machine gets
the same bits.

numpy has no float32 FMA, so ``fma32`` emulates one exactly: the product of two
float32 values is exact in double, the double sum is corrected with its exact
TwoSum error where it lands on a float32 rounding midpoint.
"""
from __future__ import annotations

import math

import numpy as np

F32 = np.float32
F64 = np.float64

LOG2E = F32(1.0 / math.log(2.0))
FLUSH = F32(-64.0)
# Taylor coefficients of 2^f: (ln 2)^k / k!, k = 0..7, rounded to float32
EXP2_COEF = [F32(math.log(2.0) ** k / math.factorial(k)) for k in range(8)]


def f32(x) -> np.ndarray:
    return np.asarray(x, dtype=F32)


def fma32(a, b, c) -> np.ndarray:
    """Correctly rounded float32 a*b + c, elementwise."""
    a64 = np.asarray(a, dtype=F32).astype(F64)
    b64 = np.asarray(b, dtype=F32).astype(F64)
    c64 = np.asarray(c, dtype=F32).astype(F64)
    p = a64 * b64                       # exact: 24-bit x 24-bit significands fit in 53 bits
    with np.errstate(invalid="ignore", over="ignore"):
        s = p + c64                     # nearest double to the exact sum
        bb = s - p                      # TwoSum: s + e == p + c exactly
        e = (p - (s - bb)) + (c64 - bb)
        r = s.astype(F32)               # nearest-even float32 of s
    r64 = r.astype(F64)
    # the float32 neighbour of r on the side of s; s can only mislead the rounding
    # when it is exactly the midpoint between r and that neighbour
    up = np.nextafter(r, F32(np.inf))
    dn = np.nextafter(r, F32(-np.inf))
    other = np.where(s > r64, up, dn)
    mid = (r64 + other.astype(F64)) * 0.5
    fix = (s == mid) & (e != 0) & (s != r64)
    hi = np.maximum(r, other)
    lo = np.minimum(r, other)
    out = np.where(fix, np.where(e > 0, hi, lo), r)
    return np.asarray(out, dtype=F32)


def exp2_poly(f) -> np.ndarray:
    """P(f) ~ 2^f for |f| <= 1/2: Horner with float32 FMAs, highest degree first."""
    f = f32(f)
    p = np.full(f.shape, EXP2_COEF[7], dtype=F32)
    for k in range(6, -1, -1):
        p = fma32(p, f, EXP2_COEF[k])
    return p


def weight(d) -> np.ndarray:
    """Unnormalised softmax weight of an exponent d = z - zmax <= 0 (float32)."""
    d = f32(d)
    keep = d >= FLUSH
    dd = np.where(keep, d, F32(0.0)).astype(F32)
    t = (dd * LOG2E).astype(F32)
    n = np.rint(t).astype(F32)          # round half to even
    f = (t - n).astype(F32)             # exact
    p = exp2_poly(f)
    w = np.ldexp(p, n.astype(np.int32)).astype(F32)   # exact power-of-two scaling (normal range)
    return np.where(keep, w, F32(0.0)).astype(F32)
