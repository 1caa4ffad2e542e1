"""A numpy model of how libqvg's update kernels form a stored centroid, in fp32: the
members are added with TwoSum compensation (a running sum S and the sum E of the rounding
errors), the mean is the fp32 quotient corrected once by the remainder, and a 16-bit
storage format rounds that mean to nearest even, with the sign of what the fp32 mean leaves
out deciding when the mean sits exactly on a midpoint of two 16-bit values.  It serves the
CPU tests of that rounding rule against the oracle at constructed ties; it is not the
oracle and the library does not use it.

fp32 operations are numpy float32 operations (round to nearest even).  A fused
multiply-add fma(a, b, c) is formed in float64, which is exact for the operands used here
(a product of two fp32 values has at most 48 significant bits, and the sums it enters
cancel to a value well inside fp64's precision)."""
import numpy as np
import torch

f32 = np.float32


def two_sum(a, b):
    s = f32(a + b)
    bb = f32(s - a)
    e = f32(f32(a - f32(s - bb)) + f32(b - bb))
    return s, e


def fma32(a, b, c):
    return f32(float(a) * float(b) + float(c))


def compensated_sum(xs):
    S, E = f32(0.0), f32(0.0)
    for x in np.asarray(xs, dtype=f32):
        S, err = two_sum(S, x)
        E = f32(E + err)
    return S, E


def mean_of(S, E, n):
    n = f32(n)
    q0 = f32(S / n)
    r = f32(fma32(-q0, n, S) + E)
    return f32(q0 + f32(r / n))


def _neighbours(v, fmt):
    """The two values of the format around fp32 v (equal when v is representable) and the
    format's round to nearest even of v."""
    if fmt == 1:
        rn = np.float16(v)
        rnf = float(rn)
        if rnf == float(v):
            return rnf, rnf, rnf
        other = np.nextafter(rn, np.float16(np.inf) if rnf < float(v) else np.float16(-np.inf))
        lo, hi = sorted((rnf, float(other)))
        return lo, hi, rnf
    t = torch.tensor([float(v)], dtype=torch.float32)
    rn = t.to(torch.bfloat16)
    rnf = float(rn.float())
    if rnf == float(v):
        return rnf, rnf, rnf
    step = 1 if (rnf < float(v)) == (rnf >= 0) else -1   # one bit pattern away from zero or towards it
    other = float((rn.view(torch.int16) + step).view(torch.bfloat16).float())
    lo, hi = sorted((rnf, other))
    return lo, hi, rnf


def store_value(v, rem, fmt):
    """The stored value of the exact mean v + rem (v its fp32 mean) in format fmt."""
    if fmt == 0:
        return f32(v)
    lo, hi, rn = _neighbours(v, fmt)
    if lo == hi or float(v) != 0.5 * (lo + hi) or rem == 0:
        return f32(rn)
    return f32(hi if rem > 0 else lo)


def stored_mean(xs, fmt):
    S, E = compensated_sum(xs)
    n = f32(len(xs))
    m = mean_of(S, E, n)
    if fmt == 0:
        return m
    return store_value(m, f32(fma32(-m, n, S) + E), fmt)
