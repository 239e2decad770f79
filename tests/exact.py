"""Exact rational / high-precision helpers used to pin the oracle.

Nothing here imports the oracle or the CUDA path: values are computed from
fractions.Fraction (exact) or decimal.Decimal (50 digits) and rounded to
binary32 by an independent round-to-nearest-even routine.
"""
from decimal import Decimal, getcontext
from fractions import Fraction

import numpy as np

getcontext().prec = 50


def f32_bits(x):
    return int(np.asarray(x, dtype=np.float32).view(np.uint32))


def bits_f32(u):
    return float(np.array([u], dtype=np.uint32).view(np.float32)[0])


def _floor_log2(a):
    """floor(log2(a)) for a positive Fraction."""
    e = a.numerator.bit_length() - a.denominator.bit_length()
    if Fraction(2) ** e > a:
        e -= 1
    elif Fraction(2) ** (e + 1) <= a:
        e += 1
    return e


def rn32(x):
    """Round an exact rational to binary32, nearest, ties to even.

    Returns (value as Python float, distance of x from the nearest rounding
    midpoint relative to |x|); the distance lets a caller tell apart the few
    results that sit too close to a midpoint for an FP64 evaluation to decide.
    """
    x = Fraction(x)
    if x == 0:
        return 0.0, Fraction(1)
    s = -1 if x < 0 else 1
    a = abs(x)
    e = _floor_log2(a)
    q = Fraction(2) ** (max(e, -126) - 23)
    n = a / q
    fl = n.numerator // n.denominator
    rem = n - fl
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and fl % 2 == 1):
        fl += 1
    mid_dist = abs(rem - Fraction(1, 2)) * q / a
    return float(s * fl * q), mid_dist


def rn32_bits(x):
    v, d = rn32(x)
    return f32_bits(np.float32(v)), d


def rne_bf16_bits_from_f32(f):
    """bf16 bits of an FP32 value by exact comparison with the two neighbours."""
    f = np.float32(f)
    u = f32_bits(f)
    lo = u & 0xFFFF0000
    x = Fraction(float(f))
    a = Fraction(bits_f32(lo))
    b = Fraction(bits_f32(lo + 0x10000)) if (lo & 0x7FFFFFFF) != 0x7F7F0000 else None
    if u & 0xFFFF == 0:
        return lo >> 16
    da, db = abs(x - a), abs(b - x)
    if da < db:
        return lo >> 16
    if db < da:
        return (lo + 0x10000) >> 16
    return (lo >> 16) if ((lo >> 16) & 1) == 0 else ((lo + 0x10000) >> 16)


def F(x):
    """Exact rational value of a float (double) or numpy float."""
    return Fraction(float(x))


def adam_bound(t, b1, b2):
    """Cauchy-Schwarz bound on |m_hat / sqrt(v_hat)| after t steps from m=v=0:
    m_t = (1-b1) sum_k b1^k g_{t-k}, v_t = (1-b2) sum_k b2^k g_{t-k}^2, so
    |m_hat/sqrt(v_hat)| <= (1-b1)/(1-b1^t) * sqrt(sum_{k<t} (b1^2/b2)^k) * sqrt((1-b2^t)/(1-b2))."""
    s = sum((b1 * b1 / b2) ** k for k in range(t))
    return (1 - b1) / (1 - b1 ** t) * (s ** 0.5) * (((1 - b2 ** t) / (1 - b2)) ** 0.5)


def D(x):
    return Decimal(Fraction(float(x)).numerator) / Decimal(Fraction(float(x)).denominator)


def dec_to_frac(d):
    return Fraction(d)
