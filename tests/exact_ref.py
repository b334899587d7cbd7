"""Exact-rational restatement of the W8A8 epilogue, used only to pin the oracle.

Every intermediate is a Python Fraction (exact); each IEEE operation of the
method is modelled as "compute the exact value, then round it once" with a
round-to-nearest-even written from the definition of a binary floating-point
format (precision p, minimum normal exponent emin, maximum exponent emax).
This shares no code or formula with oracle.c, which works on hardware floats.
"""
from __future__ import annotations

import math
import struct
from fractions import Fraction

INF = float("inf")


def round_binary(v: Fraction, p: int, emin: int, emax: int):
    """Nearest value of the binary format (p significand bits), ties to even.
    Returns a Fraction, or +-inf on overflow."""
    if v == 0:
        return Fraction(0)
    sign = -1 if v < 0 else 1
    a = abs(v)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    if Fraction(2) ** e > a:
        e -= 1
    assert Fraction(2) ** e <= a < Fraction(2) ** (e + 1)
    e = max(e, emin)                         # subnormal range keeps emin's spacing
    ulp = Fraction(2) ** (e - p + 1)
    r = round(a / ulp)                       # Fraction.__round__: half to even
    out = r * ulp
    if out >= Fraction(2) ** (emax + 1):
        return -INF if sign < 0 else INF
    return sign * out


def rn_f32(v: Fraction):
    return round_binary(v, 24, -126, 127)


def rn_bf16(v: Fraction):
    return round_binary(v, 8, -126, 127)


def f32_bits(x) -> int:
    return struct.unpack("<I", struct.pack("<f", float(x)))[0]


def bf16_bits(v) -> int:
    """Bit pattern of a value that is exactly a bf16 value (or +-inf)."""
    u = f32_bits(float(v))
    assert u & 0xFFFF == 0, v
    return u >> 16


def bf16_value(b: int) -> Fraction:
    return Fraction(struct.unpack("<f", struct.pack("<I", (int(b) & 0xFFFF) << 16))[0])


def f32_value(x) -> Fraction:
    return Fraction(float(x))


def rne_int(v: Fraction) -> int:
    return round(v)


def quantize_row(vals):
    """vals: Fractions (exact fp32 values).  Returns (codes, scale Fraction)."""
    amax = max((abs(v) for v in vals), default=Fraction(0))
    s = Fraction(1) if amax == 0 else rn_f32(amax / 127)
    codes = []
    for v in vals:
        t = rn_f32(v / s)
        codes.append(max(-127, min(127, rne_int(t))))
    return codes, s


def linear(q_rows, s_a, w_rows, s_w):
    """y[m][n] as bf16 bit patterns, from exact integer sums and single roundings."""
    out = []
    for m, qa in enumerate(q_rows):
        row = []
        for n, wr in enumerate(w_rows):
            acc = sum(int(a) * int(b) for a, b in zip(qa, wr))
            assert abs(acc) < 2 ** 31
            f0 = rn_f32(Fraction(acc))
            f1 = rn_f32(f0 * s_a[m])
            f2 = rn_f32(f1 * s_w[n])
            row.append(bf16_bits(rn_bf16(f2)))
        out.append(row)
    return out


def nearest_pow2_log(s: float) -> float:
    """Brute force: the power of two 2^j minimising |log2(s) - j| (math.log2)."""
    l2 = math.log2(s)
    best = None
    for j in range(math.floor(l2) - 1, math.floor(l2) + 3):
        d = abs(l2 - j)
        if best is None or d < best[0]:
            best = (d, j)
    return 2.0 ** best[1]


def _is_neg_zero_bits(b: int) -> bool:
    return (int(b) & 0xFFFF) == 0x8000


def _bits_of(v: Fraction, neg_zero: bool) -> int:
    if v == 0:
        return 0x8000 if neg_zero else 0x0000
    return bf16_bits(v)


def residual_rescale_row(h_bits, y_bits):
    """Exact restatement of the residual step on one row of bf16 patterns.

    t = bf16 of the exact sum h + y (one rounding); e = floor(log2 max|t|)
    (0 for an all-zero row); result = bf16 of the exact t * 2^-e.  Signed
    zeros follow IEEE: an exact-zero sum is +0 unless both addends are -0; a
    nonzero value that rounds to zero keeps its sign."""
    t = []
    for hb, yb in zip(h_bits, y_bits):
        hv, yv = bf16_value(hb), bf16_value(yb)
        s = hv + yv
        if s == 0:
            t.append((Fraction(0), _is_neg_zero_bits(hb) and _is_neg_zero_bits(yb)))
        else:
            r = rn_bf16(s)
            t.append((r, r == 0 and s < 0))
    amax = max(abs(v) for v, _ in t)
    if amax == 0:
        e = 0
    else:
        e = amax.numerator.bit_length() - amax.denominator.bit_length()
        if Fraction(2) ** e > amax:
            e -= 1
    out = []
    for v, nz in t:
        if v == 0:
            out.append(_bits_of(Fraction(0), nz))
            continue
        r = rn_bf16(v * Fraction(2) ** (-e))
        out.append(_bits_of(r, v < 0))
    return out


def relu_mul_row(g_bits, u_bits):
    """bf16 of the exact relu(g) * u per element (relu(g) = g if g > 0 else +0)."""
    out = []
    for gb, ub in zip(g_bits, u_bits):
        g, u = bf16_value(gb), bf16_value(ub)
        u_neg = (int(ub) & 0x8000) != 0
        gr = g if g > 0 else Fraction(0)
        p = gr * u
        if p == 0:
            out.append(0x8000 if u_neg else 0x0000)   # +0 * u carries u's sign
            continue
        r = rn_bf16(p)
        out.append(_bits_of(r, p < 0))
    return out


def argmax_bf16(row_bits):
    """Lowest index of the largest bf16 value (-0 == +0)."""
    best, bv = 0, bf16_value(row_bits[0])
    for n in range(1, len(row_bits)):
        v = bf16_value(row_bits[n])
        if v > bv:
            best, bv = n, v
    return best
