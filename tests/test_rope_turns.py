"""The float32 RoPE angle reduction of the absorbed-query kernel, emulated on
the host, stays within its stated bound of the exact angle.

The kernel forms cos/sin of pos * inv_freq (the rope helper of the
iotdigitaltwinplm.com listing, theta = 10000, d_r = 64) for positions below
2^24 in float32 "turns": with f_hi + f_lo the float32 head and tail of
inv_freq / (2 pi),
    n = rint(fl(p * f_hi)),  t = fma(p, f_hi, -n),  t = fma(p, f_lo, t),
and the angle is 2 pi t.  A float32 FMA is emulated exactly here: the product
of two float32 values is exact in float64, and one rounding of the exact sum
to float32 is what the FMA does.  The reference is the exact angle reduced in
extended precision (Python integers and fractions of the float64 inputs).
"""
from fractions import Fraction

import numpy as np

THETA = 10000.0
D_R = 64


def f32(x):
    return np.float32(x)


def round_f32(x: Fraction) -> np.float32:
    """The float32 nearest to the rational x (ties to even): one rounding."""
    f = np.float32(float(x))          # within one float32 step of the answer
    cands = [np.nextafter(f, np.float32(-np.inf)), f, np.nextafter(f, np.float32(np.inf))]
    best = min(cands, key=lambda c: (abs(Fraction(float(c)) - x),
                                     int(np.float32(c).view(np.uint32)) & 1))
    return np.float32(best)


def fma32(a, b, c):
    """float32 fma(a, b, c): exact a * b + c, rounded once to float32."""
    return round_f32(Fraction(float(a)) * Fraction(float(b)) + Fraction(float(c)))


def turns_f32(pos: int, inv_freq: float) -> float:
    turns = inv_freq / (2.0 * np.pi)
    f_hi = f32(turns)
    f_lo = f32(turns - float(f_hi))
    p = f32(pos)
    n = np.rint(f32(p * f_hi))
    t = fma32(p, f_hi, -n)
    t = fma32(p, f_lo, t)
    return float(t)


def exact_turns(pos: int, inv_freq: float) -> float:
    """pos * inv_freq / (2 pi), reduced to (-1/2, 1/2], in extended precision
    (inv_freq is the float64 the host forms; 2 pi to 40 digits)."""
    two_pi = Fraction("6.283185307179586476925286766559005768394")
    x = Fraction(pos) * Fraction(inv_freq) / two_pi
    frac = x - round(x)
    return float(frac)


def test_turns_reduction_is_within_its_bound():
    rng = np.random.default_rng(7224)
    inv = [THETA ** (-2.0 * i / D_R) for i in range(D_R // 2)]
    positions = [0, 1, 2, 63, 64, 4095, 8191, 131071, (1 << 24) - 1]
    positions += [int(v) for v in rng.integers(0, 1 << 24, size=40)]
    bound = 2.0 ** -23            # turns: the angle error is below 2 pi * 2^-23
    worst = 0.0
    for pos in positions:
        for f in inv:
            got, ref = turns_f32(pos, f), exact_turns(pos, f)
            d = abs(got - ref)
            d = min(d, abs(d - 1.0))                  # a whole turn apart is the same angle
            worst = max(worst, d)
            assert d < bound, (pos, f, got, ref)
    assert worst > 0.0                                # the check exercised rounding


def test_turns_reduction_leaves_small_angles_exact_enough():
    # position 1: the angle is inv_freq itself (up to the float32 head/tail split)
    for i in range(D_R // 2):
        f = THETA ** (-2.0 * i / D_R)
        assert abs(turns_f32(1, f) * 2.0 * np.pi - (f if f < np.pi else f - 2.0 * np.pi)) < 1e-6
