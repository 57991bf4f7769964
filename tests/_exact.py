"""Exact-arithmetic helpers for the oracle pins: the correctly rounded fp32
value of a rational, and inputs placed next to rounding decision points.

Pure Python (fractions) and numpy scalars; no quantized arithmetic of the
library or of the oracle is restated here -- these are the IEEE-754 rules the
pins evaluate against."""
from __future__ import annotations

from fractions import Fraction

import numpy as np


def fl32(fr: Fraction) -> np.float32:
    """Correctly rounded (nearest, ties to even) fp32 value of an exact rational."""
    fr = Fraction(fr)
    c = np.float32(float(fr))
    cands = [np.nextafter(c, np.float32(-np.inf)), c, np.nextafter(c, np.float32(np.inf))]
    best, bd = None, None
    for x in cands:
        if not np.isfinite(x):
            continue
        d = abs(Fraction(float(x)) - fr)
        if bd is None or d < bd or (d == bd and (int(np.float32(x).view(np.uint32)) & 1) == 0):
            best, bd = x, d
    return np.float32(best)


def F(x) -> Fraction:
    """The exact rational value of an fp32 / fp64 number."""
    return Fraction(float(x))


def step_ulps(x, j: int) -> np.float32:
    """x moved by j units in the last place (fp32)."""
    x = np.float32(x)
    for _ in range(abs(j)):
        x = np.nextafter(x, np.float32(np.inf if j > 0 else -np.inf))
    return np.float32(x)


def near_half_inputs(s, ks, ulps: int = 3) -> np.ndarray:
    """fp32 inputs x within `ulps` units in the last place of (k + 1/2) * s for
    each k in ks: quotients x / s that sit on, or a few roundings away from, a
    rounding decision point."""
    S = F(s)
    xs = []
    for k in ks:
        x0 = fl32(Fraction(2 * k + 1, 2) * S)
        xs.extend(step_ulps(x0, j) for j in range(-ulps, ulps + 1))
    return np.array(xs, np.float32)


def round_half_away(v: Fraction) -> int:
    """Round to nearest, ties away from zero (C's round(); not the library's rule)."""
    a = abs(v)
    r = (a.numerator * 2 + a.denominator) // (2 * a.denominator)
    return r if v >= 0 else -r
