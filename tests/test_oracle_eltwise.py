"""Pins of the oracle's standalone quantized elementwise ops and dynamic
per-row quantization.

Sources: "【量化】神经网络量化介绍" (loveleaves.github.io/p/quantization), sections
量化乘法, 量化加法, 量化激活函数 (the ops) and 量化参数选择 (最大值截断: the scale
is the largest magnitude over 127).  Pins: exact rational arithmetic (Python
Fractions) for the rescale, the page's closed forms (shared scale with M = 1;
the power-of-two "shift" variant), passivity of ReLU, and the defining
properties of the dynamic scale (the largest code is 127; every dequantized
value lies within half a step of its input).
"""
from fractions import Fraction

import numpy as np
import pytest

from _exact import F, fl32, near_half_inputs, round_half_away

pytestmark = pytest.mark.cpu


def _round_half_even(fr: Fraction) -> int:
    f = fr.numerator // fr.denominator
    rem = fr - f
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and f % 2 == 1):
        f += 1
    return f


def test_mul_matches_exact_rescale(oracle):
    """MUL = clip(round(a b M)); the fp32 product may only differ from the exact
    rational rounding where a b M lies within fp32 rounding of a half-way point."""
    rng = np.random.default_rng(1)
    a = rng.integers(-128, 128, 4000)
    b = rng.integers(-128, 128, 4000)
    for M in (0.0123, 1.0 / 96.0, 0.5):
        Mf = Fraction(float(np.float32(M)))
        got = oracle.eltwise_s8("mul", a, b, M)
        for ai, bi, g in zip(a.tolist(), b.tolist(), got.tolist()):
            exact = Fraction(ai * bi) * Mf
            want = max(-128, min(127, _round_half_even(exact)))
            frac = exact - (exact.numerator // exact.denominator)
            near_tie = abs(frac - Fraction(1, 2)) <= abs(exact) * Fraction(1, 2 ** 23)
            assert g == want or near_tie, (ai, bi, M, g, want)


def test_shift_variant_is_exact(oracle):
    """M = 2^-k (the page's integer variant: a shift by round(log2 scale_abc)):
    out = clip(round(a b / 2^k)) exactly, ties to even."""
    a = np.arange(-128, 128).repeat(256)
    b = np.tile(np.arange(-128, 128), 256)
    for k in (0, 3, 7, 10):
        got = oracle.eltwise_s8("mul", a, b, 2.0 ** -k)
        want = [max(-128, min(127, _round_half_even(Fraction(int(x) * int(y), 2 ** k)))) for x, y in zip(a, b)]
        assert got.tolist() == want


def test_add_shared_scale(oracle):
    """With the output scale equal to the shared input scale (M = 1) ADD is the
    saturating integer sum; with M = 1/2, round((a + b) / 2), ties to even."""
    a = np.arange(-128, 128).repeat(256)
    b = np.tile(np.arange(-128, 128), 256)
    assert np.array_equal(oracle.eltwise_s8("add", a, b, 1.0), np.clip(a + b, -128, 127))
    want = [_round_half_even(Fraction(int(x) + int(y), 2)) for x, y in zip(a, b)]
    assert oracle.eltwise_s8("add", a, b, 0.5).tolist() == want


def test_relu_is_passive(oracle):
    """ReLU keeps the scale: max(a, 0), no rounding; relu after ADD / MUL clamps at 0."""
    a = np.arange(-128, 128)
    assert np.array_equal(oracle.eltwise_s8("relu", a), np.maximum(a, 0))
    b = np.full_like(a, 3)
    assert np.array_equal(oracle.eltwise_s8("add", a, b, 1.0, relu=True), np.clip(a + 3, 0, 127))


def test_dynamic_quantize_properties(oracle):
    """s = max|x| / 127: the largest magnitude maps to +-127, every |q s - x| is at
    most half a step (plus fp32 slack), zero rows give zero codes and scale 0."""
    rng = np.random.default_rng(2)
    x = (rng.standard_normal((64, 300)) * rng.uniform(0.01, 10.0, (64, 1))).astype(np.float32)
    x[5] = 0.0
    x[7, 11] = -50.0
    for narrow in (False, True):
        q, s = oracle.quantize_rows_dynamic(x, narrow)
        assert s[5] == 0.0 and np.all(q[5] == 0)
        live = np.arange(64) != 5
        assert np.all(np.abs(q[live]).max(axis=1) == 127)
        assert q.min() >= (-127 if narrow else -128) and q.max() <= 127
        err = np.abs(q[live] * s[live, None].astype(np.float64) - x[live])
        assert np.all(err <= s[live, None] * (0.5 + 1e-5))
        amax = np.abs(x).max(axis=1)
        assert np.all(s == (amax / np.float32(127.0)).astype(np.float32))
        assert q[7, 11] == -127


def _dynamic_rows(rng):
    """Rows whose largest magnitude A fixes s = fl32(A / 127), the other entries
    placed a few ulps either side of (k + 1/2) s; rows with A = 127 * 2^e make s a
    power of two, so x / s is exact and (k + 1/2) s is an exact tie."""
    rows = []
    for i, A in enumerate([127.0, -127.0 * 2.0 ** -5, 3.7, 0.61, -11.3, 127.0 * 4.0, 1e-3]):
        A = np.float32(A)
        s = fl32(F(abs(A)) / 127)
        body = near_half_inputs(s, range(-127, 126, 3), ulps=2)
        body = body[np.abs(body) < abs(A)]
        row = np.concatenate([[A], body, rng.permutation(body)[:40]]).astype(np.float32)
        rows.append(rng.permutation(row))
    n = max(len(r) for r in rows)
    return np.stack([np.pad(r, (0, n - len(r))) for r in rows]).astype(np.float32)


@pytest.mark.parametrize("narrow", [False, True])
def test_dynamic_quantize_exact(oracle, narrow):
    """Quantization intro, 量化参数选择 (最大值截断) and 量化算子: the row scale is the
    correctly rounded quotient max|x| / 127, and each code is round half to even
    of the correctly rounded quotient x / s, clipped.  Inputs sit next to and on
    rounding decision points, so multiplying by a rounded reciprocal of s, or
    rounding ties away from zero, gives other codes (both are asserted present)."""
    rng = np.random.default_rng(5)
    x = _dynamic_rows(rng)
    q, s = oracle.quantize_rows_dynamic(x, narrow)
    qmin = -127 if narrow else -128
    recip_differs = away_differs = 0
    for r in range(x.shape[0]):
        amax = max(abs(F(v)) for v in x[r])
        sr = fl32(amax / 127)
        assert s[r] == sr, (r, s[r], sr)
        inv = F(fl32(1 / F(sr)))
        for c in range(x.shape[1]):
            t = F(fl32(F(x[r, c]) / F(sr)))
            want = max(qmin, min(127, _round_half_even(t)))
            assert q[r, c] == want, (r, c, float(x[r, c]), int(q[r, c]), want)
            tr = F(fl32(F(x[r, c]) * inv))
            recip_differs += max(qmin, min(127, _round_half_even(tr))) != want
            away_differs += max(qmin, min(127, round_half_away(t))) != want
    assert recip_differs > 0 and away_differs > 0


def test_eltwise_errors(oracle):
    with pytest.raises(KeyError):
        oracle.eltwise_s8("sub", np.zeros(4))
