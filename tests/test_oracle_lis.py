"""Pins of the oracle's Log-Int-Softmax and bit-shift attention product.

Source: "首个完全量化Vision Transformer的方法FQ-ViT" (aijishu.com), section 3.3
(Attention Map 的 Log2 量化; Softmax 的量化推理; Integer-only 推理; Softmax 的量化的实现).
The pins are hand-worked values (tests/golden/lis_worked_example.txt), the real
exponential and softmax the method approximates, an independent definition of
log_round (the nearest power of two), closed forms for equal rows, and the
float64 product of the dequantized attention map with V.
"""
import math
import os

import numpy as np
import pytest

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
pytestmark = pytest.mark.cpu


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return [ln.split() for ln in (l.strip() for l in f) if ln and not ln.startswith("#")]


def test_lis_golden_constants_and_exponentials(oracle):
    """Hand-worked constants and integer exponentials (section 3.3, Integer-only 推理)."""
    n = 0
    for rec in _golden("lis_worked_example.txt"):
        if rec[0] == "const":
            S, x0, b, c = float(rec[1]), int(rec[2]), int(rec[3]), int(rec[4])
            # the constants show through the exponential: e(0) = c 2^30,
            # e(-1) = (c - (b - 1)) 2^30, and x0 is where q first becomes 1
            assert oracle.lis_int_exp(0, S) == c << 30
            assert oracle.lis_int_exp(-1, S) == (c - (b - 1)) << 30
            assert oracle.lis_int_exp(x0, S) == c << 29
            assert oracle.lis_int_exp(x0 + 1, S) != c << 29
            n += 1
        elif rec[0] == "exp":
            S, x, z, sh = float(rec[1]), int(rec[2]), int(rec[3]), int(rec[4])
            assert oracle.lis_int_exp(x, S) == z << sh, rec
            n += 1
    assert n >= 10


def test_lis_golden_rows(oracle):
    """Hand-worked rows, including the round-half-to-even ties 1.5, 2.5, 5.5 (section 3.3)."""
    rows = [r for r in _golden("lis_worked_example.txt") if r[0] == "row"]
    assert len(rows) >= 8
    for rec in rows:
        S, bits = float(rec[1]), int(rec[2])
        bar = rec.index("|")
        x = np.array([int(t) for t in rec[3:bar]], np.int32)
        want = np.array([int(t) for t in rec[bar + 1:]], np.uint8)
        got = oracle.log_int_softmax(x[None, :], S, bits)[0]
        assert np.array_equal(got, want), (rec, got)


def test_log_round_is_nearest_power_of_two(oracle):
    """log_round(v) is the exponent of the power of two nearest to v, the midpoint
    1.5 * 2^b going up (section 3.3, log_round: floor(log2 v) plus one when
    v - 2^b >= 2^(b - 1)).  Checked against a brute-force search over exponents."""
    def nearest(v):
        best = 0
        for j in range(64):
            if abs(v - 2 ** j) <= abs(v - 2 ** best) and (abs(v - 2 ** j) < abs(v - 2 ** best) or j > best):
                best = j
        return best
    vals = list(range(1, 3000))
    for b in range(1, 63):
        vals += [2 ** b - 1, 2 ** b, 2 ** b + 1, 3 * 2 ** (b - 1) - 1, 3 * 2 ** (b - 1)]
    rng = np.random.default_rng(5)
    vals += [int(v) for v in rng.integers(1, 2 ** 63, 2000, dtype=np.uint64)]
    for v in vals:
        assert oracle.log_round(v) == nearest(v), v


@pytest.mark.parametrize("S", [2.0 ** -3, 2.0 ** -6, 0.0123, 2.0 ** -10])
def test_int_exp_approximates_exp(oracle, S):
    """e * a S^2 / 2^30 approximates exp(x S) (section 3.3, Integer-only 推理: the
    second-order polynomial on [-ln 2, 0] and the power-of-two scaling).  Each of the
    q halvings stands for a step of |x0_int| S instead of ln 2, which the bound allows
    for; the rest is the polynomial's and the floored constants' error."""
    a = 0.35815147
    x0 = math.floor(np.float32(-0.6931) / np.float32(S))
    drift = -x0 * S - math.log(2.0)
    for x in list(range(0, 30 * x0 - 1, -max(1, -x0 // 7))) + [-1, -2, x0, x0 + 1, x0 - 1]:
        if x < 30 * x0:
            continue
        e = oracle.lis_int_exp(x, S)
        approx = e * a * S * S / 2 ** 30
        q = x // x0
        err = abs(math.log(approx) - x * S)
        assert err <= 0.004 + 2.5 * S + q * drift, (S, x, approx, math.exp(x * S))


def test_int_exp_clamps_below_thirty_ln2(oracle):
    """Values below n x0_int (n = 30) take the exponential of n x0_int (section 3.3)."""
    S = 2.0 ** -6
    lo = oracle.lis_int_exp(30 * -45, S)
    for x in (-1351, -5000, -(2 ** 31)):
        assert oracle.lis_int_exp(x, S) == lo


def _rows(rng, rows, L, spread):
    return rng.integers(-spread, spread + 1, (rows, L)).astype(np.int32)


@pytest.mark.parametrize("S,spread", [(2.0 ** -6, 600), (0.01, 900), (2.0 ** -9, 3000)])
def test_lis_tracks_float_softmax(oracle, S, spread):
    """2^-code approximates softmax(x S) within the log_round window: log2(1/p) - k
    lies in [log2 0.75, log2 1.5) up to the rounding of v and the exponential's
    error (section 3.3, Attention Map 的 Log2 量化 and Softmax 的量化推理)."""
    rng = np.random.default_rng(11)
    x = _rows(rng, 40, 197, spread)
    k = oracle.log_int_softmax(x, S, 5).astype(np.float64)
    z = x.astype(np.float64) * S
    p = np.exp(z - z.max(axis=1, keepdims=True))
    p /= p.sum(axis=1, keepdims=True)
    # each halving of the integer exponential stands for |x0_int| S instead of ln 2
    x0 = math.floor(np.float32(-0.6931) / np.float32(S))
    drift = (-x0 * S - math.log(2.0)) / math.log(2.0)
    q = np.minimum((x.max(axis=1, keepdims=True) - x) // -x0, 30)
    slack = 0.1 + (q + q.max(axis=1, keepdims=True)) * drift
    live = (k < 32) & (p > 0)
    dev = (np.log2(1.0 / p) - k)[live]
    big = ((1.0 / p) >= 8)[live]
    sl = slack[live]
    assert np.all(dev[big] >= math.log2(0.75) - sl[big])
    assert np.all(dev[big] < math.log2(1.5) + sl[big])
    assert np.all(dev >= -1.0 - sl) and np.all(dev <= 1.6 + sl)
    # masked entries are those whose probability is below about 2^-31.4
    assert np.all(np.log2(p[k >= 32]) < -31.4 + 0.6 + (2 * 30 * drift))


def test_lis_equal_rows_and_shift_invariance(oracle):
    """A row of equal values gives v = L and code log_round(L); adding a constant to a
    row changes nothing (the maximum is subtracted first, section 3.3)."""
    S = 2.0 ** -6
    for L in (1, 2, 3, 5, 6, 11, 12, 197, 1000):
        for val in (-7, 0, 123456):
            got = oracle.log_int_softmax(np.full((1, L), val, np.int32), S, 5)[0]
            assert np.all(got == oracle.log_round(L))
    rng = np.random.default_rng(3)
    x = _rows(rng, 8, 50, 400)
    a = oracle.log_int_softmax(x, S, 4)
    b = oracle.log_int_softmax(x + np.int32(1000), S, 4)
    assert np.array_equal(a, b)


def test_lis_monotone_and_masked_at_bits(oracle):
    """Within a row, larger logits never get larger codes; codes >= 2^bits read
    as 2^bits (masked, probability 0) (section 3.3, Softmax 的量化的实现)."""
    rng = np.random.default_rng(4)
    x = _rows(rng, 16, 64, 2000)
    for bits in (1, 2, 3, 4, 5):
        k = oracle.log_int_softmax(x, 2.0 ** -6, bits)
        assert k.max() <= 2 ** bits
        for r in range(x.shape[0]):
            o = np.argsort(-x[r], kind="stable")
            assert np.all(np.diff(k[r][o].astype(int)) >= 0)
        k5 = oracle.log_int_softmax(x, 2.0 ** -6, 5).astype(int)
        assert np.array_equal(k, np.minimum(k5, 2 ** bits))


def test_lis_argument_errors(oracle):
    x = np.zeros((1, 4), np.int32)
    for S, bits in ((0.0, 4), (-1.0, 4), (float("nan"), 4), (2.0 ** -6, 0), (2.0 ** -6, 6), (50.0, 4)):
        with pytest.raises(ValueError):
            oracle.log_int_softmax(x, S, bits)
    with pytest.raises(ValueError):   # c_int >= 2^31
        oracle.log_int_softmax(x, 2.0 ** -16, 4)


@pytest.mark.parametrize("bits", [2, 3, 4])
def test_attn_shift_equals_dequantized_matmul(oracle, bits):
    """AttnQ x V as shifts equals 2^(2^bits - 1) times the float64 product of the
    dequantized map (2^-code, 0 where masked) with V (section 3.3, Attention Map 的
    Log2 量化: the MatMul becomes a BitShift)."""
    rng = np.random.default_rng(bits)
    H, Lq, Lk, d = 3, 17, 29, 8
    code = rng.integers(0, 2 ** bits + 1, (H, Lq, Lk)).astype(np.uint8)
    v = rng.integers(-128, 128, (H, Lk, d)).astype(np.int32)
    got = oracle.attn_shift_v(code, v, bits)
    deq = np.where(code < 2 ** bits, 2.0 ** -code.astype(np.float64), 0.0)
    want = np.matmul(deq, v.astype(np.float64)) * 2.0 ** (2 ** bits - 1)
    assert np.array_equal(got, want.astype(np.int64))
