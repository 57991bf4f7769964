"""Pins of the oracle's integer LayerNorm over PTF-quantized rows.

Source: "首个完全量化Vision Transformer的方法FQ-ViT" (aijishu.com), section 3.2
(LayerNorm 的量化推理; LayerNorm 的量化实现).  The pins are hand-worked rows
(tests/golden/int_layernorm_worked_example.txt), the float LayerNorm the method
approximates (with an error bound derived from M, N and the two roundings), the
PTF shift as a pre-multiplied input, and the sign symmetry of the normalisation.
"""
import os

import numpy as np
import pytest

pytestmark = pytest.mark.cpu
GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "int_layernorm_worked_example.txt")


def _golden():
    rows = []
    for line in open(GOLDEN):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        head, al, xs, ys = (p.split() for p in line.split("|"))
        rows.append(([float(v) for v in head], [int(v) for v in al], [int(v) for v in xs], [int(v) for v in ys]))
    return rows


def test_int_layernorm_golden(oracle):
    rows = _golden()
    assert len(rows) >= 4
    for (s, g, b, o), al, xs, ys in rows:
        y = oracle.int_layernorm(np.array([xs]), s, g, b, o, alpha=np.array(al, np.uint8))
        assert y[0].tolist() == ys, (s, g, b, o, al, xs, y)


def _ln_case(rng, rows, C, spread=40):
    x = rng.integers(-spread, spread + 1, size=(rows, C)).astype(np.int32)
    alpha = rng.integers(0, 4, size=C).astype(np.uint8)
    gamma = rng.uniform(0.5, 2.0, size=C).astype(np.float32) * rng.choice([-1, 1], size=C).astype(np.float32)
    beta = rng.normal(0.0, 0.5, size=C).astype(np.float32)
    o = rng.uniform(0.01, 0.05, size=C).astype(np.float32)
    return x, alpha, gamma, beta, o


@pytest.mark.parametrize("C", [8, 192, 768])
def test_int_layernorm_tracks_float_layernorm(oracle, C):
    """y o approximates gamma (x - mean) / std + beta (population std, no epsilon)
    within 0.5 + (|x'| + 1/2) a / 128 output steps, a = |gamma| / (o std) -- the
    error of M / 2^N against |A| (A = a in code units) and of B's rounding -- plus
    a small fp32 allowance (section 3.2, LayerNorm 的量化推理)."""
    rng = np.random.default_rng(C)
    s = 0.02
    x, alpha, gamma, beta, o = _ln_case(rng, 24, C)
    y = oracle.int_layernorm(x, s, gamma, beta, o, alpha=alpha)
    xp = x.astype(np.float64) * 2.0 ** alpha.astype(np.float64)
    mu = xp.mean(axis=1, keepdims=True)
    sd = xp.std(axis=1, keepdims=True)
    ref = (gamma * (xp - mu) / sd + beta) / o
    a = np.abs(gamma) / (o * sd)
    bound = 0.5 + (np.abs(xp) + 0.5) * a / 128.0 + 1e-4 * (np.abs(ref) + 1.0)
    assert np.all(np.abs(y - ref) <= bound)


def test_int_layernorm_ptf_is_a_shift(oracle):
    """Codes with factors 2^alpha give the same output as the pre-shifted codes
    with no factors (section 3.2, 阶段1: the activations are shifted by alpha)."""
    rng = np.random.default_rng(9)
    x, alpha, gamma, beta, o = _ln_case(rng, 16, 96)
    a = oracle.int_layernorm(x, 0.03, gamma, beta, o, alpha=alpha)
    b = oracle.int_layernorm(x * (1 << alpha.astype(np.int32)), 0.03, gamma, beta, o)
    assert np.array_equal(a, b)


def test_int_layernorm_sign_symmetry(oracle):
    """With beta = 0, negating a row negates its output exactly (the mean and
    B change sign; round half to even is symmetric)."""
    rng = np.random.default_rng(10)
    x, alpha, gamma, _, o = _ln_case(rng, 16, 64)
    beta = np.zeros(64, np.float32)
    a = oracle.int_layernorm(x, 0.05, gamma, beta, o, alpha=alpha)
    b = oracle.int_layernorm(-x, 0.05, gamma, beta, o, alpha=alpha)
    assert np.array_equal(a, -b)


def test_int_layernorm_unit_row(oracle):
    """A row of +-1 with gamma = o and beta = 0 is already normalised: y = x."""
    x = np.array([[1, -1] * 8, [-1, 1] * 8], np.int32)
    for s in (0.1, 0.37, 2.0 ** -7):
        y = oracle.int_layernorm(x, s, 0.02, 0.0, 0.02)
        assert np.array_equal(y, x)


def test_int_layernorm_errors(oracle):
    x = np.zeros((1, 4), np.int32)
    for kw in (dict(s=0.0, o=1.0), dict(s=float("nan"), o=1.0), dict(s=1.0, o=0.0), dict(s=1.0, o=-1.0)):
        with pytest.raises(ValueError):
            oracle.int_layernorm(x, kw["s"], 1.0, 0.0, kw["o"])
    with pytest.raises(ValueError):
        oracle.int_layernorm(x, 1.0, 1.0, 0.0, 1.0, alpha=np.array([0, 0, 31, 0], np.uint8))
    for g, b in ((float("inf"), 0.0), (float("nan"), 0.0), (1.0, float("-inf"))):
        with pytest.raises(ValueError):
            oracle.int_layernorm(x, 1.0, g, b, 1.0)


def test_int_layernorm_overflowing_scale(oracle):
    """A finite gamma whose A = (s / std) gamma / o overflows to +-inf: log2 |A|
    is infinite, so N = clamp(7 - inf) = 0 and M = clamp(inf) = 255; with
    mean 0 and beta 0, B = 0 and y = sign(A) 255 x' exactly.  The other
    channel keeps its ordinary constants (y = x for gamma = o)."""
    x = np.array([[1, -1, 1, -1], [3, -3, -3, 3]], np.int32)
    gamma = np.array([3e38, -3e38, 0.5, 0.5], np.float32)
    o = np.array([1e-3, 1e-3, 0.5, 0.5], np.float32)
    y = oracle.int_layernorm(x, 1.0, gamma, 0.0, o)
    sgn = np.array([1, -1, 1, 1])
    unit = np.sign(x)
    assert np.array_equal(y[:, :2], 255 * sgn[:2] * x[:, :2])
    assert np.array_equal(y[:, 2:], unit[:, 2:])
