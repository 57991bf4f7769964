"""Pins of the CPU oracle against what the pages and the mathematics fix.

None of these re-types the oracle's formulas: they use the pages' worked
examples (tests/golden), exact rational arithmetic (Python ints / Fractions,
oracle/brute.py), closed forms, invariants and numpy's integer matmul.
Page sources are named in each test's docstring.
"""
import math
import os
from fractions import Fraction

import numpy as np
import pytest

from oracle import brute
from _exact import F, fl32, near_half_inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
pytestmark = pytest.mark.cpu


def _golden(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append(line.split())
    return rows


# ---------------------------------------------------------------- quantize ---

def test_worked_example(oracle):
    """Quantization intro, 量化算子 / 反量化算子: 1.0 at scale 0.1 -> 10; 1 * 0.1 -> 0.1."""
    rows = {r[0]: r for r in _golden("quantize_worked_example.txt")}
    _, v, s, exp = rows["quantize"]
    q = oracle.quantize(np.array([float(v)], np.float32), oracle.SYM, "s8", scale=float(s))
    assert int(q[0]) == int(exp)
    _, v, s, exp = rows["dequantize"]
    x = oracle.dequantize(np.array([int(v)]), oracle.SYM, scale=float(s))
    assert x[0] == np.float32(float(exp))


def test_rounding_mode_table(oracle):
    """Quantization intro, 量化算子: the five tie-breaking rules at 1.5 and -2.5."""
    for row in _golden("rounding_ties.txt"):
        v = float(row[0])
        for mode, exp in enumerate(row[1:]):
            assert oracle.round_mode(v, mode) == float(exp), (v, mode)


def test_round_nonties_nearest(oracle):
    g = np.random.default_rng(7)
    for v in g.uniform(-1000, 1000, size=2000):
        frac = v - math.floor(v)
        if abs(frac - 0.5) < 1e-9:
            continue
        for mode in range(5):
            assert oracle.round_mode(v, mode) == float(math.floor(v + 0.5))


def test_library_rounding_is_half_even_column(oracle):
    """The library's quantizer takes the half-to-even column of the tie table."""
    table = _golden("rounding_ties.txt")
    xs = np.array([float(r[0]) for r in table], np.float32)
    q = oracle.quantize(xs, oracle.SYM, "s8", scale=1.0)
    assert [int(v) for v in q] == [int(r[1]) for r in table]


def test_code_ranges_and_clamp(oracle):
    """MegEngine article, 背景: UINT4 0..15, INT4 -8..7; out-of-range values clip."""
    for dt, lo, hi in _golden("code_ranges.txt"):
        narrow = dt.endswith("narrow")
        d = dt.replace("narrow", "")
        assert oracle.qrange(d, narrow) == (int(lo), int(hi))
        x = np.array([-1e9, -np.inf, float(lo) - 0.7, float(hi) + 0.7, np.inf, 1e9], np.float32)
        q = oracle.quantize(x, oracle.SYM, d, scale=1.0, narrow=narrow)
        assert list(q) == [int(lo), int(lo), int(lo), int(hi), int(hi), int(hi)]


def test_asym_offset_added_after_rounding(oracle):
    """Quantization intro, 量化模式: round(value/scale) + offset.  With value/scale =
    2.5 and offset 1 that is rint(2.5) + 1 = 3, not rint(3.5) = 4."""
    q = oracle.quantize(np.array([2.5, 0.0, -0.0], np.float32), oracle.ASYM, "u8",
                        scale=1.0, zp=1)
    assert list(q) == [3, 1, 1]
    q = oracle.quantize(np.array([0.0], np.float32), oracle.ASYM, "u8", scale=0.02, zp=128)
    assert int(q[0]) == 128


def test_nan_maps_to_zero_point(oracle):
    x = np.array([np.nan], np.float32)
    assert int(oracle.quantize(x, oracle.ASYM, "u4", scale=0.1, zp=8)[0]) == 8
    assert int(oracle.quantize(x, oracle.SYM, "s8", scale=0.1)[0]) == 0


def ieee_quotient_code(x, s, z, lo, hi):
    """The code of reading c2: one IEEE fp32 division x / s (correctly rounded,
    ties to even), then round half to even, + z, clip."""
    t = fl32(Fraction(float(x)) / Fraction(float(s)))
    return min(max(brute.round_half_even(Fraction(float(t))) + z, lo), hi)


def reciprocal_code(x, s, z, lo, hi):
    """The same with x * RN(1 / s) in place of the division (not the reading)."""
    t = fl32(Fraction(float(x)) * Fraction(float(fl32(1 / Fraction(float(s))))))
    return min(max(brute.round_half_even(Fraction(float(t))) + z, lo), hi)


@pytest.mark.parametrize("dt,scheme,z", [("s8", 0, 0), ("u8", 1, 128), ("s4", 0, 0),
                                         ("u4", 1, 8)])
def test_quantize_is_ieee_division(oracle, dt, scheme, z):
    """Quantization intro, 量化算子: q = round(x / scale), read as one IEEE fp32
    division then half-even rounding (reading c2), + offset after rounding
    (量化模式), clip.  Every code must equal that reading evaluated in exact
    rational arithmetic, including inputs placed a few ulps either side of
    (k + 1/2) * s, where multiplying by a rounded reciprocal gives another code
    (the test asserts such inputs are present)."""
    g = np.random.default_rng(11)
    lo, hi = oracle.qrange(dt)
    span = range(lo - z - 2, hi - z + 2)
    discriminating = 0
    for s in (np.float32(0.037), np.float32(0.1), np.float32(0.0071), np.float32(0.013), np.float32(3.3)):
        x = np.concatenate([g.normal(0, 3, size=500).astype(np.float32) * np.float32(s / 0.037),
                            near_half_inputs(s, span)])
        q = oracle.quantize(x, scheme, dt, scale=s, zp=z)
        for xi, qi in zip(x, q):
            want = ieee_quotient_code(xi, s, z, lo, hi)
            assert qi == want, (dt, float(s), float(xi), int(qi), want)
            discriminating += reciprocal_code(xi, s, z, lo, hi) != want
    assert discriminating > 0


def test_pow2_closed_form(oracle):
    """Quantization intro, 量化模式 (power of two): q = clip(rint(x * 2^shift)).
    x * 2^shift is exact, so the result is the exact half-even rounding."""
    g = np.random.default_rng(3)
    x = g.normal(0, 4, size=3000).astype(np.float32)
    for shift in (0, 1, 3, 5):
        q = oracle.quantize(x, oracle.POW2, "s8", shift=shift)
        for xi, qi in zip(x, q):
            t = Fraction(float(xi)) * 2 ** shift
            assert qi == min(max(brute.round_half_even(t), -128), 127)
        # dequantize of pow2: q * 2^-shift exactly
        y = oracle.dequantize(q, oracle.POW2, shift=shift)
        assert all(Fraction(float(yi)) == Fraction(int(qi), 2 ** shift) for yi, qi in zip(y, q))
    # a tie: 0.75 * 2 = 1.5 -> 2 ; -1.25 * 2 = -2.5 -> -2
    q = oracle.quantize(np.array([0.75, -1.25], np.float32), oracle.POW2, "s8", shift=1)
    assert list(q) == [2, -2]


@pytest.mark.parametrize("dt", ["s8", "u8", "s4", "u4"])
def test_roundtrip_every_code(oracle, dt):
    """quantize(dequantize(q)) == q for every representable code and scale."""
    lo, hi = oracle.qrange(dt)
    codes = np.arange(lo, hi + 1, dtype=np.int32)
    for s in (0.1, 0.0137, 3.7, 1e-4):
        z = 0 if dt.startswith("s") else (hi + 1) // 2
        scheme = oracle.SYM if z == 0 else oracle.ASYM
        x = oracle.dequantize(codes, scheme, scale=s, zp=z)
        assert np.array_equal(oracle.quantize(x, scheme, dt, scale=s, zp=z), codes)
    for shift in (0, 2, 4):
        x = oracle.dequantize(codes, oracle.POW2, shift=shift)
        if dt.startswith("s"):
            assert np.array_equal(oracle.quantize(x, oracle.POW2, dt, shift=shift), codes)


def test_dequantize_exhaustive_exact(oracle):
    """Dequantize equals the correctly rounded exact product (q - z) * s."""
    codes = np.arange(0, 256, dtype=np.int32)
    for s in (np.float32(0.1), np.float32(0.0071), np.float32(12.5)):
        x = oracle.dequantize(codes, oracle.ASYM, scale=s, zp=128)
        for q, xv in zip(codes, x):
            assert xv == fl32(Fraction(int(q) - 128) * Fraction(float(s)))


def test_per_channel_indexing(oracle):
    """Quantization intro, tensor量化与通道量化: per-channel = per-tensor on each
    channel's slice with that channel's parameters."""
    g = np.random.default_rng(5)
    x = g.normal(0, 2, size=(3, 5, 7)).astype(np.float32)
    for axis in (0, 1, 2):
        C = x.shape[axis]
        sc = g.uniform(0.01, 0.2, size=C).astype(np.float32)
        zp = g.integers(0, 255, size=C).astype(np.int32)
        q = oracle.quantize(x, oracle.ASYM, "u8", scale=sc, zp=zp, per_channel=True, axis=axis)
        y = oracle.dequantize(q, oracle.ASYM, scale=sc, zp=zp, per_channel=True, axis=axis)
        for c in range(C):
            sl = [slice(None)] * 3
            sl[axis] = c
            qc = oracle.quantize(x[tuple(sl)], oracle.ASYM, "u8", scale=sc[c], zp=zp[c])
            assert np.array_equal(q[tuple(sl)], qc)
            yc = oracle.dequantize(qc, oracle.ASYM, scale=sc[c], zp=zp[c])
            assert np.array_equal(y[tuple(sl)], yc)


def test_nibble_order(oracle):
    """Two codes per byte, element 2i in the low nibble; s4 sign-extends."""
    p = oracle.pack_nibbles(np.array([1, 2, 15, 0, -1, 7], np.int32))
    assert list(p) == [0x21, 0x0F, 0x7F]
    assert list(oracle.unpack_nibbles(np.array([0x21, 0xF8], np.uint8), signed=True)) == [1, 2, -8, -1]
    assert list(oracle.unpack_nibbles(np.array([0xF8], np.uint8), signed=False)) == [8, 15]
    g = np.random.default_rng(1)
    b = g.integers(0, 256, size=(4, 16)).astype(np.uint8)
    for signed in (0, 1):
        assert np.array_equal(oracle.pack_nibbles(oracle.unpack_nibbles(b, signed)), b)
    assert list(oracle.pack_bytes(np.array([-1, 127, -128, 200]))) == [255, 127, 128, 200]


# ---------------------------------------------------------------- GEMM -------

def test_gemm_acc_brute_force(oracle):
    """Quantization intro, 量化矩阵乘: int32 sums of products, exact."""
    g = np.random.default_rng(2)
    for (M, N, K) in [(1, 1, 1), (3, 5, 7), (4, 8, 33)]:
        A = g.integers(0, 256, size=(M, K)).astype(np.int32)
        B = g.integers(-128, 128, size=(N, K)).astype(np.int32)
        for z in (0, 128, 37):
            assert oracle.gemm_acc(A, B, z).tolist() == brute.gemm_acc(A.tolist(), B.tolist(), z)
        al = g.integers(0, 4, size=K).astype(np.int32)
        assert oracle.gemm_acc(A, B, 0, al).tolist() == brute.gemm_acc(A.tolist(), B.tolist(), 0, al)


def test_gemm_acc_numpy_int64(oracle):
    g = np.random.default_rng(4)
    M, N, K = 67, 45, 300
    A = g.integers(-128, 128, size=(M, K)).astype(np.int32)
    B = g.integers(-128, 128, size=(N, K)).astype(np.int32)
    ref = A.astype(np.int64) @ B.astype(np.int64).T
    assert np.array_equal(oracle.gemm_acc(A, B), ref)
    al = g.integers(0, 4, size=K).astype(np.int32)
    ref = (A.astype(np.int64) * (1 << al.astype(np.int64))) @ B.astype(np.int64).T
    assert np.array_equal(oracle.gemm_acc(A, B, 0, al), ref)


def test_gemm_permutation_properties(oracle):
    """MegEngine article, conv 算子優化 (Fig. 8): permuting B's columns permutes C's
    columns; permuting K (both operands alike) leaves C unchanged."""
    g = np.random.default_rng(6)
    A = g.integers(0, 256, size=(20, 48)).astype(np.int32)
    B = g.integers(-128, 128, size=(16, 48)).astype(np.int32)
    C = oracle.gemm_acc(A, B, 128)
    pn = g.permutation(16)
    assert np.array_equal(oracle.gemm_acc(A, B[pn], 128), C[:, pn])
    pk = g.permutation(48)
    assert np.array_equal(oracle.gemm_acc(A[:, pk], B[:, pk], 128), C)


def test_gemm_overflow_detected(oracle):
    A = np.full((1, 140000), -128, np.int32)
    B = np.full((1, 140000), -128, np.int32)
    with pytest.raises(OverflowError):
        oracle.gemm_acc(A, B)


def test_zero_point_fold_identity(oracle):
    """MegEngine article, 緩解精度下降: sum (q_I - Z_I) q_W = sum q_I q_W - Z_I sum q_W,
    the second term computable before inference.  With the operand centred at
    128 (as the library feeds a u8 operand to the MMA) the folded term becomes
    Z colsum - 128 colsum; both forms must give the unexpanded sum."""
    g = np.random.default_rng(8)
    A = g.integers(0, 256, size=(9, 70)).astype(np.int32)
    B = g.integers(-128, 128, size=(11, 70)).astype(np.int32)
    cs = oracle.colsum(B)
    assert np.array_equal(cs, B.sum(axis=1))
    for z in (0, 128, 3, 255):
        direct = oracle.gemm_acc(A, B, z)
        zp, *_ = oracle.fold(cs, z, 1.0, np.ones(11, np.float32), 1.0)
        assert np.array_equal(oracle.gemm_acc(A, B, 0) - zp[None, :], direct)
        assert np.array_equal(zp, z * B.sum(axis=1))
        zp_c = zp.astype(np.int64) - 128 * cs.astype(np.int64)
        assert np.array_equal(oracle.gemm_acc(A, B, 128) - zp_c[None, :], direct)


def test_fold_constants_correctly_rounded(oracle):
    """Quantization intro, 量化乘法: scale_abc = s_a s_b / s_c computed ahead, as
    fp32 multiply then fp32 divide; Bq = bias / s_o; D = s_a s_w."""
    g = np.random.default_rng(9)
    N = 64
    s_w = g.uniform(1e-3, 1e-2, size=N).astype(np.float32)
    bias = g.normal(0, 1, size=N).astype(np.float32)
    s_a, s_o = np.float32(0.02), np.float32(0.0731)
    zp, Mv, Bq, D = oracle.fold(np.zeros(N, np.int32), 0, s_a, s_w, s_o, bias)
    for n in range(N):
        p = fl32(Fraction(float(s_a)) * Fraction(float(s_w[n])))
        assert D[n] == p
        assert Mv[n] == fl32(Fraction(float(p)) / Fraction(float(s_o)))
        assert Bq[n] == fl32(Fraction(float(bias[n])) / Fraction(float(s_o)))


# ---------------------------------------------------------------- epilogues --

def test_requant_closed_form_pow2_scale(oracle):
    """Symmetric s8 x s8 with requant multiplier exactly 2^-10, no bias: every
    output is clip(round_half_even(acc / 1024))."""
    g = np.random.default_rng(10)
    A = g.integers(-128, 128, size=(32, 256)).astype(np.int32)
    B = g.integers(-128, 128, size=(24, 256)).astype(np.int32)
    acc = oracle.gemm_acc(A, B)
    _, Mv, Bq, _ = oracle.fold(oracle.colsum(B), 0, 1.0, np.ones(24, np.float32), 1024.0)
    q = oracle.requant(acc, Mv, Bq, "s8")
    for a, qv in zip(acc.ravel(), q.ravel()):
        assert qv == min(max(brute.round_half_even(Fraction(int(a), 1024)), -128), 127)
    # a few hand-made ties: 1536/1024 = 1.5 -> 2, -2560/1024 = -2.5 -> -2
    q = oracle.requant(np.array([[1536, -2560, 512, -512]], np.int32), Mv[:4], Bq[:4], "s8")
    assert q.tolist() == [[2, -2, 0, 0]]


def _requant_case(oracle, relu, residual, out_dt, seed):
    g = np.random.default_rng(seed)
    M, N, K = 6, 10, 40
    A = g.integers(0, 256, size=(M, K)).astype(np.int32)
    B = g.integers(-128, 128, size=(N, K)).astype(np.int32)
    z_a = 128
    s_a = np.float32(0.02)
    s_w = g.uniform(1e-3, 1e-2, size=N).astype(np.float32)
    bias = g.normal(0, 1, size=N).astype(np.float32)
    s_o = np.float32(0.0173)
    lo, hi = oracle.qrange(out_dt)
    z_out = 0 if out_dt == "s8" else 3
    acc = oracle.gemm_acc(A, B, z_a)
    _, Mv, Bq, _ = oracle.fold(oracle.colsum(B), 0, s_a, s_w, s_o, bias)
    res, z_res, R, s_r = None, 0, 0.0, np.float32(0.0)
    if residual:
        res = g.integers(lo, hi + 1, size=(M, N)).astype(np.int32)
        z_res = 5
        s_r = np.float32(0.0211)
        R = np.float32(s_r / s_o)
    q = oracle.requant(acc, Mv, Bq, out_dt, relu=relu, res=res, z_res=z_res, R=R, z_out=z_out)
    ex = brute.gemm_acc(A.tolist(), B.tolist(), z_a)
    near = 0
    for m in range(M):
        for n in range(N):
            real = Fraction(float(s_a)) * Fraction(float(s_w[n])) * ex[m][n]
            rr = None
            if residual:
                rr = Fraction(float(s_r)) * (int(res[m, n]) - z_res)
            e, t = brute.requant_exact(real, float(bias[n]), float(s_o), z_out, lo, hi, relu, rr)
            if e != q[m, n]:
                assert abs(e - int(q[m, n])) == 1
                assert brute.distance_to_tie(t) < (abs(t) + 1) * Fraction(1, 2 ** 19)
                near += 1
    return q, near


@pytest.mark.parametrize("relu,residual,out_dt", [(False, False, "s8"), (True, False, "u8"),
                                                  (True, True, "u8"), (False, True, "s8"),
                                                  (True, True, "u4"), (False, False, "u4")])
def test_requant_vs_exact_rational(oracle, relu, residual, out_dt):
    """The fp32 requant pipeline equals exact-rational requantization
    (dequantize everything, sum, add bias and residual, divide by S_o, round
    half even, add Z_o, clip) except within fp32 error of a tie."""
    _, near = _requant_case(oracle, relu, residual, out_dt, seed=21)
    assert near <= 1


def test_relu_is_passive(oracle):
    """Quantization intro, 量化激活函数: relu is a max with the quantized zero, so
    q_relu == max(q_plain, clip(Z_o))."""
    g = np.random.default_rng(12)
    acc = g.integers(-50000, 50000, size=(20, 16)).astype(np.int32)
    Mv = g.uniform(1e-4, 1e-3, size=16).astype(np.float32)
    Bq = g.normal(0, 3, size=16).astype(np.float32)
    for dt, z in (("u8", 7), ("s8", 0), ("u4", 8)):
        q0 = oracle.requant(acc, Mv, Bq, dt, relu=False, z_out=z)
        q1 = oracle.requant(acc, Mv, Bq, dt, relu=True, z_out=z)
        lo, hi = oracle.qrange(dt)
        assert np.array_equal(q1, np.maximum(q0, min(max(z, lo), hi)))


def test_dequant_epilogue_correctly_rounded(oracle):
    g = np.random.default_rng(13)
    acc = g.integers(-2 ** 23, 2 ** 23, size=(8, 12)).astype(np.int32)
    D = g.uniform(1e-5, 1e-3, size=12).astype(np.float32)
    bias = g.normal(0, 1, size=12).astype(np.float32)
    y = oracle.dequant_epilogue(acc, D, bias)
    for m in range(8):
        for n in range(12):
            p = fl32(Fraction(int(acc[m, n])) * Fraction(float(D[n])))
            assert y[m, n] == fl32(Fraction(float(p)) + Fraction(float(bias[n])))


# ---------------------------------------------------------------- conv -------

@pytest.mark.parametrize("geom", [(1, 5, 6, 4, 3, 3, 1, 1), (2, 4, 4, 2, 5, 3, 1, 2),
                                  (1, 3, 5, 6, 2, 1, 0, 1), (1, 6, 6, 2, 2, 3, 0, 2)])
def test_conv_direct_brute_force(oracle, geom):
    """MegEngine article, 緩解精度下降 / conv 算子優化: conv over (q_I - Z_I) q_W with
    padded taps holding the real value 0."""
    n_, h, w, c, oc, f, pad, st = geom
    g = np.random.default_rng(14)
    I = g.integers(0, 16, size=(n_, h, w, c)).astype(np.int32)
    W = g.integers(-8, 8, size=(oc, f, f, c)).astype(np.int32)
    got = oracle.conv_acc_direct(I, W, 8, (pad, pad), (st, st))
    ref = brute.conv_acc(I.tolist(), W.tolist(), 8, (pad, pad), (st, st))
    assert got.tolist() == ref


def test_conv_implicit_gemm_identity(oracle):
    """MegEngine article, conv 算子優化 (Fig. 5): explicit img2col then GEMM, with
    the zero-point term folded, equals the direct convolution."""
    g = np.random.default_rng(15)
    I = g.integers(0, 16, size=(2, 7, 9, 8)).astype(np.int32)
    W = g.integers(-8, 8, size=(6, 3, 3, 8)).astype(np.int32)
    for pad, st in (((1, 1), (1, 1)), ((1, 1), (2, 2)), ((0, 0), (1, 1))):
        direct = oracle.conv_acc_direct(I, W, 8, pad, st)
        cols = oracle.im2col(I, 3, 3, 8, pad, st)
        Bm = W.reshape(6, -1)
        acc = oracle.gemm_acc(cols, Bm, 0)
        zp, *_ = oracle.fold(oracle.colsum(Bm), 8, 1.0, np.ones(6, np.float32), 1.0)
        assert np.array_equal(acc - zp[None, :], direct)
        assert np.array_equal(oracle.gemm_acc(cols, Bm, 8), direct)


def test_conv_filter_zero_point_terms(oracle):
    """MegEngine article, 緩解精度下降, for asymmetric filters: the conv over
    (q_I - Z_I)(q_W - Z_W) is the conv with q_W less Z_W times the conv with a
    filter of ones (the input's receptive-field sum, padded taps 0), both terms
    by brute force, at full u8 ranges."""
    g = np.random.default_rng(17)
    I = g.integers(0, 256, size=(1, 5, 6, 3)).astype(np.int32)
    W = g.integers(0, 256, size=(4, 3, 3, 3)).astype(np.int32)
    z_w = np.array([0, 255, 128, 77], np.int32)
    ones = np.ones((1, 3, 3, 3), np.int32)
    for pad, st, z_in in (((1, 1), (1, 1), 100), ((0, 0), (2, 2), 255), ((1, 1), (2, 1), 0)):
        got = oracle.conv_acc_direct(I, W - z_w.reshape(-1, 1, 1, 1), z_in, pad, st)
        full = np.array(brute.conv_acc(I.tolist(), W.tolist(), z_in, pad, st), np.int64)
        rsum = np.array(brute.conv_acc(I.tolist(), ones.tolist(), z_in, pad, st), np.int64)
        assert np.array_equal(got, full - rsum * z_w[None, :])


def test_conv1x1_is_gemm(oracle):
    """A 1x1, stride-1, unpadded conv is a GEMM of the pixel matrix (numpy int64)."""
    g = np.random.default_rng(16)
    I = g.integers(0, 16, size=(2, 5, 3, 12)).astype(np.int32)
    W = g.integers(-8, 8, size=(7, 1, 1, 12)).astype(np.int32)
    got = oracle.conv_acc_direct(I, W, 8, (0, 0), (1, 1))
    ref = (I.reshape(-1, 12).astype(np.int64) - 8) @ W.reshape(7, 12).astype(np.int64).T
    assert np.array_equal(got, ref)


def test_requant_rowscale_reduces_and_scales(oracle):
    """Per-row activation scales (a dynamically quantized input feeding the GEMM):
    r = 1 is the plain requant, r = 2^k equals the plain requant with M * 2^k
    (both exact in fp32), and the result tracks the exact rational
    round(acc r M + Bq) except within fp32 error of a tie."""
    g = np.random.default_rng(40)
    acc = g.integers(-200000, 200000, size=(12, 24)).astype(np.int32)
    Mv = g.uniform(1e-5, 1e-3, size=24).astype(np.float32)
    Bq = g.normal(0, 3, size=24).astype(np.float32)
    ones = np.ones(12, np.float32)
    assert np.array_equal(oracle.requant_rowscale(acc, ones, Mv, Bq, "s8"), oracle.requant(acc, Mv, Bq, "s8"))
    r = (2.0 ** g.integers(-3, 4, size=12)).astype(np.float32)
    q = oracle.requant_rowscale(acc, r, Mv, Bq, "s8")
    for m in range(12):
        assert np.array_equal(q[m:m + 1], oracle.requant(acc[m:m + 1], Mv * r[m], Bq, "s8"))
    r = g.uniform(0.01, 0.1, size=12).astype(np.float32)
    q = oracle.requant_rowscale(acc, r, Mv, Bq, "s8")
    near = 0
    for m in range(12):
        for n in range(24):
            exact = Fraction(int(acc[m, n])) * Fraction(float(r[m])) * Fraction(float(Mv[n])) + Fraction(float(Bq[n]))
            want = min(max(brute.round_half_even(exact), -128), 127)
            if q[m, n] != want:
                frac = exact - (exact.numerator // exact.denominator)
                assert abs(frac - Fraction(1, 2)) < abs(exact) * Fraction(1, 2 ** 21) + Fraction(1, 2 ** 20)
                near += 1
    assert near <= 2


def test_nchw64_layout(oracle):
    """MegEngine 4-bit article, conv 算子優化: NCHW64 keeps each 64 consecutive
    channels of a pixel together.  With C = 64 it is NHWC itself; in general
    every element lands at [n][c // 64][h][w][c % 64] (checked by explicit loops)."""
    g = np.random.default_rng(43)
    x = g.integers(-8, 8, size=(2, 3, 5, 64))
    assert np.array_equal(oracle.nhwc_to_nchw64(x)[:, 0], x)
    x = g.integers(0, 16, size=(2, 3, 4, 192))
    y = oracle.nhwc_to_nchw64(x)
    for n in range(2):
        for h in range(3):
            for w in range(4):
                for c in range(192):
                    assert y[n, c // 64, h, w, c % 64] == x[n, h, w, c]
    with pytest.raises(ValueError):
        oracle.nhwc_to_nchw64(np.zeros((1, 2, 2, 48), np.int32))


def _rowscale_inputs(seed):
    g = np.random.default_rng(seed)
    acc = np.concatenate([g.integers(-200000, 200000, size=(10, 24)),
                          g.integers(-2 ** 31, 2 ** 31, size=(2, 24))]).astype(np.int32)
    r = g.uniform(0.01, 0.1, size=12).astype(np.float32)
    Mv = g.uniform(1e-5, 1e-3, size=24).astype(np.float32)
    bias = g.normal(0, 3, size=24).astype(np.float32)
    return acc, r, Mv, bias


def test_dequant_rowscale_steps_exact(oracle):
    """Per-row activation scales in the dequantizing epilogue (reading r32):
    d = fl(r[m] * D[n]) first, then y = fl(fl(float(acc) * d) + bias[n]) -- each
    step one correctly rounded fp32 operation, evaluated here in exact rational
    arithmetic (float(acc) rounds to nearest even above 2^24).  Grouping the
    product as (acc * r) * D instead changes many results (asserted)."""
    acc, r, D, bias = _rowscale_inputs(41)
    y = oracle.dequant_rowscale(acc, r, D, bias)
    y0 = oracle.dequant_rowscale(acc, r, D)
    regrouped = 0
    for m in range(acc.shape[0]):
        for n in range(acc.shape[1]):
            a = F(fl32(int(acc[m, n])))
            d = F(fl32(F(r[m]) * F(D[n])))
            v = fl32(a * d)
            assert y0[m, n] == v
            assert y[m, n] == fl32(F(v) + F(bias[n])), (m, n)
            regrouped += fl32(F(fl32(a * F(r[m]))) * F(D[n])) != v
    assert regrouped > 0


@pytest.mark.parametrize("relu,residual", [(False, False), (True, True)])
def test_requant_rowscale_steps_exact(oracle, relu, residual):
    """The requant with per-row scales as its fp32 steps (reading r32 with the
    requant order of 常见计算图优化, Y = Wx + (Y2 + B)): Mrow = fl(r[m] * M[n]);
    t = Bq, with a residual t = fl(fl(float(res - z_res) * R) + t); v =
    fl(fl(float(acc) * Mrow) + t); q = clip(round_half_even(v) [, max 0] +
    z_out).  Exact rational evaluation of each correctly rounded step."""
    acc, r, Mv, Bq = _rowscale_inputs(42)
    g = np.random.default_rng(43)
    res = g.integers(0, 256, size=acc.shape).astype(np.int32) if residual else None
    z_res, R, z_out = 120, np.float32(0.731), 3
    q = oracle.requant_rowscale(acc, r, Mv, Bq, "u8", relu=relu, res=res, z_res=z_res,
                                R=R if residual else 0.0, z_out=z_out)
    for m in range(acc.shape[0]):
        for n in range(acc.shape[1]):
            mrow = F(fl32(F(r[m]) * F(Mv[n])))
            t = F(Bq[n])
            if residual:
                t = F(fl32(F(fl32(F(fl32(int(res[m, n]) - z_res)) * F(R))) + t))
            v = F(fl32(F(fl32(F(fl32(int(acc[m, n]))) * mrow)) + t))
            k = brute.round_half_even(v)
            if relu:
                k = max(k, 0)
            assert q[m, n] == min(max(k + z_out, 0), 255), (m, n)


def test_requant_rowscale_on_ties(oracle):
    """Per-row scales in the requant, on rounding decision points: for each row
    the bias is chosen so that v = fl(fl(float(acc) * fl(r * M)) + Bq) is
    exactly k + 1/2 (Bq = T - p is exact for p within a factor 2 of T), so the
    result is round-half-even of a tie.  A factor formed in another order
    (fl(fl(acc * r) * M), or M / (1 / r)) moves v off the tie for many elements
    (asserted), so a reordering in the oracle shows up here."""
    g = np.random.default_rng(44)
    N = 64
    Mv = g.uniform(1e-5, 1e-3, size=N).astype(np.float32)
    other = 0
    for m in range(16):
        r = np.float32(g.uniform(0.01, 0.1))
        mrow = [F(fl32(F(r) * F(Mv[n]))) for n in range(N)]
        acc = np.array([int(round(float(g.uniform(40, 120) / float(mrow[n]))) * (1 if g.random() < 0.5 else -1))
                        for n in range(N)], np.int32)
        p = [F(fl32(F(fl32(int(acc[n]))) * mrow[n])) for n in range(N)]
        T = [Fraction(2 * int(np.floor(float(pv))) + 1, 2) for pv in p]
        Bq = np.array([fl32(T[n] - p[n]) for n in range(N)], np.float32)
        assert all(F(Bq[n]) == T[n] - p[n] for n in range(N))
        q = oracle.requant_rowscale(acc[None, :], np.array([r], np.float32), Mv, Bq, "s8")[0]
        for n in range(N):
            assert q[n] == min(max(brute.round_half_even(T[n]), -128), 127), (m, n)
            alt = F(fl32(F(fl32(F(fl32(F(fl32(int(acc[n]))) * F(r))) * F(Mv[n]))) + F(Bq[n])))
            other += alt != T[n]
    assert other > 0


@pytest.mark.parametrize("geom", [(2, 5, 6, 64, 64, 3, 1, 1), (1, 7, 4, 128, 64, 3, 1, 2), (2, 4, 6, 64, 128, 1, 0, 1)])
def test_conv_layouts(oracle, geom):
    """MegEngine 4-bit article, conv 算子優化 (the conv in NCHW64, each 64
    consecutive channels of a pixel contiguous) and NCHW: the accumulator of the
    conv with its input and output in NCHW or NCHW64 is the NHWC conv's, brute
    forced on the NHWC view of the same codes, moved by numpy transposes."""
    n_, h, w, c, oc, f, pad, st = geom
    g = np.random.default_rng(44)
    I = g.integers(0, 16, size=(n_, h, w, c)).astype(np.int32)
    W = g.integers(-8, 8, size=(oc, f, f, c)).astype(np.int32)
    ref = np.array(brute.conv_acc(I.tolist(), W.tolist(), 8, (pad, pad), (st, st)), np.int64)
    oh, ow = (h + 2 * pad - f) // st + 1, (w + 2 * pad - f) // st + 1
    ref = ref.reshape(n_, oh, ow, oc)
    got = oracle.conv_acc_layout(I, W, 8, n_, h, w, c, "nhwc", (pad, pad), (st, st))
    assert np.array_equal(got.reshape(n_, oh, ow, oc), ref)
    got = oracle.conv_acc_layout(I.transpose(0, 3, 1, 2), W, 8, n_, h, w, c, "nchw", (pad, pad), (st, st))
    assert np.array_equal(got.reshape(n_, oc, oh, ow), ref.transpose(0, 3, 1, 2))
    I64 = I.reshape(n_, h, w, c // 64, 64).transpose(0, 3, 1, 2, 4)
    got = oracle.conv_acc_layout(I64, W, 8, n_, h, w, c, "nchw64", (pad, pad), (st, st))
    assert np.array_equal(got.reshape(n_, oc // 64, oh, ow, 64),
                          ref.reshape(n_, oh, ow, oc // 64, 64).transpose(0, 3, 1, 2, 4))
    if c == 64 and oc == 64:
        # one 64-channel block: NCHW64 is NHWC itself
        got = oracle.conv_acc_layout(I, W, 8, n_, h, w, c, "nchw64", (pad, pad), (st, st))
        assert np.array_equal(got.reshape(n_, oh, ow, oc), ref)


def test_conv_layout_indices_by_hand(oracle):
    """Explicit indices: a single nonzero input code at (b, ch, y, x) and a 1x1
    filter that picks channel ch into output channel o put (q - z) w exactly at
    output (b, o, y, x) of each layout, and the zero point everywhere else."""
    n_, h, w, c, oc = 2, 3, 4, 128, 64
    b, ch, y, x, o = 1, 70, 2, 3, 5
    for layout in ("nchw", "nchw64", "nhwc"):
        I = np.zeros(n_ * h * w * c, np.int32)
        if layout == "nchw":
            I[((b * c + ch) * h + y) * w + x] = 9
        elif layout == "nchw64":
            I[(((b * (c // 64) + ch // 64) * h + y) * w + x) * 64 + ch % 64] = 9
        else:
            I[((b * h + y) * w + x) * c + ch] = 9
        W = np.zeros((oc, 1, 1, c), np.int32)
        W[o, 0, 0, ch] = 3
        acc = oracle.conv_acc_layout(I, W, 0, n_, h, w, c, layout, (0, 0), (1, 1))
        nz = np.flatnonzero(acc)
        if layout == "nchw":
            want = ((b * oc + o) * h + y) * w + x
        elif layout == "nchw64":
            want = (((b * (oc // 64) + o // 64) * h + y) * w + x) * 64 + o % 64
        else:
            want = ((b * h + y) * w + x) * oc + o
        assert nz.tolist() == [want] and acc[want] == 27, layout
