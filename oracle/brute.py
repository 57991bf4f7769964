"""Exact brute force for tiny shapes (Python integers and fractions).

TEST INFRASTRUCTURE ONLY.  Used to pin the C oracle: it shares nothing with it
but the definitions on the pages, and computes them in exact rational
arithmetic instead of fp32, so a dropped term, a wrong sign, a swapped index or
a mis-ordered rounding in the oracle shows up as a mismatch.

Sources: "【量化】神经网络量化介绍" (量化算子, 反量化算子, 量化乘法, 量化加法,
量化激活函数, 常见计算图优化 conv-add) and the MegEngine 4-bit article
(背景: r = S (q - Z); 緩解精度下降: the unexpanded conv sum).
"""
from __future__ import annotations

from fractions import Fraction
import math


def round_half_even(v: Fraction) -> int:
    f = math.floor(v)
    d = v - f
    if d < Fraction(1, 2):
        return f
    if d > Fraction(1, 2):
        return f + 1
    return f if f % 2 == 0 else f + 1


def gemm_acc(A, B, z_a=0, alpha=None):
    """Python-int triple loop: sum_k (A[m][k]-z_a) * 2^alpha_k * B[n][k]."""
    M, K = len(A), len(A[0])
    N = len(B)
    out = [[0] * N for _ in range(M)]
    for m in range(M):
        for n in range(N):
            s = 0
            for k in range(K):
                a = int(A[m][k]) - int(z_a)
                if alpha is not None:
                    a *= 2 ** int(alpha[k])
                s += a * int(B[n][k])
            out[m][n] = s
    return out


def conv_acc(I, W, z_in, pad, stride):
    """Seven-deep loop over NHWC codes I and OHWI codes W; padded taps are the
    real value 0 (they contribute nothing)."""
    n_, h, w, c = len(I), len(I[0]), len(I[0][0]), len(I[0][0][0])
    oc, fh, fw = len(W), len(W[0]), len(W[0][0])
    oh = (h + 2 * pad[0] - fh) // stride[0] + 1
    ow = (w + 2 * pad[1] - fw) // stride[1] + 1
    out = []
    for b in range(n_):
        for y in range(oh):
            for x in range(ow):
                row = []
                for o in range(oc):
                    s = 0
                    for r in range(fh):
                        for t in range(fw):
                            iy = y * stride[0] - pad[0] + r
                            ix = x * stride[1] - pad[1] + t
                            if 0 <= iy < h and 0 <= ix < w:
                                for ic in range(c):
                                    s += (int(I[b][iy][ix][ic]) - int(z_in)) * int(W[o][r][t][ic])
                    row.append(s)
                out.append(row)
    return out


def requant_exact(real_acc_scaled, bias, s_o, z_out, qmin, qmax, relu=False, res_real=None):
    """Exact requantization of one output from its real value.

    real_acc_scaled : Fraction, S_a * S_w * acc_c (the real-valued product sum)
    bias, s_o       : fp32 numbers (taken exactly as Fractions)
    res_real        : Fraction or None, the residual's real value S_r (r - Z_r)
    Returns (q, t) where t = y / S_o is the exact pre-rounding value.
    """
    y = real_acc_scaled + Fraction(bias)
    if res_real is not None:
        y += res_real
    t = y / Fraction(s_o)
    r = round_half_even(t)
    if relu:
        r = max(r, 0)
    q = min(max(r + int(z_out), qmin), qmax)
    return q, t


def distance_to_tie(t: Fraction) -> Fraction:
    """|t - (nearest k + 1/2)|: how close t is to a rounding decision point."""
    f = math.floor(t)
    return abs(t - (f + Fraction(1, 2)))
