"""numpy front end of the plain C oracle (``qnn_oracle.c``).

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg may import this module; the product (the CUDA
library and its binding) never does.  It shares no code with the CUDA path.

Every function takes and returns numpy arrays of integer *codes* (int32) or
float32 values; packing to bytes / nibbles is a separate, explicit step.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "qnn_oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "liboracle.so")

SYM, ASYM, POW2 = 0, 1, 2
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (no fp contraction, no fast-math)."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math",
           "-fopenmp", "-shared", "-fPIC", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def lib() -> ctypes.CDLL:
    global _lib
    if _lib is None:
        _lib = ctypes.CDLL(build())
        L = _lib
        i64, i32, f32, vp = ctypes.c_int64, ctypes.c_int32, ctypes.c_float, ctypes.c_void_p
        L.oracle_round_mode.restype = ctypes.c_double
        L.oracle_round_mode.argtypes = [ctypes.c_double, ctypes.c_int]
        L.oracle_quantize.argtypes = [vp, i64, i64, i64, ctypes.c_int, ctypes.c_int,
                                      vp, vp, vp, i32, i32, vp]
        L.oracle_dequantize.argtypes = [vp, i64, i64, i64, ctypes.c_int, ctypes.c_int,
                                        vp, vp, vp, vp]
        L.oracle_pack_nibbles.argtypes = [vp, i64, vp]
        L.oracle_unpack_nibbles.argtypes = [vp, i64, ctypes.c_int, vp]
        L.oracle_pack_bytes.argtypes = [vp, i64, vp]
        L.oracle_gemm_acc.argtypes = [vp, vp, i64, i64, i64, i32, vp, vp]
        L.oracle_colsum.argtypes = [vp, i64, i64, vp]
        L.oracle_fold.argtypes = [i64, i32, vp, f32, vp, ctypes.c_int, vp, f32,
                                  vp, vp, vp, vp]
        L.oracle_requant.argtypes = [vp, i64, i64, vp, vp, ctypes.c_int, vp, i32, f32,
                                     i32, i32, i32, vp]
        L.oracle_dequant_epilogue.argtypes = [vp, i64, i64, vp, vp, vp]
        L.oracle_conv_acc_direct.argtypes = [vp] * 2 + [ctypes.c_int] * 11 + [i32, vp]
        L.oracle_im2col.argtypes = [vp] + [ctypes.c_int] * 10 + [i32, vp]
        L.oracle_conv_acc_layout.argtypes = [vp] * 2 + [ctypes.c_int] * 11 + [i32, ctypes.c_int, vp]
        L.oracle_lis_int_exp.restype = i64
        L.oracle_lis_int_exp.argtypes = [i64, f32]
        L.oracle_log_round.restype = ctypes.c_int
        L.oracle_log_round.argtypes = [ctypes.c_uint64]
        L.oracle_log_int_softmax.argtypes = [vp, i64, i64, f32, ctypes.c_int, vp]
        L.oracle_attn_shift_v.argtypes = [vp, vp, i64, i64, i64, i64, ctypes.c_int, vp]
        L.oracle_int_layernorm.argtypes = [vp, i64, i64, vp, f32, vp, vp, vp, vp]
        L.oracle_eltwise_s8.argtypes = [ctypes.c_int, vp, vp, i64, f32, ctypes.c_int, vp]
        L.oracle_quantize_rows_dynamic.argtypes = [vp, i64, i64, ctypes.c_int, vp, vp]
        L.oracle_requant_rowscale.argtypes = [vp, i64, i64, vp, vp, vp, ctypes.c_int, vp, i32, f32, i32, i32,
                                              i32, vp]
        L.oracle_dequant_rowscale.argtypes = [vp, i64, i64, vp, vp, vp, vp]
        L.oracle_nhwc_to_nchw64.argtypes = [vp] + [ctypes.c_int] * 4 + [vp]
        L.oracle_set_threads.argtypes = [ctypes.c_int]
        L.oracle_get_threads.restype = ctypes.c_int
    return _lib


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dt):
    return np.ascontiguousarray(a, dtype=dt)


def set_threads(n: int) -> None:
    lib().oracle_set_threads(int(n))


def get_threads() -> int:
    return int(lib().oracle_get_threads())


# Code ranges [MG 背景: UINT4 0..15, INT4 -8..7; int8 / uint8 by their width].
RANGES = {"s8": (-128, 127), "u8": (0, 255), "s4": (-8, 7), "u4": (0, 15)}


def qrange(dt: str, narrow: bool = False):
    lo, hi = RANGES[dt]
    if narrow and dt in ("s8", "s4"):
        lo = -hi
    return lo, hi


def round_mode(v: float, mode: int) -> float:
    return float(lib().oracle_round_mode(float(v), int(mode)))


def _view(shape, axis, per_channel):
    shape = tuple(int(s) for s in shape)
    if not per_channel:
        n = int(np.prod(shape)) if shape else 1
        return 1, 1, n
    axis = axis % len(shape)
    outer = int(np.prod(shape[:axis])) if axis > 0 else 1
    inner = int(np.prod(shape[axis + 1:])) if axis + 1 < len(shape) else 1
    return outer, shape[axis], inner


def quantize(x, scheme, dt, scale=None, zp=None, shift=None, per_channel=False,
             axis=0, narrow=False):
    x = _c(x, np.float32)
    outer, C, inner = _view(x.shape, axis, per_channel)
    qmin, qmax = qrange(dt, narrow)
    sc = _c(np.atleast_1d(scale if scale is not None else 1.0), np.float32)
    z = _c(np.atleast_1d(zp if zp is not None else 0), np.int32)
    sh = _c(np.atleast_1d(shift if shift is not None else 0), np.int32)
    q = np.empty(x.shape, np.int32)
    rc = lib().oracle_quantize(_p(x), outer, C, inner, scheme, int(per_channel),
                               _p(sc), _p(z), _p(sh), qmin, qmax, _p(q))
    assert rc == 0
    return q


def dequantize(q, scheme, scale=None, zp=None, shift=None, per_channel=False, axis=0):
    q = _c(q, np.int32)
    outer, C, inner = _view(q.shape, axis, per_channel)
    sc = _c(np.atleast_1d(scale if scale is not None else 1.0), np.float32)
    z = _c(np.atleast_1d(zp if zp is not None else 0), np.int32)
    sh = _c(np.atleast_1d(shift if shift is not None else 0), np.int32)
    x = np.empty(q.shape, np.float32)
    rc = lib().oracle_dequantize(_p(q), outer, C, inner, scheme, int(per_channel),
                                 _p(sc), _p(z), _p(sh), _p(x))
    assert rc == 0
    return x


def pack_nibbles(q):
    q = _c(q, np.int32)
    assert q.shape[-1] % 2 == 0
    out = np.empty(q.shape[:-1] + (q.shape[-1] // 2,), np.uint8)
    lib().oracle_pack_nibbles(_p(q), q.size, _p(out))
    return out


def unpack_nibbles(p, signed):
    p = _c(p, np.uint8)
    q = np.empty(p.shape[:-1] + (p.shape[-1] * 2,), np.int32)
    lib().oracle_unpack_nibbles(_p(p), q.size, int(signed), _p(q))
    return q


def pack_bytes(q):
    q = _c(q, np.int32)
    out = np.empty(q.shape, np.uint8)
    lib().oracle_pack_bytes(_p(q), q.size, _p(out))
    return out


def gemm_acc(A, B, z_a=0, alpha=None):
    """acc[m, n] = sum_k (A[m,k] - z_a) * 2^alpha[k] * B[n,k] (int32, exact)."""
    A = _c(A, np.int32)
    B = _c(B, np.int32)
    M, K = A.shape
    N, K2 = B.shape
    assert K == K2
    al = None if alpha is None else _c(alpha, np.int32)
    acc = np.empty((M, N), np.int32)
    rc = lib().oracle_gemm_acc(_p(A), _p(B), M, N, K, int(z_a), _p(al), _p(acc))
    if rc != 0:
        raise OverflowError("accumulator does not fit int32")
    return acc


def colsum(B):
    B = _c(B, np.int32)
    N, K = B.shape
    out = np.empty(N, np.int32)
    lib().oracle_colsum(_p(B), N, K, _p(out))
    return out


def fold(colsum_, z_a, s_a, s_w, s_o, bias=None):
    """Returns (zp_term, M, Bq, D) as folded ahead of inference; zp_term = z_a * colsum."""
    cs = _c(colsum_, np.int32)
    N = cs.shape[0]
    sw = _c(np.atleast_1d(s_w), np.float32)
    per_ch = int(sw.shape[0] == N and N > 1)
    b = None if bias is None else _c(bias, np.float32)
    zp = np.empty(N, np.int32)
    Mv = np.empty(N, np.float32)
    Bq = np.empty(N, np.float32)
    D = np.empty(N, np.float32)
    rc = lib().oracle_fold(N, int(z_a), _p(cs), np.float32(s_a), _p(sw), per_ch, _p(b),
                           np.float32(s_o), _p(zp), _p(Mv), _p(Bq), _p(D))
    if rc != 0:
        raise OverflowError("zp_term does not fit int32")
    return zp, Mv, Bq, D


def requant(acc_c, Mv, Bq, dt_out, relu=False, res=None, z_res=0, R=0.0, z_out=0,
            narrow=False):
    acc_c = _c(acc_c, np.int32)
    rows, N = acc_c.shape
    qmin, qmax = qrange(dt_out, narrow)
    Mv = _c(Mv, np.float32)
    Bq = _c(Bq, np.float32)
    r = None if res is None else _c(res, np.int32)
    q = np.empty((rows, N), np.int32)
    lib().oracle_requant(_p(acc_c), rows, N, _p(Mv), _p(Bq), int(relu), _p(r), int(z_res),
                         np.float32(R), int(z_out), qmin, qmax, _p(q))
    return q


def dequant_epilogue(acc_c, D, bias=None):
    acc_c = _c(acc_c, np.int32)
    rows, N = acc_c.shape
    D = _c(D, np.float32)
    b = None if bias is None else _c(bias, np.float32)
    y = np.empty((rows, N), np.float32)
    lib().oracle_dequant_epilogue(_p(acc_c), rows, N, _p(D), _p(b), _p(y))
    return y


def conv_out_hw(h, w, fh, fw, ph, pw, sh, sw):
    return (h + 2 * ph - fh) // sh + 1, (w + 2 * pw - fw) // sw + 1


def conv_acc_direct(I, W, z_in, pad=(1, 1), stride=(1, 1)):
    """I: NHWC codes, W: OHWI codes -> acc [N*OH*OW, OC] (int32)."""
    I = _c(I, np.int32)
    W = _c(W, np.int32)
    n_, h, w, c = I.shape
    oc, fh, fw, c2 = W.shape
    assert c == c2
    oh, ow = conv_out_hw(h, w, fh, fw, pad[0], pad[1], stride[0], stride[1])
    acc = np.empty((n_ * oh * ow, oc), np.int32)
    rc = lib().oracle_conv_acc_direct(_p(I), _p(W), n_, h, w, c, oc, fh, fw, pad[0], pad[1],
                                      stride[0], stride[1], int(z_in), _p(acc))
    if rc != 0:
        raise OverflowError("conv accumulator out of range or bad geometry")
    return acc


LAYOUTS = {"nhwc": 0, "nchw": 1, "nchw64": 2}


def conv_acc_layout(I, W, z_in, N, H, Wd, C, layout, pad=(1, 1), stride=(1, 1)):
    """Direct conv of codes I stored in `layout` ("nhwc", "nchw", "nchw64": any array
    of N*H*Wd*C codes in that element order) with OHWI codes W; returns the int32
    accumulators as a flat array in the same layout."""
    I = _c(I, np.int32).ravel()
    W = _c(W, np.int32)
    OC, FH, FW, C2 = W.shape
    assert C2 == C and I.size == N * H * Wd * C
    OH, OW = conv_out_hw(H, Wd, FH, FW, pad[0], pad[1], stride[0], stride[1])
    acc = np.empty(N * OH * OW * OC, np.int32)
    rc = lib().oracle_conv_acc_layout(_p(I), _p(W), N, H, Wd, C, OC, FH, FW, pad[0], pad[1], stride[0], stride[1],
                                      int(z_in), LAYOUTS[layout], _p(acc))
    if rc == 1:
        raise OverflowError("conv accumulator does not fit int32")
    if rc != 0:
        raise ValueError(f"oracle_conv_acc_layout: error {rc}")
    return acc


def im2col(I, fh, fw, z_in, pad=(1, 1), stride=(1, 1)):
    I = _c(I, np.int32)
    n_, h, w, c = I.shape
    oh, ow = conv_out_hw(h, w, fh, fw, pad[0], pad[1], stride[0], stride[1])
    cols = np.empty((n_ * oh * ow, fh * fw * c), np.int32)
    rc = lib().oracle_im2col(_p(I), n_, h, w, c, fh, fw, pad[0], pad[1], stride[0],
                             stride[1], int(z_in), _p(cols))
    assert rc == 0
    return cols


# ----------------------------------------------------------------------------
# Log-Int-Softmax and the bit-shift attention product [FQ 3.3]

def lis_int_exp(x: int, S: float) -> int:
    """Integer exponential of one value x <= 0 (codes at scale S)."""
    return int(lib().oracle_lis_int_exp(int(x), float(np.float32(S))))


def log_round(v: int) -> int:
    return int(lib().oracle_log_round(int(v)))


def log_int_softmax(x, S: float, bits: int = 4):
    """Rows along the last axis of int32 codes -> uint8 log2 codes (2^bits = masked)."""
    x = _c(x, np.int32)
    L = x.shape[-1]
    rows = x.size // L if L else 0
    out = np.empty(x.shape, np.uint8)
    rc = lib().oracle_log_int_softmax(_p(x), rows, L, float(np.float32(S)), int(bits), _p(out))
    if rc != 0:
        raise ValueError(f"oracle_log_int_softmax: error {rc}")
    return out


def attn_shift_v(code, v, bits: int = 4):
    """code [H, Lq, Lk] uint8, v [H, Lk, d] int -> int64 [H, Lq, d]:
    sum_t 2^(2^bits - 1 - code) * v, masked codes (>= 2^bits) contributing 0."""
    code = _c(code, np.uint8)
    v = _c(v, np.int32)
    H, Lq, Lk = code.shape
    d = v.shape[-1]
    assert v.shape == (H, Lk, d)
    out = np.empty((H, Lq, d), np.int64)
    rc = lib().oracle_attn_shift_v(_p(code), _p(v), H, Lq, Lk, d, int(bits), _p(out))
    if rc != 0:
        raise ValueError(f"oracle_attn_shift_v: error {rc}")
    return out


# ----------------------------------------------------------------------------
# Integer LayerNorm over PTF-quantized rows [FQ 3.2]

def int_layernorm(x, s: float, gamma, beta, out_scale, alpha=None):
    """x int codes [..., C] (real x * s * 2^alpha[c]) -> int64 output codes
    (unclipped), per the integer mode of the page's QIntLayerNorm."""
    x = _c(x, np.int32)
    C = x.shape[-1]
    rows = x.size // C
    g = _c(np.broadcast_to(np.asarray(gamma, np.float32), (C,)), np.float32)
    b = _c(np.broadcast_to(np.asarray(beta, np.float32), (C,)), np.float32)
    o = _c(np.broadcast_to(np.asarray(out_scale, np.float32), (C,)), np.float32)
    al = None if alpha is None else _c(alpha, np.uint8)
    y = np.empty(x.shape, np.int64)
    rc = lib().oracle_int_layernorm(_p(x), rows, C, _p(al), float(np.float32(s)), _p(g), _p(b), _p(o), _p(y))
    if rc != 0:
        raise ValueError(f"oracle_int_layernorm: error {rc}")
    return y


# ----------------------------------------------------------------------------
# Standalone quantized elementwise ops and dynamic per-row quantization [QI]

ELTWISE = {"add": 0, "mul": 1, "relu": 2}


def eltwise_s8(op: str, a, b=None, M: float = 1.0, relu: bool = False):
    a = _c(a, np.int32)
    b = a if b is None else _c(b, np.int32)
    assert a.shape == b.shape
    out = np.empty(a.shape, np.int32)
    rc = lib().oracle_eltwise_s8(ELTWISE[op], _p(a), _p(b), a.size, float(np.float32(M)), int(relu), _p(out))
    if rc != 0:
        raise ValueError(f"oracle_eltwise_s8: error {rc}")
    return out


def quantize_rows_dynamic(x, narrow: bool = False):
    """x fp32 [rows, cols] -> (int32 codes, fp32 per-row scales max|x| / 127)."""
    x = _c(x, np.float32)
    rows, cols = x.shape
    q = np.empty(x.shape, np.int32)
    sc = np.empty(rows, np.float32)
    rc = lib().oracle_quantize_rows_dynamic(_p(x), rows, cols, int(narrow), _p(q), _p(sc))
    if rc != 0:
        raise ValueError(f"oracle_quantize_rows_dynamic: error {rc}")
    return q, sc


def requant_rowscale(acc_c, r, Mv, Bq, dt_out, relu=False, res=None, z_res=0, R=0.0, z_out=0, narrow=False):
    """requant with per-row activation scales: M[m][n] = r[m] * Mv[n] (fp32) first."""
    acc_c = _c(acc_c, np.int32)
    rows, N = acc_c.shape
    qmin, qmax = qrange(dt_out, narrow)
    rr = _c(r, np.float32)
    Mv = _c(Mv, np.float32)
    Bq = _c(Bq, np.float32)
    rs = None if res is None else _c(res, np.int32)
    q = np.empty((rows, N), np.int32)
    rc = lib().oracle_requant_rowscale(_p(acc_c), rows, N, _p(rr), _p(Mv), _p(Bq), int(relu), _p(rs), int(z_res),
                                       np.float32(R), int(z_out), qmin, qmax, _p(q))
    assert rc == 0
    return q


def dequant_rowscale(acc_c, r, D, bias=None):
    acc_c = _c(acc_c, np.int32)
    rows, N = acc_c.shape
    y = np.empty((rows, N), np.float32)
    b = None if bias is None else _c(bias, np.float32)
    lib().oracle_dequant_rowscale(_p(acc_c), rows, N, _p(_c(r, np.float32)), _p(_c(D, np.float32)), _p(b), _p(y))
    return y


def nhwc_to_nchw64(x):
    """codes [N, H, W, C] -> [N, C / 64, H, W, 64]."""
    x = _c(x, np.int32)
    N, H, W, C = x.shape
    y = np.empty((N, C // 64, H, W, 64), np.int32)
    rc = lib().oracle_nhwc_to_nchw64(_p(x), N, H, W, C, _p(y))
    if rc != 0:
        raise ValueError(f"oracle_nhwc_to_nchw64: error {rc}")
    return y
