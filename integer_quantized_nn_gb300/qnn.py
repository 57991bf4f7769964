"""Thin Python binding of libqnn.so (the C ABI in include/qnn.h).

Argument marshalling only: every function here forwards device pointers
(``tensor.data_ptr()``), host scalars and the current CUDA stream to the
function of the same name in the CUDA library and raises ``QnnError`` on a
non-OK status.  All device memory is allocated by the caller (with torch);
nothing here computes any part of the quantized path.  There is no fallback:
if the library cannot be loaded, every call raises.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

from . import build as _build

# ---- enums (mirror include/qnn.h) ------------------------------------------------
QNN_OK, QNN_ERR_INVALID_ARG, QNN_ERR_UNSUPPORTED, QNN_ERR_ALIGNMENT = 0, 1, 2, 3
QNN_ERR_OVERFLOW_RISK, QNN_ERR_CUDA, QNN_ERR_TIMEOUT = 4, 5, 6
DTYPES = {"s8": 0, "u8": 1, "s4": 2, "u4": 3, "s32": 4, "f32": 5}
SCHEMES = {"sym": 0, "asym": 1, "pow2": 2}
EPI_MODES = {"requant": 0, "dequant": 1, "s32": 2}
ELTWISE_OPS = {"add": 0, "mul": 1, "relu": 2}


class QnnError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_string(status)} ({status})")


class QParams(ctypes.Structure):
    _fields_ = [("scheme", ctypes.c_int32), ("per_channel", ctypes.c_int32),
                ("axis", ctypes.c_int32), ("narrow_range", ctypes.c_int32),
                ("scale", ctypes.c_void_p), ("zero_point", ctypes.c_void_p),
                ("shift", ctypes.c_void_p)]


class Epilogue(ctypes.Structure):
    _fields_ = [("mode", ctypes.c_int32), ("relu", ctypes.c_int32), ("out_dt", ctypes.c_int32),
                ("z_out", ctypes.c_int32), ("zp_term", ctypes.c_void_p), ("M", ctypes.c_void_p),
                ("Bq", ctypes.c_void_p), ("D", ctypes.c_void_p), ("bias", ctypes.c_void_p),
                ("residual", ctypes.c_void_p), ("res_dt", ctypes.c_int32),
                ("z_res", ctypes.c_int32), ("R", ctypes.c_float),
                ("ptf_shift", ctypes.c_void_p), ("ptf_max_shift", ctypes.c_int32),
                ("row_scale", ctypes.c_void_p)]


class ConvGeom(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in
                ("N", "H", "W", "C", "OC", "FH", "FW", "pad_h", "pad_w", "stride_h", "stride_w", "layout")]

    @property
    def OH(self):
        return (self.H + 2 * self.pad_h - self.FH) // self.stride_h + 1

    @property
    def OW(self):
        return (self.W + 2 * self.pad_w - self.FW) // self.stride_w + 1


_lib = None
_SYMBOLS = {}


def _declare(L):
    vp, i32, i64, f32, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float, ctypes.c_size_t
    c_int = ctypes.c_int
    sig = {
        "q_quantize": (c_int, [vp, vp, c_int, c_int, vp, vp, vp]),
        "q_dequantize": (c_int, [vp, c_int, vp, c_int, vp, vp, vp]),
        "qnn_gemm_packed_b_bytes": (sz, [c_int, c_int]),
        "qgemm_prepack_b": (c_int, [vp, c_int, c_int, vp, vp, vp]),
        "q_fold_epilogue": (c_int, [c_int, c_int, i32, vp, f32, vp, c_int, vp, f32, vp, vp, vp, vp, vp]),
        "qnn_gemm_workspace_bytes": (sz, [c_int, c_int]),
        "qgemm_s8": (c_int, [vp, c_int, vp, c_int, c_int, c_int, vp, vp, vp, vp, sz, vp]),
        "qgemm_pack_a": (c_int, [vp, c_int, c_int, c_int, vp, vp, sz, vp]),
        "qgemm_s8_packed": (c_int, [vp, c_int, vp, c_int, c_int, c_int, vp, vp, vp, vp]),
        "qgemm_s8_static_scratch": (c_int, [vp, c_int, vp, c_int, c_int, c_int, vp, vp, vp, vp]),
        "qnn_conv_packed_w_bytes": (sz, [vp, c_int]),
        "qconv_prepack_w": (c_int, [vp, c_int, vp, vp, vp, vp]),
        "qnn_conv_workspace_bytes": (sz, [vp, c_int]),
        "qconv_u4s4": (c_int, [vp, i32, vp, vp, vp, vp, vp, vp, sz, vp]),
        "qconv_u8s8": (c_int, [vp, i32, vp, vp, vp, vp, vp, vp, sz, vp]),
        "qconv_u8u8": (c_int, [vp, i32, vp, vp, vp, vp, vp, vp, sz, vp]),
        "qconv_prepack_w_u8": (c_int, [vp, vp, vp, vp, vp, vp]),
        "q_log_int_softmax": (c_int, [vp, i64, i64, f32, c_int, vp, vp]),
        "q_attn_shift_v": (c_int, [vp, vp, i64, c_int, c_int, c_int, c_int, vp, vp]),
        "q_int_layernorm": (c_int, [vp, i64, c_int, vp, c_int, f32, vp, vp, vp, c_int, vp, vp]),
        "q_eltwise_s8": (c_int, [c_int, vp, vp, i64, f32, c_int, vp, vp]),
        "q_quantize_rows_dynamic": (c_int, [vp, i64, i64, c_int, vp, vp, vp]),
        "qgemm_prepack_b_u8": (c_int, [vp, vp, c_int, c_int, vp, vp, vp]),
        "qgemm_prepack_b_ptf": (c_int, [vp, vp, c_int, c_int, vp, vp, vp]),
        "qnn_gemm_zw_workspace_bytes": (sz, [c_int, c_int]),
        "qgemm_zw": (c_int, [vp, c_int, vp, vp, c_int, c_int, c_int, vp, vp, vp, vp, sz, vp]),
        "q_layout_nchw64": (c_int, [vp, c_int, c_int, c_int, c_int, c_int, c_int, vp, vp]),
        "qconv_prepack_w_u4": (c_int, [vp, vp, vp, vp, vp, vp]),
        "q_lis_attn_v": (c_int, [vp, f32, vp, i64, c_int, c_int, c_int, c_int, vp, vp]),
        "qnn_status_string": (ctypes.c_char_p, [c_int]),
        "qnn_check_device_error": (c_int, [vp]),
        "qnn_selftest_wait_timeout": (c_int, [ctypes.c_uint64, vp]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(L, name)
        fn.restype = res
        fn.argtypes = args
        _SYMBOLS[name] = fn


def lib_path() -> str:
    return _build.LIB


def load(build_if_missing: bool = True) -> ctypes.CDLL:
    """Loads libqnn.so (building it first if it is missing or stale)."""
    global _lib
    if _lib is None:
        path = _build.LIB
        if build_if_missing and not _build.up_to_date():
            _build.build()
        if not os.path.exists(path):
            raise RuntimeError(f"libqnn.so not found at {path}: build it with "
                               "integer_quantized_nn_gb300.build.build()")
        L = ctypes.CDLL(path)
        _declare(L)
        _lib = L
    return _lib


def status_string(status: int) -> str:
    load()
    return _SYMBOLS["qnn_status_string"](int(status)).decode()


def _check(status: int, what: str):
    if status != QNN_OK:
        raise QnnError(status, what)


def _ptr(t) -> Optional[int]:
    if t is None:
        return None
    return int(t.data_ptr())


def _nbytes(t) -> int:
    return int(t.numel()) * int(t.element_size())


def _stream(stream) -> Optional[int]:
    if stream is not None:
        return int(getattr(stream, "cuda_stream", stream))
    import torch
    return int(torch.cuda.current_stream().cuda_stream)


def _shape(shape):
    arr = (ctypes.c_int64 * len(shape))(*[int(s) for s in shape])
    return arr


def qparams(scheme="sym", scale=None, zero_point=None, shift=None, per_channel=False, axis=0,
            narrow_range=False) -> QParams:
    return QParams(SCHEMES[scheme], int(per_channel), int(axis), int(narrow_range), _ptr(scale),
                   _ptr(zero_point), _ptr(shift))


def q_quantize(x, q, q_dt: str, params: QParams, shape=None, stream=None):
    """x: fp32 device tensor; q: uint8/int8 device tensor holding the codes
    (4-bit: packed, last dimension halved).  shape: logical shape (default x.shape)."""
    shp = tuple(x.shape) if shape is None else tuple(shape)
    load()
    _check(_SYMBOLS["q_quantize"](_ptr(x), _ptr(q), DTYPES[q_dt], len(shp), _shape(shp),
                                  ctypes.byref(params), _stream(stream)), "q_quantize")


def q_dequantize(q, q_dt: str, x, params: QParams, shape=None, stream=None):
    shp = tuple(x.shape) if shape is None else tuple(shape)
    load()
    _check(_SYMBOLS["q_dequantize"](_ptr(q), DTYPES[q_dt], _ptr(x), len(shp), _shape(shp),
                                    ctypes.byref(params), _stream(stream)), "q_dequantize")


def qnn_gemm_packed_b_bytes(N: int, K: int) -> int:
    load()
    return int(_SYMBOLS["qnn_gemm_packed_b_bytes"](int(N), int(K)))


def qgemm_prepack_b(B, B_packed, colsum=None, stream=None):
    """B: int8 [N, K] device tensor; B_packed: uint8 device tensor of
    qnn_gemm_packed_b_bytes(N, K) bytes, 1024-byte aligned."""
    N, K = B.shape
    load()
    _check(_SYMBOLS["qgemm_prepack_b"](_ptr(B), int(N), int(K), _ptr(B_packed), _ptr(colsum),
                                       _stream(stream)), "qgemm_prepack_b")


def q_fold_epilogue(N, a_dt: str, z_a: int, colsum, s_a: float, s_w, s_o: float, bias=None,
                    zp_term=None, M=None, Bq=None, D=None, w_per_channel=True, stream=None):
    load()
    _check(_SYMBOLS["q_fold_epilogue"](int(N), DTYPES[a_dt], int(z_a), _ptr(colsum), float(s_a),
                                       _ptr(s_w), int(w_per_channel), _ptr(bias), float(s_o),
                                       _ptr(zp_term), _ptr(M), _ptr(Bq), _ptr(D), _stream(stream)),
           "q_fold_epilogue")


def epilogue(mode="requant", relu=False, out_dt="s8", z_out=0, zp_term=None, M=None, Bq=None,
             D=None, bias=None, residual=None, res_dt="s8", z_res=0, R=0.0, ptf_shift=None,
             ptf_max_shift=0, row_scale=None) -> Epilogue:
    return Epilogue(EPI_MODES[mode], int(relu), DTYPES[out_dt], int(z_out), _ptr(zp_term), _ptr(M),
                    _ptr(Bq), _ptr(D), _ptr(bias), _ptr(residual), DTYPES[res_dt], int(z_res),
                    float(R), _ptr(ptf_shift), int(ptf_max_shift), _ptr(row_scale))


def qnn_gemm_workspace_bytes(M: int, K: int) -> int:
    load()
    return int(_SYMBOLS["qnn_gemm_workspace_bytes"](int(M), int(K)))


def qgemm_s8(A, a_dt: str, B_packed, M: int, N: int, K: int, epi: Epilogue, C, C_s32=None,
             workspace=None, stream=None):
    """workspace: optional uint8 device tensor of at least
    qnn_gemm_workspace_bytes(M, K) bytes (the pre-pass path); None: no scratch."""
    load()
    ws_bytes = 0 if workspace is None else _nbytes(workspace)
    _check(_SYMBOLS["qgemm_s8"](_ptr(A), DTYPES[a_dt], _ptr(B_packed), int(M), int(N), int(K),
                                ctypes.byref(epi), _ptr(C), _ptr(C_s32), _ptr(workspace),
                                ctypes.c_size_t(ws_bytes), _stream(stream)),
           "qgemm_s8")


def qgemm_pack_a(A, a_dt: str, M: int, K: int, A_packed, ptf_shift=None, stream=None):
    """Re-encodes A into A_packed (uint8 device tensor of at least
    qnn_gemm_workspace_bytes(M, K) bytes) for qgemm_s8_packed."""
    load()
    _check(_SYMBOLS["qgemm_pack_a"](_ptr(A), DTYPES[a_dt], int(M), int(K), _ptr(ptf_shift),
                                    _ptr(A_packed), ctypes.c_size_t(_nbytes(A_packed)),
                                    _stream(stream)), "qgemm_pack_a")


def qgemm_s8_packed(A_packed, a_dt: str, B_packed, M: int, N: int, K: int, epi: Epilogue, C,
                    C_s32=None, stream=None):
    load()
    _check(_SYMBOLS["qgemm_s8_packed"](_ptr(A_packed), DTYPES[a_dt], _ptr(B_packed), int(M), int(N),
                                       int(K), ctypes.byref(epi), _ptr(C), _ptr(C_s32),
                                       _stream(stream)), "qgemm_s8_packed")


QNN_GEMM_STATIC_SCRATCH_BYTES = 32 << 20


def qgemm_s8_static_scratch(A, a_dt: str, B_packed, M: int, N: int, K: int, epi: Epilogue, C,
                            C_s32=None, stream=None):
    """qgemm_s8 for callers that cannot allocate at call time: the workspace is
    the library's fixed device array (QNN_GEMM_STATIC_SCRATCH_BYTES); calls
    that overlap in time race on it."""
    load()
    _check(_SYMBOLS["qgemm_s8_static_scratch"](_ptr(A), DTYPES[a_dt], _ptr(B_packed), int(M), int(N),
                                               int(K), ctypes.byref(epi), _ptr(C), _ptr(C_s32),
                                               _stream(stream)), "qgemm_s8_static_scratch")


LAYOUTS = {"nhwc": 0, "nchw": 1, "nchw64": 2}


def conv_geom(N, H, W, C, OC, FH, FW, pad=(1, 1), stride=(1, 1), layout="nhwc") -> ConvGeom:
    return ConvGeom(N, H, W, C, OC, FH, FW, pad[0], pad[1], stride[0], stride[1], LAYOUTS[layout])


def qnn_conv_packed_w_bytes(g: ConvGeom, w_dt: str = "s4") -> int:
    load()
    return int(_SYMBOLS["qnn_conv_packed_w_bytes"](ctypes.byref(g), DTYPES[w_dt]))


def qconv_prepack_w(W, w_dt: str, g: ConvGeom, W_packed, colsum=None, stream=None):
    load()
    _check(_SYMBOLS["qconv_prepack_w"](_ptr(W), DTYPES[w_dt], ctypes.byref(g), _ptr(W_packed),
                                       _ptr(colsum), _stream(stream)), "qconv_prepack_w")


def qconv_prepack_w_u4(W, z_w, g: ConvGeom, W_packed, colsum=None, stream=None):
    """u4 filters (packed nibbles, OHWI) with per-filter zero points z_w (int32 [OC])."""
    load()
    _check(_SYMBOLS["qconv_prepack_w_u4"](_ptr(W), _ptr(z_w), ctypes.byref(g), _ptr(W_packed), _ptr(colsum),
                                           _stream(stream)), "qconv_prepack_w_u4")


def qconv_prepack_w_u8(W, z_w, g: ConvGeom, W_packed, colsum=None, stream=None):
    """u8 filters (bytes, OHWI) with per-filter zero points z_w (int32 [OC]), for qconv_u8u8."""
    load()
    _check(_SYMBOLS["qconv_prepack_w_u8"](_ptr(W), _ptr(z_w), ctypes.byref(g), _ptr(W_packed), _ptr(colsum),
                                           _stream(stream)), "qconv_prepack_w_u8")


def qnn_conv_workspace_bytes(g: ConvGeom, in_dt: str = "u4") -> int:
    load()
    return int(_SYMBOLS["qnn_conv_workspace_bytes"](ctypes.byref(g), DTYPES[in_dt]))


def qconv_u4s4(I, z_in: int, W_packed, g: ConvGeom, epi: Epilogue, O, O_s32=None, workspace=None,
               stream=None):
    """workspace: optional uint8 device tensor of at least
    qnn_conv_workspace_bytes(g, "u4") bytes (the pre-pass + TMA path)."""
    load()
    ws_bytes = 0 if workspace is None else _nbytes(workspace)
    _check(_SYMBOLS["qconv_u4s4"](_ptr(I), int(z_in), _ptr(W_packed), ctypes.byref(g),
                                  ctypes.byref(epi), _ptr(O), _ptr(O_s32), _ptr(workspace),
                                  ctypes.c_size_t(ws_bytes), _stream(stream)),
           "qconv_u4s4")


def qconv_u8s8(I, z_in: int, W_packed, g: ConvGeom, epi: Epilogue, O, O_s32=None, workspace=None, stream=None):
    """workspace: optional uint8 device tensor of at least qnn_conv_workspace_bytes(g, "u8") bytes."""
    load()
    ws_bytes = 0 if workspace is None else _nbytes(workspace)
    _check(_SYMBOLS["qconv_u8s8"](_ptr(I), int(z_in), _ptr(W_packed), ctypes.byref(g),
                                  ctypes.byref(epi), _ptr(O), _ptr(O_s32), _ptr(workspace),
                                  ctypes.c_size_t(ws_bytes), _stream(stream)),
           "qconv_u8s8")


def qconv_u8u8(I, z_in: int, W_packed, g: ConvGeom, epi: Epilogue, O, O_s32=None, workspace=None, stream=None):
    """u8 activations x u8 filters prepacked by qconv_prepack_w_u8."""
    load()
    ws_bytes = 0 if workspace is None else _nbytes(workspace)
    _check(_SYMBOLS["qconv_u8u8"](_ptr(I), int(z_in), _ptr(W_packed), ctypes.byref(g),
                                  ctypes.byref(epi), _ptr(O), _ptr(O_s32), _ptr(workspace),
                                  ctypes.c_size_t(ws_bytes), _stream(stream)),
           "qconv_u8u8")


def qgemm_prepack_b_u8(B, z_w, B_packed, colsum=None, stream=None):
    """u8 weights [N, K] with per-channel zero points z_w (int32 [N])."""
    load()
    N, K = B.shape
    _check(_SYMBOLS["qgemm_prepack_b_u8"](_ptr(B), _ptr(z_w), N, K, _ptr(B_packed), _ptr(colsum), _stream(stream)),
           "qgemm_prepack_b_u8")


def qgemm_prepack_b_ptf(B, ptf_shift, B_packed, colsum=None, stream=None):
    """s8 weights [N, K] times 2^ptf_shift[k] (u8 [K], each 0..3) folded into the image."""
    load()
    N, K = B.shape
    _check(_SYMBOLS["qgemm_prepack_b_ptf"](_ptr(B), _ptr(ptf_shift), N, K, _ptr(B_packed), _ptr(colsum),
                                           _stream(stream)), "qgemm_prepack_b_ptf")


def qnn_gemm_zw_workspace_bytes(M: int, K: int) -> int:
    load()
    return int(_SYMBOLS["qnn_gemm_zw_workspace_bytes"](int(M), int(K)))


def qgemm_zw(A, a_dt: str, B_packed, z_w, M: int, N: int, K: int, epi: Epilogue, C, C_s32=None, workspace=None,
             stream=None):
    """qgemm_s8 for u8 weights with zero points (the run-time row-sum term)."""
    load()
    ws_bytes = 0 if workspace is None else _nbytes(workspace)
    _check(_SYMBOLS["qgemm_zw"](_ptr(A), DTYPES[a_dt], _ptr(B_packed), _ptr(z_w), int(M), int(N), int(K),
                                ctypes.byref(epi), _ptr(C), _ptr(C_s32), _ptr(workspace), ws_bytes, _stream(stream)),
           "qgemm_zw")


def q_log_int_softmax(x, rows: int, L: int, S: float, bits: int, code, stream=None):
    """Log-Int-Softmax of int32 rows x [rows, L] into u8 log2 codes (2^bits: masked)."""
    load()
    _check(_SYMBOLS["q_log_int_softmax"](_ptr(x), int(rows), int(L), float(S), int(bits), _ptr(code),
                                          _stream(stream)), "q_log_int_softmax")


def q_attn_shift_v(code, v, batch: int, Lq: int, Lk: int, d: int, bits: int, out, stream=None):
    """out[b, i, j] = sum_t 2^(2^bits - 1 - code[b, i, t]) v[b, t, j] (int32)."""
    load()
    _check(_SYMBOLS["q_attn_shift_v"](_ptr(code), _ptr(v), int(batch), int(Lq), int(Lk), int(d),
                                       int(bits), _ptr(out), _stream(stream)), "q_attn_shift_v")


def q_int_layernorm(x, rows: int, C: int, s: float, gamma, beta, out_scale, y, y_dt: str = "s8",
                    alpha=None, alpha_max: int = 0, stream=None):
    """Integer LayerNorm of s8 rows x [rows, C] with PTF factors alpha (u8 [C])."""
    load()
    _check(_SYMBOLS["q_int_layernorm"](_ptr(x), int(rows), int(C), _ptr(alpha), int(alpha_max), float(s),
                                        _ptr(gamma), _ptr(beta), _ptr(out_scale), DTYPES[y_dt], _ptr(y),
                                        _stream(stream)), "q_int_layernorm")


def q_eltwise_s8(op: str, a, b, n: int, M: float, out, relu: bool = False, stream=None):
    """Quantized elementwise add / mul / relu on s8 codes."""
    load()
    _check(_SYMBOLS["q_eltwise_s8"](ELTWISE_OPS[op], _ptr(a), _ptr(b), int(n), float(M), int(relu), _ptr(out),
                                     _stream(stream)), "q_eltwise_s8")


def q_quantize_rows_dynamic(x, rows: int, cols: int, q, scale, narrow: bool = False, stream=None):
    """Per-row scale max|x| / 127 and s8 codes."""
    load()
    _check(_SYMBOLS["q_quantize_rows_dynamic"](_ptr(x), int(rows), int(cols), int(narrow), _ptr(q), _ptr(scale),
                                                _stream(stream)), "q_quantize_rows_dynamic")


def q_layout_nchw64(src, to_nchw64: bool, N: int, H: int, W: int, C: int, dt: str, dst, stream=None):
    """NHWC <-> NCHW64 block permutation of packed codes."""
    load()
    _check(_SYMBOLS["q_layout_nchw64"](_ptr(src), int(bool(to_nchw64)), int(N), int(H), int(W), int(C), DTYPES[dt],
                                        _ptr(dst), _stream(stream)), "q_layout_nchw64")


def q_lis_attn_v(x, S: float, v, batch: int, Lq: int, Lk: int, d: int, bits: int, out, stream=None):
    """Log-Int-Softmax of int32 logits x and the shift product with v in one kernel."""
    load()
    _check(_SYMBOLS["q_lis_attn_v"](_ptr(x), float(S), _ptr(v), int(batch), int(Lq), int(Lk), int(d), int(bits),
                                     _ptr(out), _stream(stream)), "q_lis_attn_v")


def qnn_check_device_error(stream=None) -> int:
    """Synchronises the stream; returns the status (does not raise)."""
    load()
    return int(_SYMBOLS["qnn_check_device_error"](_stream(stream)))


def qnn_selftest_wait_timeout(limit_ns: int, stream=None):
    load()
    _check(_SYMBOLS["qnn_selftest_wait_timeout"](int(limit_ns), _stream(stream)),
           "qnn_selftest_wait_timeout")
