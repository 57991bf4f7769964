"""Host-side checks of the C ABI (no GPU needed): the library builds for
sm_103a, loads, exports every function include/qnn.h declares, and rejects
invalid arguments before launching anything."""
import ctypes
import os
import re

import pytest

from integer_quantized_nn_gb300 import qnn

pytestmark = pytest.mark.cpu
HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "qnn.h")


def _declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = re.findall(r"^[A-Za-z_][\w\s\*]*?\b([a-z_][a-z0-9_]*)\s*\(", src, flags=re.M)
    return sorted(set(n for n in names if n not in ("if", "sizeof")))


@pytest.fixture(scope="module")
def lib():
    return qnn.load()


def test_header_declares_the_boundary():
    names = _declared_functions()
    for n in ("q_quantize", "q_dequantize", "qgemm_prepack_b", "q_fold_epilogue", "qgemm_s8",
              "qnn_gemm_workspace_bytes", "qgemm_pack_a", "qgemm_s8_packed", "qgemm_s8_static_scratch",
              "qgemm_prepack_b_ptf",
              "qconv_prepack_w", "qconv_u4s4", "qconv_u8s8", "qnn_conv_workspace_bytes",
              "q_log_int_softmax", "q_attn_shift_v", "q_lis_attn_v", "q_int_layernorm", "q_eltwise_s8",
              "q_quantize_rows_dynamic", "qgemm_prepack_b_u8", "qgemm_zw", "qnn_gemm_zw_workspace_bytes",
              "q_layout_nchw64", "qconv_prepack_w_u4", "qconv_prepack_w_u8", "qconv_u8u8", "qnn_status_string",
              "qnn_check_device_error"):
        assert n in names


def _declared_arities():
    """Function name -> number of parameters, from the header's prototypes."""
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    out = {}
    for m in re.finditer(r"^[A-Za-z_][\w\s\*]*?\b([a-z_][a-z0-9_]*)\s*\(([^)]*)\)\s*;", src, flags=re.M | re.S):
        args = m.group(2).strip()
        out[m.group(1)] = 0 if args in ("", "void") else args.count(",") + 1
    return out


def test_binding_matches_header_arity(lib):
    """Every function the binding declares exists in the header with the same
    number of parameters (a ctypes signature with a missing or extra argument
    would pass garbage across the boundary)."""
    arity = _declared_arities()
    assert len(arity) >= 30
    assert set(arity) == set(qnn._SYMBOLS), set(arity) ^ set(qnn._SYMBOLS)
    for name, fn in qnn._SYMBOLS.items():
        assert name in arity, name
        assert len(fn.argtypes) == arity[name], (name, len(fn.argtypes), arity[name])


def test_library_exports_every_declared_symbol(lib):
    missing = [n for n in _declared_functions() if not hasattr(lib, n)]
    assert not missing, missing


def test_status_strings(lib):
    assert qnn.status_string(qnn.QNN_OK) == "ok"
    assert "align" in qnn.status_string(qnn.QNN_ERR_ALIGNMENT)
    assert qnn.status_string(99) == "unknown status"


def test_invalid_arguments_rejected_on_host(lib):
    L = lib
    shape = (ctypes.c_int64 * 2)(4, 8)
    p = qnn.qparams("sym")
    # NULL tensors
    assert L.q_quantize(None, None, 0, 2, shape, ctypes.byref(p), None) == qnn.QNN_ERR_INVALID_ARG
    # bad dtype for a quantized tensor
    assert L.q_quantize(16, 16, 4, 2, shape, ctypes.byref(p), None) == qnn.QNN_ERR_INVALID_ARG
    # scheme needs a scale
    assert L.q_dequantize(16, 0, 16, 2, shape, ctypes.byref(p), None) == qnn.QNN_ERR_INVALID_ARG
    epi = qnn.epilogue("requant")
    # unsupported activation type, zero sizes
    assert L.qgemm_s8(16, 2, 1024, 4, 8, 16, ctypes.byref(epi), 16, None, None, 0, None) == qnn.QNN_ERR_UNSUPPORTED
    assert L.qgemm_s8(16, 0, 1024, 0, 8, 16, ctypes.byref(epi), 16, None, None, 0, None) == qnn.QNN_ERR_INVALID_ARG
    # K not a multiple of 16, misaligned weights
    assert L.qgemm_s8(16, 0, 1024, 4, 8, 24, ctypes.byref(epi), 16, None, None, 0, None) == qnn.QNN_ERR_ALIGNMENT
    assert L.qgemm_s8(16, 0, 1040, 4, 8, 32, ctypes.byref(epi), 16, None, None, 0, None) == qnn.QNN_ERR_ALIGNMENT
    # workspace smaller than qnn_gemm_workspace_bytes, or misaligned
    need = L.qnn_gemm_workspace_bytes(4, 32)
    assert need == 16384
    assert L.qnn_gemm_workspace_bytes(129, 65) == 2 * 2 * 16384
    assert L.qnn_gemm_workspace_bytes(0, 64) == 0
    ok_epi = qnn.epilogue("requant")
    ok_epi.M, ok_epi.Bq = 256, 512  # never dereferenced on the host
    assert L.qgemm_s8(16, 0, 1024, 4, 8, 32, ctypes.byref(ok_epi), 16, None, 4096, need - 1,
                      None) == qnn.QNN_ERR_INVALID_ARG
    assert L.qgemm_s8(16, 0, 1024, 4, 8, 32, ctypes.byref(ok_epi), 16, None, 4104, need,
                      None) == qnn.QNN_ERR_ALIGNMENT
    # the fixed-scratch form: sizes beyond its array are refused before any launch
    assert L.qnn_gemm_workspace_bytes(16384, 4096) > qnn.QNN_GEMM_STATIC_SCRATCH_BYTES
    assert L.qgemm_s8_static_scratch(16, 0, 1024, 16384, 8, 4096, ctypes.byref(ok_epi), 16, None,
                                     None) == qnn.QNN_ERR_UNSUPPORTED
    # conv workspace: its size, and a too-small one refused before any launch
    g = qnn.conv_geom(64, 56, 56, 64, 64, 3, 3)
    assert qnn.qnn_conv_workspace_bytes(g, "u4") == 64 * 56 * 56 * 64
    assert qnn.qnn_conv_workspace_bytes(g, "u8") == 2 * 64 * 56 * 56 * 64
    assert qnn.qnn_conv_workspace_bytes(g, "s8") == 0
    cneed = qnn.qnn_conv_workspace_bytes(g, "u4")
    assert L.qconv_u4s4(16, 8, 1024, ctypes.byref(g), ctypes.byref(ok_epi), 16, None, 4096, cneed - 1,
                        None) == qnn.QNN_ERR_INVALID_ARG
    assert L.qconv_u4s4(16, 8, 1024, ctypes.byref(g), ctypes.byref(ok_epi), 16, None, 4104, cneed,
                        None) == qnn.QNN_ERR_ALIGNMENT
    # the two-call form validates the same way
    assert L.qgemm_pack_a(16, 0, 4, 32, None, 4096, need - 1, None) == qnn.QNN_ERR_INVALID_ARG
    assert L.qgemm_pack_a(16, 0, 4, 24, None, 4096, need, None) == qnn.QNN_ERR_ALIGNMENT
    assert L.qgemm_pack_a(16, 1, 4, 32, 4096, 4096, need, None) == qnn.QNN_ERR_UNSUPPORTED
    assert L.qgemm_pack_a(None, 0, 4, 32, None, 4096, need, None) == qnn.QNN_ERR_INVALID_ARG
    assert L.qgemm_s8_packed(4096, 0, 1040, 4, 8, 32, ctypes.byref(ok_epi), 16, None,
                             None) == qnn.QNN_ERR_ALIGNMENT
    assert L.qgemm_prepack_b(16, 8, 24, 1024, None, None) == qnn.QNN_ERR_ALIGNMENT
    assert L.q_fold_epilogue(0, 0, 0, None, 1.0, None, 0, None, 1.0, None, None, None, None,
                             None) == qnn.QNN_ERR_INVALID_ARG
    # zero point outside the code range of the activation type
    assert L.q_fold_epilogue(8, 1, 300, 16, 1.0, 16, 0, None, 1.0, 16, None, None, None,
                             None) == qnn.QNN_ERR_INVALID_ARG
    assert L.qnn_selftest_wait_timeout(10 ** 10, None) == qnn.QNN_ERR_INVALID_ARG


def test_lis_arguments_rejected_on_host(lib):
    L = lib
    ok = qnn.QNN_OK
    # bits, lengths, scales
    assert L.q_log_int_softmax(16, 4, 8, 0.01, 0, 16, None) == qnn.QNN_ERR_INVALID_ARG
    assert L.q_log_int_softmax(16, 4, 8, 0.01, 6, 16, None) == qnn.QNN_ERR_INVALID_ARG
    assert L.q_log_int_softmax(16, 4, 0, 0.01, 4, 16, None) == qnn.QNN_ERR_INVALID_ARG
    assert L.q_log_int_softmax(16, 4, 8, 0.0, 4, 16, None) == qnn.QNN_ERR_INVALID_ARG
    assert L.q_log_int_softmax(16, 4, 8, float("inf"), 4, 16, None) == qnn.QNN_ERR_INVALID_ARG
    assert L.q_log_int_softmax(16, 4, 8, 50.0, 4, 16, None) == qnn.QNN_ERR_INVALID_ARG
    # c_int >= 2^31, and a row sum that could pass 2^64 (L c 2^30 >= 2^64)
    assert L.q_log_int_softmax(16, 4, 8, 2.0 ** -16, 4, 16, None) == qnn.QNN_ERR_OVERFLOW_RISK
    assert L.q_log_int_softmax(16, 4, 256, 2e-4, 4, 16, None) == qnn.QNN_ERR_OVERFLOW_RISK
    # nothing to do; NULL and misaligned tensors
    assert L.q_log_int_softmax(None, 0, 8, 0.01, 4, None, None) == ok
    assert L.q_log_int_softmax(None, 4, 8, 0.01, 4, 16, None) == qnn.QNN_ERR_INVALID_ARG
    assert L.q_log_int_softmax(20, 4, 8, 0.01, 4, 16, None) == qnn.QNN_ERR_ALIGNMENT
    # shift product
    assert L.q_attn_shift_v(16, 16, 1, 4, 8, 16, 5, 16, None) == qnn.QNN_ERR_INVALID_ARG
    assert L.q_attn_shift_v(16, 16, 1, 4, 8, 8, 4, 16, None) == qnn.QNN_ERR_UNSUPPORTED
    assert L.q_attn_shift_v(16, 16, 1, 4, 513, 16, 4, 16, None) == qnn.QNN_ERR_OVERFLOW_RISK
    assert L.q_attn_shift_v(16, 16, 1, 4, 512, 16, 4, 20, None) == qnn.QNN_ERR_ALIGNMENT
    assert L.q_attn_shift_v(None, None, 0, 4, 512, 16, 4, None, None) == ok


def test_int_layernorm_arguments_rejected_on_host(lib):
    L = lib
    args = lambda **k: dict(dict(x=16, rows=4, C=768, al=None, amax=0, s=0.1, g=16, b=16, o=16, dt=0, y=16), **k)

    def call(**k):
        a = args(**k)
        return L.q_int_layernorm(a["x"], a["rows"], a["C"], a["al"], a["amax"], a["s"], a["g"], a["b"], a["o"],
                                 a["dt"], a["y"], None)
    assert call(amax=4) == qnn.QNN_ERR_INVALID_ARG
    assert call(s=0.0) == qnn.QNN_ERR_INVALID_ARG
    assert call(s=float("inf")) == qnn.QNN_ERR_INVALID_ARG
    assert call(C=0) == qnn.QNN_ERR_INVALID_ARG
    assert call(dt=1) == qnn.QNN_ERR_UNSUPPORTED
    assert call(C=770) == qnn.QNN_ERR_ALIGNMENT
    assert call(C=8192, amax=3) == qnn.QNN_ERR_OVERFLOW_RISK
    assert call(rows=0, x=None, y=None) == qnn.QNN_OK
    assert call(x=None) == qnn.QNN_ERR_INVALID_ARG
    assert call(g=20) == qnn.QNN_ERR_ALIGNMENT


def test_eltwise_arguments_rejected_on_host(lib):
    L = lib
    assert L.q_eltwise_s8(3, 16, 16, 16, 1.0, 0, 16, None) == qnn.QNN_ERR_INVALID_ARG
    assert L.q_eltwise_s8(0, 16, 16, -1, 1.0, 0, 16, None) == qnn.QNN_ERR_INVALID_ARG
    assert L.q_eltwise_s8(1, 16, 16, 16, float("inf"), 0, 16, None) == qnn.QNN_ERR_INVALID_ARG
    assert L.q_eltwise_s8(0, 16, None, 16, 1.0, 0, 16, None) == qnn.QNN_ERR_INVALID_ARG
    assert L.q_eltwise_s8(0, 17, 16, 16, 1.0, 0, 16, None) == qnn.QNN_ERR_ALIGNMENT
    assert L.q_eltwise_s8(0, None, None, 0, 1.0, 0, None, None) == qnn.QNN_OK
    assert L.q_quantize_rows_dynamic(16, 2, 6, 0, 16, 16, None) == qnn.QNN_ERR_ALIGNMENT
    assert L.q_quantize_rows_dynamic(16, 2, 0, 0, 16, 16, None) == qnn.QNN_ERR_INVALID_ARG
    assert L.q_quantize_rows_dynamic(None, 2, 8, 0, 16, 16, None) == qnn.QNN_ERR_INVALID_ARG


def test_gemm_zw_arguments_rejected_on_host(lib):
    L = lib
    epi = qnn.epilogue("requant")
    epi.M, epi.Bq = 256, 512
    need = L.qnn_gemm_zw_workspace_bytes(4, 32)
    assert need == L.qnn_gemm_workspace_bytes(4, 32) + 256
    assert L.qnn_gemm_zw_workspace_bytes(300, 64) == L.qnn_gemm_workspace_bytes(300, 64) + 1280
    # no zero points, no workspace, a small one, PTF, K too large for int32
    assert L.qgemm_zw(16, 1, 1024, None, 4, 8, 32, ctypes.byref(epi), 16, None, 4096, need, None) == \
        qnn.QNN_ERR_INVALID_ARG
    assert L.qgemm_zw(16, 1, 1024, 16, 4, 8, 32, ctypes.byref(epi), 16, None, None, 0, None) == qnn.QNN_ERR_INVALID_ARG
    assert L.qgemm_zw(16, 1, 1024, 16, 4, 8, 32, ctypes.byref(epi), 16, None, 4096, need - 1, None) == \
        qnn.QNN_ERR_INVALID_ARG
    assert L.qgemm_zw(16, 1, 1024, 16, 4, 8, 40000, ctypes.byref(epi), 16, None, 4096, 1 << 40, None) == \
        qnn.QNN_ERR_OVERFLOW_RISK
    assert L.qgemm_zw(16, 1, 1024, 20, 4, 8, 32, ctypes.byref(epi), 16, None, 4096, need, None) == \
        qnn.QNN_ERR_ALIGNMENT
    assert L.qgemm_prepack_b_u8(16, None, 8, 32, 1024, None, None) == qnn.QNN_ERR_INVALID_ARG
    assert L.qgemm_prepack_b_u8(16, 16, 8, 24, 1024, None, None) == qnn.QNN_ERR_ALIGNMENT


def test_layout_arguments_rejected_on_host(lib):
    L = lib
    assert L.q_layout_nchw64(16, 1, 1, 2, 2, 96, 3, 16, None) == qnn.QNN_ERR_ALIGNMENT
    assert L.q_layout_nchw64(16, 1, 1, 2, 2, 64, 4, 16, None) == qnn.QNN_ERR_UNSUPPORTED
    assert L.q_layout_nchw64(16, 1, 1, 0, 2, 64, 3, 16, None) == qnn.QNN_ERR_INVALID_ARG
    assert L.q_layout_nchw64(None, 1, 0, 2, 2, 64, 3, None, None) == qnn.QNN_OK
    assert L.q_layout_nchw64(20, 1, 1, 2, 2, 64, 3, 16, None) == qnn.QNN_ERR_ALIGNMENT


def test_conv_u4_zero_point_prepack_rejected_on_host(lib):
    L = lib
    g = qnn.conv_geom(1, 8, 8, 64, 64, 3, 3)
    assert L.qconv_prepack_w_u4(16, None, ctypes.byref(g), 1024, None, None) == qnn.QNN_ERR_INVALID_ARG
    assert L.qconv_prepack_w_u4(16, 20, ctypes.byref(g), 1024, None, None) == qnn.QNN_ERR_ALIGNMENT
    big = qnn.conv_geom(1, 8, 8, 8320, 64, 3, 3)  # 9 * 8320 * 225 >= 2^24
    assert L.qconv_prepack_w_u4(16, 16, ctypes.byref(big), 1024, None, None) == qnn.QNN_ERR_OVERFLOW_RISK


def test_conv_u8_zero_point_rejected_on_host(lib):
    L = lib
    g = qnn.conv_geom(1, 8, 8, 64, 64, 3, 3)
    assert L.qconv_prepack_w_u8(16, None, ctypes.byref(g), 1024, None, None) == qnn.QNN_ERR_INVALID_ARG
    assert L.qconv_prepack_w_u8(16, 20, ctypes.byref(g), 1024, None, None) == qnn.QNN_ERR_ALIGNMENT
    assert L.qconv_prepack_w_u8(16, 16, ctypes.byref(g), 1040, None, None) == qnn.QNN_ERR_ALIGNMENT
    assert L.qconv_prepack_w_u8(20, 16, ctypes.byref(g), 1024, None, None) == qnn.QNN_ERR_ALIGNMENT
    odd = qnn.conv_geom(1, 8, 8, 8, 64, 3, 3)
    assert L.qconv_prepack_w_u8(16, 16, ctypes.byref(odd), 1024, None, None) == qnn.QNN_ERR_UNSUPPORTED
    # the u8 filters take the s8 image, the u4 filters the s4 one
    assert qnn.qnn_conv_packed_w_bytes(g, "u8") == qnn.qnn_conv_packed_w_bytes(g, "s8") > 0
    assert qnn.qnn_conv_packed_w_bytes(g, "u4") == qnn.qnn_conv_packed_w_bytes(g, "s4") > 0
    # 9 * 3680 * 255^2 > 2^31 - 1: refused before any launch
    epi = qnn.epilogue("requant", out_dt="u8")
    epi.M, epi.Bq = 256, 512  # never dereferenced on the host
    big = qnn.conv_geom(1, 8, 8, 3680, 64, 3, 3)
    assert L.qconv_u8u8(16, 8, 1024, ctypes.byref(big), ctypes.byref(epi), 16, None, None, 0,
                        None) == qnn.QNN_ERR_OVERFLOW_RISK


def test_packed_sizes(lib):
    # the operand image, then a 1 KB trailer of weight magnitude bounds
    assert qnn.qnn_gemm_packed_b_bytes(3072, 768) == 12 * 12 * 256 * 128 + 1024
    assert qnn.qnn_gemm_packed_b_bytes(300, 272) == 2 * 5 * 256 * 128 + 1024
    assert qnn.qnn_gemm_packed_b_bytes(0, 16) == 0


def test_struct_layouts_match_header(tmp_path):
    """The ctypes mirrors of qnn_qparams, qnn_epilogue and qnn_conv_geom have
    the C structs' size and field offsets: a C probe compiled against
    include/qnn.h (plain C, no CUDA headers) prints them."""
    import shutil
    import subprocess
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    structs = {"qnn_qparams": qnn.QParams, "qnn_epilogue": qnn.Epilogue, "qnn_conv_geom": qnn.ConvGeom}
    lines = ["#include <stdio.h>", "#include <stddef.h>", '#include "qnn.h"', "int main(void) {"]
    for cname, py in structs.items():
        lines.append(f'    printf("{cname} size %zu\\n", sizeof({cname}));')
        for fname, _ in py._fields_:
            lines.append(f'    printf("{cname} {fname} %zu\\n", offsetof({cname}, {fname}));')
    lines += ["    return 0;", "}"]
    src = tmp_path / "layout.c"
    src.write_text("\n".join(lines) + "\n")
    exe = tmp_path / "layout"
    subprocess.run([cc, "-I", os.path.dirname(HEADER), str(src), "-o", str(exe)], check=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout.split("\n")
    got = {tuple(l.split()[:2]): int(l.split()[2]) for l in out if l.strip()}
    for cname, py in structs.items():
        assert got[(cname, "size")] == ctypes.sizeof(py), cname
        for fname, _ in py._fields_:
            assert got[(cname, fname)] == getattr(py, fname).offset, (cname, fname)
