"""Shared helpers for the tests: moving arrays to the device and running the
GEMM / conv paths end to end on both sides (CUDA library and CPU oracle).

The two sides share only the seeded inputs: the CUDA side goes through the
C ABI (integer_quantized_nn_gb300.qnn), the oracle side through oracle/."""
from __future__ import annotations

import numpy as np

from integer_quantized_nn_gb300 import qnn


def torch():
    import torch as _t
    return _t


def dev(a):
    t = torch()
    return t.from_numpy(np.ascontiguousarray(a)).cuda()


def host(t):
    return t.detach().cpu().numpy()


def aligned_empty(nbytes, align=1024, dtype=None):
    """Device uint8 buffer of nbytes whose data_ptr is `align`-byte aligned."""
    t = torch()
    buf = t.empty(nbytes + align, dtype=t.uint8, device="cuda")
    off = (-buf.data_ptr()) % align
    return buf[off:off + nbytes]


def gpu_gemm_setup(B, a_dt, z_a, s_a, s_w, s_o, bias=None):
    """Prepack + fold on the device.  Returns dict of device tensors."""
    t = torch()
    N, K = B.shape
    Bd = dev(B.astype(np.int8))
    Bp = aligned_empty(qnn.qnn_gemm_packed_b_bytes(N, K))
    colsum = t.empty(N, dtype=t.int32, device="cuda")
    qnn.qgemm_prepack_b(Bd, Bp, colsum)
    sw = dev(np.asarray(s_w, np.float32).reshape(-1))
    bd = None if bias is None else dev(np.asarray(bias, np.float32))
    zp = t.empty(N, dtype=t.int32, device="cuda")
    Mv = t.empty(N, dtype=t.float32, device="cuda")
    Bq = t.empty(N, dtype=t.float32, device="cuda")
    D = t.empty(N, dtype=t.float32, device="cuda")
    qnn.q_fold_epilogue(N, a_dt, z_a, colsum, s_a, sw, s_o, bias=bd, zp_term=zp, M=Mv, Bq=Bq, D=D,
                        w_per_channel=sw.numel() == N and N > 1)
    return dict(Bd=Bd, Bp=Bp, colsum=colsum, zp=zp, M=Mv, Bq=Bq, D=D, bias=bd, sw=sw)


def library_zp_term(zp_page, colsum, centre):
    """The zero-point term in the library's operand encoding.  The oracle folds
    the page's term Z_a * colsum (sum (q - Z_a) w = sum q w - Z_a colsum); the
    library feeds a u8 operand to the MMA as q - 128 (centre 128), so the term it
    subtracts is sum (q - 128) w - sum (q - Z_a) w = (Z_a - 128) colsum =
    Z_a colsum - 128 colsum."""
    z = np.asarray(zp_page, np.int64) - int(centre) * np.asarray(colsum, np.int64)
    assert np.all(np.abs(z) < 2 ** 31)
    return z.astype(np.int32)


def oracle_fold(oracle, B, a_dt, z_a, s_a, s_w, s_o, bias=None):
    """Oracle fold (the page's zp_term = Z_a * colsum), with zp_term translated
    to the library's encoding for comparison with q_fold_epilogue."""
    cs = oracle.colsum(B.astype(np.int32))
    centre = 128 if a_dt == "u8" else 0
    zp, Mv, Bq, D = oracle.fold(cs, z_a, s_a, np.asarray(s_w, np.float32), s_o, bias)
    return library_zp_term(zp, cs, centre), Mv, Bq, D, cs


def f32_bits(a):
    return np.ascontiguousarray(a, np.float32).view(np.uint32)
