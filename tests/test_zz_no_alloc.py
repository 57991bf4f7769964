"""qgemm_s8_static_scratch (the fixed-scratch GEMM entry point) against
qgemm_s8: byte-identical outputs over two calls in a row with different shapes
and operand types, so that the second call cannot pass on what the first left
in the library's scratch array.  Kept in its own file, collected last."""
import numpy as np
import pytest

from integer_quantized_nn_gb300 import qnn, workloads
from _util import dev, host, gpu_gemm_setup, torch

pytestmark = pytest.mark.gpu


def _outputs(A, a_dt, B, z_a, s_w, s_o, bias, out_dt, alpha=None):
    t = torch()
    M, K = A.shape
    N = B.shape[0]
    g = gpu_gemm_setup(B, a_dt, z_a, 0.02, s_w, s_o, bias)
    al = None if alpha is None else dev(alpha.astype(np.uint8))
    epi = qnn.epilogue("requant", out_dt=out_dt, zp_term=None if al is not None else g["zp"],
                       M=g["M"], Bq=g["Bq"], ptf_shift=al,
                       ptf_max_shift=0 if alpha is None else int(alpha.max()))
    Ad = dev(A)
    ref = t.full((M, N), 0x5A, dtype=t.uint8, device="cuda")
    ref32 = t.zeros((M, N), dtype=t.int32, device="cuda")
    qnn.qgemm_s8(Ad, a_dt, g["Bp"], M, N, K, epi, ref, ref32)
    got = t.full((M, N), 0xA5, dtype=t.uint8, device="cuda")
    got32 = t.full((M, N), -1, dtype=t.int32, device="cuda")
    qnn.qgemm_s8_static_scratch(Ad, a_dt, g["Bp"], M, N, K, epi, got, got32)
    assert qnn.qnn_check_device_error() == qnn.QNN_OK
    return host(ref), host(ref32), host(got), host(got32)


def test_static_scratch_matches_qgemm_s8_two_calls():
    rng = np.random.default_rng(31)
    # call 1: ViT-B fc1 at full size (u8 with zero point, 19.5 MB of scratch)
    w = workloads.vit_fc1()
    r, r32, g, g32 = _outputs(w["A"], "u8", w["B"], w["z_a"], w["s_w"], w["s_o"], w["bias"], "s8")
    assert np.array_equal(g32, r32)
    assert np.array_equal(g, r)
    # call 2: a smaller, ragged s8 GEMM with PTF shifts, right after
    M, N, K = 389, 300, 272
    A = rng.integers(-128, 128, size=(M, K)).astype(np.int8)
    B = rng.integers(-128, 128, size=(N, K)).astype(np.int8)
    alpha = rng.integers(0, 4, size=K).astype(np.int32)
    s_w = rng.uniform(1e-3, 1e-2, size=N).astype(np.float32)
    bias = rng.normal(0, 1, size=N).astype(np.float32)
    r, r32, g, g32 = _outputs(A, "s8", B, 0, s_w, 0.5, bias, "s8", alpha=alpha)
    assert np.array_equal(g32, r32)
    assert np.array_equal(g, r)


def test_static_scratch_rejects_oversize():
    t = torch()
    M, K, N = 16384, 4096, 256   # needs 128 MiB > the 32 MiB array
    assert qnn.qnn_gemm_workspace_bytes(M, K) > qnn.QNN_GEMM_STATIC_SCRATCH_BYTES
    A = t.zeros((M, K), dtype=t.int8, device="cuda")
    Bp = t.zeros(qnn.qnn_gemm_packed_b_bytes(N, K) + 1024, dtype=t.uint8, device="cuda")
    off = (-Bp.data_ptr()) % 1024
    Mv = t.ones(N, dtype=t.float32, device="cuda")
    C = t.zeros((M, N), dtype=t.uint8, device="cuda")
    with pytest.raises(qnn.QnnError) as e:
        qnn.qgemm_s8_static_scratch(A, "s8", Bp[off:], M, N, K, qnn.epilogue("requant", M=Mv, Bq=Mv), C)
    assert e.value.status == qnn.QNN_ERR_UNSUPPORTED
