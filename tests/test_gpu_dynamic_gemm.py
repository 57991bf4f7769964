"""Dynamic per-token quantization feeding the GEMM: q_quantize_rows_dynamic's
per-row scales consumed by the qgemm_s8 epilogue (row_scale), against the CPU
oracle's chain (its dynamic quantization, GEMM accumulator and per-row-scale
requant / dequant); codes and fp32 bits bit-exact."""
import numpy as np
import pytest

from integer_quantized_nn_gb300 import qnn
from _util import aligned_empty, dev, host, f32_bits

pytestmark = pytest.mark.gpu


def _run(oracle, M, K, N, seed, mode, workspace, rows=None):
    t = __import__("torch")
    rng = np.random.default_rng(seed)
    x = (rng.standard_normal((M, K)) * rng.uniform(0.1, 4.0, (M, 1))).astype(np.float32)
    B = rng.integers(-128, 128, (N, K)).astype(np.int8)
    s_w = rng.uniform(1e-3, 1e-2, N).astype(np.float32)
    bias = rng.normal(0, 1, N).astype(np.float32)
    s_o = 0.05
    # dynamic quantization on the GPU
    q = t.empty((M, K), dtype=t.int8, device="cuda")
    sr = t.empty(M, dtype=t.float32, device="cuda")
    qnn.q_quantize_rows_dynamic(dev(x), M, K, q, sr)
    # weights, fold with s_a = 1: M = s_w / s_o, D = s_w
    Bp = aligned_empty(qnn.qnn_gemm_packed_b_bytes(N, K))
    cs = t.empty(N, dtype=t.int32, device="cuda")
    qnn.qgemm_prepack_b(dev(B), Bp, cs)
    Mv, Bq, D = (t.empty(N, dtype=t.float32, device="cuda") for _ in range(3))
    bd = dev(bias)
    qnn.q_fold_epilogue(N, "s8", 0, cs, 1.0, dev(s_w), s_o, bias=bd, M=Mv, Bq=Bq, D=D, w_per_channel=True)
    epi = qnn.epilogue(mode, out_dt="s8", M=Mv, Bq=Bq, D=D, bias=bd, row_scale=sr)
    C = t.zeros((M, N), dtype=t.uint8 if mode == "requant" else t.float32, device="cuda")
    ws = t.empty(qnn.qnn_gemm_workspace_bytes(M, K), dtype=t.uint8, device="cuda") if workspace else None
    qnn.qgemm_s8(q, "s8", Bp, M, N, K, epi, C, workspace=ws)
    assert qnn.qnn_check_device_error() == qnn.QNN_OK
    # the oracle's chain
    qo, so = oracle.quantize_rows_dynamic(x)
    assert np.array_equal(f32_bits(host(sr)), f32_bits(so))
    assert np.array_equal(host(q).astype(np.int32), qo)
    _, M_o, Bq_o, D_o = oracle.fold(oracle.colsum(B.astype(np.int32)), 0, 1.0, s_w, s_o, bias)
    sel = np.arange(M) if rows is None else rows
    acc = oracle.gemm_acc(qo[sel], B.astype(np.int32), 0)
    if mode == "requant":
        want = oracle.pack_bytes(oracle.requant_rowscale(acc, so[sel], M_o, Bq_o, "s8"))
        assert np.array_equal(host(C)[sel], want)
    else:
        want = oracle.dequant_rowscale(acc, so[sel], D_o, bias)
        assert np.array_equal(f32_bits(host(C)[sel]), f32_bits(want))


@pytest.mark.parametrize("mode", ["requant", "dequant"])
@pytest.mark.parametrize("workspace", [False, True])
@pytest.mark.parametrize("shape", [(256, 256, 256), (200, 208, 100), (96, 2048, 64)])
def test_dynamic_quant_gemm(oracle, mode, workspace, shape):
    M, K, N = shape
    _run(oracle, M, K, N, M + K, mode, workspace)


def test_dynamic_quant_gemm_vit_fc1(oracle):
    """The ViT-B fc1 shape (12608 x 768 -> 3072), 160 sampled rows."""
    rows = np.random.default_rng(41).choice(12608, 160, replace=False)
    _run(oracle, 12608, 768, 3072, 42, "requant", True, rows=rows)
