"""GEMM with weight zero points (Z_w != 0, the red term of the MegEngine
4-bit article, section 緩解精度下降) on the GPU against the CPU oracle: the
oracle's accumulator is sum_k (a_k - z_a)(w_k - z_w[n]) (its GEMM on the
zero-point-centred weights); int32 sums and requantized codes bit-exact."""
import numpy as np
import pytest

from integer_quantized_nn_gb300 import qnn
from _util import aligned_empty, dev, host, f32_bits, library_zp_term

pytestmark = pytest.mark.gpu


def _case(seed, M, N, K, a_dt):
    rng = np.random.default_rng(seed)
    if a_dt == "u8":
        A = np.clip(np.rint(rng.normal(128, 40, (M, K))), 0, 255).astype(np.uint8)
        z_a = int(rng.integers(0, 256))
    else:
        A = rng.integers(-128, 128, (M, K)).astype(np.int8)
        z_a = 0
    B = rng.integers(0, 256, (N, K)).astype(np.uint8)
    z_w = rng.integers(0, 256, N).astype(np.int32)
    s_w = rng.uniform(1e-3, 1e-2, N).astype(np.float32)
    bias = rng.normal(0, 1, N).astype(np.float32)
    return A, z_a, B, z_w, s_w, bias


def _run(oracle, A, a_dt, z_a, B, z_w, s_w, bias, s_a=0.02, s_o=None, rows=None):
    t = __import__("torch")
    M, K = A.shape
    N = B.shape[0]
    if s_o is None:
        s_o = float(np.float32(0.02 * 0.0055 * 255 * np.sqrt(K) * 3 / 127))
    Bp = aligned_empty(qnn.qnn_gemm_packed_b_bytes(N, K))
    cs = t.empty(N, dtype=t.int32, device="cuda")
    zwd = dev(z_w)
    qnn.qgemm_prepack_b_u8(dev(B), zwd, Bp, cs)
    zp = t.empty(N, dtype=t.int32, device="cuda")
    Mv = t.empty(N, dtype=t.float32, device="cuda")
    Bq = t.empty(N, dtype=t.float32, device="cuda")
    qnn.q_fold_epilogue(N, a_dt, z_a, cs, s_a, dev(s_w), s_o, bias=dev(bias), zp_term=zp, M=Mv, Bq=Bq,
                        w_per_channel=True)
    Bc = B.astype(np.int32) - z_w[:, None]  # the zero-point-centred weights
    cs_o = oracle.colsum(Bc)
    centre = 128 if a_dt == "u8" else 0
    zp_o, M_o, Bq_o, _ = oracle.fold(cs_o, z_a, s_a, s_w, s_o, bias)
    zp_o = library_zp_term(zp_o, cs_o, centre)
    assert np.array_equal(host(cs), cs_o)
    assert np.array_equal(host(zp), zp_o)
    assert np.array_equal(f32_bits(host(Mv)), f32_bits(M_o))
    epi = qnn.epilogue("requant", out_dt="s8", zp_term=zp, M=Mv, Bq=Bq)
    C = t.full((M, N), 0x5A, dtype=t.uint8, device="cuda")
    C32 = t.zeros((M, N), dtype=t.int32, device="cuda")
    ws = t.full((qnn.qnn_gemm_zw_workspace_bytes(M, K),), 0xFF, dtype=t.uint8, device="cuda")
    qnn.qgemm_zw(dev(A), a_dt, Bp, zwd, M, N, K, epi, C, C32, workspace=ws)
    assert qnn.qnn_check_device_error() == qnn.QNN_OK
    sel = np.arange(M) if rows is None else rows
    acc = oracle.gemm_acc(A[sel].astype(np.int32), Bc, z_a)
    assert np.array_equal(host(C32)[sel], acc)
    q = oracle.requant(acc, M_o, Bq_o, "s8")
    assert np.array_equal(host(C)[sel], oracle.pack_bytes(q))


@pytest.mark.parametrize("shape", [(256, 256, 256), (200, 100, 208), (1, 8, 16), (130, 300, 1024), (160, 96, 2048)])
@pytest.mark.parametrize("a_dt", ["u8", "s8"])
def test_gemm_zw(oracle, shape, a_dt):
    """u8 x u8 and s8 x u8, ragged M / N / K, one and two exact K chunks."""
    A, z_a, B, z_w, s_w, bias = _case(shape[0] * 7 + shape[2], *shape, a_dt)
    _run(oracle, A, a_dt, z_a, B, z_w, s_w, bias)


def test_gemm_zw_extreme_codes(oracle):
    """Every code 0 or 255 with zero points at both ends: the sums reach the
    largest magnitudes the int32 check allows for."""
    M, N, K = 128, 64, 512
    A = np.where(np.arange(M * K).reshape(M, K) % 3 == 0, 255, 0).astype(np.uint8)
    B = np.where(np.arange(N * K).reshape(N, K) % 5 == 0, 0, 255).astype(np.uint8)
    z_w = np.tile(np.array([0, 255, 128, 1], np.int32), N // 4)
    _run(oracle, A, "u8", 255, B, z_w, np.full(N, 1e-3, np.float32), np.zeros(N, np.float32), s_o=50.0)


def test_gemm_zw_vit_fc1_size(oracle):
    """u8 x u8 at the ViT-B fc1 shape (12608 x 3072 x 768), 160 sampled rows."""
    A, z_a, B, z_w, s_w, bias = _case(11, 12608, 3072, 768, "u8")
    rows = np.random.default_rng(12).choice(12608, 160, replace=False)
    _run(oracle, A, "u8", z_a, B, z_w, s_w, bias, rows=rows)
