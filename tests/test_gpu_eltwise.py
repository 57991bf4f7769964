"""Standalone quantized elementwise ops and dynamic per-row quantization on the
GPU against the CPU oracle ("【量化】神经网络量化介绍": 量化加法, 量化乘法,
量化激活函数, 量化参数选择): codes and fp32 scale bits bit-exact, through the C ABI."""
import numpy as np
import pytest

from integer_quantized_nn_gb300 import qnn
from _util import dev, host, f32_bits

pytestmark = pytest.mark.gpu


def _elt_gpu(op, a, b, M, relu):
    t = __import__("torch")
    out = t.full(a.shape, 99, dtype=t.int8, device="cuda")
    qnn.q_eltwise_s8(op, dev(a.astype(np.int8)), dev(b.astype(np.int8)), a.size, M, out, relu=relu)
    t.cuda.synchronize()
    return host(out).astype(np.int32)


@pytest.mark.parametrize("n", [1, 15, 16, 17, 1000, (1 << 20) + 7])
@pytest.mark.parametrize("op", ["add", "mul", "relu"])
def test_eltwise(oracle, n, op):
    rng = np.random.default_rng(n)
    a = rng.integers(-128, 128, n).astype(np.int32)
    b = rng.integers(-128, 128, n).astype(np.int32)
    for M, relu in ((0.0123, False), (2.0 ** -7, True), (1.0, False), (0.5, True), (37.0, False)):
        want = oracle.eltwise_s8(op, a, b, M, relu)
        assert np.array_equal(_elt_gpu(op, a, b, M, relu), want), (op, n, M, relu)


def test_eltwise_all_pairs(oracle):
    """Every pair of s8 codes, both ops, a rescale with ties (M = 1/2, 1/4)."""
    a = np.arange(-128, 128).repeat(256).astype(np.int32)
    b = np.tile(np.arange(-128, 128), 256).astype(np.int32)
    for op in ("add", "mul"):
        for M in (0.5, 0.25, 1.0 / 3.0):
            assert np.array_equal(_elt_gpu(op, a, b, M, False), oracle.eltwise_s8(op, a, b, M))


def _dyn_gpu(x, narrow):
    t = __import__("torch")
    rows, cols = x.shape
    q = t.full((rows, cols), 99, dtype=t.int8, device="cuda")
    s = t.full((rows,), -1.0, dtype=t.float32, device="cuda")
    qnn.q_quantize_rows_dynamic(dev(x), rows, cols, q, s, narrow=narrow)
    t.cuda.synchronize()
    return host(q).astype(np.int32), host(s)


@pytest.mark.parametrize("shape", [(1, 4), (3, 132), (9, 500), (37, 768), (4, 1024), (5, 1028), (64 * 197, 768)])
def test_quantize_rows_dynamic(oracle, shape):
    rng = np.random.default_rng(shape[1])
    x = (rng.standard_normal(shape) * rng.uniform(0.01, 30.0, (shape[0], 1))).astype(np.float32)
    x[0, :] = 0.0
    if shape[0] > 3:
        x[3, 1] = 1e30
        x[2, :] = -1e-30
    for narrow in (False, True):
        q, s = _dyn_gpu(x, narrow)
        wq, ws = oracle.quantize_rows_dynamic(x, narrow)
        assert np.array_equal(f32_bits(s), f32_bits(ws))
        assert np.array_equal(q, wq), f"{(q != wq).sum()} mismatches"


def test_quantize_rows_dynamic_near_half_quotients(oracle):
    """Elements whose quotient x / s lies within a few units in the last place
    of a half-integer k + 1/2 (and exactly on it): rint(RN(x / s)) must follow
    the IEEE quotient, ties to even, in every row scale's binade."""
    rng = np.random.default_rng(11)
    rows, cols = 64, 256
    amax = (2.0 ** rng.uniform(-90, 90, size=rows) * rng.uniform(1.0, 2.0, size=rows)).astype(np.float32)
    amax[:4] = [127.0, 1.0, 3.0, 254.0]
    s = (amax / np.float32(127.0)).astype(np.float32)
    k = rng.integers(-127, 127, size=(rows, cols)).astype(np.float32) + np.float32(0.5)
    x = (k * s[:, None]).astype(np.float32)
    steps = rng.integers(-3, 4, size=(rows, cols))
    for d in range(1, 4):  # nudge by up to three units in the last place either way
        x = np.where(steps >= d, np.nextafter(x, np.float32(np.inf)), x)
        x = np.where(steps <= -d, np.nextafter(x, np.float32(-np.inf)), x)
    x = np.clip(x, -amax[:, None], amax[:, None]).astype(np.float32)
    x[:, 0] = amax  # the row maximum fixes s
    for narrow in (False, True):
        q, sg = _dyn_gpu(x, narrow)
        wq, ws = oracle.quantize_rows_dynamic(x, narrow)
        assert np.array_equal(f32_bits(sg), f32_bits(ws))
        assert np.array_equal(q, wq), f"{(q != wq).sum()} mismatches"


def test_eltwise_errors():
    t = __import__("torch")
    a = t.zeros(32, dtype=t.int8, device="cuda")
    qnn.q_eltwise_s8("add", a, a, 0, 1.0, a)  # nothing to do
    with pytest.raises(qnn.QnnError):
        qnn.q_eltwise_s8("add", a[1:], a, 16, 1.0, a)
    with pytest.raises(qnn.QnnError):
        qnn.q_eltwise_s8("mul", a, a, 16, float("nan"), a)
    x = t.zeros((2, 6), dtype=t.float32, device="cuda")
    s = t.zeros(2, dtype=t.float32, device="cuda")
    with pytest.raises(qnn.QnnError):
        qnn.q_quantize_rows_dynamic(x, 2, 6, a, s)


@pytest.mark.parametrize("dt", ["u4", "s8"])
@pytest.mark.parametrize("shape", [(1, 1, 1, 64), (2, 7, 5, 192), (64, 56, 56, 256)])
def test_layout_nchw64(oracle, dt, shape):
    """NHWC <-> NCHW64 (MegEngine's conv output layout) against the oracle's
    permutation of the codes, both directions, packed bytes compared."""
    t = __import__("torch")
    N, H, W, C = shape
    rng = np.random.default_rng(C + H)
    lo, hi = (0, 15) if dt == "u4" else (-128, 127)
    codes = rng.integers(lo, hi + 1, size=shape).astype(np.int32)
    pack = oracle.pack_nibbles if dt == "u4" else oracle.pack_bytes
    src = pack(codes)
    want = pack(oracle.nhwc_to_nchw64(codes))
    d_src = dev(src)
    d_dst = t.empty(want.size, dtype=t.uint8, device="cuda")
    qnn.q_layout_nchw64(d_src, True, N, H, W, C, dt, d_dst)
    back = t.empty(src.size, dtype=t.uint8, device="cuda")
    qnn.q_layout_nchw64(d_dst, False, N, H, W, C, dt, back)
    t.cuda.synchronize()
    assert np.array_equal(host(d_dst), want.reshape(-1))
    assert np.array_equal(host(back), src.reshape(-1))
