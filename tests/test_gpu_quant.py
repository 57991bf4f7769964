"""q_quantize / q_dequantize on the GPU against the CPU oracle: bit-exact codes
(packed bytes) and bit-exact fp32 values."""
import numpy as np
import pytest

from integer_quantized_nn_gb300 import qnn, workloads
from _util import dev, host, f32_bits

pytestmark = pytest.mark.gpu

SCHEME_ID = {"sym": 0, "asym": 1, "pow2": 2}


def _params_np(rng, scheme, dt, C, oracle):
    lo, hi = oracle.qrange(dt)
    scale = rng.uniform(0.005, 0.3, size=C).astype(np.float32)
    zp = rng.integers(lo, hi + 1, size=C).astype(np.int32) if scheme == "asym" else np.zeros(C, np.int32)
    shift = rng.integers(-2, 6, size=C).astype(np.int32)
    return scale, zp, shift


def _run_quant(oracle, x, dt, scheme, per_channel, axis, narrow=False, seed=0):
    rng = np.random.default_rng(seed)
    C = x.shape[axis] if per_channel else 1
    scale, zp, shift = _params_np(rng, scheme, dt, C, oracle)
    t = __import__("torch")
    xd = dev(x)
    packed_last = x.shape[-1] // 2 if dt in ("s4", "u4") else x.shape[-1]
    qd = t.zeros(x.shape[:-1] + (packed_last,), dtype=t.uint8, device="cuda")
    sd, zd, hd = dev(scale), dev(zp), dev(shift)
    p = qnn.qparams(scheme, scale=sd, zero_point=zd, shift=hd, per_channel=per_channel,
                    axis=axis, narrow_range=narrow)
    qnn.q_quantize(xd, qd, dt, p)
    codes = oracle.quantize(x, SCHEME_ID[scheme], dt, scale=scale, zp=zp, shift=shift,
                            per_channel=per_channel, axis=axis, narrow=narrow)
    exp = oracle.pack_nibbles(codes) if dt in ("s4", "u4") else oracle.pack_bytes(codes)
    got = host(qd)
    assert np.array_equal(got, exp), f"{(got != exp).sum()} byte mismatches"
    # dequantize the GPU codes on both sides
    yd = t.empty(x.shape, dtype=t.float32, device="cuda")
    qnn.q_dequantize(qd, dt, yd, p)
    y = oracle.dequantize(codes, SCHEME_ID[scheme], scale=scale, zp=zp, shift=shift,
                          per_channel=per_channel, axis=axis)
    assert np.array_equal(f32_bits(host(yd)), f32_bits(y))


@pytest.mark.parametrize("dt", ["s8", "u8", "s4", "u4"])
@pytest.mark.parametrize("scheme", ["sym", "asym", "pow2"])
def test_quantize_per_tensor(oracle, dt, scheme):
    rng = np.random.default_rng(1)
    x = rng.normal(0, 4, size=(37, 102)).astype(np.float32)   # 3774 elements: ragged tail
    x[0, :6] = [np.nan, np.inf, -np.inf, 1e30, -1e30, 0.0]
    _run_quant(oracle, x, dt, scheme, False, 0)


@pytest.mark.parametrize("axis", [0, 1, 2, -1])
@pytest.mark.parametrize("dt", ["s8", "u4"])
def test_quantize_per_channel(oracle, axis, dt):
    rng = np.random.default_rng(2)
    x = rng.normal(0, 2, size=(3, 24, 40)).astype(np.float32)
    _run_quant(oracle, x, dt, "asym" if dt == "u4" else "sym", True, axis, seed=3)
    _run_quant(oracle, x, dt, "pow2" if dt == "s8" else "asym", True, axis, seed=4)


def test_quantize_odd_channel_layout(oracle):
    rng = np.random.default_rng(5)
    x = rng.normal(0, 2, size=(5, 7, 6)).astype(np.float32)   # inner=6, C=7: generic path
    _run_quant(oracle, x, "u8", "asym", True, 1, seed=6)
    _run_quant(oracle, x, "s8", "sym", True, 2, narrow=True, seed=7)


def test_quantize_worked_example_on_gpu(oracle):
    """Quantization intro, 量化算子: 1.0 at scale 0.1 -> 10; ties go to even."""
    t = __import__("torch")
    x = dev(np.array([1.0, 1.5, -2.5, 0.5, -0.5, 2.5, 0, 0], np.float32))
    q = t.zeros(8, dtype=t.uint8, device="cuda")
    s = dev(np.array([1.0], np.float32))
    qnn.q_quantize(x, q, "s8", qnn.qparams("sym", scale=s))
    assert host(q).view(np.int8).tolist()[:6] == [1, 2, -2, 0, 0, 2]
    s = dev(np.array([0.1], np.float32))
    qnn.q_quantize(x, q, "s8", qnn.qparams("sym", scale=s))
    assert int(host(q).view(np.int8)[0]) == 10


def test_quantize_empty_and_errors(oracle):
    t = __import__("torch")
    x = t.empty((0, 8), dtype=t.float32, device="cuda")
    q = t.empty((0, 8), dtype=t.uint8, device="cuda")
    s = dev(np.array([1.0], np.float32))
    qnn.q_quantize(x, q, "s8", qnn.qparams("sym", scale=s))
    xo = t.zeros((4, 7), dtype=t.float32, device="cuda")
    qo = t.zeros((4, 4), dtype=t.uint8, device="cuda")
    with pytest.raises(qnn.QnnError) as e:
        qnn.q_quantize(xo, qo, "u4", qnn.qparams("sym", scale=s))
    assert e.value.status == qnn.QNN_ERR_INVALID_ARG
    xm = t.zeros(64, dtype=t.float32, device="cuda")[1:]
    with pytest.raises(qnn.QnnError) as e:
        qnn.q_quantize(xm, t.zeros(63, dtype=t.uint8, device="cuda"), "s8",
                       qnn.qparams("sym", scale=s))
    assert e.value.status == qnn.QNN_ERR_ALIGNMENT


def test_quantize_rows_full_size_sampled(oracle):
    """fp32 -> s8 per-row symmetric on a 16384 x 16384 (1 GiB) tensor, as timed by
    the benchmark; sampled rows are checked against the oracle byte for byte."""
    t = __import__("torch")
    R = Ccols = 16384
    x = workloads.device_normal_f32((R, Ccols), 505, "cuda")
    scale = (x.abs().amax(dim=1) / 127.0).contiguous()
    q = t.empty((R, Ccols), dtype=t.uint8, device="cuda")
    qnn.q_quantize(x, q, "s8", qnn.qparams("sym", scale=scale, per_channel=True, axis=0))
    rows = np.random.default_rng(9).choice(R, size=24, replace=False)
    rows.sort()
    xs = host(x[rows])
    ss = host(scale[rows])
    codes = oracle.quantize(xs, 0, "s8", scale=ss, per_channel=True, axis=0)
    assert np.array_equal(host(q[rows]), oracle.pack_bytes(codes))
    del x, q
