"""Integer LayerNorm over PTF-quantized rows on the GPU against the CPU oracle
("首个完全量化Vision Transformer的方法FQ-ViT", section 3.2): output codes
bit-exact, through the C ABI."""
import os

import numpy as np
import pytest

from integer_quantized_nn_gb300 import qnn, workloads
from _util import dev, host

pytestmark = pytest.mark.gpu
GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "int_layernorm_worked_example.txt")


def _ln_gpu(x, s, gamma, beta, o, alpha=None, y_dt="s8"):
    t = __import__("torch")
    rows, C = x.shape
    alpha_max = 0 if alpha is None else int(alpha.max())
    y = t.full((rows, C), 77, dtype=t.int8 if y_dt == "s8" else t.int32, device="cuda")
    qnn.q_int_layernorm(dev(x.astype(np.int8)), rows, C, s, dev(np.asarray(gamma, np.float32)),
                        dev(np.asarray(beta, np.float32)), dev(np.asarray(o, np.float32)), y, y_dt=y_dt,
                        alpha=None if alpha is None else dev(alpha.astype(np.uint8)), alpha_max=alpha_max)
    t.cuda.synchronize()
    return host(y).astype(np.int64)


def _want(oracle, x, s, gamma, beta, o, alpha, y_dt):
    y = oracle.int_layernorm(x.astype(np.int32), s, gamma, beta, o, alpha=alpha)
    lo, hi = (-128, 127) if y_dt == "s8" else (-(2 ** 31), 2 ** 31 - 1)
    return np.clip(y, lo, hi)


def test_int_layernorm_golden():
    n = 0
    for line in open(GOLDEN):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        head, al, xs, ys = (p.split() for p in line.split("|"))
        s, g, b, o = (float(v) for v in head)
        x = np.array([[int(v) for v in xs]], np.int32)
        alpha = np.array([int(v) for v in al], np.uint8)
        C = x.shape[1]
        got = _ln_gpu(x, s, np.full(C, g), np.full(C, b), np.full(C, o), alpha=alpha, y_dt="s32")
        assert got[0].tolist() == [int(v) for v in ys], line
        n += 1
    assert n >= 5


@pytest.mark.parametrize("C", [4, 8, 64, 192, 768, 1024, 4096])
@pytest.mark.parametrize("y_dt", ["s8", "s32"])
def test_int_layernorm_random(oracle, C, y_dt):
    rng = np.random.default_rng(C)
    rows = 37
    x = np.clip(np.rint(rng.normal(0, 40, size=(rows, C))), -128, 127).astype(np.int32)
    amax = 2 if C == 4096 else 3
    alpha = rng.integers(0, amax + 1, size=C).astype(np.uint8)
    gamma = (rng.uniform(0.2, 2.0, size=C) * rng.choice([-1, 1], size=C)).astype(np.float32)
    gamma[::17] = 0.0  # A = 0: N = 31, M = 0
    beta = rng.normal(0, 0.5, size=C).astype(np.float32)
    o = rng.uniform(0.005, 0.05, size=C).astype(np.float32)
    for s, al in ((0.02, alpha), (0.37, None)):
        want = _want(oracle, x, s, gamma, beta, o, al, y_dt)
        got = _ln_gpu(x, s, gamma, beta, o, alpha=al, y_dt=y_dt)
        assert np.array_equal(got, want), f"{(got != want).sum()} mismatches"


def test_int_layernorm_edge_rows(oracle):
    """Constant rows (variance numerator 0), full-scale rows, a single outlier,
    tiny and huge gamma / o ratios."""
    C = 64
    rows = [np.full(C, -128), np.full(C, 127), np.full(C, 0), np.array([-128, 127] * 32),
            np.array([127] + [0] * 63), np.array([1, -1] * 32), np.arange(-32, 32)]
    x = np.stack(rows).astype(np.int32)
    rng = np.random.default_rng(3)
    alpha = rng.integers(0, 4, size=C).astype(np.uint8)
    for g, o in ((1.0, 0.05), (1e-6, 1.0), (50.0, 1e-3), (-2.0, 0.01)):
        gamma = np.full(C, g, np.float32)
        beta = rng.normal(0, 1, size=C).astype(np.float32)
        ov = np.full(C, o, np.float32)
        for y_dt in ("s8", "s32"):
            assert np.array_equal(_ln_gpu(x, 0.1, gamma, beta, ov, alpha=alpha, y_dt=y_dt),
                                  _want(oracle, x, 0.1, gamma, beta, ov, alpha, y_dt))


def test_int_layernorm_vit_base_full(oracle):
    """ViT-B LayerNorm at batch 64 (12608 tokens x 768 channels), the benchmark's
    size, compared in full."""
    w = workloads.vit_layernorm()
    got = _ln_gpu(w["x"].astype(np.int32), w["s"], w["gamma"], w["beta"], w["o"], alpha=w["alpha"], y_dt="s8")
    want = _want(oracle, w["x"].astype(np.int32), w["s"], w["gamma"], w["beta"], w["o"], w["alpha"], "s8")
    assert np.array_equal(got, want), f"{(got != want).sum()} mismatches"


def test_int_layernorm_errors():
    t = __import__("torch")
    x = t.zeros((4, 8), dtype=t.int8, device="cuda")
    f = t.ones(8, dtype=t.float32, device="cuda")
    y = t.zeros((4, 8), dtype=t.int8, device="cuda")
    qnn.q_int_layernorm(x, 0, 8, 0.1, f, f, f, y)  # no rows: nothing to do
    with pytest.raises(qnn.QnnError):
        qnn.q_int_layernorm(x, 4, 8, 0.1, f, f, f, y, alpha_max=4)
    with pytest.raises(qnn.QnnError):
        qnn.q_int_layernorm(x, 4, 8, 0.1, f, f, f, y, y_dt="u8")
    with pytest.raises(qnn.QnnError):
        qnn.q_int_layernorm(x, 4, 8, 0.1, f[1:], f, f, y)  # misaligned gamma


def test_int_layernorm_overflowing_and_huge_constants(oracle):
    """gamma near the fp32 maximum over a tiny o (A overflows to +-inf: N = 0,
    M = 255), and gammas / betas large enough that B leaves the 32-bit range or
    reaches the 2^62 clamp: the 64-bit form of the rounding shift."""
    rng = np.random.default_rng(5)
    C, rows = 64, 9
    x = np.clip(np.rint(rng.normal(0, 30, size=(rows, C))), -128, 127).astype(np.int32)
    x[0] = 7  # a zero-variance row next to the others
    gamma = rng.uniform(0.5, 2.0, size=C).astype(np.float32)
    gamma[0::8] = 3e38
    gamma[1::8] = -3e38
    gamma[2::8] = 1e20
    beta = rng.normal(0, 1, size=C).astype(np.float32)
    beta[3::8] = 1e25
    beta[4::8] = -3e9
    o = np.full(C, 1e-3, np.float32)
    for y_dt in ("s8", "s32"):
        got = _ln_gpu(x, 0.05, gamma, beta, o, y_dt=y_dt)
        want = _want(oracle, x, 0.05, gamma, beta, o, None, y_dt)
        assert np.array_equal(got, want), f"{(got != want).sum()} mismatches"


def test_int_layernorm_scales_across_binades(oracle):
    """Output scales and gammas spread over many binades (each o[c] = 2^U(-20, 10)
    times a random mantissa): every division by o[c] must round exactly as the
    IEEE division the printed module performs."""
    rng = np.random.default_rng(77)
    C, rows = 256, 64
    x = np.clip(np.rint(rng.normal(0, 50, size=(rows, C))), -128, 127).astype(np.int32)
    o = (2.0 ** rng.uniform(-20, 10, size=C) * rng.uniform(1.0, 2.0, size=C)).astype(np.float32)
    gamma = (2.0 ** rng.uniform(-12, 6, size=C) * rng.choice([-1, 1], size=C)).astype(np.float32)
    beta = (rng.normal(0, 1, size=C) * 2.0 ** rng.uniform(-10, 10, size=C)).astype(np.float32)
    for s in (0.013, 2.0 ** -9):
        got = _ln_gpu(x, s, gamma, beta, o, y_dt="s32")
        assert np.array_equal(got, _want(oracle, x, s, gamma, beta, o, None, "s32"))
