"""Log-Int-Softmax and the bit-shift attention product on the GPU against the
CPU oracle ("首个完全量化Vision Transformer的方法FQ-ViT", section 3.3): codes and
int32 products bit-exact, through the C ABI."""
import os

import numpy as np
import pytest

from integer_quantized_nn_gb300 import qnn, workloads
from _util import dev, host, torch

pytestmark = pytest.mark.gpu
GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "lis_worked_example.txt")


def _lis_gpu(x, S, bits):
    t = __import__("torch")
    L = x.shape[-1]
    rows = x.size // L
    xd = dev(x.reshape(rows, L))
    cd = t.full((rows, L), 0xEE, dtype=t.uint8, device="cuda")
    qnn.q_log_int_softmax(xd, rows, L, S, bits, cd)
    t.cuda.synchronize()
    return host(cd).reshape(x.shape)


def test_lis_golden_rows():
    """The hand-worked rows, ties and masks included."""
    n = 0
    for line in open(GOLDEN):
        rec = line.split()
        if not rec or rec[0] != "row":
            continue
        S, bits = float(rec[1]), int(rec[2])
        bar = rec.index("|")
        x = np.array([int(v) for v in rec[3:bar]], np.int32)[None, :]
        want = np.array([int(v) for v in rec[bar + 1:]], np.uint8)
        assert np.array_equal(_lis_gpu(x, S, bits)[0], want), rec
        n += 1
    assert n >= 8


@pytest.mark.parametrize("L", [1, 2, 31, 32, 33, 64, 65, 127, 197, 256, 257, 1000, 4099])
def test_lis_lengths(oracle, L):
    """Every register-resident row length class and the streaming path (L > 256)."""
    rng = np.random.default_rng(L)
    S = workloads.ATTN_S if L <= 197 else 2.0 ** -9
    x = np.rint(rng.normal(0.0, 2.5, size=(37, L)) / S).astype(np.int32)
    for bits in (4, 1, 5):
        assert np.array_equal(_lis_gpu(x, S, bits), oracle.log_int_softmax(x, S, bits)), bits


@pytest.mark.parametrize("S", [2.0 ** -6, 0.0123, 1.0 / 3.0, 0.75, 2.0 ** -12])
def test_lis_scales(oracle, S):
    """Scales from coarse (few integer steps per ln 2) to fine; every bit width."""
    rng = np.random.default_rng(7)
    x = np.rint(rng.normal(0.0, 3.0, size=(64, 150)) / S).astype(np.int32)
    for bits in range(1, 6):
        assert np.array_equal(_lis_gpu(x, S, bits), oracle.log_int_softmax(x, S, bits))


def test_lis_extreme_values(oracle):
    """Rows spanning the whole int32 range, constant rows and rows of exact
    powers-of-two ratios (ties of the half-to-even rounding)."""
    S = 2.0 ** -6
    rows = [np.full(40, np.iinfo(np.int32).min), np.full(40, np.iinfo(np.int32).max),
            np.array([np.iinfo(np.int32).max, np.iinfo(np.int32).min] * 20),
            np.array([0, -45, -45, -45] * 10), np.array([0] + [-45] * 9 + [-90] * 30),
            np.arange(0, -40 * 45, -45), np.array([5] * 39 + [6])]
    x = np.stack(rows).astype(np.int32)
    for bits in (2, 4, 5):
        assert np.array_equal(_lis_gpu(x, S, bits), oracle.log_int_softmax(x, S, bits))


def test_lis_empty_and_errors():
    t = __import__("torch")
    x = t.zeros((4, 8), dtype=t.int32, device="cuda")
    c = t.zeros((4, 8), dtype=t.uint8, device="cuda")
    qnn.q_log_int_softmax(x, 0, 8, 0.01, 4, c)            # no rows: nothing to do
    with pytest.raises(qnn.QnnError):
        qnn.q_log_int_softmax(x, 4, 8, 0.01, 6, c)        # bits out of range
    with pytest.raises(qnn.QnnError):
        qnn.q_log_int_softmax(x, 4, 8, 2.0 ** -16, 4, c)  # c_int >= 2^31
    with pytest.raises(qnn.QnnError):
        qnn.q_log_int_softmax(x[:, 1:], 4, 7, 0.01, 4, c)  # misaligned base


def test_lis_vit_base_full(oracle):
    """ViT-B attention maps at batch 64 (768 heads x 197 x 197), the size the
    benchmark times, compared in full."""
    t = __import__("torch")
    rows, L = 64 * 12 * 197, 197
    xd = workloads.device_attention_logits(rows, L, 1234, "cuda")
    cd = t.empty((rows, L), dtype=t.uint8, device="cuda")
    qnn.q_log_int_softmax(xd, rows, L, workloads.ATTN_S, 4, cd)
    t.cuda.synchronize()
    want = oracle.log_int_softmax(host(xd), workloads.ATTN_S, 4)
    got = host(cd)
    assert np.array_equal(got, want), f"{(got != want).sum()} mismatches"


def _shift_gpu(code, v, bits):
    t = __import__("torch")
    Bh, Lq, Lk = code.shape
    d = v.shape[-1]
    out = t.full((Bh, Lq, d), -7, dtype=t.int32, device="cuda")
    qnn.q_attn_shift_v(dev(code), dev(v), Bh, Lq, Lk, d, bits, out)
    t.cuda.synchronize()
    return host(out)


@pytest.mark.parametrize("shape", [(3, 197, 197, 64), (2, 1, 5, 16), (5, 65, 63, 80), (1, 130, 512, 48),
                                   (2, 64, 64, 64), (1, 257, 300, 128), (2, 40, 70, 144), (1, 33, 1100, 32)])
@pytest.mark.parametrize("bits", [1, 2, 3, 4])
def test_attn_shift_v(oracle, shape, bits):
    """Ragged query / token / column tiles, masked codes, every bit width; d <= 128
    with Lk <= 512 on the tensor pipe (one to four token rounds), the last two shapes
    on the CUDA-core kernel."""
    Bh, Lq, Lk, d = shape
    if Lk * 128 * 2 ** (2 ** bits - 1) > 2 ** 31:
        # beyond the int32 range of the sums: the host refuses the shape before launching
        t = torch()
        code = t.zeros((Bh, Lq, Lk), dtype=t.uint8, device="cuda")
        v = t.zeros((Bh, Lk, d), dtype=t.int8, device="cuda")
        out = t.zeros((Bh, Lq, d), dtype=t.int32, device="cuda")
        with pytest.raises(qnn.QnnError) as e:
            qnn.q_attn_shift_v(code, v, Bh, Lq, Lk, d, bits, out)
        assert e.value.status == qnn.QNN_ERR_OVERFLOW_RISK
        return
    rng = np.random.default_rng(Lq * 7 + bits)
    code = rng.integers(0, 2 ** bits + 1, size=(Bh, Lq, Lk)).astype(np.uint8)
    v = rng.integers(-128, 128, size=(Bh, Lk, d)).astype(np.int8)
    want = oracle.attn_shift_v(code, v, bits)
    assert np.array_equal(_shift_gpu(code, v, bits).astype(np.int64), want)


def test_attn_shift_v_extremes(oracle):
    """The int32 range's edge: Lk = 512 at 4 bits with every code 0 and v = -128
    reaches exactly -2^31, v = 127 the largest positive sum; Lk = 256 puts the
    tensor-pipe sums at 2^22, the edge of their exact conversion."""
    for Lk in (512, 256, 257):
        code = np.zeros((1, 3, Lk), np.uint8)
        code[0, 2, ::3] = 8  # a row of mixed halves
        for val in (-128, 127):
            v = np.full((1, Lk, 16), val, np.int8)
            want = oracle.attn_shift_v(code, v, 4)
            assert np.array_equal(_shift_gpu(code, v, 4).astype(np.int64), want)
    t = __import__("torch")
    with pytest.raises(qnn.QnnError):  # Lk = 513 could overflow int32
        qnn.q_attn_shift_v(t.zeros((1, 1, 513), dtype=t.uint8, device="cuda"),
                           t.zeros((1, 513, 16), dtype=t.int8, device="cuda"), 1, 1, 513, 16, 4,
                           t.zeros((1, 1, 16), dtype=t.int32, device="cuda"))


def test_lis_then_shift_vit_base(oracle):
    """The attention path of one ViT-B layer at batch 4: logits -> Log-Int-Softmax
    codes -> shift product with V, both stages against the oracle's."""
    t = __import__("torch")
    w = workloads.vit_attention(B=4)
    x, v, S, bits = w["x"], w["v"], w["S"], w["bits"]
    Bh, L, _ = x.shape
    d = v.shape[-1]
    xd, vd = dev(x), dev(v)
    cd = t.empty((Bh, L, L), dtype=t.uint8, device="cuda")
    od = t.empty((Bh, L, d), dtype=t.int32, device="cuda")
    qnn.q_log_int_softmax(xd, Bh * L, L, S, bits, cd)
    qnn.q_attn_shift_v(cd, vd, Bh, L, L, d, bits, od)
    t.cuda.synchronize()
    k = oracle.log_int_softmax(x, S, bits)
    assert np.array_equal(host(cd), k)
    assert np.array_equal(host(od).astype(np.int64), oracle.attn_shift_v(k, v, bits))


@pytest.mark.parametrize("shape", [(4 * 12, 197, 197, 64), (3, 130, 70, 80), (2, 1, 1, 16), (1, 200, 256, 128),
                                   (2, 64, 33, 48)])
@pytest.mark.parametrize("bits", [1, 2, 3, 4])
def test_lis_attn_fused(oracle, shape, bits):
    """q_lis_attn_v (Log-Int-Softmax into shared memory, then the shift product)
    against the oracle's two steps; ragged query, token and column tiles."""
    t = __import__("torch")
    Bh, Lq, Lk, d = shape
    rng = np.random.default_rng(Bh * 31 + Lk + bits)
    S = workloads.ATTN_S if Lk <= 197 else 2.0 ** -9  # L c_int 2^30 < 2^64 at L = 256
    x = np.rint(rng.normal(0.0, 2.5, size=(Bh, Lq, Lk)) / S).astype(np.int32)
    x[:, :, 0] += np.int32(4.0 / S)
    v = rng.integers(-128, 128, size=(Bh, Lk, d)).astype(np.int8)
    out = t.full((Bh, Lq, d), 7, dtype=t.int32, device="cuda")
    qnn.q_lis_attn_v(dev(x), S, dev(v), Bh, Lq, Lk, d, bits, out)
    t.cuda.synchronize()
    k = oracle.log_int_softmax(x, S, bits)
    want = oracle.attn_shift_v(k, v, bits)
    assert np.array_equal(host(out).astype(np.int64), want)


def test_lis_attn_fused_errors():
    t = __import__("torch")
    x = t.zeros((1, 4, 300), dtype=t.int32, device="cuda")
    v = t.zeros((1, 300, 16), dtype=t.int8, device="cuda")
    o = t.zeros((1, 4, 16), dtype=t.int32, device="cuda")
    with pytest.raises(qnn.QnnError):  # Lk > 256
        qnn.q_lis_attn_v(x, 2e-4, v, 1, 4, 300, 16, 4, o)
    with pytest.raises(qnn.QnnError):  # bits 5 has no shift product
        qnn.q_lis_attn_v(x, 2e-4, v, 1, 4, 200, 16, 5, o)


@pytest.mark.parametrize("bits", [4, 5])
def test_lis_ties_at_large_thresholds(oracle, bits):
    """Rows whose largest element has v = s / e exactly half-way below a log_round
    step L_j = 3 * 2^(j-2) (one element at 0 and n at -45 with S = 2^-6: v = 1 +
    n / 2^q for q halvings), so the half-to-even rounding decides the code at
    large thresholds as well as small ones."""
    S = 2.0 ** -6
    for q, L in ((1, 48), (1, 384), (1, 1536), (10, 3), (10, 12), (3, 24)):
        n = int((L - 1.5) * 2 ** q)
        x = np.array([[0] + [-45 * q] * n], np.int32)
        got = _lis_gpu(x, S, bits)
        want = oracle.log_int_softmax(x, S, bits)
        assert np.array_equal(got, want), (q, L, got[0, :3], want[0, :3])
