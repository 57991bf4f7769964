"""The seeded synthetic inputs: the same bytes on every call, and the shapes,
ranges and distribution parameters the input recipes state (the layer shapes
of ViT-B / ViT-L / ResNet-50 standing in for the pages' datasets)."""
import numpy as np
import pytest

from integer_quantized_nn_gb300 import workloads as wl

pytestmark = pytest.mark.cpu


def test_same_bytes_every_call():
    for make in (lambda: wl.gemm_sym(), lambda: wl.vit_fc1(M=64), lambda: wl.conv_u4(N=1, H=8, W=8),
                 lambda: wl.conv_u8(N=1, H=8, W=8), lambda: wl.vit_fc1_zw(M=64), lambda: wl.vit_layernorm(rows=32),
                 lambda: wl.vit_attention(B=1)):
        a, b = make(), make()
        for k, v in a.items():
            if isinstance(v, np.ndarray):
                assert np.array_equal(v, b[k]), k
            else:
                assert v == b[k], k


def test_workloads_draw_independent_streams():
    # distinct (workload, tensor) pairs give distinct streams
    x = wl.rng(wl.VIT_FC1, 0).integers(0, 1 << 30, 8)
    y = wl.rng(wl.VIT_FC1, 1).integers(0, 1 << 30, 8)
    z = wl.rng(wl.VIT_FC1_ZW, 0).integers(0, 1 << 30, 8)
    assert not np.array_equal(x, y) and not np.array_equal(x, z)


def test_vit_fc1_recipe():
    w = wl.vit_fc1(M=2048)
    A, B = w["A"], w["B"]
    assert A.shape == (2048, 768) and A.dtype == np.uint8
    assert B.shape == (3072, 768) and B.dtype == np.int8
    assert abs(A.mean() - 128.0) < 0.5 and abs(A.std() - 30.0) < 0.5
    assert abs(B.astype(np.float64).mean()) < 0.2 and abs(B.std() - 25.0) < 0.3
    assert w["z_a"] == 128 and w["s_a"] == 0.02
    assert ((w["s_w"] >= 1e-3) & (w["s_w"] <= 1e-2)).all()
    assert np.float32(w["s_o"]) == w["s_o"] > 0


def test_vit_fc1_zw_recipe():
    w = wl.vit_fc1_zw(M=256)
    B, z_w = w["B"], w["z_w"]
    assert B.dtype == np.uint8 and B.shape == (3072, 768)
    assert z_w.min() >= 96 and z_w.max() <= 160
    d = B.astype(np.float64) - z_w[:, None]
    assert abs(d.mean()) < 0.2 and abs(d.std() - 25.0) < 0.5


def test_conv_recipes():
    c4 = wl.conv_u4()
    assert c4["I"].shape == (64, 56, 56, 32) and c4["W"].shape == (64, 3, 3, 32)
    assert c4["res"].shape == (64, 56, 56, 32) and c4["z_in"] == 8 and c4["z_res"] == 8
    c1 = wl.conv_u4(C=256, OC=64, F=1, pad=0, residual=False, tag=1)
    assert c1["I"].shape == (64, 56, 56, 128) and c1["res"] is None
    c8 = wl.conv_u8()
    assert c8["I"].shape == (64, 56, 56, 64) and c8["W"].shape == (64, 3, 3, 64)
    assert c8["z_w"].min() >= 96 and c8["z_w"].max() <= 160 and c8["z_in"] == 128
    d = c8["W"].astype(np.float64) - c8["z_w"].reshape(-1, 1, 1, 1)
    assert abs(d.std() - 40.0) < 1.0


def test_attention_and_layernorm_recipes():
    a = wl.vit_attention(B=1)
    assert a["x"].shape == (12, 197, 197) and a["v"].shape == (12, 197, 64)
    z = a["x"].astype(np.float64) * a["S"]
    assert abs(z[:, :, 1:].std() - 2.5) < 0.05
    assert abs(z[:, :, 0].mean() - 4.0) < 0.1  # the class-token column raised by 4
    ln = wl.vit_layernorm()
    assert ln["x"].shape == (64 * 197, 768)
    frac = (ln["alpha"] == 3).mean()
    assert 0.02 < frac < 0.09 and set(np.unique(ln["alpha"])) <= {0, 3}
    assert (np.abs(ln["gamma"]) >= 0.5).all() and (np.abs(ln["gamma"]) <= 1.5).all()
    assert (ln["o"] == np.float32(0.04)).all()
