"""qconv_u4s4 / qconv_u8s8 (implicit-GEMM convolution, fused Conv_Relu /
Conv_Add_Relu) on the GPU against the CPU oracle's direct convolution:
bit-exact int32 accumulators and quantized outputs."""
import numpy as np
import pytest

from integer_quantized_nn_gb300 import qnn, workloads
from _util import dev, host, aligned_empty, f32_bits, library_zp_term, torch

pytestmark = pytest.mark.gpu


def _conv(oracle, I_pk, W_pk, geom, z_in, s_a, s_w, s_o, bias, u4=True, mode="requant",
          out_dt="u4", relu=True, z_out=0, res=None, res_dt="u4", z_res=8, s_r=None,
          full=True, pixels=None, w_zp=None):
    """Runs the conv on both sides.  I_pk / W_pk: packed u4 / s4 bytes (u4=True)
    or u8 / s8 codes (u4=False), NHWC / OHWI."""
    t = torch()
    N, H, W, C, OC, F, pad, st = geom
    g = qnn.conv_geom(N, H, W, C, OC, F, F, (pad, pad), (st, st))
    OH, OW = g.OH, g.OW
    w_dt = "s4" if u4 else "s8"
    Wd = dev(W_pk)
    Wp = aligned_empty(qnn.qnn_conv_packed_w_bytes(g, w_dt))
    colsum = t.empty(OC, dtype=t.int32, device="cuda")
    if w_zp is None:
        qnn.qconv_prepack_w(Wd, w_dt, g, Wp, colsum)
    elif u4:
        qnn.qconv_prepack_w_u4(Wd, dev(np.asarray(w_zp, np.int32)), g, Wp, colsum)
    else:
        qnn.qconv_prepack_w_u8(Wd, dev(np.asarray(w_zp, np.int32)), g, Wp, colsum)
    a_dt = "u4" if u4 else "u8"
    sw = dev(np.asarray(s_w, np.float32))
    bd = dev(np.asarray(bias, np.float32))
    zp = t.empty(OC, dtype=t.int32, device="cuda")
    Mv = t.empty(OC, dtype=t.float32, device="cuda")
    Bq = t.empty(OC, dtype=t.float32, device="cuda")
    D = t.empty(OC, dtype=t.float32, device="cuda")
    qnn.q_fold_epilogue(OC, a_dt, z_in, colsum, s_a, sw, s_o, bias=bd, zp_term=zp, M=Mv, Bq=Bq, D=D)
    R = 0.0 if s_r is None else float(np.float32(np.float32(s_r) / np.float32(s_o)))
    resd = None if res is None else dev(res)
    epi = qnn.epilogue(mode, relu=relu, out_dt=out_dt, z_out=z_out, zp_term=zp, M=Mv, Bq=Bq, D=D,
                       bias=bd, residual=resd, res_dt=res_dt, z_res=z_res, R=R)
    rows = N * OH * OW
    Id = dev(I_pk)
    # u4: both paths -- the packed input re-encoded inside the conv kernel, and
    # the input expanded into a workspace (pre-filled with 0xFF) read by TMA
    outs = []
    for path in ("fused", "workspace"):
        if mode == "requant":
            ob = OC // 2 if out_dt == "u4" else OC
            O = t.full((N, OH, OW, ob), 0x5A, dtype=t.uint8, device="cuda")
        elif mode == "dequant":
            O = t.empty((N, OH, OW, OC), dtype=t.float32, device="cuda")
        else:
            O = t.empty((N, OH, OW, OC), dtype=t.int32, device="cuda")
        O32 = t.zeros((N, OH, OW, OC), dtype=t.int32, device="cuda")
        # the workspace paths: the input expanded (u4: e4m3 bytes; u8: fp16 q - z_in)
        # into a workspace pre-filled with 0xFF and read by tensor copies
        ws = None
        if path == "workspace":
            ws = t.full((qnn.qnn_conv_workspace_bytes(g, "u4" if u4 else "u8"),), 0xFF, dtype=t.uint8,
                        device="cuda")
        if u4:
            qnn.qconv_u4s4(Id, z_in, Wp, g, epi, O, O32, workspace=ws)
        elif w_zp is None:
            qnn.qconv_u8s8(Id, z_in, Wp, g, epi, O, O32, workspace=ws)
        else:
            qnn.qconv_u8u8(Id, z_in, Wp, g, epi, O, O32, workspace=ws)
        assert qnn.qnn_check_device_error() == qnn.QNN_OK
        outs.append((path, O, O32))

    # oracle side
    if u4:
        Ic = oracle.unpack_nibbles(I_pk, signed=False)
        if w_zp is None:
            Wc = oracle.unpack_nibbles(W_pk, signed=True)
        else:  # u4 filters: the zero-point-centred codes u - z_w[oc]
            Wc = oracle.unpack_nibbles(W_pk, signed=False) - np.asarray(w_zp, np.int32).reshape(-1, 1, 1, 1)
    else:
        Ic = I_pk.astype(np.int32)
        if w_zp is None:
            Wc = W_pk.astype(np.int8).astype(np.int32)
        else:  # u8 filters: the zero-point-centred codes w - z_w[oc]
            Wc = W_pk.astype(np.uint8).astype(np.int32) - np.asarray(w_zp, np.int32).reshape(-1, 1, 1, 1)
    cs = oracle.colsum(Wc.reshape(OC, -1))
    assert np.array_equal(host(colsum), cs)
    zp_o, M_o, Bq_o, D_o = oracle.fold(cs, z_in, s_a, np.asarray(s_w, np.float32), s_o, bias)
    assert np.array_equal(host(zp), library_zp_term(zp_o, cs, 0 if u4 else 128))
    if full:
        acc = oracle.conv_acc_direct(Ic, Wc, z_in, (pad, pad), (st, st))
        sel = np.arange(rows)
    else:
        # sampled output pixels: direct conv on the receptive fields they need
        sel = pixels
        acc_all = []
        for pix in sel:
            n_, rem = divmod(int(pix), OH * OW)
            oy, ox = divmod(rem, OW)
            sub = Ic[n_:n_ + 1]
            a = oracle.conv_acc_direct(sub, Wc, z_in, (pad, pad), (st, st))
            acc_all.append(a[oy * OW + ox])
        acc = np.stack(acc_all)
    if mode == "dequant":
        y = oracle.dequant_epilogue(acc, D_o, bias)
    elif mode == "requant":
        res_codes = None
        if res is not None:
            if res_dt == "u4":
                res_codes = oracle.unpack_nibbles(res, signed=False).reshape(rows, OC)[sel]
            else:
                res_codes = res.reshape(rows, OC)[sel].astype(np.int32)
        q = oracle.requant(acc, M_o, Bq_o, out_dt, relu=relu, res=res_codes, z_res=z_res, R=R,
                           z_out=z_out)
        exp = oracle.pack_nibbles(q) if out_dt == "u4" else oracle.pack_bytes(q)
    for path, O, O32 in outs:
        got32 = host(O32).reshape(rows, OC)[sel]
        assert np.array_equal(got32, acc), f"{path}: {(got32 != acc).sum()} accumulator mismatches"
        Og = host(O)
        if mode == "s32":
            assert np.array_equal(Og.reshape(rows, OC)[sel], acc), path
        elif mode == "dequant":
            assert np.array_equal(f32_bits(Og.reshape(rows, OC)[sel]), f32_bits(y)), path
        else:
            got = Og.reshape(rows, -1)[sel]
            assert np.array_equal(got, exp), f"{path}: {(got != exp).sum()} output bytes differ"
    return acc


def _rand_u4s4(seed, N, H, W, C, OC, F, with_res=True, OH=None, OW=None):
    rng = np.random.default_rng(seed)
    I = rng.integers(0, 256, size=(N, H, W, C // 2)).astype(np.uint8)
    Wt = rng.integers(0, 256, size=(OC, F, F, C // 2)).astype(np.uint8)
    s_w = rng.uniform(1e-3, 1e-2, size=OC).astype(np.float32)
    bias = rng.normal(0, 1, size=OC).astype(np.float32)
    res = None
    if with_res:
        res = rng.integers(0, 256, size=(N, OH or H, OW or W, OC // 2)).astype(np.uint8)
    return I, Wt, s_w, bias, res


@pytest.mark.parametrize("geom", [
    (2, 9, 9, 64, 64, 3, 1, 1),      # ragged pixel tail, Conv_Add_Relu
    (1, 7, 11, 32, 96, 3, 1, 1),     # C = 32, OC = 96 (N not a multiple of 32 per piece)
    (2, 10, 10, 64, 128, 3, 1, 2),   # stride 2
    (1, 6, 6, 128, 256, 3, 0, 1),    # no padding, OC = 256
    (3, 5, 5, 64, 320, 1, 0, 1),     # 1x1, two filter blocks
])
def test_conv_u4s4_small(oracle, geom):
    N, H, W, C, OC, F, pad, st = geom
    OH = (H + 2 * pad - F) // st + 1
    OW = (W + 2 * pad - F) // st + 1
    I, Wt, s_w, bias, res = _rand_u4s4(31, N, H, W, C, OC, F, True, OH, OW)
    _conv(oracle, I, Wt, geom, 8, 0.05, s_w, 0.11, bias, res=res, s_r=0.13)


@pytest.mark.parametrize("geom,residual", [
    ((3, 7, 9, 256, 64, 1, 0, 1), True),    # 189 pixels: a ragged 128-pixel tile, Conv_Add_Relu
    ((2, 10, 13, 512, 64, 1, 0, 1), False),  # C = 512: two 256-channel units per tile
    ((1, 16, 16, 256, 48, 1, 0, 1), True),   # OC = 48: a partial 32-column piece
    ((1, 1, 1, 256, 64, 1, 0, 1), False),    # a single pixel
])
def test_conv_u4s4_1x1_tensor_copies(oracle, geom, residual):
    """1x1 convs whose packed input tiles arrive by tensor copies and are unpacked
    in shared memory (C a multiple of 256, up to 64 filters)."""
    N, H, W, C, OC, F, pad, st = geom
    I, Wt, s_w, bias, res = _rand_u4s4(37, N, H, W, C, OC, F, residual, H, W)
    _conv(oracle, I, Wt, geom, 8, 0.05, s_w, 0.11, bias, res=res, s_r=0.13)
    _conv(oracle, I, Wt, geom, 5, 0.05, s_w, 0.11, bias, mode="s32")


def test_conv_u4u4_1x1_tensor_copies(oracle):
    """The same path with u4 filters carrying per-filter zero points."""
    geom = (2, 9, 9, 256, 64, 1, 0, 1)
    I, Wt, s_w, bias, _ = _rand_u4s4(38, 2, 9, 9, 256, 64, 1, False)
    z_w = np.random.default_rng(39).integers(0, 16, size=64)
    _conv(oracle, I, Wt, geom, 8, 0.05, s_w, 0.11, bias, w_zp=z_w)


@pytest.mark.parametrize("mode", ["dequant", "s32"])
def test_conv_u4s4_modes(oracle, mode):
    geom = (1, 8, 8, 64, 64, 3, 1, 1)
    I, Wt, s_w, bias, _ = _rand_u4s4(32, 1, 8, 8, 64, 64, 3, False)
    _conv(oracle, I, Wt, geom, 5, 0.05, s_w, 0.11, bias, mode=mode)


def test_conv_u4s4_relu_u8_out(oracle):
    geom = (1, 8, 8, 64, 64, 3, 1, 1)
    I, Wt, s_w, bias, _ = _rand_u4s4(33, 1, 8, 8, 64, 64, 3, False)
    _conv(oracle, I, Wt, geom, 3, 0.05, s_w, 0.011, bias, out_dt="u8", relu=True, z_out=7)


def test_conv_u4s4_exactness_large_sums(oracle):
    """C = 1024: |acc| reaches 9216 * 120; in the e4m3 scaling (2^-9) the fp32
    sums need 20+ significant bits, so any truncation in the accumulation shows."""
    geom = (1, 6, 6, 1024, 64, 3, 1, 1)
    I = np.full((1, 6, 6, 512), 0xFF, np.uint8)            # every code 15
    Wt = np.full((64, 3, 3, 512), 0x88, np.uint8)           # every weight -8
    rng = np.random.default_rng(34)
    I[0, 2, 2, :64] = rng.integers(0, 256, size=64).astype(np.uint8)
    Wt[::3, 1, 1, :16] = 0x11                               # +1 weights mixed in
    s_w = np.full(64, 1e-3, np.float32)
    acc = _conv(oracle, I, Wt, geom, 0, 1.0, s_w, 1000.0, np.zeros(64, np.float32), mode="s32")
    assert np.abs(acc).max() >= 9216 * 100


def test_conv_resnet_3x3_full(oracle):
    """ResNet-50 stage-1 3x3 Conv_Add_Relu at full size (N=64, 56x56, 64 -> 64,
    u4 x s4, u4 residual and output), every output compared."""
    w = workloads.conv_u4()
    geom = (64, 56, 56, 64, 64, 3, 1, 1)
    _conv(oracle, w["I"], w["W"], geom, w["z_in"], w["s_a"], w["s_w"], w["s_o"], w["bias"],
          res=w["res"], z_res=w["z_res"], s_r=w["s_r"])


def test_conv_resnet_1x1_full(oracle):
    """ResNet-50 stage-1 1x1 Conv_Relu (256 -> 64 channels) at full size."""
    w = workloads.conv_u4(C=256, OC=64, F=1, pad=0, residual=False, tag=1)
    geom = (64, 56, 56, 256, 64, 1, 0, 1)
    _conv(oracle, w["I"], w["W"], geom, w["z_in"], w["s_a"], w["s_w"], w["s_o"], w["bias"])


@pytest.mark.parametrize("geom", [(2, 9, 9, 64, 64, 3, 1, 1), (1, 7, 7, 256, 128, 3, 1, 1),
                                  (1, 9, 9, 48, 64, 3, 1, 2)])
def test_conv_u8s8(oracle, geom):
    """u8 activations (zero point 100) x s8 filters; C = 256 3x3 has K = 2304,
    above one exact fp32 chunk."""
    N, H, W, C, OC, F, pad, st = geom
    OH = (H + 2 * pad - F) // st + 1
    OW = (W + 2 * pad - F) // st + 1
    rng = np.random.default_rng(35)
    I = rng.integers(0, 256, size=(N, H, W, C)).astype(np.uint8)
    Wt = rng.integers(-128, 128, size=(OC, F, F, C)).astype(np.int8)
    s_w = rng.uniform(1e-3, 1e-2, size=OC).astype(np.float32)
    bias = rng.normal(0, 1, size=OC).astype(np.float32)
    res = rng.integers(0, 256, size=(N, OH, OW, OC)).astype(np.uint8)
    _conv(oracle, I, Wt, geom, 100, 0.02, s_w, 0.07, bias, u4=False, out_dt="u8", z_out=3,
          res=res, res_dt="u8", z_res=120, s_r=0.05)


def test_conv_resnet_stem_7x7_stride2(oracle):
    """The ResNet-50 stem shape: 7x7, stride 2, padding 3 (a 64 x 64 crop of the
    224 x 224 input, batch 2).  u8 x s8 with the 3 colour channels widened to 16:
    the extra channels hold the input zero point and carry zero weights."""
    N, H, W, C, OC, F, pad, st = 2, 64, 64, 16, 64, 7, 3, 2
    OH = (H + 2 * pad - F) // st + 1
    rng = np.random.default_rng(36)
    z_in = 110
    I = np.full((N, H, W, C), z_in, np.uint8)
    I[..., :3] = rng.integers(0, 256, size=(N, H, W, 3)).astype(np.uint8)
    Wt = np.zeros((OC, F, F, C), np.int8)
    Wt[..., :3] = rng.integers(-128, 128, size=(OC, F, F, 3)).astype(np.int8)
    s_w = rng.uniform(1e-3, 1e-2, size=OC).astype(np.float32)
    bias = rng.normal(0, 1, size=OC).astype(np.float32)
    _conv(oracle, I, Wt, (N, H, W, C, OC, F, pad, st), z_in, 0.02, s_w, 0.05, bias, u4=False, out_dt="u8",
          relu=True)
    assert OH == 32


def test_conv_u4s4_7x7_stride2(oracle):
    """u4 x s4 at 7x7, stride 2, padding 3, C = 64 (K = 3136, more than one exact chunk)."""
    geom = (1, 20, 20, 64, 64, 7, 3, 2)
    I, Wt, s_w, bias, _ = _rand_u4s4(37, 1, 20, 20, 64, 64, 7, False)
    _conv(oracle, I, Wt, geom, 6, 0.05, s_w, 0.3, bias)


@pytest.mark.parametrize("geom", [(2, 9, 9, 64, 64, 3, 1, 1), (2, 10, 10, 64, 128, 3, 1, 2), (3, 5, 5, 64, 96, 1, 0, 1),
                                  (1, 12, 12, 32, 64, 7, 3, 2)])
def test_conv_u4u4(oracle, geom):
    """u4 activations x u4 filters with per-filter zero points (both operands
    asymmetric, MegEngine article 背景 / 緩解精度下降); the fused and the TMA path."""
    N, H, W, C, OC, F, pad, st = geom
    OH = (H + 2 * pad - F) // st + 1
    OW = (W + 2 * pad - F) // st + 1
    I, Wt, s_w, bias, res = _rand_u4s4(38 + C, N, H, W, C, OC, F, True, OH, OW)
    z_w = np.random.default_rng(39).integers(0, 16, size=OC).astype(np.int32)
    z_w[:2] = (0, 15)
    _conv(oracle, I, Wt, geom, 9, 0.05, s_w, 0.2, bias, res=res, s_r=0.13, w_zp=z_w)


def test_conv_u4u4_resnet_3x3_full(oracle):
    """ResNet-50 stage-1 3x3 Conv_Add_Relu at full size with u4 filters and zero points."""
    w = workloads.conv_u4()
    z_w = np.random.default_rng(44).integers(0, 16, size=64).astype(np.int32)
    geom = (64, 56, 56, 64, 64, 3, 1, 1)
    _conv(oracle, w["I"], w["W"], geom, w["z_in"], w["s_a"], w["s_w"], w["s_o"] * 2, w["bias"],
          res=w["res"], z_res=w["z_res"], s_r=w["s_r"], w_zp=z_w)


@pytest.mark.parametrize("geom", [(2, 9, 9, 64, 64, 3, 1, 1),    # K = 576: exact chunks of 512 + 64
                                  (1, 7, 7, 256, 128, 3, 1, 1),  # K = 2304: five chunks
                                  (2, 6, 6, 512, 64, 1, 0, 1),   # K = 512: one chunk, exactly full
                                  (1, 9, 9, 48, 96, 3, 1, 2)])   # stride 2, OC = 96
def test_conv_u8u8(oracle, geom):
    """u8 activations x u8 filters with per-filter zero points (MegEngine article
    背景 / 緩解精度下降): the filter values w - z_w reach 255 in magnitude."""
    N, H, W, C, OC, F, pad, st = geom
    OH = (H + 2 * pad - F) // st + 1
    OW = (W + 2 * pad - F) // st + 1
    rng = np.random.default_rng(40 + C)
    I = rng.integers(0, 256, size=(N, H, W, C)).astype(np.uint8)
    Wt = rng.integers(0, 256, size=(OC, F, F, C)).astype(np.uint8)
    z_w = rng.integers(0, 256, size=OC).astype(np.int32)
    z_w[:2] = (0, 255)
    s_w = rng.uniform(1e-3, 1e-2, size=OC).astype(np.float32)
    bias = rng.normal(0, 1, size=OC).astype(np.float32)
    res = rng.integers(0, 256, size=(N, OH, OW, OC)).astype(np.uint8)
    _conv(oracle, I, Wt, geom, 77, 0.02, s_w, 0.5, bias, u4=False, out_dt="u8", z_out=3,
          res=res, res_dt="u8", z_res=120, s_r=0.4, w_zp=z_w)


@pytest.mark.parametrize("geom", [(1, 6, 6, 512, 64, 1, 0, 1), (1, 8, 8, 64, 64, 3, 1, 1)])
def test_conv_u8u8_extreme_codes(oracle, geom):
    """The largest products of one sign: inputs 0 (centred -128) against filters
    255 with zero point 0 and filters 0 with zero point 255 (+-255), so every
    512-term chunk sum reaches 512 * 32640, just below 2^24; raw int32 out."""
    N, H, W, C, OC, F, pad, st = geom
    I = np.zeros((N, H, W, C), np.uint8)
    Wt = np.zeros((OC, F, F, C), np.uint8)
    Wt[0::2] = 255
    z_w = np.where(np.arange(OC) % 2 == 0, 0, 255).astype(np.int32)
    s_w = np.full(OC, 1e-3, np.float32)
    _conv(oracle, I, Wt, geom, 200, 0.02, s_w, 1.0, np.zeros(OC, np.float32), u4=False, mode="s32",
          w_zp=z_w)


def test_conv_u8u8_resnet_3x3_full(oracle):
    """ResNet-50 stage-1 3x3 Conv_Add_Relu at full size (64 x 56 x 56 x 64) with u8
    activations and u8 filters with per-filter zero points, compared in full."""
    w = workloads.conv_u8()
    geom = (64, 56, 56, 64, 64, 3, 1, 1)
    _conv(oracle, w["I"], w["W"], geom, w["z_in"], w["s_a"], w["s_w"], w["s_o"], w["bias"], u4=False,
          out_dt="u8", res=w["res"], res_dt="u8", z_res=w["z_res"], s_r=w["s_r"], w_zp=w["z_w"])


def test_conv_errors():
    t = torch()
    g = qnn.conv_geom(1, 8, 8, 48, 64, 3, 3)
    I = t.zeros(1024, dtype=t.uint8, device="cuda")
    Wp = aligned_empty(1 << 20)
    O = t.zeros(4096, dtype=t.uint8, device="cuda")
    Mv = t.ones(64, dtype=t.float32, device="cuda")
    epi = qnn.epilogue("requant", out_dt="u4", M=Mv, Bq=Mv)
    with pytest.raises(qnn.QnnError) as e:
        qnn.qconv_u4s4(I, 8, Wp, g, epi, O)     # C = 48 is not a multiple of 32
    assert e.value.status == qnn.QNN_ERR_UNSUPPORTED
    g = qnn.conv_geom(1, 8, 8, 64, 64, 3, 3)
    with pytest.raises(qnn.QnnError) as e:
        qnn.qconv_u4s4(I, 16, Wp, g, epi, O)    # zero point outside u4
    assert e.value.status == qnn.QNN_ERR_INVALID_ARG
    g = qnn.conv_geom(1, 2, 2, 64, 64, 5, 5, (0, 0))
    with pytest.raises(qnn.QnnError) as e:
        qnn.qconv_u4s4(I, 8, Wp, g, epi, O)     # filter larger than the padded input
    assert e.value.status == qnn.QNN_ERR_INVALID_ARG


# ---- NCHW / NCHW64 layouts -------------------------------------------------------

def _to_layout(x, layout):
    """NHWC array [N, H, W, C] -> the same codes in `layout` (a flat-able array)."""
    N, H, W, C = x.shape
    if layout == "nchw":
        return np.ascontiguousarray(x.transpose(0, 3, 1, 2))
    if layout == "nchw64":
        return np.ascontiguousarray(x.reshape(N, H, W, C // 64, 64).transpose(0, 3, 1, 2, 4))
    return np.ascontiguousarray(x)


def _from_layout(flat, layout, N, H, W, C):
    if layout == "nchw":
        return flat.reshape(N, C, H, W).transpose(0, 2, 3, 1)
    if layout == "nchw64":
        return flat.reshape(N, C // 64, H, W, 64).transpose(0, 2, 3, 1, 4).reshape(N, H, W, C)
    return flat.reshape(N, H, W, C)


def _conv_layout(oracle, geom, layout, u4=True, mode="requant", residual=True, workspace=True, seed=50,
                 z_in=None, out_dt=None):
    """The conv with input, output and residual in `layout`, against the oracle's
    direct conv in that layout (oracle.conv_acc_layout) and its requant."""
    t = torch()
    N, H, W, C, OC, F, pad, st = geom
    g = qnn.conv_geom(N, H, W, C, OC, F, F, (pad, pad), (st, st), layout=layout)
    OH, OW = g.OH, g.OW
    rng = np.random.default_rng(seed)
    if u4:
        I = rng.integers(0, 16, size=(N, H, W, C)).astype(np.int32)
        Wc = rng.integers(-8, 8, size=(OC, F, F, C)).astype(np.int32)
        z_in = 8 if z_in is None else z_in
        out_dt = out_dt or "u4"
    else:
        I = rng.integers(0, 256, size=(N, H, W, C)).astype(np.int32)
        Wc = rng.integers(-128, 128, size=(OC, F, F, C)).astype(np.int32)
        z_in = 100 if z_in is None else z_in
        out_dt = out_dt or "u8"
    res = rng.integers(0, 16 if u4 else 256, size=(N, OH, OW, OC)).astype(np.int32) if residual else None
    s_w = rng.uniform(1e-3, 1e-2, size=OC).astype(np.float32)
    bias = rng.normal(0, 1, size=OC).astype(np.float32)
    s_a, s_o = 0.05, (0.11 if u4 else 0.9)
    pk = oracle.pack_nibbles if u4 else oracle.pack_bytes
    Id = dev(pk(_to_layout(I, layout).ravel()))
    Wpk = oracle.pack_nibbles(Wc.reshape(OC, F, F, C)) if u4 else Wc.astype(np.int8)
    w_dt = "s4" if u4 else "s8"
    Wp = aligned_empty(qnn.qnn_conv_packed_w_bytes(g, w_dt))
    colsum = t.empty(OC, dtype=t.int32, device="cuda")
    qnn.qconv_prepack_w(dev(Wpk), w_dt, g, Wp, colsum)
    zp = t.empty(OC, dtype=t.int32, device="cuda")
    Mv = t.empty(OC, dtype=t.float32, device="cuda")
    Bq = t.empty(OC, dtype=t.float32, device="cuda")
    D = t.empty(OC, dtype=t.float32, device="cuda")
    qnn.q_fold_epilogue(OC, "u4" if u4 else "u8", z_in, colsum, s_a, dev(s_w), s_o, bias=dev(bias), zp_term=zp,
                        M=Mv, Bq=Bq, D=D)
    s_r = 0.13 if u4 else 1.1
    R = float(np.float32(np.float32(s_r) / np.float32(s_o)))
    res_dt = "u4" if u4 else "u8"
    resd = None if res is None else dev(pk(_to_layout(res, layout).ravel()))
    epi = qnn.epilogue(mode, relu=True, out_dt=out_dt, zp_term=zp, M=Mv, Bq=Bq, D=D, bias=dev(bias),
                       residual=resd if mode == "requant" else None, res_dt=res_dt, z_res=8 if u4 else 128, R=R)
    n_out = N * OH * OW * OC
    if mode == "requant":
        O = t.full((n_out // 2 if out_dt == "u4" else n_out,), 0x5A, dtype=t.uint8, device="cuda")
    elif mode == "dequant":
        O = t.empty(n_out, dtype=t.float32, device="cuda")
    else:
        O = t.empty(n_out, dtype=t.int32, device="cuda")
    O32 = t.zeros(n_out, dtype=t.int32, device="cuda")
    if u4:
        ws = t.full((qnn.qnn_conv_workspace_bytes(g, "u4"),), 0xFF, dtype=t.uint8, device="cuda") if workspace else None
        qnn.qconv_u4s4(Id, z_in, Wp, g, epi, O, O32, workspace=ws)
    else:
        ws = t.full((qnn.qnn_conv_workspace_bytes(g, "u8"),), 0xFF, dtype=t.uint8, device="cuda") if workspace else None
        qnn.qconv_u8s8(Id, z_in, Wp, g, epi, O, O32, workspace=ws)
    assert qnn.qnn_check_device_error() == qnn.QNN_OK
    acc = oracle.conv_acc_layout(_to_layout(I, layout), Wc, z_in, N, H, W, C, layout, (pad, pad), (st, st))
    assert np.array_equal(host(O32), acc), f"{(host(O32) != acc).sum()} accumulator mismatches"
    acc_rows = _from_layout(acc, layout, N, OH, OW, OC).reshape(-1, OC)
    _, M_o, Bq_o, D_o = oracle.fold(oracle.colsum(Wc.reshape(OC, -1)), z_in, s_a, s_w, s_o, bias)
    if mode == "s32":
        assert np.array_equal(host(O), acc)
    elif mode == "dequant":
        y = oracle.dequant_epilogue(acc_rows, D_o, bias)
        got = _from_layout(host(O), layout, N, OH, OW, OC).reshape(-1, OC)
        assert np.array_equal(f32_bits(got), f32_bits(y))
    else:
        rr = None if res is None else res.reshape(-1, OC)
        q = oracle.requant(acc_rows, M_o, Bq_o, out_dt, relu=True, res=rr, z_res=8 if u4 else 128, R=R)
        exp = (oracle.pack_nibbles if out_dt == "u4" else oracle.pack_bytes)(
            _to_layout(q.reshape(N, OH, OW, OC), layout).ravel())
        got = host(O)
        assert np.array_equal(got, exp), f"{(got != exp).sum()} output bytes differ"


@pytest.mark.parametrize("layout", ["nchw", "nchw64"])
def test_conv_u4s4_resnet_3x3_layouts_full(oracle, layout):
    """ResNet-50 stage-1 3x3 Conv_Add_Relu at full size with input, residual and
    output in NCHW and in NCHW64 (MegEngine article, conv 算子優化), every output."""
    _conv_layout(oracle, (64, 56, 56, 64, 64, 3, 1, 1), layout)


@pytest.mark.parametrize("layout,geom,workspace", [
    ("nchw", (2, 10, 12, 64, 64, 3, 1, 1), True),
    ("nchw", (2, 9, 12, 128, 64, 3, 1, 2), True),    # stride 2, ragged output rows
    ("nchw", (1, 8, 6, 256, 64, 1, 0, 1), True),     # 1x1: an NCHW input takes the pre-pass
    ("nchw64", (2, 9, 9, 64, 128, 3, 1, 1), True),
    ("nchw64", (2, 9, 9, 128, 64, 3, 1, 1), False),  # the fused path reads NCHW64 directly
    ("nchw64", (1, 7, 5, 256, 64, 1, 0, 1), False),  # 1x1, fused
])
def test_conv_u4s4_layouts(oracle, layout, geom, workspace):
    _conv_layout(oracle, geom, layout, workspace=workspace)


@pytest.mark.parametrize("layout,mode", [("nchw", "dequant"), ("nchw", "s32"), ("nchw64", "dequant")])
def test_conv_u4s4_layouts_modes(oracle, layout, mode):
    _conv_layout(oracle, (2, 8, 8, 64, 64, 3, 1, 1), layout, mode=mode, residual=False)


@pytest.mark.parametrize("layout,geom", [("nchw", (2, 9, 9, 64, 64, 3, 1, 1)), ("nchw", (1, 7, 7, 64, 96, 3, 1, 2)),
                                         ("nchw64", (2, 9, 9, 64, 64, 3, 1, 1)),
                                         ("nchw64", (1, 6, 6, 256, 128, 3, 1, 1))])
@pytest.mark.parametrize("workspace", [False, True])
def test_conv_u8s8_layouts(oracle, layout, geom, workspace):
    """u8 x s8 convs with NCHW and NCHW64 inputs / outputs: the converter warps
    (NCHW channel planes gathered) and the fp16 expansion pre-pass + tensor copies."""
    _conv_layout(oracle, geom, layout, u4=False, workspace=workspace)


def test_conv_layout_errors():
    t = torch()
    epi = qnn.epilogue("s32")
    O = t.empty(1 << 16, dtype=t.int32, device="cuda")
    I = t.zeros(1 << 16, dtype=t.uint8, device="cuda")
    Wp = aligned_empty(1 << 20)
    g = qnn.conv_geom(1, 8, 8, 64, 64, 3, 3, layout="nchw")
    with pytest.raises(qnn.QnnError) as e:   # a 4-bit NCHW input needs the pre-pass's workspace
        qnn.qconv_u4s4(I, 8, Wp, g, epi, O)
    assert e.value.status == qnn.QNN_ERR_UNSUPPORTED
    g = qnn.conv_geom(1, 8, 8, 32, 64, 3, 3, layout="nchw64")
    with pytest.raises(qnn.QnnError) as e:   # NCHW64 needs whole 64-channel blocks
        qnn.qconv_u4s4(I, 8, Wp, g, epi, O)
    assert e.value.status == qnn.QNN_ERR_INVALID_ARG
    g = qnn.conv_geom(1, 7, 7, 64, 64, 3, 3, layout="nchw")
    ws = t.empty(1 << 16, dtype=t.uint8, device="cuda")
    with pytest.raises(qnn.QnnError) as e:   # packed NCHW rows need an even width
        qnn.qconv_u4s4(I, 8, Wp, g, epi, O, workspace=ws)
    assert e.value.status == qnn.QNN_ERR_INVALID_ARG
