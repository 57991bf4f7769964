"""Seeded synthetic inputs for the quantized GEMM / implicit-GEMM conv workloads.

This module holds random draws, shapes and fixed parameters only: none of the
quantized arithmetic itself.  Both the CPU oracle and the CUDA path are fed
from it.  Every tensor is drawn from numpy ``PCG64(1000 * workload + tensor)``
so that a (workload, tensor) pair always gives the same bytes.

Packed 4-bit tensors are drawn directly as random bytes: two independent
uniform nibbles per byte are exactly "values uniform in 0..15 (or -8..7)".

Workloads (the layer shapes of the pages' models stand in for their datasets):
  gemm_sym      : s8 x s8, per-tensor symmetric, requant scale 2^-10 (256^3)
  vit_fc1       : ViT-B MLP fc1, u8 (Z=128) x s8 per-channel, 12608 x 768 x 3072
  conv3x3_u4    : ResNet-50 stage-1 3x3 Conv_Add_Relu, u4 x s4, NHWC 64x56x56x64
  conv1x1_u4    : ResNet-50 stage-1 1x1 Conv_Relu, u4 x s4, 256 -> 64 channels
  vitl_ptf      : ViT-L encoder GEMMs, s8 activations with per-channel
                  power-of-two factors (5% outlier channels x40)
  gemm_square   : s8 x s8 square GEMMs M=N=K, requant to s8
  quant_rows    : fp32 -> s8 per-row symmetric quantize of a 16384^2 tensor
  vit_attention : ViT-B self-attention maps (12 heads, 197 tokens, head dim 64):
                  int32 logit codes of Q K^T, s8 value codes, for Log-Int-Softmax
  vit_layernorm : ViT-B LayerNorm inputs (197 tokens x 768 channels), s8 codes with
                  per-channel power-of-two factors, for the integer LayerNorm
  conv_u8       : ResNet-50 stage-1 3x3 Conv_Add_Relu with u8 activations and u8
                  filters carrying per-filter zero points (both operands asymmetric)
  vit_fc1_zw    : ViT-B MLP fc1 with u8 weights carrying per-channel zero points
"""
from __future__ import annotations

import math
import numpy as np

# workload ids (seed = 1000 * id + tensor id)
GEMM_SYM, VIT_FC1, CONV_U4, VITL_PTF, SQUARE, ATTN, LNORM, CONV_U8, VIT_FC1_ZW = 1, 2, 3, 4, 5, 6, 7, 8, 9


def rng(workload: int, tensor: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(1000 * workload + tensor))


def _uniform_int(g, lo, hi, shape, dtype):
    return g.integers(lo, hi + 1, size=shape, dtype=np.int64).astype(dtype)


def _normal_codes(g, mean, std, lo, hi, shape, dtype):
    v = np.rint(g.normal(mean, std, size=shape))
    return np.clip(v, lo, hi).astype(dtype)


def gemm_sym(M=256, N=256, K=256, tag=0):
    """A, B int8 uniform in [-128, 127]; scales 1, 1 and 2^10 so that the folded
    requant multiplier is exactly 2^-10; no bias, output zero point 0."""
    g = rng(GEMM_SYM, 10 * tag + 0)
    A = _uniform_int(g, -128, 127, (M, K), np.int8)
    B = _uniform_int(rng(GEMM_SYM, 10 * tag + 1), -128, 127, (N, K), np.int8)
    return dict(A=A, B=B, a_dt="s8", z_a=0, s_a=1.0, s_w=np.ones(N, np.float32),
                bias=None, s_o=1024.0, z_out=0, out_dt="s8")


def vit_fc1(M=12608, K=768, N=3072, tag=0):
    """u8 activations round(N(128, 30)) clipped, Z_a = 128, S_a = 0.02; int8
    weights round(N(0, 25)) clipped, stored [N, K]; per-output-channel weight
    scales U(1e-3, 1e-2); bias N(0, 1).  Output scale: a closed form from the
    distribution parameters, 4 standard deviations of the real output over the
    int8 half-range (no data-dependent computation)."""
    A = _normal_codes(rng(VIT_FC1, 10 * tag + 0), 128.0, 30.0, 0, 255, (M, K), np.uint8)
    B = _normal_codes(rng(VIT_FC1, 10 * tag + 1), 0.0, 25.0, -128, 127, (N, K), np.int8)
    s_w = rng(VIT_FC1, 10 * tag + 2).uniform(1e-3, 1e-2, size=N).astype(np.float32)
    bias = rng(VIT_FC1, 10 * tag + 3).normal(0.0, 1.0, size=N).astype(np.float32)
    s_a = 0.02
    std = math.sqrt((s_a * 0.0055 * 30.0 * 25.0) ** 2 * K + 1.0)
    s_o = float(np.float32(4.0 * std / 127.0))
    return dict(A=A, B=B, a_dt="u8", z_a=128, s_a=s_a, s_w=s_w, bias=bias, s_o=s_o,
                z_out=0, out_dt="s8")


def conv_u4(N=64, H=56, W=56, C=64, OC=64, F=3, pad=1, stride=1, residual=True, tag=0):
    """NHWC packed u4 input (Z_I = 8), OHWI packed s4 weights, per-output-channel
    weight scales U(1e-3, 1e-2), bias N(0, 1), optional packed u4 residual
    (Z_r = 8, S_r = 1.25 S_o); u4 output with ReLU and Z_o = 0."""
    wl = CONV_U4
    I = rng(wl, 10 * tag + 0).integers(0, 256, size=(N, H, W, C // 2), dtype=np.int64).astype(np.uint8)
    Wt = rng(wl, 10 * tag + 1).integers(0, 256, size=(OC, F, F, C // 2), dtype=np.int64).astype(np.uint8)
    s_w = rng(wl, 10 * tag + 2).uniform(1e-3, 1e-2, size=OC).astype(np.float32)
    bias = rng(wl, 10 * tag + 3).normal(0.0, 1.0, size=OC).astype(np.float32)
    OH = (H + 2 * pad - F) // stride + 1
    OW = (W + 2 * pad - F) // stride + 1
    res = None
    if residual:
        res = rng(wl, 10 * tag + 4).integers(0, 256, size=(N, OH, OW, OC // 2),
                                             dtype=np.int64).astype(np.uint8)
    s_a = 0.02
    K = F * F * C
    # uniform codes: std of (q - 8) and of s4 weights is sqrt(255/12) ~ 4.61
    std = math.sqrt((s_a * 0.0055 * 4.61 * 4.61) ** 2 * K + 1.0)
    s_o = float(np.float32(3.0 * std / 15.0))
    return dict(I=I, W=Wt, z_in=8, s_a=s_a, s_w=s_w, bias=bias, s_o=s_o, z_out=0,
                res=res, z_res=8, s_r=float(np.float32(1.25 * s_o)), relu=True,
                pad=(pad, pad), stride=(stride, stride), F=F, out_dt="u4")


def conv_u8(N=64, H=56, W=56, C=64, OC=64, F=3, pad=1, stride=1, residual=True, tag=0):
    """NHWC u8 input codes uniform in 0..255 with Z_I = 128; OHWI u8 filters
    round(N(z_w[oc], 40)) clipped, per-filter zero points z_w uniform in 96..160;
    weight scales U(1e-3, 1e-2), bias N(0, 1); optional u8 residual uniform in
    0..255 (Z_r = 128, S_r = 1.25 S_o); u8 output with ReLU and Z_o = 0."""
    wl = CONV_U8
    I = _uniform_int(rng(wl, 10 * tag + 0), 0, 255, (N, H, W, C), np.uint8)
    z_w = _uniform_int(rng(wl, 10 * tag + 1), 96, 160, (OC,), np.int32)
    Wt = np.clip(np.rint(rng(wl, 10 * tag + 2).normal(0.0, 40.0, size=(OC, F, F, C)) + z_w.reshape(-1, 1, 1, 1)),
                 0, 255).astype(np.uint8)
    s_w = rng(wl, 10 * tag + 3).uniform(1e-3, 1e-2, size=OC).astype(np.float32)
    bias = rng(wl, 10 * tag + 4).normal(0.0, 1.0, size=OC).astype(np.float32)
    OH = (H + 2 * pad - F) // stride + 1
    OW = (W + 2 * pad - F) // stride + 1
    res = None
    if residual:
        res = _uniform_int(rng(wl, 10 * tag + 5), 0, 255, (N, OH, OW, OC), np.uint8)
    s_a = 0.02
    K = F * F * C
    # std of (q - 128) for uniform codes sqrt(65535 / 12) ~ 73.9; of w - z_w about 40
    std = math.sqrt((s_a * 0.0055 * 73.9 * 40.0) ** 2 * K + 1.0)
    s_o = float(np.float32(3.0 * std / 255.0))
    return dict(I=I, W=Wt, z_w=z_w, z_in=128, s_a=s_a, s_w=s_w, bias=bias, s_o=s_o, z_out=0,
                res=res, z_res=128, s_r=float(np.float32(1.25 * s_o)), relu=True,
                pad=(pad, pad), stride=(stride, stride), F=F, out_dt="u8")


def vit_fc1_zw(M=12608, K=768, N=3072, tag=0):
    """vit_fc1 with asymmetric u8 weights: activations as in vit_fc1 (u8, Z_a =
    128, S_a = 0.02); weights round(N(z_w[n], 25)) clipped to 0..255 with
    per-channel zero points z_w uniform in 96..160; scales, bias and the output
    scale as in vit_fc1."""
    A = _normal_codes(rng(VIT_FC1_ZW, 10 * tag + 0), 128.0, 30.0, 0, 255, (M, K), np.uint8)
    z_w = _uniform_int(rng(VIT_FC1_ZW, 10 * tag + 1), 96, 160, (N,), np.int32)
    B = np.clip(np.rint(rng(VIT_FC1_ZW, 10 * tag + 2).normal(0.0, 25.0, size=(N, K)) + z_w[:, None]),
                0, 255).astype(np.uint8)
    s_w = rng(VIT_FC1_ZW, 10 * tag + 3).uniform(1e-3, 1e-2, size=N).astype(np.float32)
    bias = rng(VIT_FC1_ZW, 10 * tag + 4).normal(0.0, 1.0, size=N).astype(np.float32)
    s_a = 0.02
    std = math.sqrt((s_a * 0.0055 * 30.0 * 25.0) ** 2 * K + 1.0)
    s_o = float(np.float32(4.0 * std / 127.0))
    return dict(A=A, B=B, z_w=z_w, a_dt="u8", z_a=128, s_a=s_a, s_w=s_w, bias=bias, s_o=s_o,
                z_out=0, out_dt="s8")


def vitl_ptf(M=12608, K=1024, N=3072, tag=0):
    """ViT-L encoder GEMM with Power-of-Two-Factor activations.  Real
    activations x ~ N(0, 1) per channel with a seeded 5% of the K channels
    multiplied by 40; per-channel shifts alpha in 0..3 and the layer-wise scale
    chosen by absmax over the drawn data (the calibration the pages describe,
    done here once as input preparation): s = max|x| / (127 * 8), alpha_c the
    smallest alpha with max|x_c| <= 127 * 2^alpha * s.  Weights int8
    round(N(0, 25)) clipped, stored [N, K]; scales U(1e-3, 1e-2); bias N(0, 1)."""
    wl = VITL_PTF
    g = rng(wl, 10 * tag + 0)
    x = g.standard_normal(size=(M, K), dtype=np.float32)
    n_out = max(1, int(round(0.05 * K)))
    outl = rng(wl, 10 * tag + 1).choice(K, size=n_out, replace=False)
    x[:, outl] *= np.float32(40.0)
    amax = np.abs(x).max(axis=0).astype(np.float64)
    s = float(np.float32(amax.max() / (127.0 * 8.0)))
    alpha = np.zeros(K, np.int32)
    for a in (3, 2, 1, 0):
        alpha[amax <= 127.0 * (2 ** a) * s] = a
    in_scale = (np.float32(s) * (2.0 ** alpha)).astype(np.float32)   # exact: power-of-two multiples
    B = _normal_codes(rng(wl, 10 * tag + 2), 0.0, 25.0, -128, 127, (N, K), np.int8)
    s_w = rng(wl, 10 * tag + 3).uniform(1e-3, 1e-2, size=N).astype(np.float32)
    bias = rng(wl, 10 * tag + 4).normal(0.0, 1.0, size=N).astype(np.float32)
    # real output std ~ sqrt(K * E[x^2] * (25 * 0.0055)^2): E[x^2] = 0.95 + 0.05 * 1600
    std = math.sqrt(K * (0.95 + 0.05 * 1600.0) * (25.0 * 0.0055) ** 2 + 1.0)
    s_o = float(np.float32(4.0 * std / 127.0))
    return dict(x=x, in_scale=in_scale, alpha=alpha, s=s, B=B, s_w=s_w, bias=bias,
                s_o=s_o, z_out=0, out_dt="s8")


VITL_SHAPES = {"qkv": (1024, 3072), "proj": (1024, 1024), "fc1": (1024, 4096),
               "fc2": (4096, 1024)}


def gemm_square(n, tag=0):
    """A, B int8 uniform in [-128, 127], M = N = K = n; requant multiplier
    2^-(ceil(log2 K) + 7) (scales 1, 1 and 2^(ceil(log2 K) + 7)), no bias."""
    A = _uniform_int(rng(SQUARE, 10 * tag + 0), -128, 127, (n, n), np.int8)
    B = _uniform_int(rng(SQUARE, 10 * tag + 1), -128, 127, (n, n), np.int8)
    e = int(math.ceil(math.log2(n))) + 7
    return dict(A=A, B=B, a_dt="s8", z_a=0, s_a=1.0, s_w=np.ones(n, np.float32), bias=None,
                s_o=float(2.0 ** e), z_out=0, out_dt="s8")


def quant_rows(rows=16384, cols=16384, tag=0):
    """x fp32 ~ N(0, 1), [rows, cols]; per-row (axis 0) symmetric scales
    max|x_row| / 127, chosen once as input preparation."""
    x = rng(SQUARE, 10 * tag + 5).standard_normal(size=(rows, cols), dtype=np.float32)
    scale = (np.abs(x).max(axis=1) / np.float32(127.0)).astype(np.float32)
    return dict(x=x, scale=scale)


# Scale of the attention logit codes: s_q s_k / sqrt(64) with s_q = s_k = 0.04
# (a product of the int8 Q and K codes over the head dimension 64).
ATTN_S = float(np.float32(0.04 * 0.04 / 8.0))


def vit_attention(B=4, H=12, L=197, d=64, tag=0):
    """Attention logits as int32 codes at scale ATTN_S: real logits N(0, 2.5) per
    element (a spread whose softmax over 197 tokens leaves most probabilities
    below 1/16 and a few near the top), plus one sink column (token 0, the class
    token) raised by 4; value codes round(N(0, 40)) clipped to s8.
    x: int32 [B*H, L, L]; v: int8 [B*H, L, d]."""
    g = rng(ATTN, 10 * tag + 0)
    z = g.normal(0.0, 2.5, size=(B * H, L, L))
    z[:, :, 0] += 4.0
    x = np.rint(z / ATTN_S).astype(np.int32)
    v = _normal_codes(rng(ATTN, 10 * tag + 1), 0.0, 40.0, -128, 127, (B * H, L, d), np.int8)
    return dict(x=x, v=v, S=ATTN_S, bits=4)


def device_attention_logits(rows, L, seed, device):
    """The vit_attention logit distribution drawn on the device (int32 [rows, L])."""
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    z = torch.randn((rows, L), generator=g, device=device, dtype=torch.float32) * 2.5
    z[:, 0] += 4.0
    return torch.round(z / ATTN_S).to(torch.int32)


def vit_layernorm(rows=64 * 197, C=768, tag=0):
    """LayerNorm input codes x = clip(round(N(0, 30))) (s8) at layer scale s = 0.02
    with per-channel factors alpha: 5% of the channels (seeded) carry 2^3, the
    inter-channel spread PTF is for; gamma = U(0.5, 1.5) with random signs,
    beta ~ N(0, 0.2); one output scale 0.04 for all channels."""
    x = _normal_codes(rng(LNORM, 10 * tag + 0), 0.0, 30.0, -128, 127, (rows, C), np.int8)
    g = rng(LNORM, 10 * tag + 1)
    alpha = np.where(g.random(C) < 0.05, 3, 0).astype(np.uint8)
    gamma = (g.uniform(0.5, 1.5, size=C) * g.choice([-1.0, 1.0], size=C)).astype(np.float32)
    beta = g.normal(0.0, 0.2, size=C).astype(np.float32)
    o = np.full(C, 0.04, np.float32)
    return dict(x=x, alpha=alpha, s=0.02, gamma=gamma, beta=beta, o=o)


def device_uniform_s8(shape, seed, device):
    """Large int8 operands drawn on the device with a seeded torch generator
    (for sizes where host generation would dominate the run)."""
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return torch.randint(-128, 128, shape, generator=g, device=device, dtype=torch.int16).to(torch.int8)


def device_normal_f32(shape, seed, device):
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return torch.randn(shape, generator=g, device=device, dtype=torch.float32)
