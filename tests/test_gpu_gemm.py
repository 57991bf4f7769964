"""qgemm_s8 (and its prepack / fold) on the GPU against the CPU oracle.

Integer accumulators and quantized outputs must match bit for bit; fp32
dequantized outputs must match bit for bit (no FMA on either side)."""
import numpy as np
import pytest

from integer_quantized_nn_gb300 import qnn, workloads
from _util import dev, host, gpu_gemm_setup, oracle_fold, f32_bits, torch

pytestmark = pytest.mark.gpu


def _run(oracle, A, a_dt, B, z_a, s_a, s_w, s_o, bias=None, mode="requant", out_dt="s8",
         z_out=0, relu=False, res=None, res_dt="s8", z_res=0, s_r=None, alpha=None,
         rows=None, want_s32=True):
    t = torch()
    M, K = A.shape
    N = B.shape[0]
    g = gpu_gemm_setup(B, a_dt, z_a, s_a, s_w, s_o, bias)
    # fold parity
    zp_o, M_o, Bq_o, D_o, cs_o = oracle_fold(oracle, B, a_dt, z_a, s_a, s_w, s_o, bias)
    assert np.array_equal(host(g["colsum"]), cs_o)
    assert np.array_equal(host(g["zp"]), zp_o)
    assert np.array_equal(f32_bits(host(g["M"])), f32_bits(M_o))
    assert np.array_equal(f32_bits(host(g["Bq"])), f32_bits(Bq_o))
    assert np.array_equal(f32_bits(host(g["D"])), f32_bits(D_o))

    Ad = dev(A)
    R = None
    resd = None
    if res is not None:
        resd = dev(res)
        R = np.float32(np.float32(s_r) / np.float32(s_o))
    al = None
    maxs = 0
    if alpha is not None:
        al = dev(alpha.astype(np.uint8))
        maxs = int(alpha.max())
    epi = qnn.epilogue(mode, relu=relu, out_dt=out_dt, z_out=z_out,
                       zp_term=None if alpha is not None else g["zp"], M=g["M"], Bq=g["Bq"],
                       D=g["D"], bias=g["bias"], residual=resd, res_dt=res_dt, z_res=z_res,
                       R=0.0 if R is None else float(R), ptf_shift=al, ptf_max_shift=maxs)
    cdt = {"requant": t.uint8, "dequant": t.float32, "s32": t.int32}[mode]
    outs = {}
    # every path: A re-encoded inside the GEMM (no workspace), by the pre-pass
    # into a workspace (pre-filled with NaN fp16 bit patterns), and the same
    # as two calls (qgemm_pack_a, qgemm_s8_packed)
    for path in ("fused", "workspace", "packed"):
        C = t.full((M, N), 0x5A if mode == "requant" else 7, dtype=cdt, device="cuda")
        C32 = t.zeros((M, N), dtype=t.int32, device="cuda") if want_s32 else None
        ws = None
        if path != "fused":
            ws = t.full((qnn.qnn_gemm_workspace_bytes(M, K),), 0xFF, dtype=t.uint8, device="cuda")
        if path == "packed":
            qnn.qgemm_pack_a(Ad, a_dt, M, K, ws, ptf_shift=al)
            qnn.qgemm_s8_packed(ws, a_dt, g["Bp"], M, N, K, epi, C, C32)
        else:
            qnn.qgemm_s8(Ad, a_dt, g["Bp"], M, N, K, epi, C, C32, workspace=ws)
        assert qnn.qnn_check_device_error() == qnn.QNN_OK
        outs[path] = (C, C32)

    sel = np.arange(M) if rows is None else rows
    A_i = A[sel].astype(np.int32)
    acc = oracle.gemm_acc(A_i, B.astype(np.int32), 0 if alpha is not None else z_a,
                          None if alpha is None else alpha.astype(np.int32))
    if mode == "requant":
        res_codes = None
        if res is not None:
            res_codes = res[sel].astype(np.int8 if res_dt == "s8" else np.uint8).astype(np.int32)
        q = oracle.requant(acc, M_o, Bq_o, out_dt, relu=relu, res=res_codes, z_res=z_res,
                           R=0.0 if R is None else R, z_out=z_out)
        exp = oracle.pack_bytes(q)
    elif mode == "dequant":
        y = oracle.dequant_epilogue(acc, D_o, bias)
    for path, (C, C32) in outs.items():
        if want_s32:
            got32 = host(C32)[sel]
            assert np.array_equal(got32, acc), f"{path}: {(got32 != acc).sum()} accumulator mismatches"
        Cg = host(C)[sel]
        if mode == "s32":
            assert np.array_equal(Cg, acc), path
        elif mode == "dequant":
            assert np.array_equal(f32_bits(Cg), f32_bits(y)), path
        else:
            assert np.array_equal(Cg, exp), f"{path}: {(Cg != exp).sum()} output mismatches"
    return acc


def test_gemm_sym_256_requant_and_s32(oracle):
    """s8 x s8 256^3, requant scale 2^-10, also emitting the raw s32."""
    w = workloads.gemm_sym()
    _run(oracle, w["A"], "s8", w["B"], 0, w["s_a"], w["s_w"], w["s_o"])


@pytest.mark.parametrize("mode", ["requant", "dequant", "s32"])
def test_gemm_ragged_u8(oracle, mode):
    """Ragged M (several 128-row tiles + tail), N not a multiple of 32, K not a
    multiple of 64: u8 activations with zero point, per-channel weights."""
    rng = np.random.default_rng(11)
    M, N, K = 389, 300, 272
    A = rng.integers(0, 256, size=(M, K)).astype(np.uint8)
    B = rng.integers(-128, 128, size=(N, K)).astype(np.int8)
    s_w = rng.uniform(1e-3, 1e-2, size=N).astype(np.float32)
    bias = rng.normal(0, 1, size=N).astype(np.float32)
    _run(oracle, A, "u8", B, 77, 0.02, s_w, 0.05, bias, mode=mode)


@pytest.mark.parametrize("out_dt,relu,z_out", [("u8", True, 9), ("s8", False, -3)])
def test_gemm_residual_relu(oracle, out_dt, relu, z_out):
    rng = np.random.default_rng(12)
    M, N, K = 260, 512, 192
    A = rng.integers(0, 256, size=(M, K)).astype(np.uint8)
    B = rng.integers(-128, 128, size=(N, K)).astype(np.int8)
    s_w = rng.uniform(1e-3, 1e-2, size=N).astype(np.float32)
    bias = rng.normal(0, 1, size=N).astype(np.float32)
    res_dt = out_dt
    lo, hi = (0, 255) if res_dt == "u8" else (-128, 127)
    res = rng.integers(lo, hi + 1, size=(M, N)).astype(np.uint8 if res_dt == "u8" else np.int8)
    _run(oracle, A, "u8", B, 128, 0.02, s_w, 0.031, bias, out_dt=out_dt, relu=relu, z_out=z_out,
         res=res, res_dt=res_dt, z_res=5, s_r=0.04)


def test_gemm_small_edge_shapes(oracle):
    rng = np.random.default_rng(13)
    for (M, N, K) in [(1, 1, 16), (7, 8, 16), (128, 256, 64), (129, 257, 80), (3, 40, 1024)]:
        A = rng.integers(-128, 128, size=(M, K)).astype(np.int8)
        B = rng.integers(-128, 128, size=(N, K)).astype(np.int8)
        _run(oracle, A, "s8", B, 0, 1.0, np.ones(N, np.float32), 2.0 ** 12)


def test_gemm_exactness_near_2_24(oracle):
    """Adversarial operands that drive every partial sum of a chunk to 2^24:
    any loss in the fp32 accumulation shows up in the raw s32 output."""
    M, N, K = 256, 256, 1024
    A = np.full((M, K), -128, np.int8)
    B = np.full((N, K), -128, np.int8)
    # rows/cols with a few +-1 mixed in at the end of K so low bits matter
    rng = np.random.default_rng(14)
    A[::2, -64:] = rng.integers(-2, 3, size=(M // 2, 64)).astype(np.int8)
    B[1::3, -32:] = rng.integers(-1, 2, size=(len(range(1, N, 3)), 32)).astype(np.int8)
    acc = _run(oracle, A, "s8", B, 0, 1.0, np.ones(N, np.float32), 2.0 ** 17, mode="s32")
    assert acc.max() == 2 ** 24


def test_gemm_exactness_u8_centred(oracle):
    """u8 operands at the extremes (0 and 255): products after centring reach
    2^14 in magnitude; K = 1024 keeps a single exact chunk."""
    M, N, K = 256, 256, 1024
    rng = np.random.default_rng(15)
    A = np.where(rng.random((M, K)) < 0.5, 0, 255).astype(np.uint8)
    A[:, :] = 0
    A[1::2] = 255
    B = np.full((N, K), -128, np.int8)
    B[::2] = 127
    _run(oracle, A, "u8", B, 3, 1.0, np.ones(N, np.float32), 2.0 ** 20, mode="s32")


@pytest.mark.parametrize("K", [2048, 3072 + 64])
def test_gemm_multi_chunk(oracle, K):
    """K above one exact chunk: fp32 chunks are drained into int32 sums."""
    rng = np.random.default_rng(16)
    M, N = 300, 384
    A = rng.integers(-128, 128, size=(M, K)).astype(np.int8)
    A[:8] = -128
    B = rng.integers(-128, 128, size=(N, K)).astype(np.int8)
    B[:8] = -128
    _run(oracle, A, "s8", B, 0, 1.0, np.ones(N, np.float32), 2.0 ** 19)


def test_gemm_ptf(oracle):
    """Power-of-Two Factor activations: A[m][k] * 2^alpha_k, alpha in 0..3."""
    w = workloads.vitl_ptf(M=300, K=512, N=256)
    t = torch()
    xd = dev(w["x"])
    Aq = t.empty(w["x"].shape, dtype=t.uint8, device="cuda")
    sc = dev(w["in_scale"])
    qnn.q_quantize(xd, Aq, "s8", qnn.qparams("sym", scale=sc, per_channel=True, axis=1))
    codes = oracle.quantize(w["x"], 0, "s8", scale=w["in_scale"], per_channel=True, axis=1)
    assert np.array_equal(host(Aq), oracle.pack_bytes(codes))
    A = codes.astype(np.int8)
    _run(oracle, A, "s8", w["B"], 0, w["s"], w["s_w"], w["s_o"], w["bias"], alpha=w["alpha"])
    # worst case: every channel shifted by 3 and extreme codes
    A2 = np.full_like(A, -128)
    al = np.full(A.shape[1], 3, np.int32)
    B2 = np.full_like(w["B"], -128)
    _run(oracle, A2, "s8", B2, 0, 1.0, np.ones(256, np.float32), 2.0 ** 24, mode="s32", alpha=al)


def test_gemm_vit_fc1_full(oracle):
    """ViT-B MLP fc1 at full size (12608 x 768 x 3072, u8 Z=128 x s8 per-channel,
    int8 out), every output element compared."""
    w = workloads.vit_fc1()
    _run(oracle, w["A"], "u8", w["B"], w["z_a"], w["s_a"], w["s_w"], w["s_o"], w["bias"])


@pytest.mark.parametrize("name", ["qkv", "proj", "fc1", "fc2"])
def test_gemm_vitl_ptf_full(oracle, name):
    """ViT-L encoder GEMMs at full size with PTF activations (the shifts applied to
    the activation codes), every output element compared with the oracle, on the
    fused, workspace and two-call paths."""
    K, N = workloads.VITL_SHAPES[name]
    w = workloads.vitl_ptf(M=12608, K=K, N=N)
    t = torch()
    xd = dev(w["x"])
    Aq = t.empty(w["x"].shape, dtype=t.uint8, device="cuda")
    qnn.q_quantize(xd, Aq, "s8", qnn.qparams("sym", scale=dev(w["in_scale"]), per_channel=True,
                                             axis=1))
    codes = oracle.quantize(w["x"], 0, "s8", scale=w["in_scale"], per_channel=True, axis=1)
    A = host(Aq).view(np.int8)
    assert np.array_equal(A.view(np.uint8), oracle.pack_bytes(codes))
    _run(oracle, A, "s8", w["B"], 0, w["s"], w["s_w"], w["s_o"], w["bias"], alpha=w["alpha"])


@pytest.mark.parametrize("n", [2048, 4096])
def test_gemm_square_full(oracle, n):
    w = workloads.gemm_square(n)
    _run(oracle, w["A"], "s8", w["B"], 0, w["s_a"], w["s_w"], w["s_o"])


def test_gemm_square_16384_sampled(oracle):
    """The largest square GEMM (16384^3): operands drawn on the device, 48
    sampled rows compared with the oracle."""
    t = torch()
    n = 16384
    A = workloads.device_uniform_s8((n, n), 5001, "cuda")
    B = workloads.device_uniform_s8((n, n), 5002, "cuda")
    from _util import aligned_empty
    Bp = aligned_empty(qnn.qnn_gemm_packed_b_bytes(n, n))
    qnn.qgemm_prepack_b(B, Bp, None)
    e = int(np.ceil(np.log2(n))) + 7
    Mv = t.full((n,), 2.0 ** -e, dtype=t.float32, device="cuda")
    Bq = t.zeros(n, dtype=t.float32, device="cuda")
    C = t.empty((n, n), dtype=t.uint8, device="cuda")
    C2 = t.empty((n, n), dtype=t.uint8, device="cuda")
    qnn.qgemm_s8(A, "s8", Bp, n, n, n, qnn.epilogue("requant", M=Mv, Bq=Bq), C)
    ws = t.empty(qnn.qnn_gemm_workspace_bytes(n, n), dtype=t.uint8, device="cuda")
    qnn.qgemm_s8(A, "s8", Bp, n, n, n, qnn.epilogue("requant", M=Mv, Bq=Bq), C2, workspace=ws)
    assert qnn.qnn_check_device_error() == qnn.QNN_OK
    rows = np.sort(np.random.default_rng(18).choice(n, 48, replace=False))
    Ah = host(A[rows]).astype(np.int32)
    Bh = host(B).astype(np.int32)
    acc = oracle.gemm_acc(Ah, Bh)
    q = oracle.requant(acc, np.full(n, 2.0 ** -e, np.float32), np.zeros(n, np.float32), "s8")
    assert np.array_equal(host(C[rows]), oracle.pack_bytes(q))
    assert np.array_equal(host(C2[rows]), oracle.pack_bytes(q))


def test_gemm_errors():
    t = torch()
    A = t.zeros((4, 24), dtype=t.int8, device="cuda")
    Bp = t.zeros(1 << 16, dtype=t.uint8, device="cuda")
    C = t.zeros((4, 8), dtype=t.uint8, device="cuda")
    Mv = t.ones(8, dtype=t.float32, device="cuda")
    epi = qnn.epilogue("requant", M=Mv, Bq=Mv)
    with pytest.raises(qnn.QnnError) as e:
        qnn.qgemm_s8(A, "s8", Bp, 4, 8, 24, epi, C)
    assert e.value.status == qnn.QNN_ERR_ALIGNMENT
    with pytest.raises(qnn.QnnError) as e:
        qnn.qgemm_s8(A, "s4", Bp, 4, 8, 16, epi, C)
    assert e.value.status == qnn.QNN_ERR_UNSUPPORTED
    with pytest.raises(qnn.QnnError) as e:
        qnn.qgemm_s8(A, "s8", Bp, 4, 8, 70000 * 16, epi, C)
    assert e.value.status in (qnn.QNN_ERR_OVERFLOW_RISK, qnn.QNN_ERR_ALIGNMENT)


def test_device_wait_timeout_reported():
    """A bounded device wait that runs out sets the status word; the host reads
    QNN_ERR_TIMEOUT and the context stays usable."""
    qnn.qnn_selftest_wait_timeout(2_000_000)  # 2 ms
    assert qnn.qnn_check_device_error() == qnn.QNN_ERR_TIMEOUT
    assert qnn.qnn_check_device_error() == qnn.QNN_OK
    t = torch()
    x = t.ones(16, device="cuda")
    assert float(x.sum()) == 16.0


def test_gemm_back_to_back_on_one_stream(oracle):
    """Weights prepacked, epilogue constants folded, A packed and the GEMM run
    back to back on one stream with no host synchronisation in between: the
    GEMM (launched as a programmatic dependent of the preceding kernel) must
    not read the fold's or the pre-pass's outputs before they are complete."""
    t = torch()
    rng = np.random.default_rng(19)
    M, N, K = 1000, 512, 768
    A = rng.integers(0, 256, size=(M, K)).astype(np.uint8)
    B = rng.integers(-128, 128, size=(N, K)).astype(np.int8)
    s_w = rng.uniform(1e-3, 1e-2, size=N).astype(np.float32)
    bias = rng.normal(0, 1, size=N).astype(np.float32)
    Ad, Bd, swd, bd = dev(A), dev(B), dev(s_w), dev(bias)
    t.cuda.synchronize()
    from _util import aligned_empty
    Bp = aligned_empty(qnn.qnn_gemm_packed_b_bytes(N, K))
    colsum = t.empty(N, dtype=t.int32, device="cuda")
    zp = t.empty(N, dtype=t.int32, device="cuda")
    Mv = t.empty(N, dtype=t.float32, device="cuda")
    Bq = t.empty(N, dtype=t.float32, device="cuda")
    ws = t.full((qnn.qnn_gemm_workspace_bytes(M, K),), 0xFF, dtype=t.uint8, device="cuda")
    C = t.full((M, N), 0x5A, dtype=t.uint8, device="cuda")
    C2 = t.full((M, N), 0x5A, dtype=t.uint8, device="cuda")
    # no host synchronisation from here to the comparison
    qnn.qgemm_prepack_b(Bd, Bp, colsum)
    qnn.q_fold_epilogue(N, "u8", 131, colsum, 0.02, swd, 0.05, bias=bd, zp_term=zp, M=Mv, Bq=Bq)
    epi = qnn.epilogue("requant", out_dt="s8", zp_term=zp, M=Mv, Bq=Bq)
    qnn.qgemm_pack_a(Ad, "u8", M, K, ws)
    qnn.qgemm_s8_packed(ws, "u8", Bp, M, N, K, epi, C)
    qnn.qgemm_s8(Ad, "u8", Bp, M, N, K, epi, C2, workspace=ws)
    assert qnn.qnn_check_device_error() == qnn.QNN_OK
    zp_o, M_o, Bq_o, _, _ = oracle_fold(oracle, B, "u8", 131, 0.02, s_w, 0.05, bias)
    acc = oracle.gemm_acc(A.astype(np.int32), B.astype(np.int32), 131)
    exp = oracle.pack_bytes(oracle.requant(acc, M_o, Bq_o, "s8"))
    assert np.array_equal(host(C), exp)
    assert np.array_equal(host(C2), exp)


def _ptf_in_weights(oracle, A, B, alpha, s_a, s_w, s_o, bias, rows=None, mode="requant"):
    """Power-of-Two Factors folded into the prepacked weights (qgemm_prepack_b_ptf)
    and the unshifted activation codes: every path must give the oracle's
    sum_k (A << alpha_k) B exactly, and the column sums sum_k B 2^alpha_k."""
    t = torch()
    M, K = A.shape
    N = B.shape[0]
    from _util import aligned_empty
    Bp = aligned_empty(qnn.qnn_gemm_packed_b_bytes(N, K))
    colsum = t.empty(N, dtype=t.int32, device="cuda")
    qnn.qgemm_prepack_b_ptf(dev(B), dev(alpha.astype(np.uint8)), Bp, colsum)
    Bsh = B.astype(np.int32) << alpha.astype(np.int32)[None, :]
    assert np.array_equal(host(colsum), oracle.colsum(Bsh))
    zp = t.empty(N, dtype=t.int32, device="cuda")
    Mv = t.empty(N, dtype=t.float32, device="cuda")
    Bq = t.empty(N, dtype=t.float32, device="cuda")
    qnn.q_fold_epilogue(N, "s8", 0, colsum, s_a, dev(np.asarray(s_w, np.float32)), s_o, bias=dev(bias), zp_term=zp,
                        M=Mv, Bq=Bq, w_per_channel=True)
    _, M_o, Bq_o, _ = oracle.fold(oracle.colsum(Bsh), 0, s_a, np.asarray(s_w, np.float32), s_o, bias)
    epi = qnn.epilogue(mode, zp_term=zp, M=Mv, Bq=Bq, out_dt="s8", ptf_max_shift=int(alpha.max()))
    Ad = dev(A)
    sel = np.arange(M) if rows is None else rows
    acc = oracle.gemm_acc(A[sel].astype(np.int32), B.astype(np.int32), 0, alpha.astype(np.int32))
    exp = oracle.pack_bytes(oracle.requant(acc, M_o, Bq_o, "s8")) if mode == "requant" else acc
    for path in ("fused", "workspace", "packed"):
        C = t.full((M, N), 0x5A, dtype=t.uint8 if mode == "requant" else t.int32, device="cuda")
        ws = t.full((qnn.qnn_gemm_workspace_bytes(M, K),), 0xFF, dtype=t.uint8, device="cuda")
        if path == "packed":
            qnn.qgemm_pack_a(Ad, "s8", M, K, ws)
            qnn.qgemm_s8_packed(ws, "s8", Bp, M, N, K, epi, C)
        else:
            qnn.qgemm_s8(Ad, "s8", Bp, M, N, K, epi, C, workspace=None if path == "fused" else ws)
        assert qnn.qnn_check_device_error() == qnn.QNN_OK, path
        got = host(C)[sel]
        assert np.array_equal(got, exp), f"{path}: {(got != exp).sum()} mismatches"


def test_gemm_ptf_in_weights(oracle):
    """FQ-ViT 3.2 Power-of-Two Factor moved onto the weights at prepack: the same
    integers as shifting the activations, on ragged and multi-step shapes."""
    w = workloads.vitl_ptf(M=300, K=512, N=256)
    codes = oracle.quantize(w["x"], 0, "s8", scale=w["in_scale"], per_channel=True, axis=1).astype(np.int8)
    _ptf_in_weights(oracle, codes, w["B"], w["alpha"], w["s"], w["s_w"], w["s_o"], w["bias"])
    rng = np.random.default_rng(30)
    M, N, K = 389, 300, 1088
    A = rng.integers(-128, 128, size=(M, K)).astype(np.int8)
    B = rng.integers(-128, 128, size=(N, K)).astype(np.int8)
    al = rng.integers(0, 4, size=K)
    _ptf_in_weights(oracle, A, B, al, 0.02, rng.uniform(1e-3, 1e-2, N), 3.0, rng.normal(0, 1, N).astype(np.float32))
    # extreme values: every product 128 * 1024, every exact run two K steps long
    A2 = np.full((256, 1024), -128, np.int8)
    B2 = np.full((256, 1024), -128, np.int8)
    _ptf_in_weights(oracle, A2, B2, np.full(1024, 3), 1.0, np.ones(256), 2.0 ** 30, np.zeros(256, np.float32),
                    mode="s32")


@pytest.mark.parametrize("name", ["qkv", "proj", "fc1", "fc2"])
def test_gemm_vitl_ptf_in_weights_full(oracle, name):
    """ViT-L GEMMs at full size with the PTF factors folded into the weights,
    every output element compared with the oracle."""
    K, N = workloads.VITL_SHAPES[name]
    w = workloads.vitl_ptf(M=12608, K=K, N=N)
    A = oracle.quantize(w["x"], 0, "s8", scale=w["in_scale"], per_channel=True, axis=1).astype(np.int8)
    _ptf_in_weights(oracle, A, w["B"], w["alpha"], w["s"], w["s_w"], w["s_o"], w["bias"])


def test_gemm_device_argument_checks():
    """Conditions only the device can see are reported by qnn_check_device_error
    as QNN_ERR_INVALID_ARG: a PTF shift byte above ptf_max_shift (fused, pre-pass
    and two-call paths); a prepack shift above 3; weights whose folded factors
    need more exact runs than the launch was planned for; a weight image whose
    trailer belongs to another K."""
    t = torch()
    from _util import aligned_empty
    M, N, K = 256, 256, 1024
    A = t.full((M, K), -128, dtype=t.int8, device="cuda")
    B = t.full((N, K), -128, dtype=t.int8, device="cuda")
    Bp = aligned_empty(qnn.qnn_gemm_packed_b_bytes(N, K))
    qnn.qgemm_prepack_b(B, Bp, None)
    C = t.empty((M, N), dtype=t.int32, device="cuda")
    ws = t.empty(qnn.qnn_gemm_workspace_bytes(M, K), dtype=t.uint8, device="cuda")
    al = t.zeros(K, dtype=t.uint8, device="cuda")
    al[700] = 3
    epi = qnn.epilogue("s32", ptf_shift=al, ptf_max_shift=1)
    assert qnn.qnn_check_device_error() == qnn.QNN_OK
    for wsp in (None, ws):
        qnn.qgemm_s8(A, "s8", Bp, M, N, K, epi, C, workspace=wsp)
        assert qnn.qnn_check_device_error() == qnn.QNN_ERR_INVALID_ARG
    qnn.qgemm_pack_a(A, "s8", M, K, ws, ptf_shift=al)
    assert qnn.qnn_check_device_error() == qnn.QNN_OK
    qnn.qgemm_s8_packed(ws, "s8", Bp, M, N, K, epi, C)
    assert qnn.qnn_check_device_error() == qnn.QNN_ERR_INVALID_ARG
    # shifts folded into the weights: a bound of 0 launches the one-run kernel,
    # which finds that these weights need runs of two K steps
    Bf = aligned_empty(qnn.qnn_gemm_packed_b_bytes(N, K))
    qnn.qgemm_prepack_b_ptf(B, t.full((K,), 3, dtype=t.uint8, device="cuda"), Bf, None)
    assert qnn.qnn_check_device_error() == qnn.QNN_OK
    for wsp in (None, ws):
        qnn.qgemm_s8(A, "s8", Bf, M, N, K, qnn.epilogue("s32"), C, workspace=wsp)
        assert qnn.qnn_check_device_error() == qnn.QNN_ERR_INVALID_ARG
        qnn.qgemm_s8(A, "s8", Bf, M, N, K, qnn.epilogue("s32", ptf_max_shift=3), C, workspace=wsp)
        assert qnn.qnn_check_device_error() == qnn.QNN_OK
        assert bool((C == 1024 * 128 * 1024).all())
    qnn.qgemm_prepack_b_ptf(B, t.full((K,), 4, dtype=t.uint8, device="cuda"), Bf, None)
    assert qnn.qnn_check_device_error() == qnn.QNN_ERR_INVALID_ARG
    # an image prepacked for K = 1024 used as K = 512 (in bounds: a smaller view)
    qnn.qgemm_s8(A[:, :512].contiguous(), "s8", Bp, M, N, 512, qnn.epilogue("s32"), C)
    assert qnn.qnn_check_device_error() == qnn.QNN_ERR_INVALID_ARG
