/*
 * qnn.h -- C ABI of the GB300 (sm_103a) linear-quantized GEMM and
 * implicit-GEMM convolution library (libqnn.so).
 *
 * Page sources cited below (title, section):
 *   [QI] "【量化】神经网络量化介绍" (loveleaves.github.io/p/quantization)
 *   [MG] MegEngine 4-bit quantization article (m.xsypw.cn/d/1897816)
 *   [FQ] "首个完全量化Vision Transformer的方法FQ-ViT" (aijishu.com)
 *
 * Conventions for every call:
 *  - Every tensor pointer is a DEVICE pointer owned by the caller; shapes,
 *    scalars and parameter structs are host values.  The library allocates
 *    nothing and keeps no hidden buffers (one device status word aside).
 *  - Calls are asynchronous on the given stream (NULL: the legacy default
 *    stream) and never synchronise, except qnn_check_device_error.
 *  - Arguments are validated on the host before any launch; a failed check
 *    returns a status and launches nothing.  Nothing aborts or throws across
 *    the ABI.  There is no CPU fallback: what the kernels cannot do returns
 *    QNN_ERR_UNSUPPORTED.
 *  - Base pointers must be 16-byte aligned (QNN_ERR_ALIGNMENT).
 *  - 4-bit tensors hold two codes per byte along their innermost dimension,
 *    element 2i in the low nibble; that dimension must be even.
 *  - Rounding is round-half-to-even throughout; fp32 arithmetic is done as the
 *    separate IEEE operations documented per call (no fused multiply-add).
 */
#ifndef QNN_H_
#define QNN_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *qnn_stream_t; /* a cudaStream_t */

typedef enum {
    QNN_OK = 0,
    QNN_ERR_INVALID_ARG = 1,   /* bad shape, NULL pointer, bad enum, bad range */
    QNN_ERR_UNSUPPORTED = 2,   /* valid request the kernels do not implement */
    QNN_ERR_ALIGNMENT = 3,     /* pointer or row pitch not 16-byte aligned */
    QNN_ERR_OVERFLOW_RISK = 4, /* the int32 accumulator could overflow */
    QNN_ERR_CUDA = 5,          /* a CUDA runtime call failed */
    QNN_ERR_TIMEOUT = 6        /* a device-side bounded wait gave up */
} qnn_status;

typedef enum { QNN_S8 = 0, QNN_U8 = 1, QNN_S4 = 2, QNN_U4 = 3, QNN_S32 = 4, QNN_F32 = 5 } qnn_dtype;

/* Quantization schemes [QI 量化模式]:
 *   QNN_SYM : q = clip(rint(x / s))
 *   QNN_ASYM: q = clip(rint(x / s) + z)          (offset added after rounding)
 *   QNN_POW2: q = clip(rint(x * 2^shift))        ("integer" quantization; the
 *             page's text writes 2 << shift, read here as 2^shift, shift being
 *             the number of fractional bits) */
typedef enum { QNN_SYM = 0, QNN_ASYM = 1, QNN_POW2 = 2 } qnn_scheme;

/* Quantization parameters, per tensor or per channel [QI tensor量化与通道量化]. */
typedef struct {
    int32_t scheme;            /* qnn_scheme */
    int32_t per_channel;       /* 0: element 0 of each array applies everywhere */
    int32_t axis;              /* channel axis when per_channel (negative counts from the end) */
    int32_t narrow_range;      /* signed codes: qmin = -qmax (int8 -127..127) */
    const float *scale;        /* device [C] or [1]: SYM, ASYM; must be > 0 */
    const int32_t *zero_point; /* device [C] or [1]: ASYM; must lie in the code range */
    const int32_t *shift;      /* device [C] or [1]: POW2; -126..126 */
} qnn_qparams;

/* Quantize [QI 量化算子, 量化模式; MG 背景 (UINT4 0..15, INT4 -8..7)].
 * x: fp32 tensor of `ndim` dims `shape` (host array), contiguous.  q: codes of
 * q_dt (S8, U8, S4, U4), same shape, contiguous (4-bit: packed along the last
 * dim).  Per element: t = x / s (IEEE fp32 divide), r = rint(t), ASYM adds
 * (float)z after rounding, POW2 uses r = rint(x * 2^shift); then the float is
 * clipped to [qmin, qmax] and stored.  NaN becomes the code of real zero (z,
 * else 0); +-Inf saturate. */
qnn_status q_quantize(const float *x, void *q, qnn_dtype q_dt, int ndim, const int64_t *shape,
                      const qnn_qparams *p, qnn_stream_t stream);

/* Dequantize [QI 反量化算子; MG 背景: r = S (q - Z)].  x = (float)(q - z) * s
 * (integer subtract, one fp32 multiply); POW2: x = q * 2^-shift (exact). */
qnn_status q_dequantize(const void *q, qnn_dtype q_dt, float *x, int ndim, const int64_t *shape,
                        const qnn_qparams *p, qnn_stream_t stream);

/* ---- ahead of inference: weight prepack and constant folding -------------- */

/* Size in bytes of the prepacked GEMM weight operand for B of shape [N, K]. */
size_t qnn_gemm_packed_b_bytes(int N, int K);

/* Prepack int8 weights B [N, K] (row-major, the Linear weight layout: output
 * channel n, input channel k) into the GEMM kernel's shared-memory operand
 * image (`B_packed`, qnn_gemm_packed_b_bytes bytes, 1024-byte aligned), and
 * write colsum[n] = sum_k B[n][k] (int32 [N]), the weight sums that the
 * zero-point cross term needs [MG 緩解精度下降].  K must be a multiple of 16.
 * The image ends with a small trailer of bounds on the weight magnitudes (per
 * K step of 64 and per column); the GEMM reads it to size the runs of K over
 * which its fp32 partial sums stay exact integers, so a B_packed must come
 * from one of the prepack calls for the same N and K (a GEMM given a trailer
 * that does not match its K reports QNN_ERR_INVALID_ARG through
 * qnn_check_device_error). */
qnn_status qgemm_prepack_b(const int8_t *B, int N, int K, void *B_packed, int32_t *colsum,
                           qnn_stream_t stream);

/* Prepack int8 weights with per-input-channel Power-of-Two Factors folded in
 * [FQ 3.2: the activation codes x_q of a PTF quantizer enter the next layer as
 * x_q * 2^alpha_k; since sum_k (a_k 2^alpha_k) B[n][k] = sum_k a_k (B[n][k]
 * 2^alpha_k), the factor can ride on the constant operand]: the image holds
 * B[n][k] * 2^ptf_shift[k] (|.| <= 1024, exact in fp16) and colsum[n] =
 * sum_k B[n][k] 2^ptf_shift[k].  ptf_shift: device u8 [K], every value 0..3 (a
 * larger one is reported as QNN_ERR_INVALID_ARG by qnn_check_device_error).
 * Call qgemm_s8 with the UNSHIFTED activation codes, epi->ptf_shift = NULL and
 * epi->ptf_max_shift = the largest shift: the result is exactly that of
 * epi->ptf_shift = ptf_shift on plain weights, without the per-call shift of
 * A. */
qnn_status qgemm_prepack_b_ptf(const int8_t *B, const uint8_t *ptf_shift, int N, int K, void *B_packed,
                               int32_t *colsum, qnn_stream_t stream);

/* Fold the per-output-channel constants ahead of inference [MG 緩解精度下降:
 * the zero-point part that does not depend on the input is computed before
 * inference; QI 量化乘法: scale_abc computed ahead].  For n in [0, N):
 *   zp_term[n] = (z_a - c_a) * colsum[n]   (int32), where c_a is the centre the
 *                kernels subtract from the activation codes as they load them:
 *                128 for U8 activations, 0 for S8, U4 (and S4)
 *   M[n]  = (s_a * s_w[n]) / s_o            fp32 multiply, then fp32 divide
 *   Bq[n] = bias[n] / s_o
 *   D[n]  = s_a * s_w[n]                    (dequantizing epilogue)
 * s_w: device [N] if w_per_channel else [1].  bias: device [N] or NULL (zero).
 * Outputs are device [N]; any of M, Bq, D may be NULL to skip it. */
qnn_status q_fold_epilogue(int N, qnn_dtype a_dt, int32_t z_a, const int32_t *colsum, float s_a,
                           const float *s_w, int w_per_channel, const float *bias, float s_o,
                           int32_t *zp_term, float *M, float *Bq, float *D, qnn_stream_t stream);

/* ---- fused epilogue -------------------------------------------------------- */

typedef enum {
    QNN_EPI_REQUANT = 0, /* quantized output of out_dt */
    QNN_EPI_DEQUANT = 1, /* fp32 output */
    QNN_EPI_S32 = 2      /* raw int32 accumulator (zero-point corrected) */
} qnn_epi_mode;

/* Per output element (row m, column n), with acc_c = acc - zp_term[n]:
 * REQUANT [QI 量化乘法, 量化加法, 量化激活函数, 常见计算图优化 (conv-add
 *         Y = Wx + (Y2 + B)); MG 算子融合優化 (Conv_Relu, Conv_Add_Relu)]:
 *     t = Bq[n];  residual: t = (float)(res[m][n] - z_res) * R + t
 *     v = (float)acc_c * M[n];  v = v + t;  r = rint(v);  relu: r = max(r, 0)
 *     q = clip(r + (float)z_out)  to out_dt's range
 * DEQUANT [QI 反量化算子]: y = (float)acc_c * D[n] + bias[n]   (fmul, fadd)
 * S32: acc_c. */
typedef struct {
    int32_t mode;            /* qnn_epi_mode */
    int32_t relu;            /* REQUANT: fused ReLU */
    int32_t out_dt;          /* REQUANT output: S8 or U8 (GEMM), U4 or U8 (conv) */
    int32_t z_out;           /* REQUANT output zero point */
    const int32_t *zp_term;  /* device [N] or NULL (zero) */
    const float *M;          /* device [N]: REQUANT */
    const float *Bq;         /* device [N]: REQUANT */
    const float *D;          /* device [N]: DEQUANT */
    const float *bias;       /* device [N] or NULL: DEQUANT */
    const void *residual;    /* device [rows, N] codes of res_dt (same layout as the
                                output), or NULL: REQUANT only */
    int32_t res_dt;          /* S8, U8 (GEMM); U4, U8 (conv) */
    int32_t z_res;           /* residual zero point, inside res_dt's code range
                                (else QNN_ERR_INVALID_ARG) */
    float R;                 /* S_res / S_out */
    const uint8_t *ptf_shift;/* device [K] per-input-channel Power-of-Two Factor
                                alpha_k [FQ 3.2]: the GEMM uses A[m][k] * 2^alpha_k;
                                S8 activations with z_a = 0 only; NULL: none */
    int32_t ptf_max_shift;   /* upper bound (0..3) on every shift: of ptf_shift, or,
                                with ptf_shift NULL, of the shifts folded into the
                                weights by qgemm_prepack_b_ptf (0: none).  A shift
                                byte above it is reported as QNN_ERR_INVALID_ARG
                                by qnn_check_device_error. */
    const float *row_scale;  /* device [rows] per-row activation scales (dynamic per-token
                                quantization, q_quantize_rows_dynamic), or NULL: the
                                per-channel factor is first scaled by the row's,
                                M[n] -> row_scale[m] * M[n] (REQUANT) and
                                D[n] -> row_scale[m] * D[n] (DEQUANT), one fp32
                                multiply; fold with s_a = 1 so that M = s_w / s_o and
                                D = s_w */
} qnn_epilogue;

/* Size in bytes of the qgemm_s8 workspace for an M x K activation operand
 * (the re-encoded A image: ceil(M / 128) * ceil(K / 64) * 16 KB); 0 if M or K
 * is not positive. */
size_t qnn_gemm_workspace_bytes(int M, int K);

/* Quantized GEMM [QI 量化矩阵乘; MG 緩解精度下降]:
 *   acc[m][n] = sum_k (A[m][k] - c_a) * 2^alpha_k * B[n][k]   exact, in int32
 * then the epilogue above with zp_term folded by q_fold_epilogue.
 * The products run on fp16 tensor cores with fp32 partial sums, which are exact
 * integers while they stay within 2^24: K is summed in runs no longer than the
 * weight magnitudes recorded at prepack allow (every K at once when
 * 128 * 2^(A's shift) * max_n sum_k |B'[n][k]| <= 2^24), the runs added in int32.
 * A: device [M, K] row-major codes of a_dt (S8 or U8); K % 16 == 0.
 * B_packed: from qgemm_prepack_b for the same N, K.
 * C: device [M, N] row-major, of out_dt (REQUANT), fp32 (DEQUANT) or int32 (S32).
 * C_s32: optional device [M, N] int32 that also receives acc_c (NULL: none).
 * workspace: optional device scratch of at least qnn_gemm_workspace_bytes(M, K)
 *   bytes (16-byte aligned), owned by the caller and overwritten by the call;
 *   with it, A is re-encoded once by a pre-pass kernel on `stream` and the GEMM
 *   streams both operands (the faster path); NULL: the GEMM re-encodes A
 *   itself (no scratch).  Results are identical.  Two calls in flight at the
 *   same time must not share a workspace.
 * Fails with QNN_ERR_OVERFLOW_RISK when K * max|a| * 2^ptf_max_shift * 128 could
 * exceed the int32 range; QNN_ERR_INVALID_ARG when workspace_bytes is too small. */
qnn_status qgemm_s8(const void *A, qnn_dtype a_dt, const void *B_packed, int M, int N, int K,
                    const qnn_epilogue *epi, void *C, int32_t *C_s32, void *workspace,
                    size_t workspace_bytes, qnn_stream_t stream);

/* The two halves of qgemm_s8 with a workspace, for callers that time them
 * apart or reuse one re-encoded A for several GEMMs that share it:
 * qgemm_pack_a writes A (codes of a_dt, [M, K], K % 16 == 0; u8 read as
 * q - 128; times 2^ptf_shift[k] when ptf_shift is not NULL, S8 only) into
 * A_packed (qnn_gemm_workspace_bytes(M, K) bytes, 16-byte aligned) as the
 * fp16 operand image: [ceil(M/128)][ceil(K/64)][128 rows][64 fp16], each
 * 128-byte row's 16-byte chunk c stored at chunk c ^ (row % 8), zero beyond M
 * and K.  qgemm_s8_packed then takes that image in place of A; a_dt and epi
 * (including ptf_shift / ptf_max_shift) must be those used for the packing. */
qnn_status qgemm_pack_a(const void *A, qnn_dtype a_dt, int M, int K, const uint8_t *ptf_shift,
                        void *A_packed, size_t A_packed_bytes, qnn_stream_t stream);
qnn_status qgemm_s8_packed(const void *A_packed, qnn_dtype a_dt, const void *B_packed, int M, int N,
                           int K, const qnn_epilogue *epi, void *C, int32_t *C_s32,
                           qnn_stream_t stream);

/* Size of the library's fixed device scratch for qgemm_s8_static_scratch:
 * 32 MiB, enough for qnn_gemm_workspace_bytes(M, K) of any M x K activation
 * with ceil(M / 128) * ceil(K / 64) <= 2048 (e.g. 12608 x 1024). */
#define QNN_GEMM_STATIC_SCRATCH_BYTES (32u << 20)

/* qgemm_s8 with a workspace, for callers that cannot allocate device memory at
 * call time (allocation is not allowed in their execution context, or their
 * allocator is not reachable from it).  The workspace is a fixed array of
 * QNN_GEMM_STATIC_SCRATCH_BYTES that belongs to the library (allocated when
 * the library's device code is loaded); the call allocates and frees nothing.
 * The pages describe no such variant; it exists only for those callers.
 * - The array's address is looked up once per device on the first call; make
 *   that first call on each device before capturing a stream.  The looked-up
 *   address is kept for the life of the process: after cudaDeviceReset (or any
 *   reset of the device's primary context, which reloads the library's device
 *   code) it is stale, so do not call this entry point on a device again after
 *   resetting it.
 * - Returns QNN_ERR_UNSUPPORTED when qnn_gemm_workspace_bytes(M, K) exceeds
 *   QNN_GEMM_STATIC_SCRATCH_BYTES; other arguments as for qgemm_s8.
 * - Every call on a device uses the same array: calls whose executions
 *   overlap (different streams, or other host threads) race on it and give
 *   wrong results.  Order them on one stream or with events.
 * Results are identical to qgemm_s8's. */
qnn_status qgemm_s8_static_scratch(const void *A, qnn_dtype a_dt, const void *B_packed, int M, int N,
                                   int K, const qnn_epilogue *epi, void *C, int32_t *C_s32,
                                   qnn_stream_t stream);

/* ---- implicit-GEMM convolution -------------------------------------------- */

/* Layouts of a conv's input, output and residual [MG conv 算子優化: the conv
 * writes NCHW64, each 64 consecutive channels of a pixel contiguous].  Element
 * (n, c, y, x) of a tensor with C channels sits at
 *   QNN_LAYOUT_NHWC  : ((n * H + y) * W + x) * C + c
 *   QNN_LAYOUT_NCHW  : ((n * C + c) * H + y) * W + x
 *   QNN_LAYOUT_NCHW64: (((n * (C / 64) + c / 64) * H + y) * W + x) * 64 + c % 64
 * counted in codes (4-bit tensors: two per byte, element 2i in the low nibble,
 * so that NCHW packs neighbouring pixels of a row together). */
typedef enum { QNN_LAYOUT_NHWC = 0, QNN_LAYOUT_NCHW = 1, QNN_LAYOUT_NCHW64 = 2 } qnn_layout;

/* Input [N, H, W, C] and output [N, OH, OW, OC] in `layout` (the residual, when
 * there is one, in the output's), OHWI weights [OC, FH, FW, C], with OH = (H +
 * 2 pad_h - FH) / stride_h + 1 (same for W).
 * GEMM view [MG conv 算子優化, Fig. 5; output transposed so that output channels
 * are contiguous]: rows p = (n, oh, ow), columns oc, reduction k = (fh, fw, c).
 * Padded taps hold the real value 0, i.e. the code z_in.
 * NCHW64 needs C and OC multiples of 64; NCHW with 4-bit codes needs W and OW
 * even. */
typedef struct {
    int32_t N, H, W, C, OC, FH, FW, pad_h, pad_w, stride_h, stride_w;
    int32_t layout;          /* qnn_layout of input, output and residual (0: NHWC) */
} qnn_conv_geom;

/* Size in bytes of the prepacked conv weight operand for weights of w_dt
 * (S4 or S8; U4 and U8, the filters with zero points, take the same size as
 * S4 and S8); 0 for an invalid geometry or type. */
size_t qnn_conv_packed_w_bytes(const qnn_conv_geom *g, qnn_dtype w_dt);

/* Prepack conv weights of w_dt (S4: packed nibbles, OHWI; S8: bytes, OHWI) into
 * the conv kernels' operand images (`W_packed`, qnn_conv_packed_w_bytes bytes,
 * 1024-byte aligned; for S4 it holds the images of both qconv_u4s4 paths and
 * the column sums) and write colsum[oc] = sum over (fh, fw, c) of W (int32
 * [OC]) when colsum is not NULL. */
qnn_status qconv_prepack_w(const void *W, qnn_dtype w_dt, const qnn_conv_geom *g, void *W_packed,
                           int32_t *colsum, qnn_stream_t stream);

/* Prepack u4 filters (packed nibbles, OHWI) with per-filter zero points z_w
 * (device int32 [OC]) for qconv_u4s4 [MG 背景: UINT4 codes are asymmetric; 緩解
 * 精度下降: with Z_w != 0 every term of the product appears].  The filters are
 * constants, so the weight zero point is taken out here: the images hold
 * u - z_w[oc] in [-15, 15] (exact in e4m3, like the s4 values) and colsum[oc] =
 * sum (u - z_w[oc]); the conv then computes sum (q - z_in)(u - z_w) with no
 * run-time term.  Same buffer size as S4 (qnn_conv_packed_w_bytes(g, QNN_S4)).
 * QNN_ERR_OVERFLOW_RISK when FH FW C 225 >= 2^24 (the kernel's fp32 sums must
 * stay exact). */
qnn_status qconv_prepack_w_u4(const void *W, const int32_t *z_w, const qnn_conv_geom *g, void *W_packed,
                              int32_t *colsum, qnn_stream_t stream);

/* Size in bytes of the conv workspace for an input of in_dt (U4, for qconv_u4s4:
 * the input expanded to one byte per channel, N * H * W * C; U8, for qconv_u8s8
 * and qconv_u8u8: one fp16 value per channel, 2 * N * H * W * C); 0 for an
 * invalid geometry or another type. */
size_t qnn_conv_workspace_bytes(const qnn_conv_geom *g, qnn_dtype in_dt);

/* u4 activations x s4 weights [MG 緩解精度下降: UINT4 input/output, INT4
 * weights, FP32 bias], Conv_Relu / Conv_Add_Relu through `epi`
 * [MG 算子融合優化].  I: packed u4 codes in g->layout (NHWC, NCHW or NCHW64); O
 * (and the residual): the same layout, out_dt U4 (packed) or U8 codes, or fp32 /
 * int32 per epi->mode; O_s32: optional int32 acc_c.  C a multiple of 32, OC even.
 * workspace: optional device scratch of at least qnn_conv_workspace_bytes(g,
 *   QNN_U4) bytes (16-byte aligned), owned by the caller and overwritten: for
 *   filters with more than one tap, a pre-pass expands the input to one byte
 *   per channel and the convolution reads its taps with tensor-memory copies
 *   (the faster path there); 1x1 filters and NULL: the convolution re-encodes
 *   the packed input itself (NHWC 1x1 stride-1 unpadded convs copy the packed
 *   codes to shared memory and unpack them there).  Results are identical.  Calls in flight at the
 *   same time must not share a workspace.  An NCHW input needs the workspace
 *   (the pre-pass reads it and writes the expanded NHWC bytes the convolution
 *   reads, for every filter size): QNN_ERR_UNSUPPORTED without one. */
qnn_status qconv_u4s4(const void *I, int32_t z_in, const void *W_packed, const qnn_conv_geom *g,
                      const qnn_epilogue *epi, void *O, int32_t *O_s32, void *workspace,
                      size_t workspace_bytes, qnn_stream_t stream);

/* u8 activations x s8 weights, same contract (I: u8 codes in g->layout; C % 16 == 0).
 * workspace: optional device scratch of at least qnn_conv_workspace_bytes(g,
 *   QNN_U8) bytes (16-byte aligned), owned by the caller and overwritten: when C
 *   is a multiple of 64 and the filter has more than one tap, a pre-pass writes
 *   the input as fp16 values q - z_in (NHWC) and the convolution reads each tap
 *   with tensor-memory copies (the faster path); otherwise, and with NULL, the
 *   convolution re-encodes the codes itself.  Results are identical. */
qnn_status qconv_u8s8(const void *I, int32_t z_in, const void *W_packed, const qnn_conv_geom *g,
                      const qnn_epilogue *epi, void *O, int32_t *O_s32, void *workspace, size_t workspace_bytes,
                      qnn_stream_t stream);

/* Prepack u8 filters (bytes, OHWI) with per-filter zero points z_w (device int32
 * [OC], each in 0..255) for qconv_u8u8 [MG 背景: asymmetric codes carry a zero
 * point; 緩解精度下降: with Z_w != 0 every term of the product appears].  As for
 * u4 filters the weight zero point is taken out here, the filters being
 * constants: the image holds w - z_w[oc] in [-255, 255] (exact in fp16) and
 * colsum[oc] = sum (w - z_w[oc]), so the conv computes sum (q - z_in)(w - z_w)
 * with no run-time term.  W 16-byte aligned, C % 16 == 0 (QNN_ERR_UNSUPPORTED
 * otherwise); W_packed 1024-byte aligned, qnn_conv_packed_w_bytes(g, QNN_U8)
 * bytes. */
qnn_status qconv_prepack_w_u8(const void *W, const int32_t *z_w, const qnn_conv_geom *g, void *W_packed,
                              int32_t *colsum, qnn_stream_t stream);

/* u8 activations x u8 filters with zero points (prepacked by qconv_prepack_w_u8),
 * the contract of qconv_u8s8.  The centred filter values reach 255 in magnitude,
 * so the kernel's exact fp32 partial sums span 512 K values instead of 1024
 * (longer filters are summed in more chunks, exactly); QNN_ERR_OVERFLOW_RISK
 * when FH FW C 255^2 > 2^31 - 1. */
qnn_status qconv_u8u8(const void *I, int32_t z_in, const void *W_packed, const qnn_conv_geom *g,
                      const qnn_epilogue *epi, void *O, int32_t *O_s32, void *workspace, size_t workspace_bytes,
                      qnn_stream_t stream);

/* ---- weight zero points (Z_w != 0) --------------------------------------------- */

/* Prepack u8 weights B [N, K] with per-output-channel zero points z_w (device
 * int32 [N]) [MG 緩解精度下降: with Z_w != 0 the product has all four terms]:
 * the image holds the centred values w - 128 (exact in fp16, like the u8
 * activations), and colsum[n] = sum_k (B[n][k] - z_w[n]) -- pass it to
 * q_fold_epilogue, which then folds (z_a - c_a) * colsum into zp_term.
 * K % 16 == 0; B_packed 1024-byte aligned (qnn_gemm_packed_b_bytes). */
qnn_status qgemm_prepack_b_u8(const uint8_t *B, const int32_t *z_w, int N, int K, void *B_packed, int32_t *colsum,
                              qnn_stream_t stream);

/* Workspace of qgemm_zw: the A image of qnn_gemm_workspace_bytes(M, K) and the
 * per-row sums (int32 [M], 256-byte padded). */
size_t qnn_gemm_zw_workspace_bytes(int M, int K);

/* qgemm_s8 for weights with zero points (prepacked by qgemm_prepack_b_u8):
 *   acc_c[m][n] = sum_k (a_k - z_a)(w_k - z_w[n])
 * = acc - zp_term[n] + (128 - z_w[n]) * rowsum[m], where acc is the product of
 * the centred codes, zp_term[n] = (z_a - c_a) colsum[n] is folded ahead, and
 * rowsum[m] = sum_k (a_k - c_a) -- the term [MG 緩解精度下降] marks as costly
 * because it depends on the input -- is summed by the A pre-pass into the
 * workspace at run time.  Then the same epilogue as qgemm_s8.  a_dt S8 or U8; no
 * PTF; workspace required (qnn_gemm_zw_workspace_bytes).  QNN_ERR_OVERFLOW_RISK
 * when K * 255 * 255 > 2^31 - 1. */
qnn_status qgemm_zw(const void *A, qnn_dtype a_dt, const void *B_packed, const int32_t *z_w, int M, int N, int K,
                    const qnn_epilogue *epi, void *C, int32_t *C_s32, void *workspace, size_t workspace_bytes,
                    qnn_stream_t stream);

/* ---- Log-Int-Softmax attention [FQ 3.3] ------------------------------------ */

/* Log-Int-Softmax [FQ 3.3: Softmax 的量化推理, Integer-only 推理, Softmax 的量化的实现]
 * over `rows` rows of L int32 logit codes x (row-major [rows][L]; real value
 * x * S, e.g. the int32 accumulator of Q K^T with S = s_q s_k / sqrt(d)).
 * code (u8 [rows][L]) receives per element the log2 code k of its attention
 * probability 2^-k, or 2^bits where the probability is quantized to 0:
 *   x0 = floor(fp32(-0.6931) / S), b = floor(fp32(b'/a') / S),
 *   c = floor(fp32(c'/a') / (S*S))  with (a', b', c') = (0.35815147, 0.96963238, 1),
 *   the ratios in double, the divisions and S*S in fp32;
 *   d = max(x - max(row), 30 x0), q = floor(d / x0), r = d - x0 q,
 *   e = (r (r + b) + c) * 2^(30 - q)   (exact integers; 0 if negative);
 *   s = sum of e over the row; v = round(s / e) (exact, half to even);
 *   k = floor(log2 v), plus one when v - 2^k >= 2^(k-1); k >= 2^bits -> 2^bits.
 * bits in 1..5.  Fails with QNN_ERR_INVALID_ARG for S not finite and positive,
 * L <= 0, or S so coarse that x0 >= 0, b <= 0 or c <= 0; QNN_ERR_OVERFLOW_RISK
 * when c >= 2^31 (S finer than about 2^-15) or L c 2^30 >= 2^64 (the row sum
 * must fit 64 bits). */
qnn_status q_log_int_softmax(const int32_t *x, int64_t rows, int64_t L, float S, int bits,
                             uint8_t *code, qnn_stream_t stream);

/* The attention-times-value product with log2 codes as shifts [FQ 3.3,
 * Attention Map 的 Log2 量化: with probabilities 2^-k the MatMul of the attention
 * map and the value codes becomes a BitShift]:
 *   out[b][i][j] = sum_t 2^(N - code[b][i][t]) * v[b][t][j],  N = 2^bits - 1,
 * masked codes (>= 2^bits) contributing 0 -- 2^N times the product of the
 * dequantized map and v, exact in int32 (the real product is out * 2^-N * s_v).
 * code: u8 [batch][Lq][Lk] (q_log_int_softmax's output); v: s8 [batch][Lk][d];
 * out: int32 [batch][Lq][d].  bits in 1..4; d % 16 == 0; batch <= 65535.
 * QNN_ERR_OVERFLOW_RISK when Lk * 128 * 2^N > 2^31 (Lk <= 512 at 4 bits).
 * d <= 128 with Lk <= 512 runs on the tensor cores (the weight split into two
 * fp16 halves, exact fp32 sums), other shapes on the CUDA cores; both exact. */
qnn_status q_attn_shift_v(const uint8_t *code, const int8_t *v, int64_t batch, int Lq, int Lk, int d,
                          int bits, int32_t *out, qnn_stream_t stream);

/* The two calls above in one kernel [FQ 3.3, Integer-only 推理: the whole
 * attention after Q K^T stays integer]: for each head, q_log_int_softmax of the
 * logit rows x (int32 [batch][Lq][Lk], scale S) and q_attn_shift_v of the
 * resulting codes with v -- the same out, bit for bit, but the log2 codes live
 * only in shared memory and never reach global memory.  Lk <= 256, d <= 128,
 * bits 1..4; the other conditions of both calls apply. */
qnn_status q_lis_attn_v(const int32_t *x, float S, const int8_t *v, int64_t batch, int Lq, int Lk, int d, int bits,
                        int32_t *out, qnn_stream_t stream);

/* ---- integer LayerNorm [FQ 3.2] --------------------------------------------- */

/* LayerNorm of `rows` rows of C s8 codes x (row-major [rows][C]) quantized with
 * the Power-of-Two Factor [FQ 3.2: LayerNorm 的量化推理, LayerNorm 的量化实现]:
 * the real value of x[r][c] is x s 2^alpha[c] (alpha: u8 [C], NULL = all 0,
 * every value <= alpha_max <= 3).  With x' = x 2^alpha, per row
 *   mean = fp32(sum x' / C) * s,  std = (s / C) * sqrt(fp32(C sum x'^2 - (sum x')^2))
 * (exact integer sums) and per channel c, in fp32 operations in this order,
 *   A = ((s / std) * gamma[c]) / o[c],  N = clamp(7 - floor(log2 |A|), 0, 31)
 *   (N = 31 for A zero or subnormal, 0 for A infinite),  M = clamp(floor(|A| 2^N), 0, 255),
 *   B = round(((beta[c] - (mean / std) * gamma[c]) / o[c]) * 2^N)  (clamped to
 *   +-2^62 first),  y = round((sign(A) M x' + B) / 2^N)   (exact; half to even)
 * where o = out_scale [C].  A row whose variance numerator is 0 gives
 * y = round(beta[c] / o[c]).  y: QNN_S8 [rows][C] (clipped to -128..127, the
 * next layer's int8 input) or QNN_S32 (clipped to the int32 range).  gamma,
 * beta, out_scale: fp32 [C], gamma and beta finite, out_scale finite and > 0 (the
 * device values are not checked; others give unspecified codes).  C % 4 == 0 (QNN_ERR_ALIGNMENT);
 * QNN_ERR_OVERFLOW_RISK when C (128 2^alpha_max)^2 >= 2^32. */
qnn_status q_int_layernorm(const int8_t *x, int64_t rows, int C, const uint8_t *alpha, int alpha_max, float s,
                           const float *gamma, const float *beta, const float *out_scale, qnn_dtype y_dt,
                           void *y, qnn_stream_t stream);

/* ---- standalone elementwise ops and dynamic quantization [QI] ----------------- */

typedef enum { QNN_ADD = 0, QNN_MUL = 1, QNN_RELU = 2 } qnn_eltwise_op;

/* Elementwise ops on n symmetric s8 codes [QI 量化加法, 量化乘法, 量化激活函数]:
 *   QNN_ADD : out = clip(rint((float)(a + b) * M))  -- a and b share one scale
 *             (the page requires it), M = s_ab / s_out
 *   QNN_MUL : out = clip(rint((float)(a * b) * M))  -- M = s_a s_b / s_out, computed
 *             ahead; M = 2^-k is the page's shift variant
 *   QNN_RELU: out = max(a, 0)                        -- passive: b and M unused
 * clip to [-128, 127], rint half to even, one fp32 multiply; relu != 0 applies
 * max(., 0) after the rescale.  a, b, out: device s8 [n], 16-byte aligned. */
qnn_status q_eltwise_s8(qnn_eltwise_op op, const int8_t *a, const int8_t *b, int64_t n, float M, int relu,
                        int8_t *out, qnn_stream_t stream);

/* Dynamic per-row symmetric quantization [QI 量化参数选择: max truncation, the scale
 * the largest magnitude over 127; 量化算子]: for each of `rows` rows of `cols`
 * fp32 values, scale[r] = max|x[r]| / 127 (IEEE fp32 division) and
 * q[r][c] = clip(rint(x[r][c] / scale[r])) (one IEEE division each) to [-128, 127],
 * or [-127, 127] with narrow != 0.  A row of zeros gets scale 0 and codes 0.
 * x must be finite.  cols % 4 == 0.  q: s8 [rows][cols]; scale: fp32 [rows]. */
qnn_status q_quantize_rows_dynamic(const float *x, int64_t rows, int64_t cols, int narrow, int8_t *q,
                                   float *scale, qnn_stream_t stream);

/* ---- layouts ------------------------------------------------------------------ */

/* NHWC <-> NCHW64 for quantized codes [MG conv 算子優化: the conv output laid out
 * NCHW64, each 64 consecutive channels of a pixel contiguous].  The convolutions
 * of this library read and write NHWC; NCHW64 tensors go through this
 * memory-bound block permutation:
 *   nchw64[n][c / 64][h][w][c % 64] = nhwc[n][h][w][c]   (to_nchw64 != 0; else back)
 * dt: S4 / U4 (two codes per byte, element 2i in the low nibble: a block is 32
 * bytes) or S8 / U8 (64 bytes).  C % 64 == 0; 16-byte aligned pointers; src and
 * dst must not overlap. */
qnn_status q_layout_nchw64(const void *src, int to_nchw64, int N, int H, int W, int C, qnn_dtype dt, void *dst,
                           qnn_stream_t stream);

/* ---- status ----------------------------------------------------------------- */

const char *qnn_status_string(qnn_status s);

/* Synchronises `stream`, then reports and clears the device status word that
 * kernels set when a bounded wait gives up (QNN_ERR_TIMEOUT) or a device-side
 * argument check fails (QNN_ERR_INVALID_ARG: a Power-of-Two-Factor shift above
 * its stated bound; a GEMM weight image whose trailer does not match its K, or
 * whose values need more exact runs than the kernel was launched for), or
 * QNN_ERR_CUDA if the stream holds a CUDA error. */
qnn_status qnn_check_device_error(qnn_stream_t stream);

/* Launches one block that waits on a barrier nothing arrives at, giving up
 * after `limit_ns` nanoseconds (<= 1e9) the way every kernel wait gives up:
 * sets the device status word and returns.  For testing the timeout path. */
qnn_status qnn_selftest_wait_timeout(uint64_t limit_ns, qnn_stream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* QNN_H_ */
