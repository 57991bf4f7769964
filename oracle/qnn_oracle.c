/*
 * qnn_oracle.c -- plain, slow, obviously-correct CPU oracle for the linear
 * integer-quantized GEMM / implicit-GEMM convolution path.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product (the CUDA library and its
 * Python binding) may link, load or call this file; only the tests, the
 * package's smoke check and the benchmark's CPU-baseline leg use it.  It
 * shares no code, header, table or constant generator with the CUDA path.
 *
 * Build: gcc -O2 -std=c11 -ffp-contract=off -fno-fast-math -fopenmp -shared -fPIC
 * (fp contraction must stay off: every fp32 operation below is one IEEE
 * round-to-nearest-even operation, in the order written).
 *
 * Sources (page title, section):
 *   [QI]  "【量化】神经网络量化介绍" (loveleaves.github.io/p/quantization):
 *         量化算子, 反量化算子, 量化模式, tensor量化与通道量化, 量化乘法,
 *         量化加法, 量化激活函数, 量化矩阵乘, 常见计算图优化 (conv-add).
 *   [MG]  MegEngine 4-bit quantization article (m.xsypw.cn/d/1897816):
 *         背景 (linear quantization, UINT4/INT4 ranges), 緩解精度下降
 *         (zero-point formula split), conv 算子優化 (img2col / implicit GEMM,
 *         Fig. 5; column permutation, Fig. 8).
 *   [FQ]  "首个完全量化Vision Transformer的方法FQ-ViT" (aijishu.com):
 *         3.2 Power-of-Two Factor (LayerNorm 的量化推理, LayerNorm 的量化实现);
 *         3.3 Log Int Softmax (Attention Map 的 Log2
 *         量化, Softmax 的量化推理, Integer-only 推理, Softmax 的量化的实现).
 *
 * Readings of points the pages leave open are stated next to the code that
 * takes them.  Parity status: every function here is pinned by tests that do
 * not re-type its formula (worked examples, closed forms, brute force in
 * exact rational arithmetic, invariants, numpy library routines).
 */
#include <math.h>
#include <stdlib.h>
#include <stdint.h>
#include <stddef.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { OR_SYM = 0, OR_ASYM = 1, OR_POW2 = 2 };
enum { OR_OK = 0, OR_ERR_RANGE = 1, OR_ERR_ARG = 2 };

void oracle_set_threads(int n)
{
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

int oracle_get_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* ---------------------------------------------------------------------------
 * Rounding modes [QI 量化算子]: the page lists five ways to round a value that
 * lies exactly half-way between two integers.  mode: 0 half to even, 1 half
 * away from zero, 2 half toward zero, 3 half down, 4 half up.  Values that are
 * not ties go to the nearest integer in every mode.  Computed in double.
 * ------------------------------------------------------------------------- */
double oracle_round_mode(double v, int mode)
{
    double f = floor(v);
    double d = v - f;
    if (d < 0.5) return f;
    if (d > 0.5) return f + 1.0;
    switch (mode) {
    case 0: return (fmod(f, 2.0) == 0.0) ? f : f + 1.0;
    case 1: return (v > 0.0) ? f + 1.0 : f;
    case 2: return (v > 0.0) ? f : f + 1.0;
    case 3: return f;
    case 4: return f + 1.0;
    default: return NAN;
    }
}

static float clamp_f(float r, float lo, float hi)
{
    return fminf(fmaxf(r, lo), hi);
}

/* ---------------------------------------------------------------------------
 * Quantize [QI 量化算子, 量化模式, tensor量化与通道量化; MG 背景].
 * x is viewed as [outer, C, inner]; with per_channel the parameters are
 * indexed by the C coordinate, otherwise element 0 is used.
 *   symmetric : q = clip(rint(x / s))
 *   asymmetric: q = clip(rint(x / s) + z)       (offset added after rounding,
 *                                                as the page writes it)
 *   power of 2: q = clip(rint(x * 2^shift))     (reading: 2^shift; the page's
 *                                                text has "2 << shift")
 * rint is round-half-to-even (default FP environment).  x / s is one IEEE
 * fp32 division.  Clipping is done in float, then converted.
 * Reading for NaN inputs (pages silent): the code of real zero (z, else 0).
 * ------------------------------------------------------------------------- */
int oracle_quantize(const float *x, int64_t outer, int64_t C, int64_t inner,
                    int scheme, int per_channel, const float *scale,
                    const int32_t *zp, const int32_t *shift, int32_t qmin,
                    int32_t qmax, int32_t *q)
{
    if (scheme < OR_SYM || scheme > OR_POW2) return OR_ERR_ARG;
#pragma omp parallel for collapse(2) schedule(static)
    for (int64_t o = 0; o < outer; ++o) {
        for (int64_t c = 0; c < C; ++c) {
            int64_t ch = per_channel ? c : 0;
            for (int64_t i = 0; i < inner; ++i) {
                int64_t idx = (o * C + c) * inner + i;
                float v = x[idx];
                int32_t z = (scheme == OR_ASYM) ? zp[ch] : 0;
                if (v != v) { q[idx] = z; continue; }
                float r;
                if (scheme == OR_POW2) {
                    float t = ldexpf(v, shift[ch]);
                    r = rintf(t);
                } else {
                    float t = v / scale[ch];
                    r = rintf(t);
                }
                if (scheme == OR_ASYM) r = r + (float)z;
                float cl = clamp_f(r, (float)qmin, (float)qmax);
                q[idx] = (int32_t)cl;
            }
        }
    }
    return OR_OK;
}

/* ---------------------------------------------------------------------------
 * Dequantize [QI 反量化算子; MG 背景: r = S (q - Z)].
 *   symmetric / asymmetric: x = (float)(q - z) * s   (integer subtract, one
 *                                                     fp32 multiply)
 *   power of 2            : x = q * 2^-shift          (exact)
 * ------------------------------------------------------------------------- */
int oracle_dequantize(const int32_t *q, int64_t outer, int64_t C, int64_t inner,
                      int scheme, int per_channel, const float *scale,
                      const int32_t *zp, const int32_t *shift, float *x)
{
    if (scheme < OR_SYM || scheme > OR_POW2) return OR_ERR_ARG;
    for (int64_t o = 0; o < outer; ++o) {
        for (int64_t c = 0; c < C; ++c) {
            int64_t ch = per_channel ? c : 0;
            for (int64_t i = 0; i < inner; ++i) {
                int64_t idx = (o * C + c) * inner + i;
                if (scheme == OR_POW2) {
                    x[idx] = ldexpf((float)q[idx], -shift[ch]);
                } else {
                    int32_t z = (scheme == OR_ASYM) ? zp[ch] : 0;
                    float d = (float)(q[idx] - z);
                    x[idx] = d * scale[ch];
                }
            }
        }
    }
    return OR_OK;
}

/* ---------------------------------------------------------------------------
 * Storage of codes.  Reading for nibble order (pages silent beyond "8 x 4-bit
 * values in one 32-bit word", MG conv 算子優化): element 2i is the low nibble
 * of byte i, element 2i+1 the high nibble; n must be even.
 * ------------------------------------------------------------------------- */
void oracle_pack_nibbles(const int32_t *q, int64_t n, uint8_t *out)
{
    for (int64_t i = 0; i < n / 2; ++i) {
        uint32_t lo = (uint32_t)q[2 * i] & 15u;
        uint32_t hi = (uint32_t)q[2 * i + 1] & 15u;
        out[i] = (uint8_t)(lo | (hi << 4));
    }
}

void oracle_unpack_nibbles(const uint8_t *p, int64_t n, int is_signed, int32_t *q)
{
    for (int64_t i = 0; i < n; ++i) {
        uint32_t b = p[i / 2];
        int32_t v = (int32_t)((i % 2 == 0) ? (b & 15u) : (b >> 4));
        if (is_signed && v >= 8) v -= 16;
        q[i] = v;
    }
}

void oracle_pack_bytes(const int32_t *q, int64_t n, uint8_t *out)
{
    for (int64_t i = 0; i < n; ++i) out[i] = (uint8_t)((uint32_t)q[i] & 255u);
}

/* ---------------------------------------------------------------------------
 * Integer GEMM accumulator [QI 量化矩阵乘: int8 in, wide multiply, wide
 * accumulate; MG 緩解精度下降: the unexpanded sum of (q_I - Z_I) q_W].
 *   acc[m][n] = sum_k (A[m][k] - z_a) * 2^alpha_k * B[n][k]
 * A is [M,K] and B is [N,K] (both row-major, codes as int32).  alpha is the
 * per-input-channel Power-of-Two Factor of [FQ 3.2] (NULL: all zero).
 * Sums are formed in int64; the result must fit int32 (else OR_ERR_RANGE).
 * ------------------------------------------------------------------------- */
int oracle_gemm_acc(const int32_t *A, const int32_t *B, int64_t M, int64_t N,
                    int64_t K, int32_t z_a, const int32_t *alpha, int32_t *acc)
{
    int bad = 0;
#pragma omp parallel for schedule(static) reduction(|:bad)
    for (int64_t m = 0; m < M; ++m) {
        for (int64_t n = 0; n < N; ++n) {
            int64_t s = 0;
            for (int64_t k = 0; k < K; ++k) {
                int64_t a = (int64_t)A[m * K + k] - z_a;
                if (alpha) a = a * ((int64_t)1 << alpha[k]);
                s += a * (int64_t)B[n * K + k];
            }
            if (s > INT32_MAX || s < INT32_MIN) bad = 1;
            acc[m * N + n] = (int32_t)s;
        }
    }
    return bad ? OR_ERR_RANGE : OR_OK;
}

/* colsum[n] = sum_k B[n][k]: the weight sums that the zero-point cross term
 * needs [MG 緩解精度下降, the part computable before inference]. */
void oracle_colsum(const int32_t *B, int64_t N, int64_t K, int32_t *colsum)
{
    for (int64_t n = 0; n < N; ++n) {
        int64_t s = 0;
        for (int64_t k = 0; k < K; ++k) s += B[n * K + k];
        colsum[n] = (int32_t)s;
    }
}

/* ---------------------------------------------------------------------------
 * Constants folded ahead of inference [MG 緩解精度下降; QI 量化乘法:
 * "scale_abc can be computed ahead"].
 *   zp_term[n] = Z_a * colsum[n]         (int32: the input-independent term
 *                                        of sum (q_a - Z_a) q_w, subtracted from
 *                                        sum q_a q_w)
 *   M[n]  = (s_a * s_w[n]) / s_o          fmul, then fdiv
 *   Bq[n] = bias[n] / s_o
 *   D[n]  = s_a * s_w[n]                  (dequantizing epilogue)
 * s_w is per output channel when w_per_channel, else s_w[0]; bias may be NULL
 * (zero).
 * ------------------------------------------------------------------------- */
int oracle_fold(int64_t N, int32_t z_a, const int32_t *colsum, float s_a,
                const float *s_w, int w_per_channel, const float *bias, float s_o,
                int32_t *zp_term, float *Mv, float *Bq, float *D)
{
    int bad = 0;
    for (int64_t n = 0; n < N; ++n) {
        int64_t z = (int64_t)z_a * (int64_t)colsum[n];
        if (z > INT32_MAX || z < INT32_MIN) bad = 1;
        zp_term[n] = (int32_t)z;
        float sw = s_w[w_per_channel ? n : 0];
        float p = s_a * sw;
        Mv[n] = p / s_o;
        float b = bias ? bias[n] : 0.0f;
        Bq[n] = b / s_o;
        D[n] = p;
    }
    return bad ? OR_ERR_RANGE : OR_OK;
}

/* ---------------------------------------------------------------------------
 * Requantizing epilogue [QI 量化乘法 (rescale by the folded scale), 量化加法
 * (residual add with a common scale), 量化激活函数 (relu is passive: a max with
 * the quantized zero), 常见计算图优化 (conv-add: Y = Wx + (Y2 + B))].
 * Per element, fp32 ops in this order, no contraction:
 *   t = Bq[n];  with residual: t = (float)(res - z_res) * R + t   (fmul, fadd)
 *   v = (float)acc_c * M[n];  v = v + t
 *   r = rint(v);  relu: r = max(r, 0)
 *   q = clip(r + (float)z_out)
 * acc_c, res and q are [rows, N] row-major; res may be NULL.
 * ------------------------------------------------------------------------- */
int oracle_requant(const int32_t *acc_c, int64_t rows, int64_t N, const float *Mv,
                   const float *Bq, int relu, const int32_t *res, int32_t z_res,
                   float R, int32_t z_out, int32_t qmin, int32_t qmax, int32_t *q)
{
    for (int64_t m = 0; m < rows; ++m) {
        for (int64_t n = 0; n < N; ++n) {
            int64_t i = m * N + n;
            float t = Bq[n];
            if (res) {
                float d = (float)(res[i] - z_res);
                float rr = d * R;
                t = rr + t;
            }
            float a = (float)acc_c[i];
            float v = a * Mv[n];
            v = v + t;
            float r = rintf(v);
            if (relu) r = fmaxf(r, 0.0f);
            float s = r + (float)z_out;
            q[i] = (int32_t)clamp_f(s, (float)qmin, (float)qmax);
        }
    }
    return OR_OK;
}

/* Per-row activation scales r[m] (a dynamically quantized input, one scale per
 * row: QI 量化参数选择's max truncation per token) feeding the requant: the
 * folded per-channel factor is multiplied by the row's scale first, in fp32,
 * M[m][n] = r[m] * Mv[n], then the requant above.  Reading: the per-row and
 * per-channel factors are combined before they meet the accumulator (the pages
 * fold one scalar s_a; with per-row scales the fold uses s_a = 1). */
int oracle_requant_rowscale(const int32_t *acc_c, int64_t rows, int64_t N, const float *r, const float *Mv,
                            const float *Bq, int relu, const int32_t *res, int32_t z_res, float R,
                            int32_t z_out, int32_t qmin, int32_t qmax, int32_t *q)
{
    float *Mrow = (float *)malloc((size_t)(N > 0 ? N : 1) * sizeof(float));
    if (!Mrow) return OR_ERR_ARG;
    for (int64_t m = 0; m < rows; ++m) {
        for (int64_t n = 0; n < N; ++n) Mrow[n] = r[m] * Mv[n];
        oracle_requant(acc_c + m * N, 1, N, Mrow, Bq, relu, res ? res + m * N : NULL, z_res, R, z_out, qmin,
                       qmax, q + m * N);
    }
    free(Mrow);
    return OR_OK;
}

/* Dequantizing epilogue [QI 反量化算子; MG 背景]: y = (float)acc_c * D[n] + bias[n]
 * as one fmul and one fadd.  bias may be NULL (zero). */
void oracle_dequant_epilogue(const int32_t *acc_c, int64_t rows, int64_t N,
                             const float *D, const float *bias, float *y)
{
    for (int64_t m = 0; m < rows; ++m) {
        for (int64_t n = 0; n < N; ++n) {
            int64_t i = m * N + n;
            float v = (float)acc_c[i] * D[n];
            float b = bias ? bias[n] : 0.0f;
            y[i] = v + b;
        }
    }
}

/* The dequantizing epilogue with per-row activation scales: y = (float)acc_c *
 * (r[m] * D[n]) + bias[n], the product r[m] * D[n] formed first in fp32. */
void oracle_dequant_rowscale(const int32_t *acc_c, int64_t rows, int64_t N, const float *r, const float *D,
                             const float *bias, float *y)
{
    for (int64_t m = 0; m < rows; ++m) {
        for (int64_t n = 0; n < N; ++n) {
            const float d = r[m] * D[n];
            const float v = (float)acc_c[m * N + n] * d;
            y[m * N + n] = v + (bias ? bias[n] : 0.0f);
        }
    }
}

/* ---------------------------------------------------------------------------
 * Convolution accumulator, direct definition [MG 緩解精度下降 (the unexpanded
 * sum of (q_I - Z_I) q_W), conv 算子優化].
 * Input I is NHWC [n][h][w][c], weights OHWI [oc][fh][fw][c], output acc is
 * [n][oh][ow][oc] (row p = (n, oh, ow), column oc).
 * Reading for padding (pages silent): a padded tap holds the real value 0,
 * whose code is z_in, so it contributes (z_in - z_in) * w = 0.
 * ------------------------------------------------------------------------- */
static int conv_out_dim(int in, int f, int pad, int stride)
{
    return (in + 2 * pad - f) / stride + 1;
}

int oracle_conv_acc_direct(const int32_t *I, const int32_t *W, int n_, int h, int w,
                           int c, int oc, int fh, int fw, int ph, int pw, int sh,
                           int sw, int32_t z_in, int32_t *acc)
{
    int oh_ = conv_out_dim(h, fh, ph, sh), ow_ = conv_out_dim(w, fw, pw, sw);
    if (oh_ <= 0 || ow_ <= 0) return OR_ERR_ARG;
    int bad = 0;
#pragma omp parallel for schedule(static) reduction(|:bad)
    for (int64_t p = 0; p < (int64_t)n_ * oh_ * ow_; ++p) {
        int b = (int)(p / ((int64_t)oh_ * ow_));
        int oy = (int)((p / ow_) % oh_);
        int ox = (int)(p % ow_);
        for (int o = 0; o < oc; ++o) {
            int64_t s = 0;
            for (int r = 0; r < fh; ++r) {
                int iy = oy * sh - ph + r;
                if (iy < 0 || iy >= h) continue;
                for (int t = 0; t < fw; ++t) {
                    int ix = ox * sw - pw + t;
                    if (ix < 0 || ix >= w) continue;
                    const int32_t *ip = I + (((int64_t)b * h + iy) * w + ix) * c;
                    const int32_t *wp = W + (((int64_t)o * fh + r) * fw + t) * c;
                    for (int ic = 0; ic < c; ++ic)
                        s += (int64_t)(ip[ic] - z_in) * (int64_t)wp[ic];
                }
            }
            if (s > INT32_MAX || s < INT32_MIN) bad = 1;
            acc[p * oc + o] = (int32_t)s;
        }
    }
    return bad ? OR_ERR_RANGE : OR_OK;
}

/* The same convolution accumulator with the input and the output in one of
 * three layouts [MG conv 算子優化: the library's conv writes NCHW64, each 64
 * consecutive channels of a pixel contiguous]; weights stay OHWI.  Element
 * (b, ch, y, x) of a tensor with C channels sits at
 *   layout 0 (NHWC)  : ((b * H + y) * W + x) * C + ch
 *   layout 1 (NCHW)  : ((b * C + ch) * H + y) * W + x
 *   layout 2 (NCHW64): (((b * (C / 64) + ch / 64) * H + y) * W + x) * 64 + ch % 64
 * (C % 64 == 0 for NCHW64).  The sum is the direct one above, with the same
 * padding reading, written out with explicit indices for each layout. */
static int64_t layout_index(int layout, int b, int ch, int y, int x, int C, int H, int W)
{
    switch (layout) {
    case 1: return (((int64_t)b * C + ch) * H + y) * W + x;
    case 2: return ((((int64_t)b * (C / 64) + ch / 64) * H + y) * W + x) * 64 + ch % 64;
    default: return (((int64_t)b * H + y) * W + x) * C + ch;
    }
}

int oracle_conv_acc_layout(const int32_t *I, const int32_t *W, int n_, int h, int w, int c, int oc, int fh, int fw,
                           int ph, int pw, int sh, int sw, int32_t z_in, int layout, int32_t *acc)
{
    int oh_ = conv_out_dim(h, fh, ph, sh), ow_ = conv_out_dim(w, fw, pw, sw);
    if (oh_ <= 0 || ow_ <= 0 || layout < 0 || layout > 2) return OR_ERR_ARG;
    if (layout == 2 && (c % 64 != 0 || oc % 64 != 0)) return OR_ERR_ARG;
    int bad = 0;
#pragma omp parallel for schedule(static) reduction(|:bad)
    for (int64_t p = 0; p < (int64_t)n_ * oh_ * ow_; ++p) {
        int b = (int)(p / ((int64_t)oh_ * ow_));
        int oy = (int)((p / ow_) % oh_);
        int ox = (int)(p % ow_);
        for (int o = 0; o < oc; ++o) {
            int64_t s = 0;
            for (int r = 0; r < fh; ++r) {
                int iy = oy * sh - ph + r;
                if (iy < 0 || iy >= h) continue;
                for (int t = 0; t < fw; ++t) {
                    int ix = ox * sw - pw + t;
                    if (ix < 0 || ix >= w) continue;
                    for (int ic = 0; ic < c; ++ic) {
                        int32_t q = I[layout_index(layout, b, ic, iy, ix, c, h, w)];
                        int32_t wt = W[(((int64_t)o * fh + r) * fw + t) * c + ic];
                        s += (int64_t)(q - z_in) * (int64_t)wt;
                    }
                }
            }
            if (s > INT32_MAX || s < INT32_MIN) bad = 1;
            acc[layout_index(layout, b, o, oy, ox, oc, oh_, ow_)] = (int32_t)s;
        }
    }
    return bad ? OR_ERR_RANGE : OR_OK;
}

/* Explicit img2col [MG conv 算子優化, Fig. 5]: cols[p][(r, t, ic)] holds the
 * input code under tap (r, t) of output pixel p, or z_in where the tap falls in
 * the padding.  K order is (fh, fw, ic), matching OHWI weights read as [OC, K]. */
int oracle_im2col(const int32_t *I, int n_, int h, int w, int c, int fh, int fw,
                  int ph, int pw, int sh, int sw, int32_t z_in, int32_t *cols)
{
    int oh_ = conv_out_dim(h, fh, ph, sh), ow_ = conv_out_dim(w, fw, pw, sw);
    if (oh_ <= 0 || ow_ <= 0) return OR_ERR_ARG;
    int64_t K = (int64_t)fh * fw * c;
    for (int64_t p = 0; p < (int64_t)n_ * oh_ * ow_; ++p) {
        int b = (int)(p / ((int64_t)oh_ * ow_));
        int oy = (int)((p / ow_) % oh_);
        int ox = (int)(p % ow_);
        for (int r = 0; r < fh; ++r)
            for (int t = 0; t < fw; ++t)
                for (int ic = 0; ic < c; ++ic) {
                    int iy = oy * sh - ph + r, ix = ox * sw - pw + t;
                    int32_t v = z_in;
                    if (iy >= 0 && iy < h && ix >= 0 && ix < w)
                        v = I[(((int64_t)b * h + iy) * w + ix) * c + ic];
                    cols[p * K + ((int64_t)r * fw + t) * c + ic] = v;
                }
    }
    return OR_OK;
}

/* ---------------------------------------------------------------------------
 * Log-Int-Softmax [FQ 3.3].  Each row of integer logit codes x (real values
 * x * S) becomes a row of log2 codes k: the attention probability is 2^-k, or 0
 * where k = 2^bits (the mask).  Steps, in the page's order:
 *   1. x <- x - max(x) over the row (Softmax 的量化推理: subtract the maximum);
 *   2. an integer exponential of every x (int_exp below) and their sum s;
 *   3. v = round(s / e) for every element's exponential e (1 / probability);
 *   4. k = log_round(v); k >= 2^bits is masked (probability 0).
 * Readings (the page prints the algorithm as floating-point tensor code of an
 * integer-only method):
 *   - integer steps are exact integer arithmetic;
 *   - the constants derived from S -- floor(-0.6931 / S), floor((b/a) / S),
 *     floor((c/a) / S^2) -- are fp32 operations, as in the printed code (an fp32
 *     scale; the coefficient ratios b/a and c/a computed in double, then rounded
 *     to fp32 when combined with the scale);
 *   - round(s / e) rounds the exact rational half to even;
 *   - an element whose exponential is 0 has v = infinity: masked. */
typedef struct {
    int64_t x0_int, b_int, c_int;
} lis_consts;

static lis_consts lis_constants(float S)
{
    /* second-order approximation a r^2 + b r + c of exp on [-ln 2, 0] */
    const double a = 0.35815147, b = 0.96963238, c = 1.0;
    lis_consts k;
    const float s2 = S * S;
    k.x0_int = (int64_t)floorf((float)-0.6931 / S);
    k.b_int = (int64_t)floorf((float)(b / a) / S);
    k.c_int = (int64_t)floorf((float)(c / a) / s2);
    return k;
}

/* Integer exponential of x <= 0 (Integer-only 推理): x is clamped to 30 * x0_int,
 * split as x = q * x0_int + r with q = floor(x / x0_int) and r in (x0_int, 0], the
 * polynomial z = r (r + b_int) + c_int evaluated on r, and z scaled by 2^(30 - q).
 * The result times a S^2 / 2^30 approximates exp(x S). */
int64_t oracle_lis_int_exp(int64_t x, float S)
{
    const lis_consts k = lis_constants(S);
    const int64_t n = 30;
    if (x < n * k.x0_int) x = n * k.x0_int;
    /* floor(x / x0_int) for x <= 0 < -x0_int: the exact quotient is >= 0 */
    const int64_t q = x / k.x0_int;  /* both non-positive: C truncation is the floor */
    const int64_t r = x - k.x0_int * q;
    const int64_t z = r * (r + k.b_int) + k.c_int;
    const int64_t e = z * ((int64_t)1 << (n - q));
    return e > 0 ? e : 0;
}

/* round(v) for v = num / den > 0, half to even, exact. */
static uint64_t round_ratio_half_even(uint64_t num, uint64_t den)
{
    uint64_t q = num / den, rem = num % den;
    if (2 * rem > den || (2 * rem == den && (q & 1))) ++q;
    return q;
}

/* log_round [FQ 3.3, Softmax 的量化的实现]: big = floor(log2 v), plus one when
 * v - 2^big >= 2^(big - 1); v >= 1.  Reading: evaluated exactly on the integer v
 * (the printed code takes log2 in floating point). */
int oracle_log_round(uint64_t v)
{
    int big = 0;
    while (big < 63 && (v >> (big + 1)) != 0) ++big;
    if (big >= 1 && v - ((uint64_t)1 << big) >= ((uint64_t)1 << (big - 1))) ++big;
    return big;
}

/* The whole row operation; code[i] = k for k < 2^bits, else 2^bits (masked:
 * probability 0).  Returns OR_ERR_ARG for a non-positive or non-finite S, bits
 * outside 1..5, L <= 0 or constants with x0_int >= 0, b_int <= 0 or c_int <= 0
 * (S too coarse), and OR_ERR_RANGE for c_int >= 2^31 (S finer than about 2^-15)
 * or when L exponentials of the largest value, c_int * 2^30 each (the
 * exponential of 0), could reach 2^64. */
int oracle_log_int_softmax(const int32_t *x, int64_t rows, int64_t L, float S, int bits,
                           uint8_t *code)
{
    if (!(S > 0.0f) || !isfinite(S) || bits < 1 || bits > 5 || L <= 0 || rows < 0)
        return OR_ERR_ARG;
    const lis_consts k = lis_constants(S);
    if (k.x0_int >= 0 || k.c_int <= 0 || k.b_int <= 0) return OR_ERR_ARG;
    if (k.c_int >= ((int64_t)1 << 31)) return OR_ERR_RANGE;
    if ((unsigned __int128)k.c_int * ((uint64_t)1 << 30) * (uint64_t)L >> 64) return OR_ERR_RANGE;
    const int kmax = 1 << bits;
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r) {
        const int32_t *xr = x + r * L;
        int32_t mx = xr[0];
        for (int64_t i = 1; i < L; ++i)
            if (xr[i] > mx) mx = xr[i];
        uint64_t s = 0;
        for (int64_t i = 0; i < L; ++i) s += (uint64_t)oracle_lis_int_exp((int64_t)xr[i] - mx, S);
        for (int64_t i = 0; i < L; ++i) {
            const uint64_t e = (uint64_t)oracle_lis_int_exp((int64_t)xr[i] - mx, S);
            int kk = kmax;
            if (e != 0) {
                kk = oracle_log_round(round_ratio_half_even(s, e));
                if (kk > kmax) kk = kmax;
            }
            code[r * L + i] = (uint8_t)kk;
        }
    }
    return OR_OK;
}

/* AttnQ x V as bit shifts [FQ 3.3, Attention Map 的 Log2 量化: the MatMul between
 * the log2-quantized attention map and the value codes becomes shifts].  With
 * attention probabilities 2^-k (k < 2^bits; k = 2^bits is zero):
 *   out[i][j] = sum_t 2^(2^bits - 1 - k[i][t]) * v[t][j]     (int64, exact)
 * i.e. 2^(2^bits - 1) times the product of the dequantized map and the value
 * codes.  Reading (the page's equation is missing from the text): the product
 * is kept exact, a left shift of v into the wider sum, rather than shifting v
 * right and truncating. */
int oracle_attn_shift_v(const uint8_t *code, const int32_t *v, int64_t heads, int64_t Lq, int64_t Lk,
                        int64_t d, int bits, int64_t *out)
{
    if (bits < 1 || bits > 5) return OR_ERR_ARG;
    const int64_t kmax = (int64_t)1 << bits;
#pragma omp parallel for collapse(2) schedule(static)
    for (int64_t h = 0; h < heads; ++h)
        for (int64_t i = 0; i < Lq; ++i) {
            const uint8_t *cr = code + (h * Lq + i) * Lk;
            for (int64_t j = 0; j < d; ++j) {
                int64_t acc = 0;
                for (int64_t t = 0; t < Lk; ++t) {
                    if (cr[t] >= kmax) continue;
                    acc += v[(h * Lk + t) * d + j] * ((int64_t)1 << (kmax - 1 - cr[t]));
                }
                out[(h * Lq + i) * d + j] = acc;
            }
        }
    return OR_OK;
}

/* ---------------------------------------------------------------------------
 * Integer LayerNorm over PTF-quantized rows [FQ 3.2, LayerNorm 的量化推理 and
 * LayerNorm 的量化实现, the integer mode of the printed module].  Row r of C codes
 * x (real value x * s * 2^alpha[c]; alpha NULL = all 0):
 *   1. x' = x * 2^alpha[c]                    (the PTF shift; exact integers)
 *   2. mean = fp32(sum x' / C) * s;  std = (s / C) * sqrt(fp32(C sum x'^2 - (sum x')^2))
 *   3. per channel c: A = ((s / std) * gamma[c]) / o[c]; sign, a = |A|;
 *      N = clamp(7 - floor(log2 a), 0, 31); M = clamp(floor(a * 2^N), 0, 255);
 *      B = round(((beta[c] - (mean / std) * gamma[c]) / o[c]) * 2^N)
 *   4. y = round((sign * M * x' + B) / 2^N)
 * (o = the output scale).  Readings: the integer sums and C sum x'^2 - (sum x')^2
 * are exact (int64) -- the page computes them as float tensors; the float steps
 * are single fp32 operations in the printed order (division, multiplication,
 * IEEE sqrt); floor(log2 a) is the exact binary exponent of a (N = 31 for
 * a == 0 or subnormal a; N = 0 for a = +inf, whose log2 is infinite, which
 * finite gamma reaches when (s / std) gamma overflows); both round() are half
 * to even, on the exact value; a
 * row whose variance numerator is 0 (all x' equal; the page divides by zero)
 * gives M = N = 0 and B = round(beta[c] / o[c]).  y is not clipped here: the
 * consumer's quantizer clips it.  B is rounded after clamping to +-2^62.
 * Returns OR_ERR_ARG for C <= 0, s or an o[c] not finite and positive, a
 * gamma[c] or beta[c] not finite, or alpha > 30. */
static int64_t round_shift_half_even(int64_t num, int N)
{
    if (N == 0) return num;
    const int64_t q = num >> N;  /* floor: arithmetic shift (gcc) */
    const int64_t rem = num - q * ((int64_t)1 << N);
    const int64_t half = (int64_t)1 << (N - 1);
    return (rem > half || (rem == half && (q & 1))) ? q + 1 : q;
}

/* round half to even of an fp32 value, clamped to +-2^62 first (a bound no
 * real LayerNorm constant reaches; it keeps sign * M * x' + B inside int64). */
static int64_t rint_to_i64(float v)
{
    const float lim = 4611686018427387904.0f; /* 2^62 */
    if (v > lim) v = lim;
    if (v < -lim) v = -lim;
    return (int64_t)nearbyintf(v); /* default mode: half to even */
}

int oracle_int_layernorm(const int32_t *x, int64_t rows, int64_t C, const uint8_t *alpha, float s,
                         const float *gamma, const float *beta, const float *o, int64_t *y)
{
    if (C <= 0 || rows < 0 || !(s > 0.0f) || !isfinite(s)) return OR_ERR_ARG;
    for (int64_t c = 0; c < C; ++c) {
        if (!(o[c] > 0.0f) || !isfinite(o[c])) return OR_ERR_ARG;
        if (!isfinite(gamma[c]) || !isfinite(beta[c])) return OR_ERR_ARG;
        if (alpha && alpha[c] > 30) return OR_ERR_ARG;
    }
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r) {
        const int32_t *xr = x + r * C;
        int64_t sum = 0, sum2 = 0;
        for (int64_t c = 0; c < C; ++c) {
            const int64_t v = (int64_t)xr[c] * ((int64_t)1 << (alpha ? alpha[c] : 0));
            sum += v;
            sum2 += v * v;
        }
        const int64_t var_num = C * sum2 - sum * sum;
        const float Cf = (float)C;
        const float mean = ((float)sum / Cf) * s;
        const float stdv = (s / Cf) * sqrtf((float)var_num);
        const float s_over_std = s / stdv;
        const float mean_over_std = mean / stdv;
        for (int64_t c = 0; c < C; ++c) {
            const int64_t v = (int64_t)xr[c] * ((int64_t)1 << (alpha ? alpha[c] : 0));
            int64_t M = 0, B;
            int N = 0, sign = 0;
            if (var_num == 0) {
                B = rint_to_i64(beta[c] / o[c]);
            } else {
                const float A = (s_over_std * gamma[c]) / o[c];
                sign = (A > 0.0f) - (A < 0.0f);
                const float a = fabsf(A);
                if (isinf(a)) {
                    N = 0;
                } else if (a == 0.0f || !isnormal(a)) {
                    N = 31;
                } else {
                    const int e = ilogbf(a);
                    N = 7 - e < 0 ? 0 : (7 - e > 31 ? 31 : 7 - e);
                }
                const float m = floorf(ldexpf(a, N));
                M = m < 0.0f ? 0 : (m > 255.0f ? 255 : (int64_t)m);
                const float t = ((beta[c] - mean_over_std * gamma[c]) / o[c]);
                B = rint_to_i64(ldexpf(t, N));
            }
            y[r * C + c] = round_shift_half_even(sign * M * v + B, N);
        }
    }
    return OR_OK;
}

/* ---------------------------------------------------------------------------
 * Standalone quantized elementwise ops on s8 codes [QI 量化乘法, 量化加法,
 * 量化激活函数], symmetric (zero points 0):
 *   MUL : out = clip(rint((float)(a * b) * M)),  M = s_a s_b / s_c computed ahead
 *   ADD : out = clip(rint((float)(a + b) * M)),  M = s_ab / s_c, the operands
 *         sharing one scale s_ab (the page requires it)
 *   RELU: out = max(a, 0)   (a passive op: same scale in and out, no rounding)
 * then, with relu set, max(out, 0).  Readings: the rescale is a multiplication by
 * the precomputed fp32 M (the page divides by scale_abc = 1 / M; the library's
 * requant epilogue multiplies too); clip to [-128, 127]; rint is half to even.
 * The integer variant of the page (a shift by round(log2 scale_abc)) is the case
 * M = 2^-k, exact in fp32.  op: 0 ADD, 1 MUL, 2 RELU. */
int oracle_eltwise_s8(int op, const int32_t *a, const int32_t *b, int64_t n, float M, int relu, int32_t *out)
{
    if (op < 0 || op > 2) return OR_ERR_ARG;
    for (int64_t i = 0; i < n; ++i) {
        int32_t v;
        if (op == 2) {
            v = a[i] > 0 ? a[i] : 0;
        } else {
            const int32_t t = op == 0 ? a[i] + b[i] : a[i] * b[i];
            const float r = rintf((float)t * M);
            v = (int32_t)clamp_f(r, -128.0f, 127.0f);
        }
        if (relu && v < 0) v = 0;
        out[i] = v;
    }
    return OR_OK;
}

/* Dynamic per-row symmetric quantization [QI 量化参数选择, 最大值截断: the scale
 * is the largest magnitude over 127 -- the page writes -127 for symmetry; QI
 * 量化算子: q = clip(round(x / s))]:  s[r] = max_c |x[r][c]| / 127 (one fp32
 * division), q = clip(rint(x / s[r]), qmin, qmax) (one IEEE division each, as in
 * oracle_quantize).  A row of zeros gets s = 0 and codes 0.  narrow selects
 * [-127, 127], else [-128, 127].  Inputs must be finite. */
int oracle_quantize_rows_dynamic(const float *x, int64_t rows, int64_t cols, int narrow, int32_t *q, float *scale)
{
    if (rows < 0 || cols <= 0) return OR_ERR_ARG;
    const float qmin = narrow ? -127.0f : -128.0f;
    for (int64_t r = 0; r < rows; ++r) {
        const float *xr = x + r * cols;
        float amax = 0.0f;
        for (int64_t c = 0; c < cols; ++c) amax = fmaxf(amax, fabsf(xr[c]));
        const float sc = amax / 127.0f;
        scale[r] = sc;
        for (int64_t c = 0; c < cols; ++c)
            q[r * cols + c] = sc == 0.0f ? 0 : (int32_t)clamp_f(rintf(xr[c] / sc), qmin, 127.0f);
    }
    return OR_OK;
}

/* ---------------------------------------------------------------------------
 * NHWC <-> NCHW64 [MG conv 算子優化: the output is written in NCHW64, each 64
 * consecutive output channels of a pixel contiguous].  On codes (one int32 per
 * element): nchw64[n][cb][h][w][j] = nhwc[n][h][w][64 cb + j], C % 64 == 0. */
int oracle_nhwc_to_nchw64(const int32_t *src, int N, int H, int W, int C, int32_t *dst)
{
    if (N < 0 || H <= 0 || W <= 0 || C <= 0 || C % 64) return OR_ERR_ARG;
    const int CB = C / 64;
    for (int n = 0; n < N; ++n)
        for (int h = 0; h < H; ++h)
            for (int w = 0; w < W; ++w)
                for (int c = 0; c < C; ++c) {
                    const int cb = c / 64, j = c % 64;
                    dst[((((int64_t)n * CB + cb) * H + h) * W + w) * 64 + j] =
                        src[(((int64_t)n * H + h) * W + w) * C + c];
                }
    return OR_OK;
}
