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
 *         3.2 Power-of-Two Factor.
 *
 * Readings of points the pages leave open are stated next to the code that
 * takes them.  Parity status: every function here is pinned by tests that do
 * not re-type its formula (worked examples, closed forms, brute force in
 * exact rational arithmetic, invariants, numpy library routines).
 */
#include <math.h>
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
 *   zp_term[n] = zcoef * colsum[n]       (int32; zcoef = Z_a - c_a where c_a is
 *                                        the centre the library subtracts from
 *                                        a u8 operand, see the library header)
 *   M[n]  = (s_a * s_w[n]) / s_o          fmul, then fdiv
 *   Bq[n] = bias[n] / s_o
 *   D[n]  = s_a * s_w[n]                  (dequantizing epilogue)
 * s_w is per output channel when w_per_channel, else s_w[0]; bias may be NULL
 * (zero).
 * ------------------------------------------------------------------------- */
int oracle_fold(int64_t N, int32_t zcoef, const int32_t *colsum, float s_a,
                const float *s_w, int w_per_channel, const float *bias, float s_o,
                int32_t *zp_term, float *Mv, float *Bq, float *D)
{
    int bad = 0;
    for (int64_t n = 0; n < N; ++n) {
        int64_t z = (int64_t)zcoef * (int64_t)colsum[n];
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
