// qnn_quant.cu -- q_quantize / q_dequantize: memory-bound elementwise kernels.
//
// Quantize [QI 量化算子, 量化模式, tensor量化与通道量化]: per element,
//   sym : q = clip(rint(x / s))          (IEEE fp32 divide, round half to even)
//   asym: q = clip(rint(x / s) + z)      (offset added after rounding)
//   pow2: q = clip(rint(x * 2^shift))
// Dequantize [QI 反量化算子; MG 背景]: x = (float)(q - z) * s, pow2 x = q * 2^-shift.
// ([QI] "【量化】神经网络量化介绍"; [MG] MegEngine 4-bit quantization article.)
//
// The tensor is viewed as rows x columns with the column count a multiple of
// 8: per tensor (one row), per channel along rows (a channel per row: the
// channel axis is not the last one) or per channel along columns (the last
// axis is the channel axis).  Each thread handles groups of 8 consecutive
// elements, two groups in flight: two 16-byte streaming loads of fp32 and one
// 8-byte (8-bit codes) or 4-byte (4-bit codes) store.  Scheme, code width and
// channel layout are template parameters, so the loop carries no branches.
// Other layouts (channel blocks not a multiple of 8 long) take a scalar kernel.
//
// Rounding and clipping run in the integer domain: r = cvt.rni(t) is rint(t)
// for |t| < 2^31 and saturates beyond, the zero point is a saturating add, and
// the clip to [qmin, qmax] is two integer min / max -- the same codes as the
// fp32 clip of rint(t) + z for every finite t, for +-Inf (saturation) and for
// NaN (cvt gives 0, so NaN maps to z, the code of real zero).
#include <cuda_runtime.h>
#include <cstdint>
#include "qnn_internal.h"

namespace qnn {
namespace {

enum { CM_TENSOR = 0, CM_ROW = 1, CM_COL = 2 };

struct QArgs {
    const float *x;
    uint8_t *q;
    float *y;           // dequantize output
    const uint8_t *qi;  // dequantize input
    int64_t n;          // elements
    int64_t R, L;       // vector view: R rows of L elements, L % 8 == 0
    int64_t C, inner;   // channel of element i: (i / inner) % C
    int per_channel, scheme, bits, is_signed;
    const float *scale;
    const int32_t *zp;
    const int32_t *shift;
    int32_t qmin, qmax;
};

__device__ __forceinline__ int32_t cvt_rni(float f)
{
    int32_t d;
    asm("cvt.rni.s32.f32 %0, %1;" : "=r"(d) : "f"(f));
    return d;
}

__device__ __forceinline__ int32_t add_sat(int32_t a, int32_t b)
{
    int32_t d;
    asm("add.sat.s32 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

// d = c << 16 | b << 8 | a for 8-bit codes (a, b already inside the code
// range, so the saturation of the packing instruction never changes them)
template <int SIGNED>
__device__ __forceinline__ uint32_t pack8(int32_t a, int32_t b, uint32_t c)
{
    uint32_t d;
    if (SIGNED)
        asm("cvt.pack.sat.s8.s32.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(b), "r"(a), "r"(c));
    else
        asm("cvt.pack.sat.u8.s32.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(b), "r"(a), "r"(c));
    return d;
}

// d = c << 8 | b << 4 | a for 4-bit codes
template <int SIGNED>
__device__ __forceinline__ uint32_t pack4(int32_t a, int32_t b, uint32_t c)
{
    uint32_t d;
    if (SIGNED)
        asm("cvt.pack.sat.s4.s32.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(b), "r"(a), "r"(c));
    else
        asm("cvt.pack.sat.u4.s32.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(b), "r"(a), "r"(c));
    return d;
}

// 2^e as an fp32 value, -126 <= e <= 127
__device__ __forceinline__ float pow2f(int32_t e) { return __int_as_float((e + 127) << 23); }

// Per-channel parameters, as the scheme needs them.
template <int SCHEME>
struct Prm {
    float s;     // scale (sym / asym) or 2^(+-shift) (pow2)
    int32_t z;
};

template <int SCHEME, bool DEQ>
__device__ __forceinline__ Prm<SCHEME> load_prm(const QArgs &a, int64_t ch)
{
    Prm<SCHEME> p;
    if (SCHEME == QNN_POW2) {
        const int32_t sh = __ldg(a.shift + ch);
        p.s = pow2f(DEQ ? -sh : sh);
    } else {
        p.s = __ldg(a.scale + ch);
    }
    p.z = (SCHEME == QNN_ASYM) ? __ldg(a.zp + ch) : 0;
    return p;
}

template <int SCHEME>
__device__ __forceinline__ int32_t quant1(const QArgs &a, float x, const Prm<SCHEME> &p)
{
    const float t = (SCHEME == QNN_POW2) ? __fmul_rn(x, p.s) : __fdiv_rn(x, p.s);
    int32_t r = cvt_rni(t);
    if (SCHEME == QNN_ASYM) r = add_sat(r, p.z);
    return min(max(r, a.qmin), a.qmax);
}

template <int SCHEME>
__device__ __forceinline__ float dequant1(int32_t q, const Prm<SCHEME> &p)
{
    if (SCHEME == QNN_POW2) return __fmul_rn((float)q, p.s);  // exact power-of-two scaling
    return __fmul_rn((float)(q - p.z), p.s);
}

template <int SCHEME, int BITS, int SIGNED, int CM>
__device__ __forceinline__ void quant_group(const QArgs &a, const Prm<SCHEME> &pr, uint8_t *qrow, int64_t col0,
                                            float4 v0, float4 v1)
{
    const float v[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
    int32_t c[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        if (CM == CM_COL) {
            c[j] = quant1<SCHEME>(a, v[j], load_prm<SCHEME, false>(a, col0 + j));
        } else {
            c[j] = quant1<SCHEME>(a, v[j], pr);
        }
    }
    if (BITS == 8) {
        const uint32_t lo = pack8<SIGNED>(c[0], c[1], pack8<SIGNED>(c[2], c[3], 0));
        const uint32_t hi = pack8<SIGNED>(c[4], c[5], pack8<SIGNED>(c[6], c[7], 0));
        __stcs(reinterpret_cast<uint2 *>(qrow + col0), make_uint2(lo, hi));
    } else {
        const uint32_t w = pack4<SIGNED>(
            c[0], c[1], pack4<SIGNED>(c[2], c[3], pack4<SIGNED>(c[4], c[5], pack4<SIGNED>(c[6], c[7], 0))));
        __stcs(reinterpret_cast<unsigned int *>(qrow + col0 / 2), w);
    }
}

template <int SCHEME, int BITS, int SIGNED, int CM>
__global__ void __launch_bounds__(256) quantize2d_kernel(const QArgs a)
{
    const int64_t G = a.L / 8;
    const int64_t gx = (int64_t)gridDim.x * blockDim.x;
    Prm<SCHEME> pr{};
    if (CM == CM_TENSOR) pr = load_prm<SCHEME, false>(a, 0);
    for (int64_t r = blockIdx.y; r < a.R; r += gridDim.y) {
        if (CM == CM_ROW) pr = load_prm<SCHEME, false>(a, r % a.C);
        const float4 *xr = reinterpret_cast<const float4 *>(a.x + r * a.L);
        uint8_t *qrow = a.q + (BITS == 8 ? r * a.L : r * a.L / 2);
        for (int64_t g = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; g < G; g += 2 * gx) {
            const int64_t g2 = g + gx;
            const float4 v0 = __ldcs(xr + 2 * g), v1 = __ldcs(xr + 2 * g + 1);
            float4 w0 = v0, w1 = v1;
            const bool two = g2 < G;
            if (two) {
                w0 = __ldcs(xr + 2 * g2);
                w1 = __ldcs(xr + 2 * g2 + 1);
            }
            quant_group<SCHEME, BITS, SIGNED, CM>(a, pr, qrow, g * 8, v0, v1);
            if (two) quant_group<SCHEME, BITS, SIGNED, CM>(a, pr, qrow, g2 * 8, w0, w1);
        }
    }
}

__device__ __forceinline__ int32_t code_at(const QArgs &a, const uint8_t *src, int64_t i)
{
    int32_t v;
    if (a.bits == 8) {
        v = src[i];
        if (a.is_signed && v >= 128) v -= 256;
    } else {
        const uint32_t b = src[i / 2];
        v = (int32_t)((i & 1) ? (b >> 4) : (b & 15u));
        if (a.is_signed && v >= 8) v -= 16;
    }
    return v;
}

template <int SCHEME>
__device__ __forceinline__ Prm<SCHEME> prm_generic(const QArgs &a, int64_t i, bool deq)
{
    const int64_t ch = a.per_channel ? (i / a.inner) % a.C : 0;
    return deq ? load_prm<SCHEME, true>(a, ch) : load_prm<SCHEME, false>(a, ch);
}

// Scalar path: any channel layout, and the last n % 8 elements of a per-tensor
// view (elements [begin, n)).  Threads own whole bytes of 4-bit outputs.
template <int SCHEME>
__global__ void __launch_bounds__(256) quantize_scalar_kernel(const QArgs a, int64_t begin)
{
    const int64_t step = (int64_t)gridDim.x * blockDim.x;
    if (a.bits == 8) {
        for (int64_t i = begin + (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < a.n; i += step)
            a.q[i] = (uint8_t)(quant1<SCHEME>(a, a.x[i], prm_generic<SCHEME>(a, i, false)) & 255);
    } else {
        for (int64_t b = begin / 2 + (int64_t)blockIdx.x * blockDim.x + threadIdx.x; 2 * b < a.n; b += step) {
            const int32_t c0 = quant1<SCHEME>(a, a.x[2 * b], prm_generic<SCHEME>(a, 2 * b, false));
            const int32_t c1 = quant1<SCHEME>(a, a.x[2 * b + 1], prm_generic<SCHEME>(a, 2 * b + 1, false));
            a.q[b] = (uint8_t)((c0 & 15) | ((c1 & 15) << 4));
        }
    }
}

template <int SCHEME, int BITS, int SIGNED, int CM>
__global__ void __launch_bounds__(256) dequantize2d_kernel(const QArgs a)
{
    const int64_t G = a.L / 8;
    const int64_t gx = (int64_t)gridDim.x * blockDim.x;
    Prm<SCHEME> pr{};
    if (CM == CM_TENSOR) pr = load_prm<SCHEME, true>(a, 0);
    for (int64_t r = blockIdx.y; r < a.R; r += gridDim.y) {
        if (CM == CM_ROW) pr = load_prm<SCHEME, true>(a, r % a.C);
        const uint8_t *qrow = a.qi + (BITS == 8 ? r * a.L : r * a.L / 2);
        float4 *yr = reinterpret_cast<float4 *>(a.y + r * a.L);
        for (int64_t g = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; g < G; g += gx) {
            int32_t c[8];
            if (BITS == 8) {
                const uint2 w = __ldcs(reinterpret_cast<const uint2 *>(qrow + g * 8));
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    c[j] = SIGNED ? (int32_t)(int8_t)(w.x >> (8 * j)) : (int32_t)((w.x >> (8 * j)) & 255u);
                    c[4 + j] = SIGNED ? (int32_t)(int8_t)(w.y >> (8 * j)) : (int32_t)((w.y >> (8 * j)) & 255u);
                }
            } else {
                const uint32_t w = __ldcs(reinterpret_cast<const unsigned int *>(qrow + g * 4));
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    c[j] = SIGNED ? ((int32_t)(w << (28 - 4 * j)) >> 28) : (int32_t)((w >> (4 * j)) & 15u);
            }
            float o[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                if (CM == CM_COL)
                    o[j] = dequant1<SCHEME>(c[j], load_prm<SCHEME, true>(a, g * 8 + j));
                else
                    o[j] = dequant1<SCHEME>(c[j], pr);
            }
            __stcs(yr + 2 * g, make_float4(o[0], o[1], o[2], o[3]));
            __stcs(yr + 2 * g + 1, make_float4(o[4], o[5], o[6], o[7]));
        }
    }
}

template <int SCHEME>
__global__ void __launch_bounds__(256) dequantize_scalar_kernel(const QArgs a, int64_t begin)
{
    const int64_t step = (int64_t)gridDim.x * blockDim.x;
    for (int64_t i = begin + (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < a.n; i += step)
        a.y[i] = dequant1<SCHEME>(code_at(a, a.qi, i), prm_generic<SCHEME>(a, i, true));
}

qnn_status prepare(const void *x, const void *q, int q_dt, int ndim, const int64_t *shape,
                   const qnn_qparams *p, QArgs *a)
{
    if (!shape || !p || ndim < 1 || ndim > 16) return QNN_ERR_INVALID_ARG;
    int64_t n = 1;
    for (int i = 0; i < ndim; ++i) {
        if (shape[i] < 0) return QNN_ERR_INVALID_ARG;
        n *= shape[i];
    }
    a->n = n;
    if (n == 0) return QNN_OK;  // nothing to do; pointers of empty tensors may be null
    if (!x || !q) return QNN_ERR_INVALID_ARG;
    int32_t lo, hi;
    if (!qrange(q_dt, p->narrow_range, &lo, &hi)) return QNN_ERR_INVALID_ARG;
    if (p->scheme < QNN_SYM || p->scheme > QNN_POW2) return QNN_ERR_INVALID_ARG;
    if (p->scheme == QNN_POW2 && !p->shift) return QNN_ERR_INVALID_ARG;
    if (p->scheme != QNN_POW2 && !p->scale) return QNN_ERR_INVALID_ARG;
    if (p->scheme == QNN_ASYM && !p->zero_point) return QNN_ERR_INVALID_ARG;
    const int bits = (q_dt == QNN_S4 || q_dt == QNN_U4) ? 4 : 8;
    if (bits == 4 && (shape[ndim - 1] % 2) != 0) return QNN_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(q)) return QNN_ERR_ALIGNMENT;
    a->bits = bits;
    a->is_signed = (q_dt == QNN_S8 || q_dt == QNN_S4);
    a->scheme = p->scheme;
    a->per_channel = p->per_channel ? 1 : 0;
    a->scale = p->scale;
    a->zp = p->zero_point;
    a->shift = p->shift;
    a->qmin = lo;
    a->qmax = hi;
    a->C = 1;
    a->inner = 1;
    if (a->per_channel) {
        const int ax = p->axis < 0 ? p->axis + ndim : p->axis;
        if (ax < 0 || ax >= ndim) return QNN_ERR_INVALID_ARG;
        int64_t inner = 1;
        for (int i = ax + 1; i < ndim; ++i) inner *= shape[i];
        a->C = shape[ax];
        a->inner = inner;
    }
    return QNN_OK;
}

// Channel layout of the vector view, or -1 if the scalar kernel is needed.
int channel_mode(QArgs &a)
{
    if (!a.per_channel) {
        a.R = 1;
        a.L = a.n - a.n % 8;
        return CM_TENSOR;
    }
    if (a.inner % 8 == 0) {
        a.R = a.n / a.inner;
        a.L = a.inner;
        return CM_ROW;
    }
    if (a.inner == 1 && a.C % 8 == 0) {
        a.R = a.n / a.C;
        a.L = a.C;
        return CM_COL;
    }
    return -1;
}

dim3 grid2d(const QArgs &a, int per_thread_groups)
{
    const int64_t target = (int64_t)sm_count() * 8;
    const int64_t G = a.L / 8;
    int64_t gx = (G + 256LL * per_thread_groups - 1) / (256LL * per_thread_groups);
    if (gx < 1) gx = 1;
    if (gx > target) gx = target;
    int64_t gy = target / gx;
    if (gy < 1) gy = 1;
    if (gy > a.R) gy = a.R;
    if (gy > 65535) gy = 65535;
    return dim3((unsigned)gx, (unsigned)gy, 1);
}

int grid1d(int64_t n)
{
    int64_t b = (n + 255) / 256;
    const int64_t cap = (int64_t)sm_count() * 8;
    if (b > cap) b = cap;
    return b < 1 ? 1 : (int)b;
}

template <int SCHEME>
qnn_status launch_quant(QArgs &a, cudaStream_t s)
{
    const int cm = channel_mode(a);
    if (cm < 0) {
        quantize_scalar_kernel<SCHEME><<<grid1d(a.n), 256, 0, s>>>(a, 0);
        return launch_status();
    }
    if (a.L > 0) {
        const dim3 grid = grid2d(a, 2);
#define QNN_Q2D(B, S, M) quantize2d_kernel<SCHEME, B, S, M><<<grid, 256, 0, s>>>(a)
#define QNN_Q2D_CM(B, S)                               \
    do {                                               \
        if (cm == CM_TENSOR) QNN_Q2D(B, S, CM_TENSOR); \
        else if (cm == CM_ROW) QNN_Q2D(B, S, CM_ROW);  \
        else QNN_Q2D(B, S, CM_COL);                    \
    } while (0)
        if (a.bits == 8) {
            if (a.is_signed) QNN_Q2D_CM(8, 1);
            else QNN_Q2D_CM(8, 0);
        } else {
            if (a.is_signed) QNN_Q2D_CM(4, 1);
            else QNN_Q2D_CM(4, 0);
        }
#undef QNN_Q2D_CM
#undef QNN_Q2D
        if (launch_status() != QNN_OK) return QNN_ERR_CUDA;
    }
    const int64_t done = a.R * a.L;
    if (done < a.n) {  // per-tensor tail of n % 8 elements
        quantize_scalar_kernel<SCHEME><<<1, 256, 0, s>>>(a, done);
        return launch_status();
    }
    return QNN_OK;
}

template <int SCHEME>
qnn_status launch_dequant(QArgs &a, cudaStream_t s)
{
    const int cm = channel_mode(a);
    if (cm < 0) {
        dequantize_scalar_kernel<SCHEME><<<grid1d(a.n), 256, 0, s>>>(a, 0);
        return launch_status();
    }
    if (a.L > 0) {
        const dim3 grid = grid2d(a, 1);
#define QNN_D2D(B, S, M) dequantize2d_kernel<SCHEME, B, S, M><<<grid, 256, 0, s>>>(a)
#define QNN_D2D_CM(B, S)                      \
    do {                                      \
        if (cm == CM_TENSOR) QNN_D2D(B, S, CM_TENSOR); \
        else if (cm == CM_ROW) QNN_D2D(B, S, CM_ROW);  \
        else QNN_D2D(B, S, CM_COL);                    \
    } while (0)
        if (a.bits == 8) {
            if (a.is_signed) QNN_D2D_CM(8, 1);
            else QNN_D2D_CM(8, 0);
        } else {
            if (a.is_signed) QNN_D2D_CM(4, 1);
            else QNN_D2D_CM(4, 0);
        }
#undef QNN_D2D_CM
#undef QNN_D2D
        if (launch_status() != QNN_OK) return QNN_ERR_CUDA;
    }
    const int64_t done = a.R * a.L;
    if (done < a.n) {
        dequantize_scalar_kernel<SCHEME><<<1, 256, 0, s>>>(a, done);
        return launch_status();
    }
    return QNN_OK;
}

}  // namespace
}  // namespace qnn

extern "C" qnn_status q_quantize(const float *x, void *q, qnn_dtype q_dt, int ndim,
                                 const int64_t *shape, const qnn_qparams *p, qnn_stream_t stream)
{
    qnn::QArgs a{};
    qnn_status st = qnn::prepare(x, q, q_dt, ndim, shape, p, &a);
    if (st != QNN_OK || a.n == 0) return st;
    a.x = x;
    a.q = static_cast<uint8_t *>(q);
    cudaStream_t s = (cudaStream_t)stream;
    switch (a.scheme) {
    case QNN_SYM: return qnn::launch_quant<QNN_SYM>(a, s);
    case QNN_ASYM: return qnn::launch_quant<QNN_ASYM>(a, s);
    default: return qnn::launch_quant<QNN_POW2>(a, s);
    }
}

extern "C" qnn_status q_dequantize(const void *q, qnn_dtype q_dt, float *x, int ndim,
                                   const int64_t *shape, const qnn_qparams *p, qnn_stream_t stream)
{
    qnn::QArgs a{};
    qnn_status st = qnn::prepare(x, q, q_dt, ndim, shape, p, &a);
    if (st != QNN_OK || a.n == 0) return st;
    a.qi = static_cast<const uint8_t *>(q);
    a.y = x;
    cudaStream_t s = (cudaStream_t)stream;
    switch (a.scheme) {
    case QNN_SYM: return qnn::launch_dequant<QNN_SYM>(a, s);
    case QNN_ASYM: return qnn::launch_dequant<QNN_ASYM>(a, s);
    default: return qnn::launch_dequant<QNN_POW2>(a, s);
    }
}
