// qnn_quant.cu -- q_quantize / q_dequantize: memory-bound elementwise kernels.
//
// Quantize [QI 量化算子, 量化模式, tensor量化与通道量化]: per element,
//   sym : q = clip(rint(x / s))          (IEEE fp32 divide, round half to even)
//   asym: q = clip(rint(x / s) + z)      (offset added after rounding)
//   pow2: q = clip(rint(x * 2^shift))
// Dequantize [QI 反量化算子; MG 背景]: x = (float)(q - z) * s, pow2 x = q * 2^-shift.
// ([QI] "【量化】神经网络量化介绍"; [MG] MegEngine 4-bit quantization article.)
//
// Each thread handles groups of 8 consecutive elements: two 16-byte streaming
// loads of fp32 and one 8-byte (8-bit codes) or 4-byte (4-bit codes) store,
// or the reverse for dequantize.  Grid-stride over groups, two groups in
// flight per thread; a scalar tail handles the last n % 8 elements.
#include <cuda_runtime.h>
#include <cstdint>
#include "qnn_internal.h"

namespace qnn {
namespace {

struct QArgs {
    const float *x;
    uint8_t *q;
    float *y;           // dequantize output
    const uint8_t *qi;  // dequantize input
    int64_t n;          // elements
    int64_t C, inner;   // channel view [outer, C, inner]
    int per_channel, scheme, bits, is_signed;
    int group_mode;     // 0: channel constant over a group, 1: consecutive channels, 2: generic
    const float *scale;
    const int32_t *zp;
    const int32_t *shift;
    float qmin, qmax;
};

__device__ __forceinline__ int64_t chan_of(const QArgs &a, int64_t idx)
{
    return a.per_channel ? (idx / a.inner) % a.C : 0;
}

__device__ __forceinline__ int32_t quant_one(const QArgs &a, float v, int64_t ch)
{
    const int32_t z = (a.scheme == QNN_ASYM) ? __ldg(a.zp + ch) : 0;
    if (v != v) return z;
    float r;
    if (a.scheme == QNN_POW2) {
        r = rintf(ldexpf(v, __ldg(a.shift + ch)));
    } else {
        r = rintf(__fdiv_rn(v, __ldg(a.scale + ch)));
    }
    if (a.scheme == QNN_ASYM) r = __fadd_rn(r, (float)z);
    return (int32_t)fminf(fmaxf(r, a.qmin), a.qmax);
}

__device__ __forceinline__ float dequant_one(const QArgs &a, int32_t q, int64_t ch)
{
    if (a.scheme == QNN_POW2) return ldexpf((float)q, -__ldg(a.shift + ch));
    const int32_t z = (a.scheme == QNN_ASYM) ? __ldg(a.zp + ch) : 0;
    return __fmul_rn((float)(q - z), __ldg(a.scale + ch));
}

__device__ __forceinline__ int64_t group_chan(const QArgs &a, int64_t idx0, int j)
{
    if (!a.per_channel) return 0;
    if (a.group_mode == 0) return (idx0 / a.inner) % a.C;
    if (a.group_mode == 1) return (idx0 % a.C) + j;
    return chan_of(a, idx0 + j);
}

__device__ __forceinline__ void quant_group(const QArgs &a, int64_t g, float4 v0, float4 v1)
{
    const int64_t idx0 = g * 8;
    const float v[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
    int32_t c[8];
    if (a.per_channel && a.group_mode == 0) {
        const int64_t ch = (idx0 / a.inner) % a.C;
#pragma unroll
        for (int j = 0; j < 8; ++j) c[j] = quant_one(a, v[j], ch);
    } else {
#pragma unroll
        for (int j = 0; j < 8; ++j) c[j] = quant_one(a, v[j], group_chan(a, idx0, j));
    }
    if (a.bits == 8) {
        uint32_t lo = (c[0] & 255) | ((c[1] & 255) << 8) | ((c[2] & 255) << 16) | ((uint32_t)c[3] << 24);
        uint32_t hi = (c[4] & 255) | ((c[5] & 255) << 8) | ((c[6] & 255) << 16) | ((uint32_t)c[7] << 24);
        __stcs(reinterpret_cast<uint2 *>(a.q + idx0), make_uint2(lo, hi));
    } else {
        uint32_t w = 0;
#pragma unroll
        for (int j = 0; j < 8; ++j) w |= (uint32_t)(c[j] & 15) << (4 * j);
        __stcs(reinterpret_cast<unsigned int *>(a.q + idx0 / 2), w);
    }
}

__global__ void __launch_bounds__(256) quantize_kernel(const QArgs a)
{
    const int64_t ngroups = a.n / 8;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t g = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; g < ngroups; g += 2 * stride) {
        const int64_t g2 = g + stride;
        const float4 *p = reinterpret_cast<const float4 *>(a.x) + 2 * g;
        float4 v0 = __ldcs(p), v1 = __ldcs(p + 1), w0, w1;
        const bool two = g2 < ngroups;
        if (two) {
            const float4 *p2 = reinterpret_cast<const float4 *>(a.x) + 2 * g2;
            w0 = __ldcs(p2);
            w1 = __ldcs(p2 + 1);
        }
        quant_group(a, g, v0, v1);
        if (two) quant_group(a, g2, w0, w1);
    }
    // tail: at most 7 elements, handled by thread 0 of block 0
    if (blockIdx.x == 0 && threadIdx.x == 0) {
        for (int64_t i = ngroups * 8; i < a.n; ++i) {
            const int32_t c = quant_one(a, a.x[i], chan_of(a, i));
            if (a.bits == 8) {
                a.q[i] = (uint8_t)(c & 255);
            } else {
                uint8_t b = a.q[i / 2];
                b = (i & 1) ? (uint8_t)((b & 0x0F) | ((c & 15) << 4)) : (uint8_t)((b & 0xF0) | (c & 15));
                a.q[i / 2] = b;
            }
        }
    }
}

__device__ __forceinline__ int32_t code_at(const QArgs &a, uint32_t word, int j)
{
    // word holds 4 byte codes (bits == 8) or 8 nibble codes (bits == 4)
    int32_t v;
    if (a.bits == 8) {
        v = (int32_t)((word >> (8 * j)) & 255u);
        if (a.is_signed && v >= 128) v -= 256;
    } else {
        v = (int32_t)((word >> (4 * j)) & 15u);
        if (a.is_signed && v >= 8) v -= 16;
    }
    return v;
}

__global__ void __launch_bounds__(256) dequantize_kernel(const QArgs a)
{
    const int64_t ngroups = a.n / 8;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t g = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; g < ngroups; g += stride) {
        const int64_t idx0 = g * 8;
        int32_t c[8];
        if (a.bits == 8) {
            const uint2 w = __ldcs(reinterpret_cast<const uint2 *>(a.qi + idx0));
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                c[j] = code_at(a, w.x, j);
                c[4 + j] = code_at(a, w.y, j);
            }
        } else {
            const uint32_t w = __ldcs(reinterpret_cast<const unsigned int *>(a.qi + idx0 / 2));
#pragma unroll
            for (int j = 0; j < 8; ++j) c[j] = code_at(a, w, j);
        }
        float o[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) o[j] = dequant_one(a, c[j], group_chan(a, idx0, j));
        float4 *p = reinterpret_cast<float4 *>(a.y + idx0);
        __stcs(p, make_float4(o[0], o[1], o[2], o[3]));
        __stcs(p + 1, make_float4(o[4], o[5], o[6], o[7]));
    }
    if (blockIdx.x == 0 && threadIdx.x == 0) {
        for (int64_t i = ngroups * 8; i < a.n; ++i) {
            uint32_t b = a.qi[a.bits == 8 ? i : i / 2];
            int32_t v = (a.bits == 8) ? code_at(a, b, 0) : code_at(a, b, (int)(i & 1));
            a.y[i] = dequant_one(a, v, chan_of(a, i));
        }
    }
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
    a->n = n;
    a->bits = bits;
    a->is_signed = (q_dt == QNN_S8 || q_dt == QNN_S4);
    a->scheme = p->scheme;
    a->per_channel = p->per_channel ? 1 : 0;
    a->scale = p->scale;
    a->zp = p->zero_point;
    a->shift = p->shift;
    a->qmin = (float)lo;
    a->qmax = (float)hi;
    a->C = 1;
    a->inner = 1;
    a->group_mode = 0;
    if (a->per_channel) {
        int ax = p->axis < 0 ? p->axis + ndim : p->axis;
        if (ax < 0 || ax >= ndim) return QNN_ERR_INVALID_ARG;
        int64_t inner = 1;
        for (int i = ax + 1; i < ndim; ++i) inner *= shape[i];
        a->C = shape[ax] > 0 ? shape[ax] : 1;
        a->inner = inner > 0 ? inner : 1;
        if (a->inner % 8 == 0) a->group_mode = 0;
        else if (a->inner == 1 && a->C % 8 == 0) a->group_mode = 1;
        else a->group_mode = 2;
    }
    return QNN_OK;
}

int grid_for(int64_t n)
{
    const int64_t groups = (n + 7) / 8;
    int64_t blocks = (groups + 255) / 256;
    const int64_t cap = (int64_t)sm_count() * 8;
    if (blocks > cap) blocks = cap;
    return blocks < 1 ? 1 : (int)blocks;
}

}  // namespace
}  // namespace qnn

extern "C" qnn_status q_quantize(const float *x, void *q, qnn_dtype q_dt, int ndim,
                                 const int64_t *shape, const qnn_qparams *p, qnn_stream_t stream)
{
    qnn::QArgs a{};
    qnn_status st = qnn::prepare(x, q, q_dt, ndim, shape, p, &a);
    if (st != QNN_OK) return st;
    if (a.n == 0) return QNN_OK;
    a.x = x;
    a.q = static_cast<uint8_t *>(q);
    qnn::quantize_kernel<<<qnn::grid_for(a.n), 256, 0, (cudaStream_t)stream>>>(a);
    return qnn::launch_status();
}

extern "C" qnn_status q_dequantize(const void *q, qnn_dtype q_dt, float *x, int ndim,
                                   const int64_t *shape, const qnn_qparams *p, qnn_stream_t stream)
{
    qnn::QArgs a{};
    qnn_status st = qnn::prepare(x, q, q_dt, ndim, shape, p, &a);
    if (st != QNN_OK) return st;
    if (a.n == 0) return QNN_OK;
    a.qi = static_cast<const uint8_t *>(q);
    a.y = x;
    qnn::dequantize_kernel<<<qnn::grid_for(a.n), 256, 0, (cudaStream_t)stream>>>(a);
    return qnn::launch_status();
}
