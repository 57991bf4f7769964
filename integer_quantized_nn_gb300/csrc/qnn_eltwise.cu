// qnn_eltwise.cu -- standalone quantized elementwise ops and dynamic per-row
// quantization: memory-bound kernels.
//
// q_eltwise_s8 [QI] "【量化】神经网络量化介绍", sections 量化乘法 / 量化加法 /
// 量化激活函数: on symmetric s8 codes,
//   ADD : clip(rint((a + b) * M))   (operands sharing one scale; M = s_ab / s_c)
//   MUL : clip(rint((a * b) * M))   (M = s_a s_b / s_c, computed ahead)
//   RELU: max(a, 0)                 (passive: scale unchanged)
// with an optional ReLU after the rescale.  The integer sum or product is exact in
// fp32 (|t| <= 2^14); one fp32 multiply, round half to even, clip to [-128, 127].
// Each thread handles 16 elements per step: two 16-byte loads and one 16-byte
// store; a grid-stride loop, the n % 16 tail by the first threads.
//
// q_layout_nchw64: NHWC <-> NCHW64 [MG conv 算子優化: outputs in NCHW64, 64
// consecutive channels of a pixel contiguous] for packed 4-bit or 8-bit codes:
// a permutation of blocks of 64 channels (32 or 64 bytes), moved as 16-byte
// chunks, one per thread and step, both sides coalesced along the block.
//
// q_quantize_rows_dynamic [QI 量化参数选择 (最大值截断), 量化算子]: per row the
// scale max|x| / 127 (one IEEE division), then q = clip(rint(x / s)), the code of
// the IEEE quotient (formed through the row's reciprocal, with the IEEE division
// wherever that could decide the code differently -- see dyn_quant4); a zero row
// gets scale 0 and codes 0.  One warp per row: rows of up to 1024 values are
// held in registers (one read), longer ones read twice (the second time from
// cache); 4 floats per lane and step, codes stored as 4-byte words.
#include <cuda_runtime.h>
#include <algorithm>
#include <cstdint>
#include "qnn_internal.h"

namespace qnn {
namespace {

constexpr unsigned kFull = 0xffffffffu;

template <int OP>
__device__ __forceinline__ int32_t elt(int32_t a, int32_t b, float M, bool relu)
{
    int32_t v;
    if constexpr (OP == QNN_RELU) {
        v = max(a, 0);
    } else {
        const int32_t t = OP == QNN_ADD ? a + b : a * b;
        v = min(max(__float2int_rn(__fmul_rn((float)t, M)), -128), 127);
    }
    return relu ? max(v, 0) : v;
}

template <int OP>
__global__ void __launch_bounds__(256) eltwise_s8_kernel(const int8_t *__restrict__ a, const int8_t *__restrict__ b,
                                                         int64_t n, float M, int relu, int8_t *__restrict__ out)
{
    const int64_t nv = n >> 4;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < nv; i += stride) {
        const uint4 av = __ldcs(reinterpret_cast<const uint4 *>(a) + i);
        uint4 bv = av;
        if constexpr (OP != QNN_RELU) bv = __ldcs(reinterpret_cast<const uint4 *>(b) + i);
        const uint32_t aw[4] = {av.x, av.y, av.z, av.w}, bw[4] = {bv.x, bv.y, bv.z, bv.w};
        uint32_t ow[4];
#pragma unroll
        for (int w = 0; w < 4; ++w) {
            uint32_t o = 0;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int32_t x = (int32_t)(int8_t)(aw[w] >> (8 * q)), y = (int32_t)(int8_t)(bw[w] >> (8 * q));
                o |= (uint32_t)(uint8_t)elt<OP>(x, y, M, relu != 0) << (8 * q);
            }
            ow[w] = o;
        }
        __stcs(reinterpret_cast<uint4 *>(out) + i, make_uint4(ow[0], ow[1], ow[2], ow[3]));
    }
    const int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (t < (n & 15)) {
        const int64_t k = (nv << 4) + t;
        out[k] = (int8_t)elt<OP>(a[k], OP == QNN_RELU ? 0 : b[k], M, relu != 0);
    }
}

// The row's scale s = max|x| / 127 and its reciprocal route.  The code is
// rint(RN(x / s)).  With s a normal number well inside the range, q0 =
// RN(x RN(1 / s)) carries two roundings of relative size 2^-24, so
// |q0 - RN(x / s)| < 1.6 2^-23 |q0| (plus a subnormal ulp, only where |q0| is far
// below 1/2).  When q0 lies more than 2^-20 |q0| away from every half-integer,
// RN(x / s) lies strictly inside the same unit interval around rint(q0), so both
// round to the same integer; the rare elements nearer a half-integer, and whole
// rows with an extreme scale, take the IEEE division.
struct DynScale {
    float s, y;
    bool recip;
};

__device__ __forceinline__ DynScale dyn_scale(float amax)
{
    DynScale d;
    d.s = __fdiv_rn(amax, 127.0f);
    d.recip = d.s >= 0x1p-100f && d.s <= 0x1p100f;
    d.y = d.recip ? __frcp_rn(d.s) : 0.0f;
    return d;
}

__device__ __forceinline__ float abs_max4(float m, const float4 &v)
{
    return fmaxf(m, fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w))));
}

// four codes of one 16-byte group, packed little-endian
__device__ __forceinline__ uint32_t dyn_quant4(const float4 &v, const DynScale &d, int32_t qmin)
{
    const float vs[4] = {v.x, v.y, v.z, v.w};
    int32_t c[4];
    bool near = !d.recip;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const float q0 = __fmul_rn(vs[j], d.y);
        const float dist = fabsf(__fsub_rn(q0, rintf(q0)));  // exact: |q0| < 2^23
        near = near || __fsub_rn(0.5f, dist) <= 0x1p-20f * fabsf(q0);
        c[j] = __float2int_rn(q0);
    }
    if (near) {
#pragma unroll
        for (int j = 0; j < 4; ++j) c[j] = d.s == 0.0f ? 0 : __float2int_rn(__fdiv_rn(vs[j], d.s));
    }
    uint32_t o = 0;
#pragma unroll
    for (int j = 0; j < 4; ++j) o |= (uint32_t)(uint8_t)min(max(c[j], qmin), 127) << (8 * j);
    return o;
}

// One warp per row.  R > 0: the row (at most 32 R groups of 4 values) is read
// once into registers, all its loads in flight together; R = 0: any length, the
// row read twice (the second time from cache).
template <int R>
__global__ void __launch_bounds__(256) quantize_rows_dynamic_kernel(const float *__restrict__ x, int64_t rows,
                                                                    int64_t cols, int narrow, int8_t *__restrict__ q,
                                                                    float *__restrict__ scale)
{
    const int lane = threadIdx.x & 31;
    const int64_t words = cols >> 2;
    const int32_t qmin = narrow ? -127 : -128;
    for (int64_t row = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; row < rows;
         row += ((int64_t)gridDim.x * blockDim.x) >> 5) {
        const float4 *xr = reinterpret_cast<const float4 *>(x + row * cols);
        uint32_t *qr = reinterpret_cast<uint32_t *>(q + row * cols);
        float amax = 0.0f;
        if constexpr (R > 0) {
            float4 v[R];
#pragma unroll
            for (int u = 0; u < R; ++u) {
                const int k = lane + 32 * u;
                v[u] = k < words ? __ldcs(xr + k) : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
                amax = abs_max4(amax, v[u]);
            }
            // magnitudes are non-negative: their bit patterns order like the values
            amax = __uint_as_float(__reduce_max_sync(kFull, __float_as_uint(amax)));
            const DynScale d = dyn_scale(amax);
            if (lane == 0) scale[row] = d.s;
#pragma unroll
            for (int u = 0; u < R; ++u) {
                const int k = lane + 32 * u;
                if (k < words) __stcs(qr + k, dyn_quant4(v[u], d, qmin));
            }
        } else {
            for (int64_t k = lane; k < words; k += 32) amax = abs_max4(amax, __ldg(xr + k));
            amax = __uint_as_float(__reduce_max_sync(kFull, __float_as_uint(amax)));
            const DynScale d = dyn_scale(amax);
            if (lane == 0) scale[row] = d.s;
            for (int64_t k = lane; k < words; k += 32) __stcs(qr + k, dyn_quant4(__ldcs(xr + k), d, qmin));
        }
    }
}

// chunk i of the destination (16 bytes); blk = bytes per 64-channel block.
template <bool TO_NCHW64>
__global__ void __launch_bounds__(256) nchw64_kernel(const uint4 *__restrict__ src, uint4 *__restrict__ dst,
                                                     int64_t chunks, int H, int W, int CB, int cpb)
{
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < chunks;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int j = (int)(i % cpb);  // chunk within a block
        const int64_t blk = i / cpb;    // destination block index
        int64_t s;
        if (TO_NCHW64) {
            // dst block (n, cb, h, w) <- src block (n, h, w, cb)
            const int w = (int)(blk % W);
            const int64_t t1 = blk / W;
            const int h = (int)(t1 % H);
            const int64_t t2 = t1 / H;
            const int cb = (int)(t2 % CB);
            const int64_t n = t2 / CB;
            s = (((n * H + h) * W + w) * CB + cb) * cpb + j;
        } else {
            // dst block (n, h, w, cb) <- src block (n, cb, h, w)
            const int cb = (int)(blk % CB);
            const int64_t t1 = blk / CB;
            const int w = (int)(t1 % W);
            const int64_t t2 = t1 / W;
            const int h = (int)(t2 % H);
            const int64_t n = t2 / H;
            s = (((n * CB + cb) * H + h) * W + w) * cpb + j;
        }
        __stcs(dst + i, __ldcs(src + s));
    }
}

int grid_for(int64_t work, int per_block)
{
    const int64_t want = (work + per_block - 1) / per_block;
    return (int)std::max<int64_t>(1, std::min<int64_t>(want, (int64_t)sm_count() * 8));
}

}  // namespace
}  // namespace qnn

extern "C" qnn_status q_eltwise_s8(qnn_eltwise_op op, const int8_t *a, const int8_t *b, int64_t n, float M,
                                   int relu, int8_t *out, qnn_stream_t stream)
{
    using namespace qnn;
    if (n < 0 || (op != QNN_ADD && op != QNN_MUL && op != QNN_RELU)) return QNN_ERR_INVALID_ARG;
    if (op != QNN_RELU && !(M == M && M < INFINITY && M > -INFINITY)) return QNN_ERR_INVALID_ARG;
    if (n == 0) return QNN_OK;
    if (!a || !out || (op != QNN_RELU && !b)) return QNN_ERR_INVALID_ARG;
    if (!aligned16(a) || !aligned16(out) || (op != QNN_RELU && !aligned16(b))) return QNN_ERR_ALIGNMENT;
    const int grid = grid_for(std::max<int64_t>(n >> 4, 16), 256);
    cudaStream_t s = (cudaStream_t)stream;
    switch (op) {
    case QNN_ADD: eltwise_s8_kernel<QNN_ADD><<<grid, 256, 0, s>>>(a, b, n, M, relu, out); break;
    case QNN_MUL: eltwise_s8_kernel<QNN_MUL><<<grid, 256, 0, s>>>(a, b, n, M, relu, out); break;
    default: eltwise_s8_kernel<QNN_RELU><<<grid, 256, 0, s>>>(a, a, n, M, relu, out); break;
    }
    return launch_status();
}

extern "C" qnn_status q_quantize_rows_dynamic(const float *x, int64_t rows, int64_t cols, int narrow, int8_t *q,
                                              float *scale, qnn_stream_t stream)
{
    using namespace qnn;
    if (rows < 0 || cols <= 0) return QNN_ERR_INVALID_ARG;
    if (cols % 4 != 0) return QNN_ERR_ALIGNMENT;
    if (rows == 0) return QNN_OK;
    if (!x || !q || !scale) return QNN_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(q) || !aligned16(scale)) return QNN_ERR_ALIGNMENT;
    // the smallest register-resident row that holds cols / 4 groups, else two passes
    const int64_t words = cols / 4;
    auto launch = [&](auto kern) {
        int per_sm = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, 256, 0) != cudaSuccess || per_sm < 1)
            per_sm = 1;
        // one wave of resident blocks, 8 rows (warps) per block
        const int grid = (int)std::max<int64_t>(1, std::min<int64_t>((rows + 7) / 8, (int64_t)sm_count() * per_sm));
        kern<<<grid, 256, 0, (cudaStream_t)stream>>>(x, rows, cols, narrow, q, scale);
    };
    if (words <= 32) launch(quantize_rows_dynamic_kernel<1>);
    else if (words <= 64) launch(quantize_rows_dynamic_kernel<2>);
    else if (words <= 128) launch(quantize_rows_dynamic_kernel<4>);
    else if (words <= 192) launch(quantize_rows_dynamic_kernel<6>);
    else if (words <= 256) launch(quantize_rows_dynamic_kernel<8>);
    else launch(quantize_rows_dynamic_kernel<0>);
    return launch_status();
}

extern "C" qnn_status q_layout_nchw64(const void *src, int to_nchw64, int N, int H, int W, int C, qnn_dtype dt,
                                      void *dst, qnn_stream_t stream)
{
    using namespace qnn;
    if (N < 0 || H <= 0 || W <= 0 || C <= 0) return QNN_ERR_INVALID_ARG;
    int bits;
    switch (dt) {
    case QNN_S4: case QNN_U4: bits = 4; break;
    case QNN_S8: case QNN_U8: bits = 8; break;
    default: return QNN_ERR_UNSUPPORTED;
    }
    if (C % 64 != 0) return QNN_ERR_ALIGNMENT;
    if (N == 0) return QNN_OK;
    if (!src || !dst) return QNN_ERR_INVALID_ARG;
    if (!aligned16(src) || !aligned16(dst)) return QNN_ERR_ALIGNMENT;
    const int cpb = bits * 64 / 8 / 16;  // 16-byte chunks per 64-channel block: 2 or 4
    const int64_t chunks = (int64_t)N * H * W * (C / 64) * cpb;
    const int grid = grid_for(chunks, 256);
    cudaStream_t s = (cudaStream_t)stream;
    if (to_nchw64)
        nchw64_kernel<true><<<grid, 256, 0, s>>>(static_cast<const uint4 *>(src), static_cast<uint4 *>(dst), chunks,
                                                  H, W, C / 64, cpb);
    else
        nchw64_kernel<false><<<grid, 256, 0, s>>>(static_cast<const uint4 *>(src), static_cast<uint4 *>(dst),
                                                   chunks, H, W, C / 64, cpb);
    return launch_status();
}
