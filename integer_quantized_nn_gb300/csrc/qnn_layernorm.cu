// qnn_layernorm.cu -- q_int_layernorm: integer LayerNorm over PTF-quantized rows.
//
// [FQ] "首个完全量化Vision Transformer的方法FQ-ViT" (aijishu.com), section 3.2
// (LayerNorm 的量化推理, LayerNorm 的量化实现): the LayerNorm input is quantized
// with one layer scale s and per-channel power-of-two factors 2^alpha; the row
// statistics come from the shifted integer codes x' = x 2^alpha, and each
// output is an integer multiply-add and a rounding shift:
//   mean = (sum x' / C) s,  std = (s / C) sqrt(C sum x'^2 - (sum x')^2)
//   A = (s / std) gamma / o,  N = clamp(7 - floor(log2 |A|), 0, 31),
//   M = clamp(floor(|A| 2^N), 0, 255),  B = round((beta - (mean / std) gamma) / o 2^N)
//   y = round((sign(A) M x' + B) / 2^N)
// The integer sums and the variance numerator are exact; the float steps are
// single IEEE fp32 operations in that order; both roundings are half to even.
//
// One warp per row, a grid-stride loop over rows.  Pass 1 reads the row as
// 4-byte words (4 codes per lane and step), shifts by alpha and reduces sum x'
// and sum x'^2 with warp reductions; one lane's worth of fp32 work gives the row
// constants; pass 2 re-reads the row (from cache) with the per-channel gamma,
// beta, o and alpha (vector loads), forms the four channels' A, N, M and B
// without branches, and takes the 32-bit rounding shift when all four fit (the
// 64-bit one only for extreme constants); 4 outputs per step.  The op is bound
// by instruction issue (two IEEE divisions per element among them), not bytes.
#include <cuda_runtime.h>
#include <algorithm>
#include <cstdint>
#include "qnn_internal.h"

namespace qnn {
namespace {

constexpr unsigned kFull = 0xffffffffu;
constexpr int kLnWarps = 8;

struct LnArgs {
    const int8_t *x;
    const uint8_t *alpha;  // [C] or nullptr
    const float *gamma, *beta, *o;
    void *y;
    int64_t rows;
    int C;
    float s;
};

__device__ __forceinline__ int64_t round_shift_he(int64_t num, int N)
{
    if (N == 0) return num;
    const int64_t q = num >> N;
    const int64_t rem = num - (q << N);
    const int64_t half = 1ll << (N - 1);
    return (rem > half || (rem == half && (q & 1))) ? q + 1 : q;
}

__device__ __forceinline__ float pow2f(int n) { return __int_as_float((n + 127) << 23); }

template <bool S8>
__global__ void __launch_bounds__(kLnWarps * 32) int_layernorm_kernel(const __grid_constant__ LnArgs a)
{
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const int words = a.C >> 2;
    for (int64_t row = (int64_t)blockIdx.x * kLnWarps + w; row < a.rows; row += (int64_t)gridDim.x * kLnWarps) {
        const uint32_t *xr = reinterpret_cast<const uint32_t *>(a.x + row * a.C);
        int32_t sum = 0;
        uint32_t sum2 = 0;
        for (int k = lane; k < words; k += 32) {
            const uint32_t xw = __ldg(xr + k);
            const uint32_t aw = a.alpha ? __ldg(reinterpret_cast<const uint32_t *>(a.alpha) + k) : 0u;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int32_t v = (int32_t)(int8_t)(xw >> (8 * q)) * (1 << ((aw >> (8 * q)) & 0xffu));
                sum += v;
                sum2 += (uint32_t)(v * v);
            }
        }
        sum = __reduce_add_sync(kFull, sum);
        sum2 = __reduce_add_sync(kFull, sum2);
        const int64_t var_num = (int64_t)a.C * (int64_t)sum2 - (int64_t)sum * (int64_t)sum;
        const float Cf = (float)a.C;
        const float mean = __fmul_rn(__fdiv_rn((float)sum, Cf), a.s);
        const float stdv = __fmul_rn(__fdiv_rn(a.s, Cf), __fsqrt_rn(__ll2float_rn(var_num)));
        const float sos = __fdiv_rn(a.s, stdv);
        const float mos = __fdiv_rn(mean, stdv);
#pragma unroll 2
        for (int k = lane; k < words; k += 32) {
            const uint32_t xw = __ldg(xr + k);
            const uint32_t aw = a.alpha ? __ldg(reinterpret_cast<const uint32_t *>(a.alpha) + k) : 0u;
            const float4 g4 = __ldg(reinterpret_cast<const float4 *>(a.gamma) + k);
            const float4 b4 = __ldg(reinterpret_cast<const float4 *>(a.beta) + k);
            const float4 o4 = __ldg(reinterpret_cast<const float4 *>(a.o) + k);
            const float gs[4] = {g4.x, g4.y, g4.z, g4.w}, bs[4] = {b4.x, b4.y, b4.z, b4.w},
                        os[4] = {o4.x, o4.y, o4.z, o4.w};
            // the four channels' constants first, straight-line, then one test for the
            // 32-bit form of the rounding shift (|M x'| < 2^18, |B| < 2^30, N <= 30)
            int32_t v[4], M[4], N[4];  // M signed: sign(A) M
            float bt[4];               // B before rounding
            bool fits = true;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                v[q] = (int32_t)(int8_t)(xw >> (8 * q)) * (1 << ((aw >> (8 * q)) & 0xffu));
                if (var_num == 0) {
                    M[q] = 0;
                    N[q] = 0;
                    bt[q] = __fdiv_rn(bs[q], os[q]);
                } else {
                    const float A = __fdiv_rn(__fmul_rn(sos, gs[q]), os[q]);
                    const float am = fabsf(A);
                    // 7 - floor(log2 am) from the biased exponent: 0 (zero or subnormal)
                    // clamps to 31, 255 (infinite) to 0
                    const int ex = (__float_as_int(am) >> 23) & 0xff;
                    N[q] = min(max(134 - ex, 0), 31);
                    const int32_t m = min(__float2int_rd(fminf(__fmul_rn(am, pow2f(N[q])), 256.0f)), 255);
                    M[q] = A < 0.0f ? -m : m;
                    const float t = __fdiv_rn(__fsub_rn(bs[q], __fmul_rn(mos, gs[q])), os[q]);
                    bt[q] = __fmul_rn(t, pow2f(N[q]));
                }
                fits = fits && fabsf(bt[q]) < 1073741824.0f && N[q] <= 30;
            }
            int32_t yv[4];
            if (fits) {
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    // half-even division by 2^N: floor((num + 2^(N-1) - 1 + (quotient & 1)) / 2^N)
                    const int32_t num = M[q] * v[q] + __float2int_rn(bt[q]);
                    const int32_t bias = ((1 << N[q]) >> 1) - 1 + ((num >> N[q]) & 1);
                    yv[q] = N[q] == 0 ? num : (num + bias) >> N[q];
                }
            } else {
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const float lim = 4611686018427387904.0f;  // 2^62: B is rounded after this clamp
                    const int64_t B = __float2ll_rn(fminf(fmaxf(bt[q], -lim), lim));
                    const int64_t y64 = round_shift_he((int64_t)M[q] * v[q] + B, N[q]);
                    yv[q] = (int32_t)min(max(y64, (int64_t)INT32_MIN), (int64_t)INT32_MAX);
                }
            }
            if constexpr (S8) {
                uint32_t ow = 0;
#pragma unroll
                for (int q = 0; q < 4; ++q) ow |= ((uint32_t)(uint8_t)(int8_t)min(max(yv[q], -128), 127)) << (8 * q);
                reinterpret_cast<uint32_t *>(a.y)[row * words + k] = ow;
            } else {
                reinterpret_cast<int4 *>(a.y)[row * words + k] = make_int4(yv[0], yv[1], yv[2], yv[3]);
            }
        }
    }
}

}  // namespace
}  // namespace qnn

extern "C" qnn_status q_int_layernorm(const int8_t *x, int64_t rows, int C, const uint8_t *alpha, int alpha_max,
                                      float s, const float *gamma, const float *beta, const float *out_scale,
                                      qnn_dtype y_dt, void *y, qnn_stream_t stream)
{
    using namespace qnn;
    if (rows < 0 || C <= 0 || alpha_max < 0 || alpha_max > 3) return QNN_ERR_INVALID_ARG;
    if (!(s > 0.0f) || !(s < INFINITY)) return QNN_ERR_INVALID_ARG;
    if (y_dt != QNN_S8 && y_dt != QNN_S32) return QNN_ERR_UNSUPPORTED;
    if (C % 4 != 0) return QNN_ERR_ALIGNMENT;
    // sum x'^2 <= C (128 2^alpha_max)^2 must fit 32 bits
    if ((uint64_t)C * (uint64_t)(128u << alpha_max) * (uint64_t)(128u << alpha_max) >= (1ull << 32))
        return QNN_ERR_OVERFLOW_RISK;
    if (rows == 0) return QNN_OK;
    if (!x || !gamma || !beta || !out_scale || !y) return QNN_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(gamma) || !aligned16(beta) || !aligned16(out_scale) || !aligned16(y) ||
        (alpha && !aligned16(alpha)))
        return QNN_ERR_ALIGNMENT;
    LnArgs a{x, alpha, gamma, beta, out_scale, y, rows, C, s};
    const int64_t want = (rows + kLnWarps - 1) / kLnWarps;
    cudaStream_t st = (cudaStream_t)stream;
    // one wave of resident blocks (the grid-stride loop covers the rest)
    auto launch = [&](auto kern) {
        int per_sm = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kLnWarps * 32, 0) != cudaSuccess ||
            per_sm < 1)
            per_sm = 1;
        const int grid = (int)std::min<int64_t>(want, (int64_t)sm_count() * per_sm);
        kern<<<grid, kLnWarps * 32, 0, st>>>(a);
    };
    if (y_dt == QNN_S8) launch(int_layernorm_kernel<true>);
    else launch(int_layernorm_kernel<false>);
    return launch_status();
}
