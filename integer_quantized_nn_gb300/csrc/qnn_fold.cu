// qnn_fold.cu -- work done once per weight tensor, ahead of inference:
// prepacking the GEMM weight operand (s8; u8 centred at 128; u8 less per-row
// zero points for the u8 conv filters), the weight column sums and the folded
// epilogue constants.
//
// Folding [MG 緩解精度下降: the zero-point part that does not depend on the
// input is computed before inference; QI 量化乘法: scale_abc = s_a s_b / s_c is
// computed ahead].
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <cstdint>
#include "qnn_gemm_layout.h"
#include "qnn_internal.h"

namespace qnn {
namespace {

// One thread per 16-byte chunk of the packed image.  MODE says what B holds and
// which value of each code goes into the image:
//   kPackS8   : s8 codes, as they are;
//   kPackU8   : u8 codes, centred: w - 128 (the byte with its top bit flipped, read as s8);
//   kPackU8Zw : u8 codes less their row's zero point: w - z_w[n], in [-255, 255].
// All are integers of at most 255 in magnitude, exact in fp16.
constexpr int kPackS8 = 0, kPackU8 = 1, kPackU8Zw = 2;

template <int MODE>
__device__ __forceinline__ int packed_code(const int8_t *B, int64_t idx, const int32_t *z_w, int n)
{
    if constexpr (MODE == kPackS8) return B[idx];
    else if constexpr (MODE == kPackU8) return (int8_t)(B[idx] ^ 0x80);
    else return (int)(uint8_t)B[idx] - z_w[n];
}

template <int MODE>
__global__ void prepack_b_kernel(const int8_t *__restrict__ B, int N, int K, uint8_t *__restrict__ out,
                                 int64_t nchunks, const int32_t *__restrict__ z_w)
{
    using namespace gemm;
    const int KT = ksteps(K);
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < nchunks;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int cphys = (int)(i & 7);
        const int64_t row_all = i >> 3;           // (nb, ks, r)
        const int r = (int)(row_all % BN);
        const int64_t blk = row_all / BN;         // nb * KT + ks
        const int ks = (int)(blk % KT);
        const int nb = (int)(blk / KT);
        const int c = cphys ^ (r & 7);
        const int n = nb * BN + r;
        const int k0 = ks * BK + c * 8;
        uint32_t w[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            int v0 = 0, v1 = 0;
            if (n < N && k0 + 2 * j < K) v0 = packed_code<MODE>(B, (int64_t)n * K + k0 + 2 * j, z_w, n);
            if (n < N && k0 + 2 * j + 1 < K) v1 = packed_code<MODE>(B, (int64_t)n * K + k0 + 2 * j + 1, z_w, n);
            const uint32_t h0 = __half_as_ushort(__int2half_rn(v0));
            const uint32_t h1 = __half_as_ushort(__int2half_rn(v1));
            w[j] = h0 | (h1 << 16);
        }
        *reinterpret_cast<uint4 *>(out + i * 16) = make_uint4(w[0], w[1], w[2], w[3]);
    }
}

// One warp per output channel.
__global__ void colsum_s8_kernel(const int8_t *__restrict__ B, int N, int K, int32_t *__restrict__ colsum)
{
    const int warp = (int)((blockIdx.x * (int64_t)blockDim.x + threadIdx.x) >> 5);
    const int lane = threadIdx.x & 31;
    if (warp >= N) return;
    int32_t s = 0;
    for (int k = lane; k < K; k += 32) s += B[(int64_t)warp * K + k];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    if (lane == 0) colsum[warp] = s;
}

// u8 weights with zero points: colsum[n] = sum_k (B[n][k] - z_w[n]).  One warp per channel.
__global__ void colsum_u8_kernel(const uint8_t *__restrict__ B, const int32_t *__restrict__ z_w, int N, int K,
                                 int32_t *__restrict__ colsum)
{
    const int warp = (int)((blockIdx.x * (int64_t)blockDim.x + threadIdx.x) >> 5);
    const int lane = threadIdx.x & 31;
    if (warp >= N) return;
    int32_t s = 0;
    for (int k = lane; k < K; k += 32) s += (int32_t)B[(int64_t)warp * K + k];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    if (lane == 0) colsum[warp] = s - K * z_w[warp];
}

__global__ void fold_kernel(int N, int32_t zcoef, const int32_t *__restrict__ colsum, float s_a,
                            const float *__restrict__ s_w, int w_per_channel,
                            const float *__restrict__ bias, float s_o, int32_t *zp_term, float *M,
                            float *Bq, float *D)
{
    const int n = blockIdx.x * blockDim.x + threadIdx.x;
    if (n >= N) return;
    if (zp_term) zp_term[n] = zcoef * colsum[n];
    const float sw = s_w[w_per_channel ? n : 0];
    const float p = __fmul_rn(s_a, sw);
    if (M) M[n] = __fdiv_rn(p, s_o);
    if (Bq) Bq[n] = __fdiv_rn(bias ? bias[n] : 0.0f, s_o);
    if (D) D[n] = p;
}

}  // namespace
}  // namespace qnn

extern "C" size_t qnn_gemm_packed_b_bytes(int N, int K)
{
    if (N <= 0 || K <= 0) return 0;
    return qnn::gemm::packed_b_bytes(N, K);
}

extern "C" qnn_status qgemm_prepack_b(const int8_t *B, int N, int K, void *B_packed, int32_t *colsum,
                                      qnn_stream_t stream)
{
    if (!B || !B_packed || N <= 0 || K <= 0) return QNN_ERR_INVALID_ARG;
    if (K % 16 != 0) return QNN_ERR_ALIGNMENT;
    if ((reinterpret_cast<uintptr_t>(B_packed) & 1023u) != 0) return QNN_ERR_ALIGNMENT;
    if (!qnn::aligned16(B)) return QNN_ERR_ALIGNMENT;
    const int64_t nchunks = (int64_t)(qnn::gemm::packed_b_bytes(N, K) / 16);
    int64_t blocks = (nchunks + 255) / 256;
    if (blocks > 65535) blocks = 65535;
    cudaStream_t s = (cudaStream_t)stream;
    qnn::prepack_b_kernel<qnn::kPackS8><<<(int)blocks, 256, 0, s>>>(B, N, K, static_cast<uint8_t *>(B_packed),
                                                                     nchunks, nullptr);
    if (qnn::launch_status() != QNN_OK) return QNN_ERR_CUDA;
    if (colsum) {
        const int64_t threads = (int64_t)N * 32;
        qnn::colsum_s8_kernel<<<(int)((threads + 255) / 256), 256, 0, s>>>(B, N, K, colsum);
        return qnn::launch_status();
    }
    return QNN_OK;
}

extern "C" qnn_status qgemm_prepack_b_u8(const uint8_t *B, const int32_t *z_w, int N, int K, void *B_packed,
                                         int32_t *colsum, qnn_stream_t stream)
{
    if (!B || !B_packed || !z_w || N <= 0 || K <= 0) return QNN_ERR_INVALID_ARG;
    if (K % 16 != 0) return QNN_ERR_ALIGNMENT;
    if ((reinterpret_cast<uintptr_t>(B_packed) & 1023u) != 0) return QNN_ERR_ALIGNMENT;
    if (!qnn::aligned16(B) || !qnn::aligned16(z_w)) return QNN_ERR_ALIGNMENT;
    const int64_t nchunks = (int64_t)(qnn::gemm::packed_b_bytes(N, K) / 16);
    int64_t blocks = (nchunks + 255) / 256;
    if (blocks > 65535) blocks = 65535;
    cudaStream_t s = (cudaStream_t)stream;
    qnn::prepack_b_kernel<qnn::kPackU8><<<(int)blocks, 256, 0, s>>>(reinterpret_cast<const int8_t *>(B), N, K,
                                                                     static_cast<uint8_t *>(B_packed), nchunks,
                                                                     nullptr);
    if (qnn::launch_status() != QNN_OK) return QNN_ERR_CUDA;
    if (colsum) {
        const int64_t threads = (int64_t)N * 32;
        qnn::colsum_u8_kernel<<<(int)((threads + 255) / 256), 256, 0, s>>>(B, z_w, N, K, colsum);
        return qnn::launch_status();
    }
    return QNN_OK;
}

namespace qnn {
// The u8 conv filters [OC, K] with per-filter zero points: image of w - z_w[n]
// and colsum[n] = sum_k (w - z_w[n]).  Arguments checked by the caller.
qnn_status prepack_b_u8_minus_zw(const uint8_t *B, const int32_t *z_w, int N, int K, void *B_packed,
                                 int32_t *colsum, cudaStream_t s)
{
    const int64_t nchunks = (int64_t)(gemm::packed_b_bytes(N, K) / 16);
    int64_t blocks = (nchunks + 255) / 256;
    if (blocks > 65535) blocks = 65535;
    prepack_b_kernel<kPackU8Zw><<<(int)blocks, 256, 0, s>>>(reinterpret_cast<const int8_t *>(B), N, K,
                                                            static_cast<uint8_t *>(B_packed), nchunks, z_w);
    if (launch_status() != QNN_OK) return QNN_ERR_CUDA;
    if (colsum) {
        const int64_t threads = (int64_t)N * 32;
        colsum_u8_kernel<<<(int)((threads + 255) / 256), 256, 0, s>>>(B, z_w, N, K, colsum);
        return launch_status();
    }
    return QNN_OK;
}
}  // namespace qnn

extern "C" qnn_status q_fold_epilogue(int N, qnn_dtype a_dt, int32_t z_a, const int32_t *colsum,
                                      float s_a, const float *s_w, int w_per_channel,
                                      const float *bias, float s_o, int32_t *zp_term, float *M,
                                      float *Bq, float *D, qnn_stream_t stream)
{
    if (N <= 0 || !s_w) return QNN_ERR_INVALID_ARG;
    if (zp_term && !colsum) return QNN_ERR_INVALID_ARG;
    int32_t centre;
    switch (a_dt) {
    case QNN_U8: centre = 128; break;
    case QNN_S8: case QNN_U4: case QNN_S4: centre = 0; break;
    default: return QNN_ERR_INVALID_ARG;
    }
    int32_t lo, hi;
    qnn::qrange(a_dt, 0, &lo, &hi);
    if (z_a < lo || z_a > hi) return QNN_ERR_INVALID_ARG;
    if (!(s_o > 0.0f)) return QNN_ERR_INVALID_ARG;
    qnn::fold_kernel<<<(N + 255) / 256, 256, 0, (cudaStream_t)stream>>>(
        N, z_a - centre, colsum, s_a, s_w, w_per_channel, bias, s_o, zp_term, M, Bq, D);
    return qnn::launch_status();
}
