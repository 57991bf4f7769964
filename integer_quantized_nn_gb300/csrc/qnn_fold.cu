// qnn_fold.cu -- work done once per weight tensor, ahead of inference:
// prepacking the GEMM weight operand (s8; u8 centred at 128; u8 less per-row
// zero points for the u8 conv filters; s8 times per-input-channel
// Power-of-Two Factors), its trailer of magnitude bounds, the weight column
// sums and the folded epilogue constants.
//
// Folding [MG 緩解精度下降: the zero-point part that does not depend on the
// input is computed before inference; QI 量化乘法: scale_abc = s_a s_b / s_c is
// computed ahead].
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <cstdint>
#include "qnn_gemm_layout.h"
#include "qnn_internal.h"
#include "qnn_ptx.cuh"

namespace qnn {
namespace {

// What B holds and which value of each code goes into the image (MODE):
//   kPackS8   : s8 codes, as they are;
//   kPackU8   : u8 codes, centred: w - 128 (the byte with its top bit flipped, read as s8);
//   kPackU8Zw : u8 codes less their row's zero point: w - z_w[n], in [-255, 255];
//   kPackPtf  : s8 codes times the Power-of-Two Factor of their input channel,
//               w * 2^alpha[k] [FQ 3.2: the activation codes are multiplied by
//               2^alpha before the product; the factor is moved onto the
//               constant operand, sum_k (a_k 2^alpha_k) w_k = sum_k a_k (w_k 2^alpha_k)],
//               |w 2^alpha| <= 1024 for alpha <= 3.
// All are integers of at most 2048 in magnitude, exact in fp16.
constexpr int kPackS8 = 0, kPackU8 = 1, kPackU8Zw = 2, kPackPtf = 3;

struct PackSrc {
    const int8_t *B;       // [N, K] codes
    const int32_t *z_w;    // kPackU8Zw: [N]
    const uint8_t *ptf;    // kPackPtf: [K] shifts (validated by trailer_kernel; 0..3)
    int N, K;
};

template <int MODE>
__device__ __forceinline__ int packed_code(const PackSrc &s, int n, int k)
{
    const int64_t idx = (int64_t)n * s.K + k;
    if constexpr (MODE == kPackS8) return s.B[idx];
    else if constexpr (MODE == kPackU8) return (int8_t)(s.B[idx] ^ 0x80);
    else if constexpr (MODE == kPackU8Zw) return (int)(uint8_t)s.B[idx] - s.z_w[n];
    else return (int)s.B[idx] * (1 << (s.ptf[k] & 15u));
}

// One thread per 16-byte chunk of the packed image.
template <int MODE>
__global__ void prepack_b_kernel(const PackSrc src, uint8_t *__restrict__ out, int64_t nchunks)
{
    using namespace gemm;
    const int N = src.N, K = src.K;
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
            if (n < N && k0 + 2 * j < K) v0 = packed_code<MODE>(src, n, k0 + 2 * j);
            if (n < N && k0 + 2 * j + 1 < K) v1 = packed_code<MODE>(src, n, k0 + 2 * j + 1);
            const uint32_t h0 = __half_as_ushort(__int2half_rn(v0));
            const uint32_t h1 = __half_as_ushort(__int2half_rn(v1));
            w[j] = h0 | (h1 << 16);
        }
        *reinterpret_cast<uint4 *>(out + i * 16) = make_uint4(w[0], w[1], w[2], w[3]);
    }
}

__device__ __forceinline__ int warp_sum(int v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// The image's trailer (zeroed beforehand): one warp per column n forms the sum
// of |value| over each K step of 64 and over all of K, and folds them into the
// trailer's maxima.  With kPackPtf, warp 0 also records the largest shift and
// flags shifts above 3 (device status word: invalid argument).
template <int MODE>
__global__ void trailer_kernel(const PackSrc src, int32_t *__restrict__ tr, uint32_t *status)
{
    using namespace gemm;
    const int warp = (int)((blockIdx.x * (int64_t)blockDim.x + threadIdx.x) >> 5);
    const int lane = threadIdx.x & 31;
    const int KT = ksteps(src.K);
    if (warp == 0) {
        if (MODE == kPackPtf) {
            int amax = 0;
            for (int k = lane; k < src.K; k += 32) amax = max(amax, (int)src.ptf[k]);
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) amax = max(amax, __shfl_xor_sync(0xffffffffu, amax, o));
            if (lane == 0) {
                if (amax > 3 && status) atomicOr(status, kStatusBadArg);
                atomicMax(tr + TR_SHIFT_MAX, amax);
            }
        }
        if (lane == 0) {
            tr[TR_MAGIC] = TRAILER_MAGIC;
            tr[TR_KT] = KT;
        }
    }
    if (warp >= src.N) return;
    int32_t smax = 0;
    int64_t tot = 0;
    for (int s = 0; s < KT; ++s) {
        int v = 0;
        for (int j = lane; j < BK; j += 32) {
            const int k = s * BK + j;
            if (k < src.K) v += abs(packed_code<MODE>(src, warp, k));
        }
        v = warp_sum(v);
        smax = max(smax, v);
        tot += v;
    }
    if (lane == 0) {
        atomicMax(tr + TR_STEP_MAX, smax);
        atomicMax(tr + TR_TOTAL_MAX, (int32_t)(tot < INT32_MAX ? tot : INT32_MAX));
    }
}

// colsum[n] = sum_k of the image values.  One warp per output channel.
template <int MODE>
__global__ void colsum_code_kernel(const PackSrc src, int32_t *__restrict__ colsum)
{
    const int warp = (int)((blockIdx.x * (int64_t)blockDim.x + threadIdx.x) >> 5);
    const int lane = threadIdx.x & 31;
    if (warp >= src.N) return;
    int32_t s = 0;
    for (int k = lane; k < src.K; k += 32) s += packed_code<MODE>(src, warp, k);
    s = warp_sum(s);
    if (lane == 0) colsum[warp] = s;
}

// Image, then trailer, of B in the form MODE on stream s.
template <int MODE>
qnn_status pack_b(const PackSrc &src, void *B_packed, cudaStream_t s)
{
    const int64_t nchunks = (int64_t)(gemm::packed_b_image_bytes(src.N, src.K) / 16);
    int64_t blocks = (nchunks + 255) / 256;
    if (blocks > 65535) blocks = 65535;
    uint8_t *out = static_cast<uint8_t *>(B_packed);
    prepack_b_kernel<MODE><<<(int)blocks, 256, 0, s>>>(src, out, nchunks);
    if (launch_status() != QNN_OK) return QNN_ERR_CUDA;
    int32_t *tr = reinterpret_cast<int32_t *>(out + gemm::packed_b_image_bytes(src.N, src.K));
    if (cudaMemsetAsync(tr, 0, gemm::TRAILER_BYTES, s) != cudaSuccess) return QNN_ERR_CUDA;
    const int64_t threads = (int64_t)src.N * 32;
    trailer_kernel<MODE><<<(int)((threads + 255) / 256), 256, 0, s>>>(src, tr, status_word());
    return launch_status();
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
    cudaStream_t s = (cudaStream_t)stream;
    const qnn::PackSrc src{B, nullptr, nullptr, N, K};
    qnn_status st = qnn::pack_b<qnn::kPackS8>(src, B_packed, s);
    if (st != QNN_OK || !colsum) return st;
    const int64_t threads = (int64_t)N * 32;
    qnn::colsum_code_kernel<qnn::kPackS8><<<(int)((threads + 255) / 256), 256, 0, s>>>(src, colsum);
    return qnn::launch_status();
}

extern "C" qnn_status qgemm_prepack_b_ptf(const int8_t *B, const uint8_t *ptf_shift, int N, int K, void *B_packed,
                                          int32_t *colsum, qnn_stream_t stream)
{
    if (!B || !ptf_shift || !B_packed || N <= 0 || K <= 0) return QNN_ERR_INVALID_ARG;
    if (K % 16 != 0) return QNN_ERR_ALIGNMENT;
    if ((reinterpret_cast<uintptr_t>(B_packed) & 1023u) != 0) return QNN_ERR_ALIGNMENT;
    if (!qnn::aligned16(B) || !qnn::aligned16(ptf_shift)) return QNN_ERR_ALIGNMENT;
    cudaStream_t s = (cudaStream_t)stream;
    const qnn::PackSrc src{B, nullptr, ptf_shift, N, K};
    qnn_status st = qnn::pack_b<qnn::kPackPtf>(src, B_packed, s);
    if (st != QNN_OK || !colsum) return st;
    const int64_t threads = (int64_t)N * 32;
    qnn::colsum_code_kernel<qnn::kPackPtf><<<(int)((threads + 255) / 256), 256, 0, s>>>(src, colsum);
    return qnn::launch_status();
}

extern "C" qnn_status qgemm_prepack_b_u8(const uint8_t *B, const int32_t *z_w, int N, int K, void *B_packed,
                                         int32_t *colsum, qnn_stream_t stream)
{
    if (!B || !B_packed || !z_w || N <= 0 || K <= 0) return QNN_ERR_INVALID_ARG;
    if (K % 16 != 0) return QNN_ERR_ALIGNMENT;
    if ((reinterpret_cast<uintptr_t>(B_packed) & 1023u) != 0) return QNN_ERR_ALIGNMENT;
    if (!qnn::aligned16(B) || !qnn::aligned16(z_w)) return QNN_ERR_ALIGNMENT;
    cudaStream_t s = (cudaStream_t)stream;
    const qnn::PackSrc src{reinterpret_cast<const int8_t *>(B), z_w, nullptr, N, K};
    qnn_status st = qnn::pack_b<qnn::kPackU8>(src, B_packed, s);
    if (st != QNN_OK || !colsum) return st;
    const int64_t threads = (int64_t)N * 32;
    qnn::colsum_u8_kernel<<<(int)((threads + 255) / 256), 256, 0, s>>>(B, z_w, N, K, colsum);
    return qnn::launch_status();
}

namespace qnn {
// The u8 conv filters [OC, K] with per-filter zero points: image of w - z_w[n]
// and colsum[n] = sum_k (w - z_w[n]).  Arguments checked by the caller.
qnn_status prepack_b_u8_minus_zw(const uint8_t *B, const int32_t *z_w, int N, int K, void *B_packed,
                                 int32_t *colsum, cudaStream_t s)
{
    const PackSrc src{reinterpret_cast<const int8_t *>(B), z_w, nullptr, N, K};
    qnn_status st = pack_b<kPackU8Zw>(src, B_packed, s);
    if (st != QNN_OK || !colsum) return st;
    const int64_t threads = (int64_t)N * 32;
    colsum_u8_kernel<<<(int)((threads + 255) / 256), 256, 0, s>>>(B, z_w, N, K, colsum);
    return launch_status();
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
