// qnn_gemm_layout.h -- tile geometry of the quantized GEMM kernel and of its
// prepacked weight operand (shared by the prepack and the GEMM kernel).
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

namespace qnn {
namespace gemm {

constexpr int BM = 128;           // rows of A per tile (TMEM lanes)
constexpr int BN = 256;           // output columns per tile (MMA N)
constexpr int BK = 64;            // K per pipeline stage: 64 fp16 = one 128-byte swizzle row
constexpr int ROW_BYTES = BK * 2; // bytes per operand row per stage
constexpr int A_STAGE_BYTES = BM * ROW_BYTES;  // 16 KB
constexpr int B_STAGE_BYTES = BN * ROW_BYTES;  // 32 KB

// Longest run of K-steps whose fp32 partial sums stay exact integers: with
// |a| <= 128 and |b| <= 128 a product is at most 2^14 and 16 steps of 64
// products reach at most 2^24.
constexpr int MAX_EXACT_STEPS = 16;

__host__ __device__ inline int ksteps(int K) { return (K + BK - 1) / BK; }
__host__ __device__ inline int ntiles(int N) { return (N + BN - 1) / BN; }

// Prepacked B: for each 256-column block nb and K-step ks, a contiguous
// BN x 128-byte image of fp16 values in the 128-byte swizzled K-major layout
// (chunk c of row r at chunk c ^ (r % 8)); zero beyond N and K.  A trailer of
// TRAILER_BYTES follows the image: the magnitude bounds of the values written
// (below), from which the GEMM derives how many K steps its fp32 partial sums
// can take exactly.
inline size_t packed_b_image_bytes(int N, int K)
{
    return (size_t)ntiles(N) * (size_t)ksteps(K) * (size_t)B_STAGE_BYTES;
}

constexpr int TRAILER_BYTES = 1024;
constexpr int32_t TRAILER_MAGIC = 0x31424E51;  // "QNB1"
// int32 words of the trailer
enum {
    TR_MAGIC = 0,       // TRAILER_MAGIC once the prepack has written the trailer
    TR_KT = 1,          // K steps of the image
    TR_STEP_MAX = 2,    // max over columns n and K steps s of sum_{k in s} |w'[n][k]|
    TR_TOTAL_MAX = 3,   // max over columns n of sum_k |w'[n][k]|
    TR_SHIFT_MAX = 4,   // largest Power-of-Two-Factor shift folded into the values (0: none)
};

inline size_t packed_b_bytes(int N, int K)
{
    return packed_b_image_bytes(N, K) + TRAILER_BYTES;
}

// Largest number of consecutive K steps whose fp32 partial sums of products
// a * w' stay exact integers (magnitude <= 2^24) for every activation code with
// |a| <= amax, given the trailer bounds: every K when the whole column sum
// allows it, else 2^24 / (amax * step_max) steps (at least 1).
__host__ __device__ inline int certified_chunk_steps(int32_t step_max, int32_t total_max, int64_t amax, int KT)
{
    const int64_t lim = (int64_t)1 << 24;
    if ((int64_t)total_max * amax <= lim) return KT;
    const int64_t l = lim / ((int64_t)step_max * amax);
    return l < 1 ? 1 : (l > KT ? KT : (int)l);
}

}  // namespace gemm
}  // namespace qnn
