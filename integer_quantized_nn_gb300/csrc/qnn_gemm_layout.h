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
// (chunk c of row r at chunk c ^ (r % 8)); zero beyond N and K.
inline size_t packed_b_bytes(int N, int K)
{
    return (size_t)ntiles(N) * (size_t)ksteps(K) * (size_t)B_STAGE_BYTES;
}

}  // namespace gemm
}  // namespace qnn
