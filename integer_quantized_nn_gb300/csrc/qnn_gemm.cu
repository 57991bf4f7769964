// qnn_gemm.cu -- qgemm_s8: quantized GEMM with a fused requantizing /
// dequantizing epilogue on the sm_103a tensor cores.
//
// Computes [QI 量化矩阵乘: int8 inputs, wide products, int32 sums, requantize;
// MG 緩解精度下降: the zero-point part folded ahead of inference]
//     acc[m][n] = sum_k (A[m][k] - c_a) * 2^alpha_k * B[n][k]          (exact)
//     acc_c     = acc - zp_term[n]
// then the REQUANT / DEQUANT / S32 epilogue of qnn.h.
//
// sm_103a has no integer tcgen05 MMA, so the product runs exactly on the fp16
// one: every int8 code (and every PTF-shifted code, |a 2^alpha| <= 1024) is an
// exact fp16 value, every product is exact in fp32, and an fp32 sum of
// integers is exact while its magnitude stays <= 2^24.  The K loop is cut into
// chunks whose partial sums provably stay within 2^24: by default (16 >>
// ptf_max_shift) steps of 64, or longer as the prepack's trailer certifies from
// the weight values actually stored (qnn_gemm_layout.h); each chunk
// accumulates in its own TMEM buffer and the epilogue warps add the chunk
// results in int32.  A u8 operand is read as (q - 128) so that every
// operand is in [-128, 127]; the fold puts the 128 back through zp_term.
// The kernel itself is qnn_mma_kernel.cuh; this file holds the converter of
// the A rows, the A pre-pass and the host entry point.
//
// With a workspace, A is re-encoded once by a memory-bound pre-pass into the
// fp16 operand image (the same swizzled layout as the weights) and the GEMM
// kernel streams both operands with bulk copies; without one, converter warps
// re-encode A inside the GEMM kernel for every output-column tile.
#include <atomic>
#include "qnn_mma_kernel.cuh"

namespace qnn {
namespace mk {

// Whether any of 16 shift bytes exceeds `bound` (the host's ptf_max_shift, on
// which the exact-chunk length rests).
__device__ __forceinline__ bool ptf_bytes_above(uint4 a, uint32_t bound)
{
    const uint32_t b4 = bound * 0x01010101u;
    return (__vcmpgtu4(a.x, b4) | __vcmpgtu4(a.y, b4) | __vcmpgtu4(a.z, b4) | __vcmpgtu4(a.w, b4)) != 0u;
}

// fp16x2 multipliers 2^alpha for the two alpha bytes selected by `sel`.
__device__ __forceinline__ uint32_t pow2_half2(uint32_t alpha4, uint32_t sel)
{
    return (prmt(alpha4, 0u, sel) << 10) + 0x3C003C00u;
}

// 16 int8 / uint8 codes -> 16 fp16 values (q - 128 for u8, q for s8): each
// byte goes into the low mantissa bits of fp16 1024, then 1024 + 128 is
// subtracted (s8 codes are first flipped to offset binary).  Exact.
__device__ __forceinline__ void bytes_to_half(uint4 v, uint32_t flip, uint32_t (&h)[8])
{
    const uint32_t w[4] = {v.x ^ flip, v.y ^ flip, v.z ^ flip, v.w ^ flip};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        h[2 * i] = hsub2_u32(prmt(w[i], 0x64646464u, 0x4140u), 0x64806480u);
        h[2 * i + 1] = hsub2_u32(prmt(w[i], 0x64646464u, 0x4342u), 0x64806480u);
    }
}

template <bool PTF>
struct GemmOp : OpBase {
    static constexpr bool TMA_A = false;
    static constexpr bool F8 = false;
    static constexpr int SCALE_LOG2 = 0;
    static constexpr int DEPTH = 4;        // units of A rows in flight, in registers
    static constexpr int DEPTH_MULTI = 3;
    static constexpr int STG_BYTES = 16;   // no staging ring
    static constexpr bool REG_RING = true;
    struct Unit {
        uint4 v[4];
        uint4 alpha;
    };
    struct State {
        UnitCursor c;
    };

    // Units are loaded in order, one call each; the cursor follows them.
    template <int D>
    __device__ static void load(const Params &p, State &st, const uint4 *, int j, bool valid, int sub,
                                int rbase, Unit &u)
    {
        if (!valid) return;
        if (j == 0) st.c.begin(p);
        else st.c.next(p);
        const int m0 = st.c.mb * BM;
        const int k0 = st.c.ks * 64 + sub * 16;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int m = m0 + q * 32 + rbase;
            if (m < p.M && k0 < p.K)
                u.v[q] = ldg_nc_v4(p.A + (int64_t)m * p.K + k0);
            else
                u.v[q] = make_uint4(0, 0, 0, 0);
        }
        if (PTF) u.alpha = (k0 < p.K) ? ldg_nc_v4(p.ptf + k0) : make_uint4(0, 0, 0, 0);
    }

    template <int D>
    __device__ static void store(const Params &p, State &, const uint4 *, uint32_t a_stage, int, int sub,
                                 int rbase, const Unit &u)
    {
        const uint32_t flip = p.a_u8 ? 0u : 0x80808080u;
        uint32_t mul[8];
        if (PTF) {
            const uint32_t al[4] = {u.alpha.x, u.alpha.y, u.alpha.z, u.alpha.w};
            if (ptf_bytes_above(u.alpha, (uint32_t)p.ptf_max)) atomicOr(p.status, kStatusBadArg);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                mul[2 * i] = pow2_half2(al[i], 0x4140u);
                mul[2 * i + 1] = pow2_half2(al[i], 0x4342u);
            }
        }
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int row = q * 32 + rbase;
            uint32_t h[8];
            bytes_to_half(u.v[q], flip, h);
            if (PTF) {
#pragma unroll
                for (int i = 0; i < 8; ++i) h[i] = hmul2_u32(h[i], mul[i]);
            }
            const uint32_t rowaddr = a_stage + row * ROW_BYTES;
            sts_v4(rowaddr + (((2 * sub) ^ (row & 7)) << 4), h[0], h[1], h[2], h[3]);
            sts_v4(rowaddr + (((2 * sub + 1) ^ (row & 7)) << 4), h[4], h[5], h[6], h[7]);
        }
    }
};

// A operand already in the fp16 image: the producer copies it.
struct GemmPackedOp : OpBase {
    static constexpr bool TMA_A = true;
    static constexpr bool F8 = false;
    static constexpr int SCALE_LOG2 = 0;
    static constexpr int STG_BYTES = 16;
    __device__ static uint32_t a_bytes(const Params &) { return A_STAGE_BYTES; }
    __device__ static void load_a(const Params &p, const UnitCursor &c, PState &, int, uint32_t dst, uint32_t bar)
    {
        bulk_g2s(dst, p.Ap + ((int64_t)c.mb * p.KT + c.ks) * A_STAGE_BYTES, A_STAGE_BYTES, bar);
    }
};

// Pre-pass: A [M, K] (s8, or u8 read as q - 128; times 2^alpha_k with PTF)
// -> fp16 image [num_m][KT][128 rows][128 B], chunk c of row r at chunk
// c ^ (r % 8), zero beyond M and K.  A thread converts 16 codes (two chunks):
// threadIdx.x walks the 16-code groups of a row (coalesced 16-byte reads; four
// consecutive threads fill one 128-byte image row), threadIdx.y and the grid's
// y dimension walk the rows.  All index arithmetic is 32-bit.
// ROWSUM: also accumulate rowsum[m] += sum of the row's centred codes (a - 128 for
// u8, a for s8) -- the per-row factor of a weight zero point's term; rowsum
// must be zero on entry.  Lanes holding the same row combine their 16-code
// partial sums with one warp reduction before a single atomic add.
template <bool PTF, bool ROWSUM>
__global__ void __launch_bounds__(256) pack_a_kernel(const uint8_t *__restrict__ A, int M, int K, int KT,
                                                     int rows_pad, int a_u8, const uint8_t *__restrict__ ptf,
                                                     uint8_t *__restrict__ out, int32_t *__restrict__ rowsum,
                                                     int ptf_max, uint32_t *status)
{
    const int groups = KT * 4;  // 16-code groups per padded row
    const int g = blockIdx.x * blockDim.x + threadIdx.x;
    if (g >= groups) return;
    const int k0 = g * 16;
    const uint32_t flip = a_u8 ? 0u : 0x80808080u;
    uint32_t mul[8];
    if (PTF) {
        const uint4 al = (k0 < K) ? ldg_nc_v4(ptf + k0) : make_uint4(0, 0, 0, 0);
        if (blockIdx.y == 0 && threadIdx.y == 0 && ptf_bytes_above(al, (uint32_t)ptf_max)) atomicOr(status, kStatusBadArg);
        const uint32_t a4[4] = {al.x, al.y, al.z, al.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            mul[2 * j] = pow2_half2(a4[j], 0x4140u);
            mul[2 * j + 1] = pow2_half2(a4[j], 0x4342u);
        }
    }
    const int ks = g >> 2;
    const int c = (g & 3) * 2;
    const int stride = gridDim.y * blockDim.y;
    // two rows per iteration, both loads issued before either is converted
    for (int m = blockIdx.y * blockDim.y + threadIdx.y; m < rows_pad; m += 2 * stride) {
        const int mr[2] = {m, m + stride};
        uint4 v[2];
#pragma unroll
        for (int e = 0; e < 2; ++e)
            v[e] = (mr[e] < M && k0 < K) ? ldg_nc_v4(A + (size_t)mr[e] * (size_t)K + k0) : make_uint4(0, 0, 0, 0);
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            if (mr[e] >= rows_pad) break;
            uint32_t h[8];
            // rows past M and codes past K are zero images (fp16 +0)
            if (mr[e] < M && k0 < K) {
                bytes_to_half(v[e], flip, h);
                if (PTF) {
#pragma unroll
                    for (int j = 0; j < 8; ++j) h[j] = hmul2_u32(h[j], mul[j]);
                }
            } else {
#pragma unroll
                for (int j = 0; j < 8; ++j) h[j] = 0;
            }
            if (ROWSUM) {
                int32_t part = 0;
                if (mr[e] < M && k0 < K) {
                    // offset-binary bytes (centred value + 128), summed 4 at a time
                    const uint32_t fl = a_u8 ? 0u : 0x80808080u;
                    uint32_t acc = 0;
                    acc = __dp4a(v[e].x ^ fl, 0x01010101u, acc);
                    acc = __dp4a(v[e].y ^ fl, 0x01010101u, acc);
                    acc = __dp4a(v[e].z ^ fl, 0x01010101u, acc);
                    acc = __dp4a(v[e].w ^ fl, 0x01010101u, acc);
                    part = (int32_t)acc - 16 * 128;
                }
                const unsigned same = __match_any_sync(__activemask(), mr[e]);
                part = __reduce_add_sync(same, part);
                if ((threadIdx.x + threadIdx.y * blockDim.x) % 32 == (unsigned)(__ffs(same) - 1) && mr[e] < M && part != 0)
                    atomicAdd(rowsum + mr[e], part);
            }
            const int r = mr[e] & (BM - 1);
            uint8_t *row = out + ((size_t)((mr[e] / BM) * KT + ks) * BM + r) * ROW_BYTES;
            *reinterpret_cast<uint4 *>(row + ((c ^ (r & 7)) << 4)) = make_uint4(h[0], h[1], h[2], h[3]);
            *reinterpret_cast<uint4 *>(row + (((c + 1) ^ (r & 7)) << 4)) = make_uint4(h[4], h[5], h[6], h[7]);
        }
    }
}

inline size_t packed_a_bytes(int M, int K)
{
    return (size_t)((M + BM - 1) / BM) * (size_t)qnn::gemm::ksteps(K) * (size_t)A_STAGE_BYTES;
}

}  // namespace mk
}  // namespace qnn

extern "C" size_t qnn_gemm_workspace_bytes(int M, int K)
{
    if (M <= 0 || K <= 0) return 0;
    return qnn::mk::packed_a_bytes(M, K);
}

namespace qnn {
namespace mk {

// Validation and Params shared by the three GEMM entry points.  A may be the
// codes (fused path) or the packed image (A_is_packed); the epilogue's PTF
// fields decide the exact-chunk length either way.
static qnn_status gemm_params(const void *A, qnn_dtype a_dt, const void *B_packed, int M, int N, int K,
                              const qnn_epilogue *e, void *C, int32_t *C_s32, Params &p)
{
    if (!A || !B_packed || !e || !C) return QNN_ERR_INVALID_ARG;
    if (M <= 0 || N <= 0 || K <= 0) return QNN_ERR_INVALID_ARG;
    if (a_dt != QNN_S8 && a_dt != QNN_U8) return QNN_ERR_UNSUPPORTED;
    if (K % 16 != 0) return QNN_ERR_ALIGNMENT;
    if (!qnn::aligned16(A) || !qnn::aligned16(C) || (C_s32 && !qnn::aligned16(C_s32)))
        return QNN_ERR_ALIGNMENT;
    if ((reinterpret_cast<uintptr_t>(B_packed) & 1023u) != 0) return QNN_ERR_ALIGNMENT;

    p = Params{};
    p.A = static_cast<const uint8_t *>(A);
    p.a_u8 = (a_dt == QNN_U8);
    p.Bp = static_cast<const uint8_t *>(B_packed);
    p.M = M;
    p.N = N;
    p.K = K;
    p.KT = qnn::gemm::ksteps(K);
    p.num_m = (M + BM - 1) / BM;
    p.C = C;
    p.C32 = C_s32;
    p.vec_ok = (N % 32 == 0);
    qnn_status st = setup_epilogue(e, false, p);
    if (st != QNN_OK) return st;

    // shift: bound on the Power-of-Two-Factor shifts, applied here to A
    // (ptf_shift) or already folded into the weights (qgemm_prepack_b_ptf:
    // ptf_shift NULL, ptf_max_shift the bound)
    if (e->ptf_max_shift < 0 || e->ptf_max_shift > 3) return QNN_ERR_INVALID_ARG;
    const int shift = e->ptf_max_shift;
    if (e->ptf_shift) {
        if (a_dt != QNN_S8 || e->zp_term) return QNN_ERR_UNSUPPORTED;
        if (!qnn::aligned16(e->ptf_shift)) return QNN_ERR_ALIGNMENT;
        p.ptf = e->ptf_shift;
        p.ptf_max = shift;
        p.a_shift = shift;
    }
    // |acc_c| <= K * 255 * 128 * 2^shift must stay inside int32
    if ((int64_t)K * 255 * 128 * (1 << shift) > (int64_t)INT32_MAX) return QNN_ERR_OVERFLOW_RISK;
    p.chunk_steps = qnn::gemm::MAX_EXACT_STEPS >> shift;
    p.nchunks = (p.KT + p.chunk_steps - 1) / p.chunk_steps;
    p.btrail = reinterpret_cast<const int32_t *>(static_cast<const uint8_t *>(B_packed) +
                                                 qnn::gemm::packed_b_image_bytes(N, K));
    return QNN_OK;
}

static qnn_status launch_pack_a(const uint8_t *A, int M, int K, int a_u8, const uint8_t *ptf, int ptf_max,
                                uint8_t *out, cudaStream_t s, int32_t *rowsum = nullptr)
{
    uint32_t *status = qnn::status_word();
    if (!status) return QNN_ERR_CUDA;
    const int KT = qnn::gemm::ksteps(K);
    const int rows_pad = ((M + BM - 1) / BM) * BM;
    const int groups = KT * 4;
    // 256 threads: up to 64 groups of a row x 4 (or more) rows
    const int bx = groups >= 64 ? 64 : groups;
    const int by = 256 / bx;
    const dim3 block(bx, by);
    const int gx = (groups + bx - 1) / bx;
    int gy = (rows_pad + by - 1) / by;
    gy = (gy + 1) / 2;  // two rows per thread and iteration
    const int want = qnn::sm_count() * 32;  // enough blocks in flight; rows loop beyond
    if (gy > 65535) gy = 65535;
    if ((int64_t)gx * gy > want && gy > 1) {
        gy = (want + gx - 1) / gx;
        if (gy < 1) gy = 1;
    }
    const dim3 grid(gx, gy);
    if (rowsum)
        pack_a_kernel<false, true><<<grid, block, 0, s>>>(A, M, K, KT, rows_pad, a_u8, nullptr, out, rowsum, 0, status);
    else if (ptf)
        pack_a_kernel<true, false><<<grid, block, 0, s>>>(A, M, K, KT, rows_pad, a_u8, ptf, out, nullptr, ptf_max,
                                                          status);
    else
        pack_a_kernel<false, false><<<grid, block, 0, s>>>(A, M, K, KT, rows_pad, a_u8, nullptr, out, nullptr, 0,
                                                           status);
    return qnn::launch_status();
}

static qnn_status launch_gemm(Params &p, bool packed, cudaStream_t s)
{
    p.status = qnn::status_word();
    if (!p.status) return QNN_ERR_CUDA;
    const bool multi = p.nchunks > 1;
    if (packed) {
        p.Ap = p.A;
        if (!multi) return launch<GemmPackedOp, 256, false>(p, s);
        return launch<GemmPackedOp, 256, true>(p, s);
    }
    if (!p.ptf) {
        if (!multi) return launch<GemmOp<false>, 256, false>(p, s);
        return launch<GemmOp<false>, 128, true>(p, s);
    }
    if (!multi) return launch<GemmOp<true>, 256, false>(p, s);
    return launch<GemmOp<true>, 128, true>(p, s);
}

}  // namespace mk
}  // namespace qnn

// ---- fixed scratch variant ---------------------------------------------------
// For callers that must not allocate device memory at call time (allocation
// is not allowed inside their execution context, or their allocator is not
// reachable from it): the re-encoded A lives in one file-scope device array
// of QNN_GEMM_STATIC_SCRATCH_BYTES, allocated with the module.
namespace qnn {
namespace mk {

static __device__ __align__(256) uint8_t g_gemm_scratch[QNN_GEMM_STATIC_SCRATCH_BYTES];

constexpr int kScratchDevices = 64;
static std::atomic<uintptr_t> g_scratch_addr[kScratchDevices];

// Device address of the scratch array on the current device, looked up once
// per device; nullptr if the lookup failed.
static uint8_t *static_scratch()
{
    int d = -1;
    if (cudaGetDevice(&d) != cudaSuccess || d < 0 || d >= kScratchDevices) return nullptr;
    uintptr_t a = g_scratch_addr[d].load(std::memory_order_acquire);
    if (a == 0) {
        void *ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_gemm_scratch) != cudaSuccess) {
            (void)cudaGetLastError();
            return nullptr;
        }
        a = reinterpret_cast<uintptr_t>(ptr);
        g_scratch_addr[d].store(a, std::memory_order_release);
    }
    return reinterpret_cast<uint8_t *>(a);
}

}  // namespace mk
}  // namespace qnn

extern "C" qnn_status qgemm_s8_static_scratch(const void *A, qnn_dtype a_dt, const void *B_packed, int M,
                                              int N, int K, const qnn_epilogue *e, void *C, int32_t *C_s32,
                                              qnn_stream_t stream)
{
    using namespace qnn::mk;
    Params p;
    qnn_status st = gemm_params(A, a_dt, B_packed, M, N, K, e, C, C_s32, p);
    if (st != QNN_OK) return st;
    if (packed_a_bytes(M, K) > (size_t)QNN_GEMM_STATIC_SCRATCH_BYTES) return QNN_ERR_UNSUPPORTED;
    uint8_t *ws = static_scratch();
    if (!ws) return QNN_ERR_CUDA;
    // nothing has to start at zero: the pre-pass writes every byte the GEMM reads
    cudaStream_t s = (cudaStream_t)stream;
    st = launch_pack_a(p.A, M, K, p.a_u8, p.ptf, p.ptf_max, ws, s);
    if (st != QNN_OK) return st;
    p.A = ws;
    return launch_gemm(p, true, s);
}

extern "C" qnn_status qgemm_pack_a(const void *A, qnn_dtype a_dt, int M, int K, const uint8_t *ptf_shift,
                                   void *A_packed, size_t A_packed_bytes, qnn_stream_t stream)
{
    using namespace qnn::mk;
    if (!A || !A_packed || M <= 0 || K <= 0) return QNN_ERR_INVALID_ARG;
    if (a_dt != QNN_S8 && a_dt != QNN_U8) return QNN_ERR_UNSUPPORTED;
    if (ptf_shift && a_dt != QNN_S8) return QNN_ERR_UNSUPPORTED;
    if (K % 16 != 0) return QNN_ERR_ALIGNMENT;
    if (!qnn::aligned16(A) || !qnn::aligned16(A_packed) || (ptf_shift && !qnn::aligned16(ptf_shift)))
        return QNN_ERR_ALIGNMENT;
    if (A_packed_bytes < packed_a_bytes(M, K)) return QNN_ERR_INVALID_ARG;
    // the shift bytes are checked against the largest allowed shift, 3
    return launch_pack_a(static_cast<const uint8_t *>(A), M, K, a_dt == QNN_U8, ptf_shift, 3,
                         static_cast<uint8_t *>(A_packed), (cudaStream_t)stream);
}

extern "C" qnn_status qgemm_s8_packed(const void *A_packed, qnn_dtype a_dt, const void *B_packed, int M,
                                      int N, int K, const qnn_epilogue *e, void *C, int32_t *C_s32,
                                      qnn_stream_t stream)
{
    using namespace qnn::mk;
    Params p;
    const qnn_status st = gemm_params(A_packed, a_dt, B_packed, M, N, K, e, C, C_s32, p);
    if (st != QNN_OK) return st;
    return launch_gemm(p, true, (cudaStream_t)stream);
}

extern "C" size_t qnn_gemm_zw_workspace_bytes(int M, int K)
{
    if (M <= 0 || K <= 0) return 0;
    return qnn::mk::packed_a_bytes(M, K) + (((size_t)M * 4 + 255) & ~(size_t)255);
}

extern "C" qnn_status qgemm_zw(const void *A, qnn_dtype a_dt, const void *B_packed, const int32_t *z_w, int M,
                               int N, int K, const qnn_epilogue *e, void *C, int32_t *C_s32, void *workspace,
                               size_t workspace_bytes, qnn_stream_t stream)
{
    using namespace qnn::mk;
    Params p;
    qnn_status st = gemm_params(A, a_dt, B_packed, M, N, K, e, C, C_s32, p);
    if (st != QNN_OK) return st;
    if (p.ptf) return QNN_ERR_UNSUPPORTED;
    if (!z_w) return QNN_ERR_INVALID_ARG;
    if (!qnn::aligned16(z_w)) return QNN_ERR_ALIGNMENT;
    // |sum_k (a - z_a)(w - z_w)| <= K * 255 * 255 must stay inside int32
    if ((int64_t)K * 255 * 255 > (int64_t)INT32_MAX) return QNN_ERR_OVERFLOW_RISK;
    if (!workspace || workspace_bytes < qnn_gemm_zw_workspace_bytes(M, K)) return QNN_ERR_INVALID_ARG;
    if (!qnn::aligned16(workspace)) return QNN_ERR_ALIGNMENT;
    cudaStream_t s = (cudaStream_t)stream;
    uint8_t *img = static_cast<uint8_t *>(workspace);
    int32_t *rowsum = reinterpret_cast<int32_t *>(img + packed_a_bytes(M, K));
    if (cudaMemsetAsync(rowsum, 0, (size_t)M * 4, s) != cudaSuccess) return QNN_ERR_CUDA;
    st = launch_pack_a(p.A, M, K, p.a_u8, nullptr, 0, img, s, rowsum);
    if (st != QNN_OK) return st;
    p.A = img;
    p.zw = z_w;
    p.rowsum = rowsum;
    return launch_gemm(p, true, s);
}

extern "C" qnn_status qgemm_s8(const void *A, qnn_dtype a_dt, const void *B_packed, int M, int N,
                               int K, const qnn_epilogue *e, void *C, int32_t *C_s32,
                               void *workspace, size_t workspace_bytes, qnn_stream_t stream)
{
    using namespace qnn::mk;
    Params p;
    qnn_status st = gemm_params(A, a_dt, B_packed, M, N, K, e, C, C_s32, p);
    if (st != QNN_OK) return st;
    if (!workspace) return launch_gemm(p, false, (cudaStream_t)stream);
    if (workspace_bytes < packed_a_bytes(M, K)) return QNN_ERR_INVALID_ARG;
    if (!qnn::aligned16(workspace)) return QNN_ERR_ALIGNMENT;
    cudaStream_t s = (cudaStream_t)stream;
    st = launch_pack_a(p.A, M, K, p.a_u8, p.ptf, p.ptf_max, static_cast<uint8_t *>(workspace), s);
    if (st != QNN_OK) return st;
    p.A = static_cast<const uint8_t *>(workspace);
    return launch_gemm(p, true, s);
}
