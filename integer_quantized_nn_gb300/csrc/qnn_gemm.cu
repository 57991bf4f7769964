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
// chunks of at most (16 >> ptf_max_shift) steps of 64 (|sum| <= 2^24); each
// chunk accumulates in its own TMEM buffer and the epilogue warps add the
// chunk results in int32.  A u8 operand is read as (q - 128) so that every
// operand is in [-128, 127]; the fold puts the 128 back through zp_term.
//
// Warp roles (512 threads, one CTA per SM, persistent over 128 x 256 tiles):
//   warps 0-3  : converters -- load A rows from global memory (16-byte loads,
//                one unit ahead), convert int8 -> fp16 (byte permute into the
//                exponent of 1024, subtract 1024 + 128), apply 2^alpha, store
//                into the 128-byte swizzled K-major stage buffer.
//   warp 4     : TMA producer -- one bulk copy per stage of the prepacked fp16
//                weight tile (already in the swizzled image).
//   warp 5     : TMEM owner and MMA issuer -- 4 x tcgen05.mma (128x256x16)
//                per stage into one of two 256-column fp32 accumulators.
//   warps 8-15 : epilogue -- tcgen05.ld, fp32 -> int32, chunk sums, then the
//                fused requant / dequant math and 16-byte stores of each
//                thread's 32 consecutive output columns.
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <cstdint>
#include "qnn_gemm_layout.h"
#include "qnn_internal.h"
#include "qnn_ptx.cuh"

namespace qnn {
namespace gemm {

constexpr int STAGES = 4;
constexpr int NUM_THREADS = 512;
constexpr int PRODUCER_WARP = 4;
constexpr int MMA_WARP = 5;
constexpr int EPI_WARP0 = 8;
constexpr int NUM_EPI_WARPS = 8;
constexpr uint32_t TMEM_COLS = 512;

struct Params {
    const uint8_t *A;
    const uint8_t *Bp;
    int M, N, K, KT, num_m, num_tiles;
    int a_u8;
    int chunk_steps, nchunks;
    int mode, relu, z_out;
    float qmin, qmax;
    const int32_t *zp;
    const float *Mv;
    const float *Bq;
    const float *D;
    const float *bias;
    const uint8_t *res;
    int res_signed, z_res;
    float R;
    const uint8_t *ptf;
    void *C;
    int32_t *C32;
    int vec_ok;  // N % 32 == 0: every 32-column piece is whole and 16-byte aligned
    uint32_t *status;
};

template <int TBN>
struct __align__(1024) Smem {
    uint8_t a[STAGES][A_STAGE_BYTES];
    uint8_t b[STAGES][TBN * ROW_BYTES];
    uint64_t a_full[STAGES];
    uint64_t b_full[STAGES];
    uint64_t empty[STAGES];
    uint64_t acc_full[2];
    uint64_t acc_empty[2];
    uint64_t mma_done;
    uint32_t tmem_base;
};

template <int TBN>
constexpr size_t smem_bytes() { return sizeof(Smem<TBN>) + 1024; }

// ---------------------------------------------------------------- converter
struct AUnit {
    uint4 v[4];
    uint4 alpha;
};

template <bool PTF>
__device__ __forceinline__ void load_unit(const Params &p, int j, int sub, int rbase, AUnit &u)
{
    const int t = blockIdx.x + (j / p.KT) * gridDim.x;
    const int ks = j % p.KT;
    const int m0 = (t % p.num_m) * BM;
    const int k0 = ks * BK + sub * 16;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const int m = m0 + q * 32 + rbase;
        if (m < p.M && k0 < p.K)
            u.v[q] = ldg_nc_v4(p.A + (int64_t)m * p.K + k0);
        else
            u.v[q] = make_uint4(0, 0, 0, 0);
    }
    if (PTF) {
        if (k0 < p.K)
            u.alpha = ldg_nc_v4(p.ptf + k0);
        else
            u.alpha = make_uint4(0, 0, 0, 0);
    }
}

// fp16x2 multipliers 2^alpha for the two alpha bytes selected by `sel`.
__device__ __forceinline__ uint32_t pow2_half2(uint32_t alpha4, uint32_t sel)
{
    return (prmt(alpha4, 0u, sel) << 10) + 0x3C003C00u;
}

template <bool PTF>
__device__ __forceinline__ void store_unit(const Params &p, uint32_t a_stage, int sub, int rbase,
                                           const AUnit &u)
{
    const uint32_t flip = p.a_u8 ? 0u : 0x80808080u;  // s8 -> offset binary
    uint32_t mul[8];
    if (PTF) {
        const uint32_t al[4] = {u.alpha.x, u.alpha.y, u.alpha.z, u.alpha.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            mul[2 * i] = pow2_half2(al[i], 0x4140u);
            mul[2 * i + 1] = pow2_half2(al[i], 0x4342u);
        }
    }
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const int row = q * 32 + rbase;
        const uint32_t w[4] = {u.v[q].x ^ flip, u.v[q].y ^ flip, u.v[q].z ^ flip, u.v[q].w ^ flip};
        uint32_t h[8];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            // bytes -> fp16 (1024 + byte), then subtract 1024 + 128: exact
            h[2 * i] = hsub2_u32(prmt(w[i], 0x64646464u, 0x4140u), 0x64806480u);
            h[2 * i + 1] = hsub2_u32(prmt(w[i], 0x64646464u, 0x4342u), 0x64806480u);
            if (PTF) {
                h[2 * i] = hmul2_u32(h[2 * i], mul[2 * i]);
                h[2 * i + 1] = hmul2_u32(h[2 * i + 1], mul[2 * i + 1]);
            }
        }
        const uint32_t rowaddr = a_stage + row * ROW_BYTES;
        const int c0 = 2 * sub, c1 = 2 * sub + 1;
        sts_v4(rowaddr + ((c0 ^ (row & 7)) << 4), h[0], h[1], h[2], h[3]);
        sts_v4(rowaddr + ((c1 ^ (row & 7)) << 4), h[4], h[5], h[6], h[7]);
    }
}

template <int TBN, bool PTF>
__device__ __forceinline__ bool convert_one(const Params &p, Smem<TBN> &s, int j, int sub, int rbase,
                                            const AUnit &u)
{
    const int stage = j % STAGES;
    const uint32_t ph = (uint32_t)(j / STAGES) & 1u;
    if (!mbar_wait(smem_u32(&s.empty[stage]), ph ^ 1u, p.status)) return false;
    store_unit<PTF>(p, smem_u32(&s.a[stage][0]), sub, rbase, u);
    fence_proxy_async_smem();
    __syncwarp();
    if ((threadIdx.x & 31) == 0) mbar_arrive(smem_u32(&s.a_full[stage]));
    return true;
}

template <int TBN, bool PTF>
__device__ void converter_role(const Params &p, Smem<TBN> &s, int units)
{
    const int tid = threadIdx.x;  // 0..127
    const int sub = tid & 3;
    const int rbase = tid >> 2;
    AUnit u0, u1;
    if (units > 0) load_unit<PTF>(p, 0, sub, rbase, u0);
    for (int j = 0; j < units; j += 2) {
        if (j + 1 < units) load_unit<PTF>(p, j + 1, sub, rbase, u1);
        if (!convert_one<TBN, PTF>(p, s, j, sub, rbase, u0)) return;
        if (j + 1 < units) {
            if (j + 2 < units) load_unit<PTF>(p, j + 2, sub, rbase, u0);
            if (!convert_one<TBN, PTF>(p, s, j + 1, sub, rbase, u1)) return;
        }
    }
}

// ---------------------------------------------------------------- producer
template <int TBN>
__device__ void producer_role(const Params &p, Smem<TBN> &s, int units)
{
    int issued_stage_parity_ok = 1;
    int j = 0;
    for (; j < units; ++j) {
        const int stage = j % STAGES;
        const uint32_t ph = (uint32_t)(j / STAGES) & 1u;
        if (!mbar_wait(smem_u32(&s.empty[stage]), ph ^ 1u, p.status)) {
            issued_stage_parity_ok = 0;
            break;
        }
        const int t = blockIdx.x + (j / p.KT) * gridDim.x;
        const int ks = j % p.KT;
        // output columns n0 .. n0 + TBN - 1 live in the 256-row packed block n0 / 256
        const int n0 = (t / p.num_m) * TBN;
        const uint8_t *src = p.Bp + ((int64_t)(n0 / BN) * p.KT + ks) * B_STAGE_BYTES +
                             (int64_t)(n0 % BN) * ROW_BYTES;
        const uint32_t bar = smem_u32(&s.b_full[stage]);
        mbar_arrive_expect_tx(bar, TBN * ROW_BYTES);
        bulk_g2s(smem_u32(&s.b[stage][0]), src, TBN * ROW_BYTES, bar);
    }
    if (!issued_stage_parity_ok) {
        // wind down: let the copies already issued land before the CTA exits
        for (int i = (j > STAGES ? j - STAGES : 0); i < j; ++i) {
            const int stage = i % STAGES;
            const uint32_t ph = (uint32_t)(i / STAGES) & 1u;
            if (!mbar_wait(smem_u32(&s.b_full[stage]), ph, p.status)) break;
        }
    }
}

// ---------------------------------------------------------------- MMA
template <int TBN>
__device__ void mma_role(const Params &p, Smem<TBN> &s, int my_tiles, uint32_t tmem)
{
    constexpr uint32_t IDESC = idesc_f32acc(0, 0, BM, TBN);
    uint32_t u = 0;  // accumulation chunk counter
    uint32_t abuf = 0;
    bool ok = true;
    for (int i = 0; i < my_tiles && ok; ++i) {
        for (int ks = 0; ks < p.KT; ++ks) {
            const int j = i * p.KT + ks;
            const int stage = j % STAGES;
            const uint32_t ph = (uint32_t)(j / STAGES) & 1u;
            const bool first = (ks % p.chunk_steps) == 0;
            if (first) {
                abuf = u & 1u;
                if (!mbar_wait(smem_u32(&s.acc_empty[abuf]), ((u >> 1) & 1u) ^ 1u, p.status)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
            }
            if (!mbar_wait(smem_u32(&s.a_full[stage]), ph, p.status) ||
                !mbar_wait(smem_u32(&s.b_full[stage]), ph, p.status)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const uint32_t a0 = smem_u32(&s.a[stage][0]);
            const uint32_t b0 = smem_u32(&s.b[stage][0]);
            const uint32_t d = tmem + abuf * TBN;
#pragma unroll
            for (int kk = 0; kk < BK / 16; ++kk) {
                mma_f16_ss(d, sdesc_sw128(a0 + kk * 32), sdesc_sw128(b0 + kk * 32), IDESC,
                           (first && kk == 0) ? 0u : 1u);
            }
            mma_commit(smem_u32(&s.empty[stage]));
            const bool last = ((ks % p.chunk_steps) == p.chunk_steps - 1) || (ks == p.KT - 1);
            if (last) {
                mma_commit(smem_u32(&s.acc_full[abuf]));
                ++u;
            }
        }
    }
    // make sure every MMA issued has completed before the CTA winds down
    mma_commit(smem_u32(&s.mma_done));
    (void)mbar_wait(smem_u32(&s.mma_done), 0u, p.status);
}

// ---------------------------------------------------------------- epilogue
__device__ __forceinline__ void st_v4(void *ptr, uint32_t a, uint32_t b, uint32_t c, uint32_t d)
{
    *reinterpret_cast<uint4 *>(ptr) = make_uint4(a, b, c, d);
}

// Requant / dequant / raw store of 32 consecutive columns n0.. of row m.
// Works in place on `ac` (the raw accumulators on entry) to keep the register
// footprint of the multi-chunk epilogue small.
__device__ __forceinline__ void epilogue_piece(const Params &p, int m, int n0, int32_t (&ac)[32])
{
    if (m >= p.M || n0 >= p.N) return;
    const bool vec = p.vec_ok;
    if (p.zp) {
#pragma unroll
        for (int i = 0; i < 32; ++i)
            if (vec || n0 + i < p.N) ac[i] -= __ldg(p.zp + n0 + i);
    }
    const int64_t base = (int64_t)m * p.N + n0;
    if (p.C32) {
        if (vec) {
#pragma unroll
            for (int i = 0; i < 32; i += 4)
                st_v4(p.C32 + base + i, ac[i], ac[i + 1], ac[i + 2], ac[i + 3]);
        } else {
            for (int i = 0; i < 32 && n0 + i < p.N; ++i) p.C32[base + i] = ac[i];
        }
    }
    if (p.mode == QNN_EPI_S32) {
        int32_t *C = static_cast<int32_t *>(p.C);
        if (vec) {
#pragma unroll
            for (int i = 0; i < 32; i += 4) st_v4(C + base + i, ac[i], ac[i + 1], ac[i + 2], ac[i + 3]);
        } else {
            for (int i = 0; i < 32 && n0 + i < p.N; ++i) C[base + i] = ac[i];
        }
        return;
    }
    if (p.mode == QNN_EPI_DEQUANT) {
        float *C = static_cast<float *>(p.C);
#pragma unroll
        for (int i = 0; i < 32; ++i) {
            const int n = (vec || n0 + i < p.N) ? n0 + i : n0;
            const float b = p.bias ? __ldg(p.bias + n) : 0.0f;
            ac[i] = __float_as_int(__fadd_rn(__fmul_rn(__int2float_rn(ac[i]), __ldg(p.D + n)), b));
        }
        if (vec) {
#pragma unroll
            for (int i = 0; i < 32; i += 4) st_v4(C + base + i, ac[i], ac[i + 1], ac[i + 2], ac[i + 3]);
        } else {
            for (int i = 0; i < 32 && n0 + i < p.N; ++i) C[base + i] = __int_as_float(ac[i]);
        }
        return;
    }
    // REQUANT
    uint32_t rw[8];
    if (p.res) {
        if (vec) {
            const uint4 r0 = ldg_nc_v4(p.res + base), r1 = ldg_nc_v4(p.res + base + 16);
            rw[0] = r0.x; rw[1] = r0.y; rw[2] = r0.z; rw[3] = r0.w;
            rw[4] = r1.x; rw[5] = r1.y; rw[6] = r1.z; rw[7] = r1.w;
        } else {
#pragma unroll
            for (int i = 0; i < 8; ++i) rw[i] = 0;
            for (int i = 0; i < 32 && n0 + i < p.N; ++i)
                rw[i >> 2] |= (uint32_t)p.res[base + i] << (8 * (i & 3));
        }
    }
    const float zo = (float)p.z_out;
    uint32_t ow[8];
#pragma unroll
    for (int w = 0; w < 8; ++w) {
        uint32_t word = 0;
#pragma unroll
        for (int b = 0; b < 4; ++b) {
            const int i = 4 * w + b;
            const int n = (vec || n0 + i < p.N) ? n0 + i : n0;
            float t = __ldg(p.Bq + n);
            if (p.res) {
                int32_t rv = (int32_t)((rw[w] >> (8 * b)) & 255u);
                if (p.res_signed && rv >= 128) rv -= 256;
                t = __fadd_rn(__fmul_rn(__int2float_rn(rv - p.z_res), p.R), t);
            }
            const float v = __fadd_rn(__fmul_rn(__int2float_rn(ac[i]), __ldg(p.Mv + n)), t);
            float r = rintf(v);
            if (p.relu) r = fmaxf(r, 0.0f);
            const float c = fminf(fmaxf(__fadd_rn(r, zo), p.qmin), p.qmax);
            word |= ((uint32_t)__float2int_rn(c) & 255u) << (8 * b);
        }
        ow[w] = word;
    }
    uint8_t *C = static_cast<uint8_t *>(p.C);
    if (vec) {
        st_v4(C + base, ow[0], ow[1], ow[2], ow[3]);
        st_v4(C + base + 16, ow[4], ow[5], ow[6], ow[7]);
    } else {
        for (int i = 0; i < 32 && n0 + i < p.N; ++i) C[base + i] = (uint8_t)(ow[i >> 2] >> (8 * (i & 3)));
    }
}

// TBN == 256: one accumulation chunk per tile; each epilogue thread owns one
// row and 128 columns, converted and stored 32 at a time straight from TMEM.
// TBN == 128: K is cut into exact chunks; each thread keeps int32 sums for its
// row and 64 columns in registers across the chunks.
template <int TBN, bool MULTI>
__device__ void epilogue_role(const Params &p, Smem<TBN> &s, int my_tiles, uint32_t tmem)
{
    constexpr int COLS = TBN / 2;       // columns per epilogue thread
    constexpr int PIECES = COLS / 32;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int quad = warp & 3;                 // TMEM lanes 32*quad .. +31
    const int half = (warp - EPI_WARP0) >> 2;  // columns COLS*half .. +COLS-1
    uint32_t u = 0;
    for (int i = 0; i < my_tiles; ++i) {
        const int t = blockIdx.x + i * gridDim.x;
        const int m = (t % p.num_m) * BM + quad * 32 + lane;
        const int nbase = (t / p.num_m) * TBN + half * COLS;
        if (!MULTI) {
            const uint32_t abuf = u & 1u;
            if (!mbar_wait(smem_u32(&s.acc_full[abuf]), (u >> 1) & 1u, p.status)) return;
            tc_fence_after();
            const uint32_t taddr = tmem + ((uint32_t)(quad * 32) << 16) + abuf * TBN + half * COLS;
#pragma unroll 1
            for (int jp = 0; jp < PIECES; ++jp) {
                uint32_t r[32];
                tmem_ld32(taddr + jp * 32, r);
                tmem_ld_wait();
                int32_t acc[32];
#pragma unroll
                for (int k = 0; k < 32; ++k) acc[k] = __float2int_rn(__uint_as_float(r[k]));
                if (jp == PIECES - 1) {
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(smem_u32(&s.acc_empty[abuf]));
                }
                epilogue_piece(p, m, nbase + jp * 32, acc);
            }
            ++u;
        } else {
            int32_t acc[PIECES][32];
            for (int c = 0; c < p.nchunks; ++c) {
                const uint32_t abuf = u & 1u;
                if (!mbar_wait(smem_u32(&s.acc_full[abuf]), (u >> 1) & 1u, p.status)) return;
                tc_fence_after();
                const uint32_t taddr = tmem + ((uint32_t)(quad * 32) << 16) + abuf * TBN + half * COLS;
#pragma unroll
                for (int jp = 0; jp < PIECES; ++jp) {
                    uint32_t r[32];
                    tmem_ld32(taddr + jp * 32, r);
                    tmem_ld_wait();
#pragma unroll
                    for (int k = 0; k < 32; ++k) {
                        const int32_t v = __float2int_rn(__uint_as_float(r[k]));
                        acc[jp][k] = (c == 0) ? v : acc[jp][k] + v;
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&s.acc_empty[abuf]));
                ++u;
            }
#pragma unroll
            for (int jp = 0; jp < PIECES; ++jp) epilogue_piece(p, m, nbase + jp * 32, acc[jp]);
        }
    }
}

// ---------------------------------------------------------------- kernel
template <int TBN, bool MULTI, bool PTF>
__global__ void __launch_bounds__(NUM_THREADS, 1) qgemm_kernel(const __grid_constant__ Params p)
{
    extern __shared__ uint8_t smem_raw[];
    Smem<TBN> &s = *reinterpret_cast<Smem<TBN> *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                  ~static_cast<uintptr_t>(1023));
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int i = 0; i < STAGES; ++i) {
            mbar_init(smem_u32(&s.a_full[i]), 4);
            mbar_init(smem_u32(&s.b_full[i]), 1);
            mbar_init(smem_u32(&s.empty[i]), 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(smem_u32(&s.acc_full[i]), 1);
            mbar_init(smem_u32(&s.acc_empty[i]), NUM_EPI_WARPS);
        }
        mbar_init(smem_u32(&s.mma_done), 1);
        fence_mbar_init();
    }
    if (warp == MMA_WARP) {
        tmem_alloc(smem_u32(&s.tmem_base), 2 * TBN);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = s.tmem_base;

    const int my_tiles =
        (blockIdx.x < p.num_tiles) ? (p.num_tiles - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;
    const int units = my_tiles * p.KT;

    // register split (multi-chunk kernel): 128*96 + 128*56 + 256*176 = 64512 <= 65536
    if (warp < 4) {
        if (MULTI) regs_dec<96>();
        converter_role<TBN, PTF>(p, s, units);
    } else if (warp < 8) {
        if (MULTI) regs_dec<56>();
        if (warp == PRODUCER_WARP && lane == 0) producer_role<TBN>(p, s, units);
        if (warp == MMA_WARP && lane == 0) mma_role<TBN>(p, s, my_tiles, tmem);
        __syncwarp();
    } else {
        if (MULTI) regs_inc<176>();
        epilogue_role<TBN, MULTI>(p, s, my_tiles, tmem);
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == MMA_WARP) tmem_dealloc(tmem, 2 * TBN);
}

template <int TBN, bool MULTI, bool PTF>
qnn_status launch(Params p, cudaStream_t stream)
{
    static bool attr_set[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return QNN_ERR_CUDA;
    constexpr size_t SMEM = smem_bytes<TBN>();
    if (!attr_set[dev]) {
        if (cudaFuncSetAttribute(qgemm_kernel<TBN, MULTI, PTF>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM) != cudaSuccess)
            return QNN_ERR_CUDA;
        attr_set[dev] = true;
    }
    p.num_tiles = p.num_m * ((p.N + TBN - 1) / TBN);
    int grid = qnn::sm_count();
    if (grid > p.num_tiles) grid = p.num_tiles;
    qgemm_kernel<TBN, MULTI, PTF><<<grid, NUM_THREADS, SMEM, stream>>>(p);
    return launch_status();
}

}  // namespace gemm
}  // namespace qnn

extern "C" qnn_status qgemm_s8(const void *A, qnn_dtype a_dt, const void *B_packed, int M, int N,
                               int K, const qnn_epilogue *e, void *C, int32_t *C_s32,
                               qnn_stream_t stream)
{
    using namespace qnn::gemm;
    if (!A || !B_packed || !e || !C) return QNN_ERR_INVALID_ARG;
    if (M <= 0 || N <= 0 || K <= 0) return QNN_ERR_INVALID_ARG;
    if (a_dt != QNN_S8 && a_dt != QNN_U8) return QNN_ERR_UNSUPPORTED;
    if (K % 16 != 0) return QNN_ERR_ALIGNMENT;
    if (!qnn::aligned16(A) || !qnn::aligned16(C) || (C_s32 && !qnn::aligned16(C_s32)))
        return QNN_ERR_ALIGNMENT;
    if ((reinterpret_cast<uintptr_t>(B_packed) & 1023u) != 0) return QNN_ERR_ALIGNMENT;

    Params p{};
    p.A = static_cast<const uint8_t *>(A);
    p.Bp = static_cast<const uint8_t *>(B_packed);
    p.M = M;
    p.N = N;
    p.K = K;
    p.KT = ksteps(K);
    p.num_m = (M + BM - 1) / BM;
    p.a_u8 = (a_dt == QNN_U8);
    p.mode = e->mode;
    p.relu = e->relu ? 1 : 0;
    p.z_out = e->z_out;
    p.zp = e->zp_term;
    p.Mv = e->M;
    p.Bq = e->Bq;
    p.D = e->D;
    p.bias = e->bias;
    p.C = C;
    p.C32 = C_s32;
    p.vec_ok = (N % 32 == 0);

    switch (e->mode) {
    case QNN_EPI_REQUANT: {
        if (!e->M || !e->Bq) return QNN_ERR_INVALID_ARG;
        if (e->out_dt != QNN_S8 && e->out_dt != QNN_U8) return QNN_ERR_UNSUPPORTED;
        int32_t lo, hi;
        qnn::qrange(e->out_dt, 0, &lo, &hi);
        if (e->z_out < lo || e->z_out > hi) return QNN_ERR_INVALID_ARG;
        p.qmin = (float)lo;
        p.qmax = (float)hi;
        if (e->residual) {
            if (e->res_dt != QNN_S8 && e->res_dt != QNN_U8) return QNN_ERR_UNSUPPORTED;
            if (!qnn::aligned16(e->residual)) return QNN_ERR_ALIGNMENT;
            p.res = static_cast<const uint8_t *>(e->residual);
            p.res_signed = (e->res_dt == QNN_S8);
            p.z_res = e->z_res;
            p.R = e->R;
        }
        break;
    }
    case QNN_EPI_DEQUANT:
        if (!e->D) return QNN_ERR_INVALID_ARG;
        if (e->residual) return QNN_ERR_UNSUPPORTED;
        break;
    case QNN_EPI_S32:
        if (e->residual) return QNN_ERR_UNSUPPORTED;
        break;
    default:
        return QNN_ERR_INVALID_ARG;
    }

    int shift = 0;
    if (e->ptf_shift) {
        if (a_dt != QNN_S8 || e->zp_term) return QNN_ERR_UNSUPPORTED;
        if (e->ptf_max_shift < 0 || e->ptf_max_shift > 3) return QNN_ERR_INVALID_ARG;
        if (!qnn::aligned16(e->ptf_shift)) return QNN_ERR_ALIGNMENT;
        shift = e->ptf_max_shift;
        p.ptf = e->ptf_shift;
    }
    // |acc_c| <= K * 255 * 128 * 2^shift must stay inside int32
    if ((int64_t)K * 255 * 128 * (1 << shift) > (int64_t)INT32_MAX) return QNN_ERR_OVERFLOW_RISK;
    p.chunk_steps = MAX_EXACT_STEPS >> shift;
    p.nchunks = (p.KT + p.chunk_steps - 1) / p.chunk_steps;

    p.status = qnn::status_word();
    if (!p.status) return QNN_ERR_CUDA;
    cudaStream_t s = (cudaStream_t)stream;
    const bool multi = p.nchunks > 1;
    const bool ptf = p.ptf != nullptr;
    if (!multi && !ptf) return launch<256, false, false>(p, s);
    if (!multi && ptf) return launch<256, false, true>(p, s);
    if (multi && !ptf) return launch<128, true, false>(p, s);
    return launch<128, true, true>(p, s);
}
