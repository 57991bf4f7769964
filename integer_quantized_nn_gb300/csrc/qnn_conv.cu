// qnn_conv.cu -- implicit-GEMM quantized convolution (qconv_u4s4, qconv_u8s8,
// qconv_u8u8) and its weight prepack (s4 / s8 filters, and u4 / u8 filters with
// per-filter zero points, taken out at prepack).
//
// [MG conv 算子優化, Fig. 5] a convolution of an (N, IH, IW, C) input with
// (OC, FH, FW, C) filters is the product of the (N*OH*OW) x (FH*FW*C) patch
// matrix with the (FH*FW*C) x OC filter matrix; the implicit form never
// writes the patch matrix: each block re-lays the input out while moving it
// from global to shared memory.  The output is computed transposed, pixels x
// channels, so that a thread's accumulators are consecutive output channels
// of one pixel and pack straight into NHWC bytes or nibbles [MG conv 算子優化:
// output transposition, 16 consecutive 4-bit channels per thread].
//
// Operands on the tensor cores:
//   u4 x s4: a u4 code c zero-extended into a byte is exactly the e4m3
//            encoding of c / 512 (codes 0..7 are the subnormals c * 2^-9, 8..15
//            the first binade), so unpacking is two masks per 8 codes; the s4
//            weights are prepacked as exact e4m3 integers.  kind::f8f6f4 sums
//            the exact products c * w * 2^-9 in fp32 (|sum| < 2^24 * 2^-9 for any
//            K below 139810) and the epilogue multiplies by 512.  The two masks
//            deliver each group of 8 channels in the order 0,2,4,6,1,3,5,7; the
//            weight prepack uses the same order, which leaves every sum unchanged.
//   u8 x s8: bytes to fp16 exactly as in the GEMM (kind::f16), q - 128; u8
//            filters less their zero points (u8u8) reach 255 in magnitude, so
//            their exact fp32 chunks are half as long (512 products).
// Padded taps read the code z_in (the real value 0 [reading of the pages]),
// so the folded zero-point term applies to every tap alike.
#include <cuda_fp8.h>
#include <cudaTypedefs.h>
#include <atomic>
#include <type_traits>
#include "qnn_mma_kernel.cuh"

namespace qnn {
namespace mk {

constexpr int KMAX_U4_EXACT = 139810;  // 2^24 / (15 * 8): exact fp32 sums of u4 x s4 products

// Per-thread im2col cursor: the 4 pixels (rows) this thread fetches in the
// current tile and the (fh, fw, c0) position of its 16-byte group in K.
struct ConvState {
    int img[4];   // n * H of the row's image, or -1 past the last pixel
    int nim[4];   // n
    int ih0[4];
    int iw0[4];
    int c0, fh, fw;
    UnitCursor c;    // the unit being loaded
    uint64_t kinds;  // per staging slot (8 bits): what each of the 4 rows holds, 2 bits each
};

// Places the cursor at linear K position kpos = (fh * FW + fw) * C + c0.
__device__ __forceinline__ void conv_seek(const Params &p, ConvState &st, int kpos)
{
    const int tap = kpos / p.Cin;
    st.c0 = kpos - tap * p.Cin;
    st.fh = tap / p.FW;
    st.fw = tap - st.fh * p.FW;
}

template <int GROUP_ELEMS, int STEP_ELEMS>
__device__ __forceinline__ void conv_cursor(const Params &p, ConvState &st, int j, int sub, int rbase)
{
    if (j == 0) st.c.begin(p);
    else st.c.next(p);
    if (st.c.kl == 0) {
        const int m0 = st.c.mb * BM;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int r = m0 + q * 32 + rbase;
            if (r < p.M) {
                const int n = r / p.OHW;
                const int rem = r - n * p.OHW;
                const int oh = rem / p.OW;
                const int ow = rem - oh * p.OW;
                st.img[q] = n * p.H;
                st.nim[q] = n;
                st.ih0[q] = oh * p.sh - p.ph;
                st.iw0[q] = ow * p.sw - p.pw;
            } else {
                st.img[q] = -1;
                st.nim[q] = 0;
                st.ih0[q] = 0;
                st.iw0[q] = 0;
            }
        }
        conv_seek(p, st, st.c.ks * STEP_ELEMS + sub * GROUP_ELEMS);
    } else if (st.c.ks == 0) {
        conv_seek(p, st, sub * GROUP_ELEMS);  // the K walk wrapped around
    } else {
        st.c0 += STEP_ELEMS;
        while (st.c0 >= p.Cin) {
            st.c0 -= p.Cin;
            if (++st.fw == p.FW) {
                st.fw = 0;
                ++st.fh;
            }
        }
    }
}

// What a row of the unit holds: input bytes fetched by cp.async, the padding
// pattern, or zeros (past the last pixel or past the last tap).
enum { ROW_DATA = 0, ROW_PAD = 1, ROW_ZERO = 2 };

__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// The im2col converters fetch each unit's input rows with cp.async into a
// per-thread staging ring of D units in shared memory ([slot][q][thread] x 16
// bytes), so D - 1 units of loads are in flight while one is converted.
template <int ELEM_BITS, int GROUP_ELEMS, int STEP_ELEMS, int D>
struct ConvStaging : OpBase {
    static constexpr bool CACHE_COLS = true;
    static constexpr bool LAYOUTS = true;
    static constexpr int DEPTH = D;
    static constexpr int DEPTH_MULTI = D;
    static constexpr int STG_BYTES = D * 4 * 128 * 16;
    static constexpr bool TMA_A = false;
    static constexpr bool REG_RING = false;
    struct Unit {};
    using State = ConvState;

    template <int DD>
    __device__ static void load(const Params &p, State &st, const uint4 *stg, int j, bool valid, int sub,
                                int rbase, Unit &u)
    {
        if (valid) {
            conv_cursor<GROUP_ELEMS, STEP_ELEMS>(p, st, j, sub, rbase);
            const int slot = j % DD;
            uint32_t kinds = 0;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                uint32_t kind = ROW_ZERO;
                if (st.img[q] >= 0 && st.fh < p.FH) {
                    const int ih = st.ih0[q] + st.fh;
                    const int iw = st.iw0[q] + st.fw;
                    if (ih < 0 || ih >= p.H || iw < 0 || iw >= p.W) {
                        kind = ROW_PAD;
                    } else {
                        kind = ROW_DATA;
                        const int64_t elem = ((int64_t)(st.img[q] + ih) * p.W + iw) * p.Cin + st.c0;
                        const uint32_t dst = smem_u32(stg + (slot * 4 + q) * 128 + threadIdx.x);
                        cp_async16(dst, p.A + (ELEM_BITS == 4 ? elem / 2 : elem));
                    }
                }
                kinds |= kind << (2 * q);
            }
            const int sh = 8 * slot;
            st.kinds = (st.kinds & ~(0xFFull << sh)) | ((uint64_t)kinds << sh);
        }
        cp_async_commit();  // one group per unit, empty past the end
    }

    // Before a unit is converted: its copy group must have landed.
    template <int DD>
    __device__ static void wait_unit() { cp_async_wait<DD - 1>(); }

    // The 16 input bytes of row q of unit j (after its group has landed).
    __device__ static uint4 fetched(const Params &p, const ConvState &st, const uint4 *stg, int slot, int q,
                                    const Unit &)
    {
        const uint32_t kind = (uint32_t)(st.kinds >> (8 * slot + 2 * q)) & 3u;
        if (kind == ROW_DATA) return stg[(slot * 4 + q) * 128 + threadIdx.x];
        if (kind == ROW_PAD) return make_uint4(p.pad_word, p.pad_word, p.pad_word, p.pad_word);
        return make_uint4(0, 0, 0, 0);
    }
};

// The same im2col fetch into a register ring: each unit's four 16-byte row
// groups are loaded with plain non-coherent loads DEPTH - 1 units ahead
// (padding and zero rows are resolved when the unit is loaded).
template <int ELEM_BITS, int GROUP_ELEMS, int STEP_ELEMS>
struct ConvRegRing : OpBase {
    static constexpr bool CACHE_COLS = true;
    static constexpr bool LAYOUTS = true;
    static constexpr int DEPTH = 4;
    static constexpr int DEPTH_MULTI = 3;
    static constexpr int STG_BYTES = 16;  // no staging ring
    static constexpr bool TMA_A = false;
    static constexpr bool REG_RING = true;
    struct Unit {
        uint4 v[4];
    };
    using State = ConvState;

    template <int DD>
    __device__ static void load(const Params &p, State &st, const uint4 *, int j, bool valid, int sub,
                                int rbase, Unit &u)
    {
        if (!valid) return;
        conv_cursor<GROUP_ELEMS, STEP_ELEMS>(p, st, j, sub, rbase);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            uint4 v = make_uint4(0, 0, 0, 0);
            if (st.img[q] >= 0 && st.fh < p.FH) {
                const int ih = st.ih0[q] + st.fh;
                const int iw = st.iw0[q] + st.fw;
                if (ih < 0 || ih >= p.H || iw < 0 || iw >= p.W) {
                    v = make_uint4(p.pad_word, p.pad_word, p.pad_word, p.pad_word);
                } else if (p.layout == QNN_LAYOUT_NCHW) {
                    // 8-bit codes only (the host sends 4-bit NCHW inputs through the
                    // expansion pre-pass): the group's 16 channels, one per plane
                    const int64_t plane = (int64_t)p.H * p.W;
                    const uint8_t *src = p.A + ((int64_t)st.nim[q] * p.Cin + st.c0) * plane + (int64_t)ih * p.W + iw;
                    uint32_t w4[4] = {0, 0, 0, 0};
#pragma unroll
                    for (int j = 0; j < 16; ++j) w4[j >> 2] |= (uint32_t)__ldg(src + j * plane) << (8 * (j & 3));
                    v = make_uint4(w4[0], w4[1], w4[2], w4[3]);
                } else {
                    // NHWC; NCHW64 keeps a group's channels together inside its 64-channel block
                    const int64_t elem =
                        p.layout == QNN_LAYOUT_NHWC
                            ? ((int64_t)(st.img[q] + ih) * p.W + iw) * p.Cin + st.c0
                            : ((((int64_t)st.nim[q] * (p.Cin >> 6) + (st.c0 >> 6)) * p.H + ih) * p.W + iw) * 64 +
                                  (st.c0 & 63);
                    v = ldg_nc_v4(p.A + (ELEM_BITS == 4 ? elem / 2 : elem));
                }
            }
            u.v[q] = v;
        }
    }

    template <int DD>
    __device__ static void wait_unit() {}

    __device__ static uint4 fetched(const Params &, const ConvState &, const uint4 *, int, int q, const Unit &u)
    {
        return u.v[q];
    }
};

// D = 0: register ring; D > 0: shared-memory staging ring of D units.
template <int ELEM_BITS, int GROUP_ELEMS, int STEP_ELEMS, int D>
using ConvFetch = typename std::conditional<D == 0, ConvRegRing<ELEM_BITS, GROUP_ELEMS, STEP_ELEMS>,
                                            ConvStaging<ELEM_BITS, GROUP_ELEMS, STEP_ELEMS, D>>::type;

template <int D>
struct ConvU4Op : ConvFetch<4, 32, 128, D> {
    using Base = ConvFetch<4, 32, 128, D>;
    static constexpr bool F8 = true;
    static constexpr int SCALE_LOG2 = 9;

    template <int DD>
    __device__ static void store(const Params &p, ConvState &st, const uint4 *stg, uint32_t a_stage, int j,
                                 int sub, int rbase, const typename Base::Unit &u)
    {
        Base::template wait_unit<DD>();
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int row = q * 32 + rbase;
            const uint4 v = Base::fetched(p, st, stg, j % DD, q, u);
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
            uint32_t b[8];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                b[2 * i] = w[i] & 0x0F0F0F0Fu;             // channels 0, 2, 4, 6 of the 8
                b[2 * i + 1] = (w[i] >> 4) & 0x0F0F0F0Fu;  // channels 1, 3, 5, 7
            }
            const uint32_t rowaddr = a_stage + row * ROW_BYTES;
            sts_v4(rowaddr + (((2 * sub) ^ (row & 7)) << 4), b[0], b[1], b[2], b[3]);
            sts_v4(rowaddr + (((2 * sub + 1) ^ (row & 7)) << 4), b[4], b[5], b[6], b[7]);
        }
    }
};

// ---- 1x1 u4 conv fed by copies of the packed input -------------------------------
// A 1x1, stride-1, unpadded convolution is the GEMM of the NHWC pixel matrix
// [N*H*W, C] with the filters [MG conv 算子優化: the implicit GEMM of a 1x1
// filter needs no img2col].  The packed u4 input is brought to shared memory as
// it lies in global memory, 128 pixels x 256 channels (16 KB) per unit, into a
// staging ring of DEPTH slots, by asynchronous copies; the converter warps then
// unpack the nibbles into the e4m3 operand stage shared-memory to shared-memory
// [MG conv 算子優化: INT4 values unpacked on their way to the tensor cores], and
// the filters stay resident.  Global memory is read once, 16 bytes at a time
// or in 16 KB boxes, and never through registers.
//   THREAD_COPY (C = 256, a pixel's codes are one 128-byte row): every
//     converter thread copies (cp.async, 16 bytes each) exactly the 8 chunks it
//     will unpack, so no thread waits for another's copies.
//   otherwise (C a multiple of 256): one tiled 2-D TMA box of 128 pixels x 128
//     bytes per unit (128-byte swizzled), issued by warp 0 once the four warps
//     have released the slot; full / empty mbarriers per slot.
template <bool THREAD_COPY>
struct ConvU4PackedOp : OpBase {
    static constexpr bool CACHE_COLS = true;
    static constexpr bool LAYOUTS = false;     // taken for NHWC tensors only
    static constexpr bool TMA_A = false;
    static constexpr bool F8 = true;
    static constexpr int SCALE_LOG2 = 9;
    static constexpr int SUB = 2;              // two K steps of 128 channels per unit
    static constexpr int STAGES = 3;
    static constexpr bool RESB = true;
    static constexpr int B_RES_BYTES = 32768;  // filters of up to 512 channels x 64 outputs
    static constexpr bool ROTATE_K = false;    // resident filters are indexed by the unit's K position
    static constexpr int DEPTH = 4;            // staging slots (units of packed input in flight)
    static constexpr int DEPTH_MULTI = 4;
    static constexpr bool REG_RING = false;
    static constexpr int SLOT = BM * 128;      // 128 pixels x 128 packed bytes
    static constexpr int STG_BYTES = DEPTH * SLOT + 1024;  // slots, then 2 * DEPTH mbarriers
    struct Unit {};
    struct State {
        UnitCursor c;
    };

    __device__ static uint64_t *slot_full(uint4 *stg) { return reinterpret_cast<uint64_t *>(stg + DEPTH * SLOT / 16); }
    __device__ static uint64_t *slot_empty(uint4 *stg) { return slot_full(stg) + DEPTH; }

    __device__ static void init(uint4 *stg)
    {
        for (int i = 0; i < DEPTH; ++i) {
            mbar_init(smem_u32(slot_full(stg) + i), 1);
            mbar_init(smem_u32(slot_empty(stg) + i), 4);  // the four converter warps
        }
    }

    // Unit jn's input into slot jn % DEPTH (valid: jn is one of this CTA's units).
    template <int DD>
    __device__ static bool load(const Params &p, State &st, const uint4 *stg_c, int jn, bool valid, int sub, int rbase,
                                Unit &)
    {
        uint4 *stg = const_cast<uint4 *>(stg_c);
        const int slot = jn % DEPTH;
        if constexpr (THREAD_COPY) {
            // one copy group per unit (empty past the end); rows past the last
            // pixel are zero-filled
            if (valid) {
                if (jn == 0) st.c.begin(p, false);
                else st.c.next(p);
                const uint32_t dst = smem_u32(stg + slot * (SLOT / 16));
#pragma unroll
                for (int t = 0; t < SUB; ++t) {
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const int row = q * 32 + rbase;
                        const int pix = st.c.mb * BM + row;
                        const int chunk = 4 * t + sub;
                        const bool in = pix < p.M;
                        const uint8_t *src = p.A + (int64_t)(in ? pix : 0) * 128 + chunk * 16;
                        asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst + row * 128 + chunk * 16),
                                     "l"(src), "r"(in ? 16 : 0)
                                     : "memory");
                    }
                }
            }
            asm volatile("cp.async.commit_group;" ::: "memory");
            return true;
        } else {
            if (!valid) return true;
            if (jn == 0) st.c.begin(p, false);
            else st.c.next(p);
            if (threadIdx.x >= 32) return true;
            const uint32_t use = (uint32_t)(jn / DEPTH);
            if (!warp_wait_idle(smem_u32(slot_empty(stg) + slot), (use & 1u) ^ 1u, p.status)) return false;
            if (threadIdx.x == 0) {
                const uint32_t bar = smem_u32(slot_full(stg) + slot);
                mbar_arrive_expect_tx(bar, (uint32_t)SLOT);
                tma_load_2d(smem_u32(stg + slot * (SLOT / 16)), &p.tmap, st.c.ks * 128, st.c.mb * BM, bar);
            }
            __syncwarp();
            return true;
        }
    }

    // Unit j: wait for its input, unpack 4 rows x 2 K steps of 32 channels per
    // thread (two masks per 8 codes: channels 0,2,4,6 then 1,3,5,7, the order of
    // the weight image), then release the slot.
    template <int DD>
    __device__ static bool store(const Params &p, State &, const uint4 *stg_c, uint32_t a_stage, int j, int sub,
                                 int rbase, const Unit &)
    {
        uint4 *stg = const_cast<uint4 *>(stg_c);
        const int slot = j % DEPTH;
        if constexpr (THREAD_COPY) {
            asm volatile("cp.async.wait_group %0;" ::"n"(DEPTH - 1) : "memory");
        } else {
            if (!warp_wait_idle(smem_u32(slot_full(stg) + slot), (uint32_t)(j / DEPTH) & 1u, p.status)) return false;
        }
        const uint32_t src = smem_u32(stg + slot * (SLOT / 16));
#pragma unroll
        for (int t = 0; t < SUB; ++t) {
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int row = q * 32 + rbase;
                const int chunk = THREAD_COPY ? 4 * t + sub : (4 * t + sub) ^ (row & 7);
                const uint4 v = lds_v4(src + row * 128 + (chunk << 4));
                const uint32_t w[4] = {v.x, v.y, v.z, v.w};
                uint32_t b[8];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    b[2 * i] = w[i] & 0x0F0F0F0Fu;
                    b[2 * i + 1] = (w[i] >> 4) & 0x0F0F0F0Fu;
                }
                const uint32_t rowaddr = a_stage + t * (BM * ROW_BYTES) + row * ROW_BYTES;
                sts_v4(rowaddr + (((2 * sub) ^ (row & 7)) << 4), b[0], b[1], b[2], b[3]);
                sts_v4(rowaddr + (((2 * sub + 1) ^ (row & 7)) << 4), b[4], b[5], b[6], b[7]);
            }
        }
        if constexpr (!THREAD_COPY) {
            __syncwarp();
            if ((threadIdx.x & 31) == 0) mbar_arrive(smem_u32(slot_empty(stg) + slot));
        }
        return true;
    }
};

template <int D>
struct ConvU8Op : ConvFetch<8, 16, 64, D> {
    using Base = ConvFetch<8, 16, 64, D>;
    static constexpr bool F8 = false;
    static constexpr int SCALE_LOG2 = 0;

    template <int DD>
    __device__ static void store(const Params &p, ConvState &st, const uint4 *stg, uint32_t a_stage, int j,
                                 int sub, int rbase, const typename Base::Unit &u)
    {
        Base::template wait_unit<DD>();
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int row = q * 32 + rbase;
            const uint4 v = Base::fetched(p, st, stg, j % DD, q, u);
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
            uint32_t h[8];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                h[2 * i] = hsub2_u32(prmt(w[i], 0x64646464u, 0x4140u), 0x64806480u);
                h[2 * i + 1] = hsub2_u32(prmt(w[i], 0x64646464u, 0x4342u), 0x64806480u);
            }
            const uint32_t rowaddr = a_stage + row * ROW_BYTES;
            sts_v4(rowaddr + (((2 * sub) ^ (row & 7)) << 4), h[0], h[1], h[2], h[3]);
            sts_v4(rowaddr + (((2 * sub + 1) ^ (row & 7)) << 4), h[4], h[5], h[6], h[7]);
        }
    }
};

// ---- weight prepack of s4 filters into the e4m3 operand image -----------------
// Image: for each 256-filter block and K step of 128, 256 rows x 128 bytes,
// 128-byte swizzled, zero beyond OC and K; byte position 8g + j of a row holds
// the weight of K index 8g + {0,2,4,6,1,3,5,7}[j].
// With z_w (u4 filters with per-filter zero points) the weight is the centred
// nibble u - z_w[oc] in [-15, 15], exact in e4m3 like the s4 values; else the
// nibble read as s4.
__device__ __forceinline__ int filter_value(uint8_t byte, int k, const int32_t *z_w, int n)
{
    int v = (k & 1) ? (byte >> 4) : (byte & 15);
    if (z_w) return v - z_w[n];
    return v >= 8 ? v - 16 : v;
}

__global__ void prepack_w_s4_kernel(const uint8_t *__restrict__ W, int OC, int K, int KT,
                                    uint8_t *__restrict__ out, int64_t nchunks, const int32_t *__restrict__ z_w)
{
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < nchunks;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int cphys = (int)(i & 7);
        const int64_t row_all = i >> 3;
        const int r = (int)(row_all % 256);
        const int64_t blk = row_all / 256;
        const int ks = (int)(blk % KT);
        const int nb = (int)(blk / KT);
        const int c = cphys ^ (r & 7);
        const int n = nb * 256 + r;
        uint32_t w[4] = {0, 0, 0, 0};
#pragma unroll
        for (int b = 0; b < 16; ++b) {
            const int kpos = ks * 128 + c * 16 + b;
            const int j = kpos & 7;
            const int k = (kpos & ~7) + ((j < 4) ? 2 * j : 2 * (j - 4) + 1);
            uint32_t code = 0;
            if (n < OC && k < K) {
                const int v = filter_value(W[((int64_t)n * K + k) >> 1], k, z_w, n);
                code = (uint32_t)__nv_cvt_float_to_fp8((float)v, __NV_SATFINITE, __NV_E4M3);
            }
            w[b >> 2] |= code << (8 * (b & 3));
        }
        *reinterpret_cast<uint4 *>(out + i * 16) = make_uint4(w[0], w[1], w[2], w[3]);
    }
}

// colsum[oc] = sum over (fh, fw, c) of the s4 weights; one warp per filter.
__global__ void colsum_s4_kernel(const uint8_t *__restrict__ W, int OC, int K, int32_t *__restrict__ colsum,
                                 const int32_t *__restrict__ z_w)
{
    const int warp = (int)((blockIdx.x * (int64_t)blockDim.x + threadIdx.x) >> 5);
    const int lane = threadIdx.x & 31;
    if (warp >= OC) return;
    int32_t s = 0;
    for (int k = lane; k < K; k += 32) s += filter_value(W[((int64_t)warp * K + k) >> 1], k, z_w, warp);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    if (lane == 0) colsum[warp] = s;
}

inline bool geom_ok(const qnn_conv_geom *g)
{
    if (!g) return false;
    if (g->N <= 0 || g->H <= 0 || g->W <= 0 || g->C <= 0 || g->OC <= 0 || g->FH <= 0 || g->FW <= 0)
        return false;
    if (g->pad_h < 0 || g->pad_w < 0 || g->stride_h <= 0 || g->stride_w <= 0) return false;
    const int oh = (g->H + 2 * g->pad_h - g->FH) / g->stride_h + 1;
    const int ow = (g->W + 2 * g->pad_w - g->FW) / g->stride_w + 1;
    if (g->H + 2 * g->pad_h < g->FH || g->W + 2 * g->pad_w < g->FW || oh <= 0 || ow <= 0) return false;
    if (g->layout < QNN_LAYOUT_NHWC || g->layout > QNN_LAYOUT_NCHW64) return false;
    if (g->layout == QNN_LAYOUT_NCHW64 && (g->C % 64 != 0 || g->OC % 64 != 0)) return false;
    const int64_t rows = (int64_t)g->N * oh * ow;
    const int64_t K = (int64_t)g->FH * g->FW * g->C;
    const int64_t in = (int64_t)g->N * g->H * g->W * g->C;
    return rows < (1ll << 31) && K < (1ll << 24) && in < (1ll << 40);
}

inline size_t packed_w_u4_bytes(const qnn_conv_geom *g)
{
    const int K = g->FH * g->FW * g->C;
    return (size_t)((g->OC + 255) / 256) * (size_t)((K + 127) / 128) * (size_t)gemm::B_STAGE_BYTES;
}

inline size_t round1k(size_t b) { return (b + 1023) & ~(size_t)1023; }

// The TMA conv's weight image (0 when C is not a multiple of 32).
inline size_t tma_w_bytes(const qnn_conv_geom *g)
{
    if (g->C % 32 != 0) return 0;
    const int cb = (g->C % 128 == 0) ? 128 : (g->C % 64 == 0 ? 64 : 32);
    return (size_t)((g->OC + 255) / 256) * (size_t)g->FH * g->FW * (g->C / cb) * 256 * cb;
}

// W_packed of s4 weights: [fused-path image][TMA image][colsum, int32 x OC], 1 KB aligned parts.
inline size_t tma_w_offset(const qnn_conv_geom *g) { return round1k(packed_w_u4_bytes(g)); }
inline size_t colsum_offset(const qnn_conv_geom *g) { return tma_w_offset(g) + round1k(tma_w_bytes(g)); }
inline size_t packed_w_u4_total(const qnn_conv_geom *g) { return colsum_offset(g) + round1k((size_t)g->OC * 4); }

// W_packed of 8-bit filters: [GEMM image of [OC, K] + its trailer][colsum, int32 x OC], 1 KB aligned parts.
inline size_t colsum8_offset(const qnn_conv_geom *g)
{
    return round1k(gemm::packed_b_bytes(g->OC, g->FH * g->FW * g->C));
}
inline size_t packed_w_8_total(const qnn_conv_geom *g) { return colsum8_offset(g) + round1k((size_t)g->OC * 4); }

// Staging depth: 8 units for tiles up to 128 columns (64 KB of staging), 2 for
// 256-column tiles, whose units carry 4x the MMA work (and shared memory is full).
// ---- u4 conv fed by TMA (with a workspace) --------------------------------------
// A pre-pass expands the packed u4 input into bytes holding the e4m3 encoding of
// (q - z_in) / 512 (exact: |q - z_in| <= 15; the byte is |q - z_in| with the
// sign in bit 7), so that a zero byte is the real value 0.  The implicit GEMM
// then needs no re-encoding: for each output tile -- TN images x TH rows x TW
// columns of output pixels, at most 128 -- and each unit -- one filter tap x CB
// input channels -- one tiled TMA box of the expanded tensor, shifted by the
// tap and strided by the conv stride, lands as the swizzled K-major A stage;
// taps that fall in the padding read zeros.  The kernel's sum is therefore
// sum (q - z_in) * w; the epilogue adds z_in * colsum back before subtracting
// zp_term, so acc_c is the same as on the fused path.

// Bytes (= input channels) per operand row for C channels.
inline int tma_cb(int C) { return C % 128 == 0 ? 128 : (C % 64 == 0 ? 64 : 32); }

// Resident weights (64-column tiles, the whole filter bank in at most 64 KB).
constexpr int TMA_B_RES = 65536;

// Stages that fit in about 192 KB of shared memory with `t` K steps per
// stage, streamed or resident weights.
constexpr int tma_stages(int cb, int tbn, int t, bool resb, int bank = TMA_B_RES)
{
    const int per = t * BM * cb + (resb ? 0 : t * tbn * cb);
    const int n = (196608 - (resb ? bank : 0)) / per;
    return n > 15 ? 15 : n;
}

// Resident filter bank of the fp16 (u8) TMA conv: up to 10 K steps of 64 channels
// for 64 filters (a 3x3 filter over 64 channels is 9).
constexpr int TMA_B_RES16 = 81920;

// EB: bytes per element of the expanded input -- 1 (e4m3 of u4 codes, kind::f8f6f4)
// or 2 (fp16 of u8 codes less z_in, kind::f16); a row of a stage is CB elements.
template <int CB, int TBN_, int T, bool RES, int EB = 1>
struct ConvTmaOp : OpBase {
    static constexpr bool CACHE_COLS = true;
    static constexpr bool LAYOUTS = true;
    static constexpr bool TMA_A = true;
    static constexpr bool F8 = EB == 1;
    static constexpr int SCALE_LOG2 = EB == 1 ? 9 : 0;
    static constexpr int ROW = CB * EB;
    static constexpr int SUB = T;
    static constexpr bool RESB = RES;
    static constexpr int B_RES_BYTES = RES ? (EB == 2 ? TMA_B_RES16 : TMA_B_RES) : 0;
    static constexpr int STAGES = tma_stages(CB * EB, TBN_, T, RES, B_RES_BYTES);
    static constexpr int STG_BYTES = 16;

    __device__ static uint32_t a_bytes(const Params &p) { return (uint32_t)(ROW * p.TW * p.TH * p.TN); }

    // Units walk K from 0 in every tile (no per-CTA rotation), so the tap and
    // channel block advance by counting; a tile's box origin is decoded once.
    static constexpr bool ROTATE_K = false;
    struct PState {
        int mb = -1;            // tile whose origin is cached
        int w0, h0, n0;         // box origin of tap (0, 0), channel block 0
        int fh, fw, cblk;       // position of the next unit in K
    };

    // Box of K step t of unit c (steps are walked in order: t = 0 .. SUB - 1 of each unit).
    __device__ static void load_a(const Params &p, const UnitCursor &c, PState &ps, int t, uint32_t dst,
                                  uint32_t bar)
    {
        if (c.mb != ps.mb) {
            const int tx = c.mb % p.tiles_x;
            const int rest = c.mb / p.tiles_x;
            const int ty = rest % p.tiles_y;
            const int tn = rest / p.tiles_y;
            ps.mb = c.mb;
            ps.w0 = tx * p.TW * p.sw - p.pw;
            ps.h0 = ty * p.TH * p.sh - p.ph;
            ps.n0 = tn * p.TN;
        }
        if (c.ks == 0 && t == 0) {
            ps.fh = 0;
            ps.fw = 0;
            ps.cblk = 0;
        }
        tma_load_4d(dst, &p.tmap, ps.cblk * CB, ps.w0 + ps.fw, ps.h0 + ps.fh, ps.n0, bar);
        if (++ps.cblk == p.cbn) {
            ps.cblk = 0;
            if (++ps.fw == p.FW) {
                ps.fw = 0;
                ++ps.fh;
            }
        }
    }

    // Row r of a tile is output pixel (n, oh, ow) in box order (w fastest).
    struct RowInfo {
        int nl, hl, wl;  // position in the box; nl = TN marks a row outside it
    };
    __device__ static RowInfo row_info(const Params &p, int r)
    {
        const int per = p.TW * p.TH;
        RowInfo ri;
        ri.nl = r / per;
        const int rr = r - ri.nl * per;
        ri.hl = rr / p.TW;
        ri.wl = rr - ri.hl * p.TW;
        return ri;
    }
    // Output row of box row ri in tile mb, or M (skipped) outside the output.
    __device__ static int out_row(const Params &p, int mb, const RowInfo &ri)
    {
        const int tx = mb % p.tiles_x;
        const int rest = mb / p.tiles_x;
        const int ty = rest % p.tiles_y;
        const int tn = rest / p.tiles_y;
        const int n = tn * p.TN + ri.nl;
        const int oh = ty * p.TH + ri.hl;
        const int ow = tx * p.TW + ri.wl;
        if (ri.nl >= p.TN || n >= p.Nimg || oh >= p.OH || ow >= p.OW) return p.M;
        return (n * p.OH + oh) * p.OW + ow;
    }
};

// Input expansion: 16 packed bytes (32 u4 codes, low nibble first) per thread
// -> 32 bytes of e4m3((q - z) / 512) in channel order: the byte |q - z| with
// the sign in bit 7.  Four codes are handled per 32-bit operation: biasing
// every byte by 16 keeps q + 16 - z in 1..31, so bytes never borrow from one
// another; bit 4 then tells q >= z.
__device__ __forceinline__ uint32_t e4m3_centred4(uint32_t q4, uint32_t zz)
{
    const uint32_t d = (q4 | 0x10101010u) - zz;               // q + 16 - z per byte
    const uint32_t ge = (d >> 4) & 0x01010101u;               // 1 where q >= z
    const uint32_t m = ge * 0xFFu;                            // 0xFF where q >= z
    const uint32_t pos = d & 0x0F0F0F0Fu;                     // q - z (q >= z)
    const uint32_t neg = ((0x10101010u - pos) & 0x0F0F0F0Fu) | 0x80808080u;  // 0x80 | (z - q) (q < z)
    return (pos & m) | (neg & ~m);
}

__global__ void expand_u4_kernel(const uint8_t *__restrict__ in, int64_t n16, uint32_t z, uint8_t *__restrict__ out)
{
    const uint32_t zz = z * 0x01010101u;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n16;
         i += (int64_t)gridDim.x * blockDim.x) {
        const uint4 v = ldg_nc_v4(in + i * 16);
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
        uint32_t o[8];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const uint32_t ev = e4m3_centred4(w[j] & 0x0F0F0F0Fu, zz);         // codes 0, 2, 4, 6
            const uint32_t od = e4m3_centred4((w[j] >> 4) & 0x0F0F0F0Fu, zz);  // codes 1, 3, 5, 7
            o[2 * j] = prmt(ev, od, 0x5140u);      // codes 0, 1, 2, 3
            o[2 * j + 1] = prmt(ev, od, 0x7362u);  // codes 4, 5, 6, 7
        }
        uint4 *dst = reinterpret_cast<uint4 *>(out + i * 32);
        dst[0] = make_uint4(o[0], o[1], o[2], o[3]);
        dst[1] = make_uint4(o[4], o[5], o[6], o[7]);
    }
}

// The same expansion from inputs in the other layouts, written in NHWC (the
// convolution reads taps of the NHWC bytes); e4m3 of (q - z) / 512 is the byte
// |q - z| with the sign in bit 7.
__device__ __forceinline__ uint32_t e4m3_centred1(uint32_t q, uint32_t z)
{
    return q >= z ? q - z : (0x80u | (z - q));
}

// NCHW64: [N][C / 64][H][W][32 bytes] -> [N][H][W][C]; one thread per 16 input
// bytes (32 channels of one pixel), 32 output bytes.
__global__ void expand_u4_nchw64_kernel(const uint8_t *__restrict__ in, int64_t n16, int HW, int CB, uint32_t z,
                                        uint8_t *__restrict__ out)
{
    const uint32_t zz = z * 0x01010101u;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n16;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t blk = i >> 1;  // (n, cb, pixel)
        const int half = (int)(i & 1);
        const int pix = (int)(blk % HW);
        const int64_t t = blk / HW;
        const int cb = (int)(t % CB);
        const int64_t n = t / CB;
        const uint4 v = ldg_nc_v4(in + i * 16);
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
        uint32_t o[8];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const uint32_t ev = e4m3_centred4(w[j] & 0x0F0F0F0Fu, zz);
            const uint32_t od = e4m3_centred4((w[j] >> 4) & 0x0F0F0F0Fu, zz);
            o[2 * j] = prmt(ev, od, 0x5140u);
            o[2 * j + 1] = prmt(ev, od, 0x7362u);
        }
        uint4 *dst = reinterpret_cast<uint4 *>(out + ((n * HW + pix) * (int64_t)CB * 64 + cb * 64 + half * 32));
        dst[0] = make_uint4(o[0], o[1], o[2], o[3]);
        dst[1] = make_uint4(o[4], o[5], o[6], o[7]);
    }
}

// NCHW: [N][C][H][W / 2 bytes] -> [N][H][W][C]; one block per image row (n, h):
// the row of every channel plane is read into shared memory (C * W / 2 bytes),
// then each thread writes 16 channels of one pixel (16 bytes).
__global__ void expand_u4_nchw_kernel(const uint8_t *__restrict__ in, int H, int W, int C, uint32_t z,
                                      uint8_t *__restrict__ out)
{
    extern __shared__ uint8_t rowbuf[];
    const int n = blockIdx.x / H;
    const int h = blockIdx.x - n * H;
    const int rb = W / 2;  // bytes of one plane row
    for (int i = threadIdx.x; i < C * rb; i += blockDim.x) {
        const int c = i / rb;
        const int x = i - c * rb;
        rowbuf[i] = __ldg(in + (((int64_t)n * C + c) * H + h) * rb + x);
    }
    __syncthreads();
    const int groups = C / 16;
    uint8_t *orow = out + ((int64_t)n * H + h) * W * (int64_t)C;
    for (int i = threadIdx.x; i < W * groups; i += blockDim.x) {
        const int w = i / groups;
        const int c0 = (i - w * groups) * 16;
        uint32_t o[4] = {0, 0, 0, 0};
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            const uint32_t q = (rowbuf[(c0 + j) * rb + (w >> 1)] >> (4 * (w & 1))) & 15u;
            o[j >> 2] |= e4m3_centred1(q, z) << (8 * (j & 3));
        }
        *reinterpret_cast<uint4 *>(orow + (int64_t)w * C + c0) = make_uint4(o[0], o[1], o[2], o[3]);
    }
}

// u8 codes -> fp16 values q - z (exact: |q - z| <= 255), written NHWC, for the
// tensor-copy path of the u8 convs: each byte is placed in the mantissa of fp16
// 1024 and 1024 + z subtracted.  A zero fp16 (the tensor copy's fill outside the
// input) is then the real value 0, the padding reading.
__device__ __forceinline__ void u8_to_half_centred(uint4 v, uint32_t zh2, uint32_t (&h)[8])
{
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        h[2 * i] = hsub2_u32(prmt(w[i], 0x64646464u, 0x4140u), zh2);
        h[2 * i + 1] = hsub2_u32(prmt(w[i], 0x64646464u, 0x4342u), zh2);
    }
}

// NHWC or NCHW64 input: one thread per 16 input bytes (16 channels of one pixel).
template <bool NCHW64>
__global__ void expand_u8_kernel(const uint8_t *__restrict__ in, int64_t n16, int HW, int C, uint32_t zh2,
                                 uint8_t *__restrict__ out)
{
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n16;
         i += (int64_t)gridDim.x * blockDim.x) {
        int64_t o;
        if (NCHW64) {
            const int64_t blk = i >> 2;  // (n, cb, pixel)
            const int quarter = (int)(i & 3);
            const int pix = (int)(blk % HW);
            const int64_t t = blk / HW;
            const int CB = C / 64;
            const int cb = (int)(t % CB);
            const int64_t n = t / CB;
            o = (n * HW + pix) * (int64_t)C + cb * 64 + quarter * 16;
        } else {
            o = i * 16;
        }
        uint32_t h[8];
        u8_to_half_centred(ldg_nc_v4(in + i * 16), zh2, h);
        uint4 *dst = reinterpret_cast<uint4 *>(out + o * 2);
        dst[0] = make_uint4(h[0], h[1], h[2], h[3]);
        dst[1] = make_uint4(h[4], h[5], h[6], h[7]);
    }
}

// NCHW input: one block per image row (n, h); the row of every channel plane
// through shared memory (C * W bytes), then 16 channels of one pixel per thread.
__global__ void expand_u8_nchw_kernel(const uint8_t *__restrict__ in, int H, int W, int C, uint32_t zh2,
                                      uint8_t *__restrict__ out)
{
    extern __shared__ uint8_t rowbuf8[];
    const int n = blockIdx.x / H;
    const int h = blockIdx.x - n * H;
    for (int i = threadIdx.x; i < C * W; i += blockDim.x) {
        const int c = i / W;
        const int x = i - c * W;
        rowbuf8[i] = __ldg(in + (((int64_t)n * C + c) * H + h) * W + x);
    }
    __syncthreads();
    const int groups = C / 16;
    uint8_t *orow = out + (((int64_t)n * H + h) * W * (int64_t)C) * 2;
    for (int i = threadIdx.x; i < W * groups; i += blockDim.x) {
        const int w = i / groups;
        const int c0 = (i - w * groups) * 16;
        uint32_t b4[4] = {0, 0, 0, 0};
#pragma unroll
        for (int j = 0; j < 16; ++j) b4[j >> 2] |= (uint32_t)rowbuf8[(c0 + j) * W + w] << (8 * (j & 3));
        uint32_t hh[8];
        u8_to_half_centred(make_uint4(b4[0], b4[1], b4[2], b4[3]), zh2, hh);
        uint4 *dst = reinterpret_cast<uint4 *>(orow + ((int64_t)w * C + c0) * 2);
        dst[0] = make_uint4(hh[0], hh[1], hh[2], hh[3]);
        dst[1] = make_uint4(hh[4], hh[5], hh[6], hh[7]);
    }
}

// Weight image of the TMA conv: for each 256-filter block and unit (tap, CB
// channels), 256 rows x CB bytes of e4m3 weights in channel order, in the
// CB-byte swizzled layout (chunk c of row r at chunk c ^ ((r * CB / 128) %
// (CB / 16))); zero beyond OC.  One thread per 16-byte chunk.
__global__ void prepack_w_s4_tma_kernel(const uint8_t *__restrict__ W, int OC, int C, int CB, int KT,
                                        uint8_t *__restrict__ out, int64_t nchunks, const int32_t *__restrict__ z_w)
{
    const int cpr = CB / 16;
    const int cbn = C / CB;
    const int K = KT * CB;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < nchunks;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int cphys = (int)(i % cpr);
        const int64_t row_all = i / cpr;
        const int r = (int)(row_all % 256);
        const int64_t blk = row_all / 256;
        const int ks = (int)(blk % KT);
        const int nb = (int)(blk / KT);
        const int c = cphys ^ (((r * CB) >> 7) & (cpr - 1));
        const int n = nb * 256 + r;
        const int tap = ks / cbn;
        const int k0 = tap * C + (ks - tap * cbn) * CB + c * 16;
        uint32_t w[4] = {0, 0, 0, 0};
        if (n < OC) {
#pragma unroll
            for (int b = 0; b < 16; ++b) {
                const int k = k0 + b;
                const int v = filter_value(W[((int64_t)n * K + k) >> 1], k, z_w, n);
                const uint32_t code = (uint32_t)__nv_cvt_float_to_fp8((float)v, __NV_SATFINITE, __NV_E4M3);
                w[b >> 2] |= code << (8 * (b & 3));
            }
        }
        *reinterpret_cast<uint4 *>(out + i * 16) = make_uint4(w[0], w[1], w[2], w[3]);
    }
}

template <template <int> class Op, int TBN>
qnn_status conv_launch(const Params &p, cudaStream_t s)
{
    if constexpr (!Op<0>::F8) {
        // K cut into exact chunks: int32 chunk sums of 64 columns per thread
        if (p.nchunks > 1) return launch<Op<0>, 128, true>(p, s);
    }
    return launch<Op<0>, TBN, false>(p, s);
}

// Output tile shape for the TMA conv: TW x TH x TN pixels (at most 128, box
// sides within the TMA limit of 256 elements after striding) that wastes the
// fewest of the 128 accumulator rows over the whole output; ties go to the
// wider tile (longer contiguous input rows).
inline void choose_tiles(int N, int OH, int OW, int sw, int sh, int &TW, int &TH, int &TN, bool even_tw = false)
{
    int64_t best = -1;
    TW = TH = TN = 1;
    for (int tw = even_tw ? 2 : 1; tw <= 128 && tw * sw <= 256; tw += even_tw ? 2 : 1) {
        for (int th = 1; tw * th <= 128 && th * sh <= 256; ++th) {
            int tn = 128 / (tw * th);
            if (tn > N) tn = N;
            const int64_t tiles = (int64_t)((OW + tw - 1) / tw) * ((OH + th - 1) / th) * ((N + tn - 1) / tn);
            // score: fewest tiles; then the wider tile
            const int64_t score = (int64_t)1 << 40;
            const int64_t sc = score - tiles * 1024 + tw;
            if (sc > best) {
                best = sc;
                TW = tw;
                TH = th;
                TN = tn;
            }
        }
    }
}

// The driver's tensor-map encoder, looked up once through the runtime (the
// library does not link the driver library, so that it loads on hosts
// without a GPU driver); nullptr if unavailable.
static PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder()
{
    static std::atomic<PFN_cuTensorMapEncodeTiled_v12000> fn{nullptr};
    PFN_cuTensorMapEncodeTiled_v12000 f = fn.load(std::memory_order_acquire);
    if (!f) {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess || !ptr) {
            (void)cudaGetLastError();
            return nullptr;
        }
        f = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
        fn.store(f, std::memory_order_release);
    }
    return f;
}

template <int CB, int TBN, int T, bool RES>
qnn_status conv_tma_launch(Params p, cudaStream_t s)
{
    p.KT /= T;  // units per tile
    p.chunk_steps = p.KT;
    return launch<ConvTmaOp<CB, TBN, T, RES>, TBN, false>(p, s);
}

// The u8 convs on the expanded fp16 input: one K step (64 channels of one tap)
// per unit, streamed weights (the GEMM image of the filters), exact chunks as
// long as the weight image's trailer certifies for activations up to p.amax.
template <int TBN>
qnn_status conv_tma_u8_launch(Params p, bool wide_w, cudaStream_t s)
{
    // the host's bound, for |q - z_in| <= 255 and |w| <= 128 (s8) or 255 (u8 less z_w)
    p.chunk_steps = wide_w ? 4 : 8;
    p.nchunks = (p.KT + p.chunk_steps - 1) / p.chunk_steps;
    if (TBN == 64 && (int64_t)p.KT * TBN * 128 <= TMA_B_RES16)
        return launch<ConvTmaOp<64, TBN, 1, true, 2>, TBN, true>(p, s);  // filters resident
    return launch<ConvTmaOp<64, TBN, 1, false, 2>, TBN, true>(p, s);
}

// 64-column tiles group 3, 2 or 1 K steps per unit and keep the weights
// resident when they fit; wider tiles stream one step per unit.
template <int TBN>
qnn_status conv_tma_dispatch(const Params &p, int cb, cudaStream_t s)
{
    if constexpr (TBN == 64) {
        const int steps = p.KT;
        if ((int64_t)steps * TBN * cb <= TMA_B_RES) {
            const int t = steps % 3 == 0 ? 3 : (steps % 2 == 0 ? 2 : 1);
            if (cb == 128) {
                if (t == 3) return conv_tma_launch<128, TBN, 3, true>(p, s);
                if (t == 2) return conv_tma_launch<128, TBN, 2, true>(p, s);
                return conv_tma_launch<128, TBN, 1, true>(p, s);
            }
            if (cb == 64) {
                if (t == 3) return conv_tma_launch<64, TBN, 3, true>(p, s);
                if (t == 2) return conv_tma_launch<64, TBN, 2, true>(p, s);
                return conv_tma_launch<64, TBN, 1, true>(p, s);
            }
            if (t == 3) return conv_tma_launch<32, TBN, 3, true>(p, s);
            if (t == 2) return conv_tma_launch<32, TBN, 2, true>(p, s);
            return conv_tma_launch<32, TBN, 1, true>(p, s);
        }
    }
    if (cb == 128) return conv_tma_launch<128, TBN, 1, false>(p, s);
    if (cb == 64) return conv_tma_launch<64, TBN, 1, false>(p, s);
    return conv_tma_launch<32, TBN, 1, false>(p, s);
}

// The 1x1 u4 conv on asynchronous copies of the packed input (p holds the fused
// path's parameters): with C = 256 per-thread 16-byte copies; otherwise a 2-D
// tensor map over the packed NHWC input viewed as [pixels][C / 2 bytes], boxes
// of 128 pixels x 128 bytes (256 channels), 128-byte swizzled.
static qnn_status conv1x1_bulk_launch(Params p, const qnn_conv_geom *g, cudaStream_t s)
{
    if (g->C == 256) {
        // a pixel's codes are one 128-byte row: each thread copies its own chunks
        p.KT = 1;
        p.chunk_steps = 1;
        p.nchunks = 1;
        return launch<ConvU4PackedOp<true>, 64, false>(p, s);
    }
    const PFN_cuTensorMapEncodeTiled_v12000 encode = tensor_map_encoder();
    if (!encode) return QNN_ERR_CUDA;
    const cuuint64_t row_bytes = (cuuint64_t)g->C / 2;
    cuuint64_t dims[2] = {row_bytes, (cuuint64_t)p.M};
    cuuint64_t strides[1] = {row_bytes};
    cuuint32_t box[2] = {128, (cuuint32_t)BM};
    cuuint32_t estr[2] = {1, 1};
    if (encode(&p.tmap, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t *>(p.A), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return QNN_ERR_CUDA;
    p.KT = g->C / 256;  // units (256 channels) per tile
    p.chunk_steps = p.KT;
    p.nchunks = 1;
    return launch<ConvU4PackedOp<false>, 64, false>(p, s);
}

// The u8 convs with a workspace: the input expanded to fp16 (q - z_in) in NHWC,
// then one tiled 4-D TMA box (64 channels x TW x TH x TN pixels, 128-byte rows)
// per filter tap, as for u4.  The sum is sum (q - z_in) w; the epilogue adds
// (z_in - 128) colsum back (the fold's zp_term is for codes centred at 128), so
// acc_c is that of the fused path.
static qnn_status conv_tma_u8_run(Params p, const qnn_conv_geom *g, int32_t z_in, const void *W_packed,
                                  void *workspace, int oh, int ow, bool wide_w, cudaStream_t s)
{
    const bool nchw = g->layout == QNN_LAYOUT_NCHW;
    const uint32_t zh = 0x6400u + (uint32_t)z_in;  // fp16 1024 + z_in
    const uint32_t zh2 = zh | (zh << 16);
    uint8_t *xw = static_cast<uint8_t *>(workspace);
    const int64_t n16 = (int64_t)g->N * g->H * g->W * g->C / 16;
    int64_t blocks = (n16 + 255) / 256;
    const int64_t cap = (int64_t)sm_count() * 16;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    if (g->layout == QNN_LAYOUT_NHWC) {
        expand_u8_kernel<false><<<(int)blocks, 256, 0, s>>>(p.A, n16, g->H * g->W, g->C, zh2, xw);
    } else if (g->layout == QNN_LAYOUT_NCHW64) {
        expand_u8_kernel<true><<<(int)blocks, 256, 0, s>>>(p.A, n16, g->H * g->W, g->C, zh2, xw);
    } else {
        const size_t rowbuf = (size_t)g->C * g->W;
        if (rowbuf > 48 * 1024 || (int64_t)g->N * g->H > INT32_MAX) return QNN_ERR_UNSUPPORTED;
        expand_u8_nchw_kernel<<<g->N * g->H, 256, rowbuf, s>>>(p.A, g->H, g->W, g->C, zh2, xw);
    }
    if (launch_status() != QNN_OK) return QNN_ERR_CUDA;
    int TW, TH, TN;
    choose_tiles(g->N, oh, ow, g->stride_w, g->stride_h, TW, TH, TN, nchw);
    cuuint64_t dims[4] = {(cuuint64_t)g->C, (cuuint64_t)g->W, (cuuint64_t)g->H, (cuuint64_t)g->N};
    cuuint64_t strides[3] = {(cuuint64_t)g->C * 2, (cuuint64_t)g->W * g->C * 2, (cuuint64_t)g->H * g->W * g->C * 2};
    cuuint32_t box[4] = {64, (cuuint32_t)(TW * g->stride_w), (cuuint32_t)(TH * g->stride_h), (cuuint32_t)TN};
    cuuint32_t estr[4] = {1, (cuuint32_t)g->stride_w, (cuuint32_t)g->stride_h, 1};
    const PFN_cuTensorMapEncodeTiled_v12000 encode = tensor_map_encoder();
    if (!encode) return QNN_ERR_CUDA;
    if (encode(&p.tmap, CU_TENSOR_MAP_DATA_TYPE_UINT16, 4, workspace, dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return QNN_ERR_CUDA;
    p.Nimg = g->N;
    p.OH = oh;
    p.TW = TW;
    p.TH = TH;
    p.TN = TN;
    p.tiles_x = (ow + TW - 1) / TW;
    p.tiles_y = (oh + TH - 1) / TH;
    p.num_m = p.tiles_x * p.tiles_y * ((g->N + TN - 1) / TN);
    p.cbn = g->C / 64;
    p.KT = g->FH * g->FW * p.cbn;  // K steps of 64 channels = units
    p.Bp = static_cast<const uint8_t *>(W_packed);
    p.btrail = reinterpret_cast<const int32_t *>(static_cast<const uint8_t *>(W_packed) +
                                                 gemm::packed_b_image_bytes(g->OC, g->FH * g->FW * g->C));
    p.amax = z_in > 255 - z_in ? z_in : 255 - z_in;
    if (p.amax == 0) p.amax = 1;
    p.zcs = reinterpret_cast<const int32_t *>(static_cast<const uint8_t *>(W_packed) + colsum8_offset(g));
    p.z_cs = z_in - 128;
    if (g->OC <= 64) return conv_tma_u8_launch<64>(p, wide_w, s);
    if (g->OC <= 128) return conv_tma_u8_launch<128>(p, wide_w, s);
    return conv_tma_u8_launch<256>(p, wide_w, s);
}

// u4: qconv_u4s4; else the u8 conv, whose filter values reach 255 in magnitude
// when wide_w (u8 filters less their zero points) and 128 otherwise (s8).
template <template <int> class Op>
qnn_status conv_run(const void *I, int32_t z_in, const void *W_packed, const qnn_conv_geom *g,
                    const qnn_epilogue *e, void *O, int32_t *O_s32, void *workspace, size_t workspace_bytes,
                    qnn_stream_t stream, bool u4, bool wide_w = false)
{
    if (!I || !W_packed || !e || !O) return QNN_ERR_INVALID_ARG;
    if (!geom_ok(g)) return QNN_ERR_INVALID_ARG;
    if (g->C % (u4 ? 32 : 16) != 0) return QNN_ERR_UNSUPPORTED;
    if (g->OC % 2 != 0) return QNN_ERR_INVALID_ARG;
    if (z_in < 0 || z_in > (u4 ? 15 : 255)) return QNN_ERR_INVALID_ARG;
    if (e->ptf_shift) return QNN_ERR_UNSUPPORTED;
    if (!aligned16(I) || !aligned16(O) || (O_s32 && !aligned16(O_s32))) return QNN_ERR_ALIGNMENT;
    if ((reinterpret_cast<uintptr_t>(W_packed) & 1023u) != 0) return QNN_ERR_ALIGNMENT;

    Params p{};
    const int oh = (g->H + 2 * g->pad_h - g->FH) / g->stride_h + 1;
    const int ow = (g->W + 2 * g->pad_w - g->FW) / g->stride_w + 1;
    p.A = static_cast<const uint8_t *>(I);
    p.H = g->H;
    p.W = g->W;
    p.Cin = g->C;
    p.OHW = oh * ow;
    p.OW = ow;
    p.FH = g->FH;
    p.FW = g->FW;
    p.ph = g->pad_h;
    p.pw = g->pad_w;
    p.sh = g->stride_h;
    p.sw = g->stride_w;
    p.pad_word = u4 ? (uint32_t)z_in * 0x11111111u : (uint32_t)z_in * 0x01010101u;
    p.Bp = static_cast<const uint8_t *>(W_packed);
    p.M = g->N * oh * ow;
    p.N = g->OC;
    p.K = g->FH * g->FW * g->C;
    p.KT = u4 ? (p.K + 127) / 128 : (p.K + 63) / 64;
    p.num_m = (p.M + BM - 1) / BM;
    p.C = O;
    p.C32 = O_s32;
    p.vec_ok = (g->OC % 32 == 0);
    p.layout = g->layout;
    const bool nchw = g->layout == QNN_LAYOUT_NCHW;
    qnn_status st = setup_epilogue(e, true, p);
    if (st != QNN_OK) return st;
    if (p.mode == QNN_EPI_REQUANT && p.out_bits == 4 && e->out_dt != QNN_U4) return QNN_ERR_UNSUPPORTED;
    // NCHW packs 4-bit codes along W: pixel pairs of even widths share bytes
    if (nchw && u4 && (g->W % 2 != 0 || ow % 2 != 0)) return QNN_ERR_INVALID_ARG;
    if (nchw && p.res && p.res_bits == 4 && ow % 2 != 0) return QNN_ERR_INVALID_ARG;
    if (nchw && p.mode == QNN_EPI_REQUANT && p.out_bits == 4 && ow % 2 != 0) return QNN_ERR_INVALID_ARG;
    // exact fp32 chunk sums: u4 x s4 products are at most 120, centred u8 x s8 at most
    // 2^14, centred u8 x (u8 - z_w) below 2^15 (half as many steps per chunk)
    if (u4) {
        p.chunk_steps = KMAX_U4_EXACT / 128;
        if ((int64_t)p.K * 240 > (int64_t)INT32_MAX) return QNN_ERR_OVERFLOW_RISK;
    } else if (wide_w) {
        p.chunk_steps = gemm::MAX_EXACT_STEPS / 2;
        // |(q - z_in)(w - z_w)| <= 255^2 per tap
        if ((int64_t)p.K * 255 * 255 > (int64_t)INT32_MAX) return QNN_ERR_OVERFLOW_RISK;
    } else {
        p.chunk_steps = gemm::MAX_EXACT_STEPS;
        if ((int64_t)p.K * 255 * 128 > (int64_t)INT32_MAX) return QNN_ERR_OVERFLOW_RISK;
    }
    p.nchunks = (p.KT + p.chunk_steps - 1) / p.chunk_steps;
    if (u4 && p.nchunks > 1) return QNN_ERR_UNSUPPORTED;
    // the workspace path pays one expansion pass over the input, which only
    // filters with several taps (each input pixel read by several of them) repay
    // (a 4-bit NCHW input always takes the pre-pass, which reorders it to NHWC)
    if (workspace && g->FH * g->FW == 1 && !(u4 && nchw)) workspace = nullptr;
    if (u4 && nchw && !workspace) return QNN_ERR_UNSUPPORTED;
    // u8 inputs take the tensor-copy path when their channels fill 64-channel K steps
    if (workspace && !u4 && g->C % 64 != 0) workspace = nullptr;
    if (workspace) {
        if (workspace_bytes < (size_t)g->N * g->H * g->W * g->C * (u4 ? 1 : 2)) return QNN_ERR_INVALID_ARG;
        if (!aligned16(workspace)) return QNN_ERR_ALIGNMENT;
        if (g->stride_h > 8 || g->stride_w > 8) return QNN_ERR_UNSUPPORTED;
    }
    p.status = status_word();
    if (!p.status) return QNN_ERR_CUDA;
    cudaStream_t s = (cudaStream_t)stream;
    if (workspace && !u4) return conv_tma_u8_run(p, g, z_in, W_packed, workspace, oh, ow, wide_w, s);
    if (workspace) {
        // expanded input, then the tensor map over it: dims (C, W, H, N), bytes
        const int64_t n16 = (int64_t)g->N * g->H * g->W * g->C / 32;
        int64_t blocks = (n16 + 255) / 256;
        const int64_t cap = (int64_t)sm_count() * 16;
        if (blocks > cap) blocks = cap;
        if (blocks < 1) blocks = 1;
        uint8_t *xw = static_cast<uint8_t *>(workspace);
        if (g->layout == QNN_LAYOUT_NHWC) {
            expand_u4_kernel<<<(int)blocks, 256, 0, s>>>(p.A, n16, (uint32_t)z_in, xw);
        } else if (g->layout == QNN_LAYOUT_NCHW64) {
            expand_u4_nchw64_kernel<<<(int)blocks, 256, 0, s>>>(p.A, n16, g->H * g->W, g->C / 64, (uint32_t)z_in, xw);
        } else {
            const size_t rowbuf = (size_t)g->C * (g->W / 2);
            if (rowbuf > 48 * 1024 || (int64_t)g->N * g->H > INT32_MAX) return QNN_ERR_UNSUPPORTED;
            expand_u4_nchw_kernel<<<g->N * g->H, 256, rowbuf, s>>>(p.A, g->H, g->W, g->C, (uint32_t)z_in, xw);
        }
        if (launch_status() != QNN_OK) return QNN_ERR_CUDA;
        const int cb = tma_cb(g->C);
        int TW, TH, TN;
        choose_tiles(g->N, oh, ow, g->stride_w, g->stride_h, TW, TH, TN, nchw);
        cuuint64_t dims[4] = {(cuuint64_t)g->C, (cuuint64_t)g->W, (cuuint64_t)g->H, (cuuint64_t)g->N};
        cuuint64_t strides[3] = {(cuuint64_t)g->C, (cuuint64_t)g->W * g->C, (cuuint64_t)g->H * g->W * g->C};
        cuuint32_t box[4] = {(cuuint32_t)cb, (cuuint32_t)(TW * g->stride_w), (cuuint32_t)(TH * g->stride_h),
                             (cuuint32_t)TN};
        cuuint32_t estr[4] = {1, (cuuint32_t)g->stride_w, (cuuint32_t)g->stride_h, 1};
        const CUtensorMapSwizzle swz = cb == 128 ? CU_TENSOR_MAP_SWIZZLE_128B
                                                 : (cb == 64 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_32B);
        const PFN_cuTensorMapEncodeTiled_v12000 encode = tensor_map_encoder();
        if (!encode) return QNN_ERR_CUDA;
        if (encode(&p.tmap, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, workspace, dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return QNN_ERR_CUDA;
        p.Nimg = g->N;
        p.OH = oh;
        p.TW = TW;
        p.TH = TH;
        p.TN = TN;
        p.tiles_x = (ow + TW - 1) / TW;
        p.tiles_y = (oh + TH - 1) / TH;
        p.num_m = p.tiles_x * p.tiles_y * ((g->N + TN - 1) / TN);
        p.cbn = g->C / cb;
        p.KT = g->FH * g->FW * p.cbn;
        p.nchunks = 1;
        p.chunk_steps = p.KT;
        p.Bp = static_cast<const uint8_t *>(W_packed) + tma_w_offset(g);
        p.zcs = reinterpret_cast<const int32_t *>(static_cast<const uint8_t *>(W_packed) + colsum_offset(g));
        p.z_cs = z_in;
        if (g->OC <= 64) return conv_tma_dispatch<64>(p, cb, s);
        if (g->OC <= 128) return conv_tma_dispatch<128>(p, cb, s);
        return conv_tma_dispatch<256>(p, cb, s);
    }
    if (u4 && g->layout == QNN_LAYOUT_NHWC && g->FH == 1 && g->FW == 1 && g->stride_h == 1 && g->stride_w == 1 &&
        g->pad_h == 0 && g->pad_w == 0 &&
        g->C % 256 == 0 && (int64_t)(g->C / 128) * 64 * 128 <= ConvU4PackedOp<true>::B_RES_BYTES && g->OC <= 64)
        return conv1x1_bulk_launch(p, g, s);
    if (g->OC <= 64) return conv_launch<Op, 64>(p, s);
    if (g->OC <= 128) return conv_launch<Op, 128>(p, s);
    return conv_launch<Op, 256>(p, s);
}

}  // namespace mk
}  // namespace qnn

extern "C" size_t qnn_conv_packed_w_bytes(const qnn_conv_geom *g, qnn_dtype w_dt)
{
    if (!qnn::mk::geom_ok(g)) return 0;
    // u4 / u8 filters with zero points (qconv_prepack_w_u4 / _u8) take the images of s4 / s8
    if (w_dt == QNN_S4 || w_dt == QNN_U4) return qnn::mk::packed_w_u4_total(g);
    if (w_dt == QNN_S8 || w_dt == QNN_U8) return qnn::mk::packed_w_8_total(g);
    return 0;
}

namespace qnn {
namespace mk {
// The 4-bit filter images and column sums; z_w: u4 filters with per-filter zero
// points (device int32 [OC]), or null for s4 filters.
static qnn_status prepack_w4(const void *W, const int32_t *z_w, const qnn_conv_geom *g, void *W_packed,
                             int32_t *colsum, qnn_stream_t stream);
}  // namespace mk
}  // namespace qnn

extern "C" qnn_status qconv_prepack_w(const void *W, qnn_dtype w_dt, const qnn_conv_geom *g,
                                      void *W_packed, int32_t *colsum, qnn_stream_t stream)
{
    if (!W || !W_packed || !qnn::mk::geom_ok(g)) return QNN_ERR_INVALID_ARG;
    const int K = g->FH * g->FW * g->C;
    if (w_dt == QNN_S8) {
        // filters [OC][FH][FW][C] are the GEMM operand B [OC, K]; the column sums
        // also go into the image (the tensor-copy path adds z_in * colsum back)
        int32_t *cs_img = reinterpret_cast<int32_t *>(static_cast<uint8_t *>(W_packed) + qnn::mk::colsum8_offset(g));
        qnn_status st = qgemm_prepack_b(static_cast<const int8_t *>(W), g->OC, K, W_packed, cs_img, stream);
        if (st != QNN_OK || !colsum) return st;
        return cudaMemcpyAsync(colsum, cs_img, (size_t)g->OC * 4, cudaMemcpyDeviceToDevice, (cudaStream_t)stream) ==
                       cudaSuccess
                   ? QNN_OK
                   : QNN_ERR_CUDA;
    }
    if (w_dt != QNN_S4) return QNN_ERR_UNSUPPORTED;
    return qnn::mk::prepack_w4(W, nullptr, g, W_packed, colsum, stream);
}

namespace qnn {
qnn_status prepack_b_u8_minus_zw(const uint8_t *B, const int32_t *z_w, int N, int K, void *B_packed,
                                 int32_t *colsum, cudaStream_t s);
}  // namespace qnn

extern "C" qnn_status qconv_prepack_w_u8(const void *W, const int32_t *z_w, const qnn_conv_geom *g, void *W_packed,
                                         int32_t *colsum, qnn_stream_t stream)
{
    if (!W || !W_packed || !z_w || !qnn::mk::geom_ok(g)) return QNN_ERR_INVALID_ARG;
    if (g->C % 16 != 0) return QNN_ERR_UNSUPPORTED;
    if ((reinterpret_cast<uintptr_t>(W_packed) & 1023u) != 0) return QNN_ERR_ALIGNMENT;
    if (!qnn::aligned16(W) || !qnn::aligned16(z_w)) return QNN_ERR_ALIGNMENT;
    // filters [OC][FH][FW][C] are the GEMM operand B [OC, K]; column sums into the image too
    int32_t *cs_img = reinterpret_cast<int32_t *>(static_cast<uint8_t *>(W_packed) + qnn::mk::colsum8_offset(g));
    qnn_status st = qnn::prepack_b_u8_minus_zw(static_cast<const uint8_t *>(W), z_w, g->OC, g->FH * g->FW * g->C,
                                               W_packed, cs_img, (cudaStream_t)stream);
    if (st != QNN_OK || !colsum) return st;
    return cudaMemcpyAsync(colsum, cs_img, (size_t)g->OC * 4, cudaMemcpyDeviceToDevice, (cudaStream_t)stream) ==
                   cudaSuccess
               ? QNN_OK
               : QNN_ERR_CUDA;
}

extern "C" qnn_status qconv_prepack_w_u4(const void *W, const int32_t *z_w, const qnn_conv_geom *g, void *W_packed,
                                         int32_t *colsum, qnn_stream_t stream)
{
    if (!W || !W_packed || !z_w || !qnn::mk::geom_ok(g)) return QNN_ERR_INVALID_ARG;
    if (!qnn::aligned16(z_w)) return QNN_ERR_ALIGNMENT;
    // |u - z_w| <= 15: every fp32 sum in the kernel's 2^-9 units stays exact while
    // K * 15 * 15 < 2^24
    if ((int64_t)g->FH * g->FW * g->C * 225 >= (1ll << 24)) return QNN_ERR_OVERFLOW_RISK;
    return qnn::mk::prepack_w4(W, z_w, g, W_packed, colsum, stream);
}

static qnn_status qnn::mk::prepack_w4(const void *W, const int32_t *z_w, const qnn_conv_geom *g, void *W_packed,
                                      int32_t *colsum, qnn_stream_t stream)
{
    const int K = g->FH * g->FW * g->C;
    if (g->C % 2 != 0) return QNN_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(W_packed) & 1023u) != 0) return QNN_ERR_ALIGNMENT;
    const int KT = (K + 127) / 128;
    const int64_t nchunks = (int64_t)(qnn::mk::packed_w_u4_bytes(g) / 16);
    int64_t blocks = (nchunks + 255) / 256;
    if (blocks > 65535) blocks = 65535;
    cudaStream_t s = (cudaStream_t)stream;
    uint8_t *wp = static_cast<uint8_t *>(W_packed);
    qnn::mk::prepack_w_s4_kernel<<<(int)blocks, 256, 0, s>>>(static_cast<const uint8_t *>(W), g->OC, K,
                                                               KT, wp, nchunks, z_w);
    if (qnn::launch_status() != QNN_OK) return QNN_ERR_CUDA;
    // the TMA conv's image and the column sums follow the fused-path image
    const size_t tb = qnn::mk::tma_w_bytes(g);
    if (tb) {
        const int cb = qnn::mk::tma_cb(g->C);
        const int64_t tchunks = (int64_t)(tb / 16);
        int64_t tblocks = (tchunks + 255) / 256;
        if (tblocks > 65535) tblocks = 65535;
        qnn::mk::prepack_w_s4_tma_kernel<<<(int)tblocks, 256, 0, s>>>(
            static_cast<const uint8_t *>(W), g->OC, g->C, cb, g->FH * g->FW * (g->C / cb),
            wp + qnn::mk::tma_w_offset(g), tchunks, z_w);
        if (qnn::launch_status() != QNN_OK) return QNN_ERR_CUDA;
    }
    const int64_t threads = (int64_t)g->OC * 32;
    int32_t *cs_img = reinterpret_cast<int32_t *>(wp + qnn::mk::colsum_offset(g));
    qnn::mk::colsum_s4_kernel<<<(int)((threads + 255) / 256), 256, 0, s>>>(static_cast<const uint8_t *>(W),
                                                                          g->OC, K, cs_img, z_w);
    if (qnn::launch_status() != QNN_OK) return QNN_ERR_CUDA;
    if (colsum) {
        if (cudaMemcpyAsync(colsum, cs_img, (size_t)g->OC * 4, cudaMemcpyDeviceToDevice, s) != cudaSuccess)
            return QNN_ERR_CUDA;
    }
    return QNN_OK;
}

extern "C" size_t qnn_conv_workspace_bytes(const qnn_conv_geom *g, qnn_dtype in_dt)
{
    if (!qnn::mk::geom_ok(g)) return 0;
    // the input expanded to one e4m3 byte (u4) or one fp16 value (u8) per channel
    if (in_dt == QNN_U4) return (size_t)g->N * g->H * g->W * g->C;
    if (in_dt == QNN_U8) return (size_t)g->N * g->H * g->W * g->C * 2;
    return 0;
}

extern "C" qnn_status qconv_u4s4(const void *I, int32_t z_in, const void *W_packed,
                                 const qnn_conv_geom *g, const qnn_epilogue *e, void *O,
                                 int32_t *O_s32, void *workspace, size_t workspace_bytes,
                                 qnn_stream_t stream)
{
    return qnn::mk::conv_run<qnn::mk::ConvU4Op>(I, z_in, W_packed, g, e, O, O_s32, workspace,
                                                workspace_bytes, stream, true);
}

extern "C" qnn_status qconv_u8s8(const void *I, int32_t z_in, const void *W_packed,
                                 const qnn_conv_geom *g, const qnn_epilogue *e, void *O,
                                 int32_t *O_s32, void *workspace, size_t workspace_bytes, qnn_stream_t stream)
{
    return qnn::mk::conv_run<qnn::mk::ConvU8Op>(I, z_in, W_packed, g, e, O, O_s32, workspace, workspace_bytes,
                                                stream, false);
}

extern "C" qnn_status qconv_u8u8(const void *I, int32_t z_in, const void *W_packed,
                                 const qnn_conv_geom *g, const qnn_epilogue *e, void *O,
                                 int32_t *O_s32, void *workspace, size_t workspace_bytes, qnn_stream_t stream)
{
    return qnn::mk::conv_run<qnn::mk::ConvU8Op>(I, z_in, W_packed, g, e, O, O_s32, workspace, workspace_bytes,
                                                stream, false, true);
}
