// qnn_lis.cu -- Log-Int-Softmax and the bit-shift attention product.
//
// [FQ] "首个完全量化Vision Transformer的方法FQ-ViT" (aijishu.com), section 3.3:
//   Softmax 的量化推理 / Integer-only 推理: softmax over a row of integer logit
//     codes x (real value x * S) with integer arithmetic only: subtract the row
//     maximum, an integer exponential (a second-order polynomial on a remainder
//     in (-ln 2, 0] scaled by a power of two), the integer sum of the row;
//   Softmax 的量化的实现: the attention probability is quantized to a log2 code
//     k = log_round(round(sum / e)), k >= 2^bits meaning probability 0;
//   Attention Map 的 Log2 量化: with probabilities 2^-k the product of the
//     attention map with the value codes is a shift per term.
//
// q_log_int_softmax: one warp per row.  Per element the exponential is
//   e = z * 2^(30 - q), q = floor(d / x0_int), r = d - x0_int q,
//   z = r (r + b_int) + c_int, d = max(x - max(x), 30 x0_int)
// in exact integers (q by a multiply-high with a host-computed reciprocal).  The
// row sum s is a u64 warp reduction.  The code is not formed from v = round(s /
// e) per element: round(v) reaches a step L_j of log_round (2, 3, 6, 12, ...,
// 3 * 2^(j-2)) exactly when v + 1/2 > L_j, so an fp32 estimate of v + 1/2 gives
// the count of steps from its exponent and first mantissa bit; where that
// estimate lies within fp32 error of a step, exact 128-bit comparisons of 2s
// with (2L - 1) e decide.  That equals log_round(round(s/e)) exactly, half-to-
// even ties included.
//
// q_attn_shift_v: out[b][i][j] = sum_t 2^(2^bits - 1 - k[b][i][t]) v[b][t][j]
// over unmasked codes, exact in int32 (the host rejects shapes that could
// overflow).  For d <= 128 and Lk <= 512 it runs on the tensor pipe (below);
// otherwise on the CUDA cores: a 64 x 64 output tile per block, 4 x 4 per
// thread, the weights 2^(N - k) expanded into shared memory per 64 tokens.
//
// q_lis_attn_v: the tensor-pipe kernel with its shared code tile filled by
// Log-Int-Softmax of the CTA's logit rows instead of a copy of stored codes.
#include <cuda_runtime.h>
#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdint>
#include "qnn_internal.h"
#include "qnn_ptx.cuh"

namespace qnn {
namespace {

constexpr unsigned kFull = 0xffffffffu;
constexpr int kLisWarps = 8;

struct LisArgs {
    const int32_t *x;
    uint8_t *code;
    int64_t rows, L;
    uint32_t x0n;     // -x0_int (> 0)
    uint32_t ndmax;   // 30 |x0_int|: the clamp of max(x) - x
    int32_t b, c;     // b_int, c_int
    uint32_t qm;      // floor(nd / x0n) = mulhi(nd, qm) >> ql for nd <= 30 x0n < 2^21
    uint32_t ql;      // (x0n == 1: qm = 0, q = nd)
    int kmax;         // 2^bits
};

// Integer exponential of x - mx (mx the row maximum) and its fp32 value.  The
// host has checked that 0 < z <= c_int < 2^31 for every remainder, so z is
// formed in 32 bits.
__device__ __forceinline__ uint64_t lis_exp(int32_t x, int32_t mx, const LisArgs &a, float &ef)
{
    // nd = -(max(x - mx, 30 x0_int)): mx >= x, so the unsigned difference is exact
    const uint32_t nd = min((uint32_t)mx - (uint32_t)x, a.ndmax);
    const uint32_t q = a.qm ? __umulhi(nd, a.qm) >> a.ql : nd;
    const int32_t r = (int32_t)(nd - q * a.x0n);
    // the page's remainder is -r (in (x0_int, 0]): z = (-r)(-r + b) + c
    const int32_t z = a.c - r * (a.b - r);
    const uint32_t sh = 30u - q;
    // z scaled by 2^sh through the exponent field of its fp32 value
    ef = __int_as_float(__float_as_int(__int2float_rn(z)) + (int32_t)(sh << 23));
    // (z << sh) as two words: z < 2^31, sh <= 30
    const uint32_t lo = (uint32_t)z << sh, hi = __funnelshift_l((uint32_t)z, 0u, sh);
    return ((uint64_t)hi << 32) | lo;
}

// round_half_even(s / e) >= L  <=>  2s > (2L - 1) e, or equality with L even
// (exact: 2s has 65 bits, (2L - 1) e at most 95).
__device__ __forceinline__ bool ratio_reaches(uint64_t s, uint64_t e, uint64_t L)
{
    const uint64_t D = 2 * L - 1;
    const uint64_t plo = D * e, phi = __umul64hi(D, e);
    const uint64_t slo = s << 1, shi = s >> 63;
    if (shi != phi) return shi > phi;
    if (slo != plo) return slo > plo;
    return (L & 1) == 0;
}

// L_j, the values of v at which log_round steps up: L_1 = 2, L_j = 3 * 2^(j-2).
__device__ __forceinline__ uint64_t step_value(int j) { return j <= 1 ? 2ull : (3ull << (j - 2)); }

// Code of one exponential e (fp32 value ef) in a row whose sum is s (fp32 value
// sf): the number k of thresholds j <= kmax with round_half_even(s / e) >= L_j,
// L_1 = 2 and L_j = 3 * 2^(j-2).  round(v) >= L exactly when v + 1/2 > L (ties:
// to even), so with the fp32 estimate w of v = s / e (relative error below
// 2^-21) and u = w + 1/2, k = #{j : L_j < u}: from u's exponent E and first
// mantissa bit, ((t + 1) >> 1) - 127 with t = 2 (E + 127) + that bit, and 0 below
// 2.  Every L_j is 2 or has the mantissa 1.5, so u lies near a threshold only
// when its mantissa is within 32 units (2^-18.6 relative, well above the error)
// of 1.5, 1 or 2; those rare cases return `near` and are settled by
// lis_code_exact around kh.
__device__ __forceinline__ int lis_code_fast(float sf, float ef, int kmax, int &kh, bool &near)
{
    const float u = __fadd_rn(__fdividef(sf, ef), 0.5f);
    const int bu = __float_as_int(u);
    const int m = bu & 0x7FFFFF;
    const int t = bu >> 22;
    kh = t >= 256 ? min(((t + 1) >> 1) - 127, kmax + 1) : 0;
    near = abs(m - 0x400000) <= 32 || m <= 32 || m >= 0x7FFFFF - 32;
    return min(kh, kmax);
}

// The exact count around kh: v lies within one threshold of kh either way.
__device__ __noinline__ int lis_code_exact(uint64_t s, uint64_t e, int kh, int kmax)
{
    int k = kh >= 1 ? kh - 1 + (int)ratio_reaches(s, e, step_value(kh)) : 0;
    k += (int)ratio_reaches(s, e, step_value(kh + 1));
    return min(k, kmax);
}

// Sum over the warp of per-lane u64 values whose total is below 2^64, as three
// limbs of 22, 22 and 20 bits, each summed by one warp reduction (below 2^27).
__device__ __forceinline__ uint64_t warp_sum_u64(uint64_t v)
{
    const uint32_t l0 = __reduce_add_sync(kFull, (uint32_t)v & 0x3FFFFFu);
    const uint32_t l1 = __reduce_add_sync(kFull, (uint32_t)(v >> 22) & 0x3FFFFFu);
    const uint32_t l2 = __reduce_add_sync(kFull, (uint32_t)(v >> 44));
    return (uint64_t)l0 + ((uint64_t)l1 << 22) + ((uint64_t)l2 << 44);
}

// R > 0: rows of L <= 32 R held in registers.  R == 0: any L, three passes over
// the row (the later two from cache).
template <int R>
__global__ void __launch_bounds__(kLisWarps * 32) log_int_softmax_kernel(const __grid_constant__ LisArgs a)
{
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const int64_t L = a.L;
    for (int64_t row = (int64_t)blockIdx.x * kLisWarps + w; row < a.rows;
         row += (int64_t)gridDim.x * kLisWarps) {
        const int32_t *xr = a.x + row * L;
        uint8_t *cr = a.code + row * L;
        if constexpr (R > 0) {
            int32_t xv[R];
            int32_t mx = INT32_MIN;
            const int Li = (int)L;  // <= 256 here
#pragma unroll
            for (int j = 0; j < R; ++j) {
                const int i = lane + 32 * j;
                xv[j] = i < Li ? __ldcs(xr + i) : INT32_MIN;
                mx = max(mx, xv[j]);
            }
            mx = __reduce_max_sync(kFull, mx);
            uint64_t ev[R];
            float ef[R];
            uint64_t s = 0;
#pragma unroll
            for (int j = 0; j < R; ++j) {
                ev[j] = lis_exp(xv[j], mx, a, ef[j]);
                if (lane + 32 * j < Li) s += ev[j];
            }
            s = warp_sum_u64(s);
            const float sf = __ull2float_rn(s);
            int kc[R], khs[R];
            bool nr[R];
#pragma unroll
            for (int j = 0; j < R; ++j) kc[j] = lis_code_fast(sf, ef[j], a.kmax, khs[j], nr[j]);
#pragma unroll
            for (int j = 0; j < R; ++j) {
                // the exact comparisons only where an estimate fell near a half-way point
                if (__any_sync(kFull, nr[j]) && nr[j]) kc[j] = lis_code_exact(s, ev[j], khs[j], a.kmax);
                const int i = lane + 32 * j;
                if (i < Li) __stcs(cr + i, (uint8_t)kc[j]);
            }
        } else {
            int32_t mx = INT32_MIN;
            for (int64_t i = lane; i < L; i += 32) mx = max(mx, __ldg(xr + i));
            mx = __reduce_max_sync(kFull, mx);
            uint64_t s = 0;
            float ef;
            for (int64_t i = lane; i < L; i += 32) s += lis_exp(__ldg(xr + i), mx, a, ef);
            s = warp_sum_u64(s);
            const float sf = __ull2float_rn(s);
            for (int64_t i = lane; i < L; i += 32) {
                const uint64_t e = lis_exp(__ldg(xr + i), mx, a, ef);
                int kh;
                bool nr;
                int k = lis_code_fast(sf, ef, a.kmax, kh, nr);
                if (nr) k = lis_code_exact(s, e, kh, a.kmax);
                __stcs(cr + i, (uint8_t)k);
            }
        }
    }
}

// ---------------------------------------------------------------------------
// bit-shift product
constexpr int kShT = 64;  // tokens per chunk
constexpr int kShM = 64;  // query rows per block
constexpr int kShN = 64;  // value columns per block

struct ShiftArgs {
    const uint8_t *code;  // [B][Lq][Lk]
    const int8_t *v;      // [B][Lk][d]
    int32_t *out;         // [B][Lq][d]
    int Lq, Lk, d, kmax;
};

__global__ void __launch_bounds__(256) attn_shift_v_kernel(ShiftArgs a)
{
    __shared__ __align__(16) int32_t Ws[kShT][kShM + 4];   // weights 2^(N - k), [t][row]
    __shared__ __align__(16) int8_t Vs[kShT][kShN];        // value codes, [t][col]
    const int tid = threadIdx.x;
    const int tx = tid & 15, ty = tid >> 4;                 // 4 cols x 4 rows per thread
    const int64_t b = blockIdx.z;
    const int i0 = blockIdx.x * kShM, j0 = blockIdx.y * kShN;
    const uint8_t *cb = a.code + b * (int64_t)a.Lq * a.Lk;
    const int8_t *vb = a.v + b * (int64_t)a.Lk * a.d;
    const int nsh = a.kmax - 1;
    int32_t acc[4][4] = {};
    for (int t0 = 0; t0 < a.Lk; t0 += kShT) {
        // weights: a thread per (token, 4 rows): four coalesced byte loads (one per
        // row, consecutive tokens across the warp) and one 16-byte store; the row
        // pitch of 68 words keeps the eight stores of a quarter warp on distinct banks
        for (int e = tid; e < kShT * (kShM / 4); e += 256) {
            const int t = e % kShT, r4 = (e / kShT) * 4;
            const int tt = t0 + t;
            int32_t wv[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int i = i0 + r4 + q;
                wv[q] = 0;
                if (i < a.Lq && tt < a.Lk) {
                    const int k = cb[(int64_t)i * a.Lk + tt];
                    wv[q] = k < a.kmax ? (1 << (nsh - k)) : 0;
                }
            }
            *reinterpret_cast<int4 *>(&Ws[t][r4]) = make_int4(wv[0], wv[1], wv[2], wv[3]);
        }
        // values: 4 bytes per thread-step (d % 4 == 0 and j0 + c < d checked per word)
        for (int e = tid; e < kShT * (kShN / 4); e += 256) {
            const int t = e / (kShN / 4), c4 = (e % (kShN / 4)) * 4;
            const int tt = t0 + t, j = j0 + c4;
            uint32_t word = 0;
            if (tt < a.Lk && j < a.d) word = *reinterpret_cast<const uint32_t *>(vb + (int64_t)tt * a.d + j);
            *reinterpret_cast<uint32_t *>(&Vs[t][c4]) = word;
        }
        __syncthreads();
        const int tn = min(kShT, a.Lk - t0);
        for (int t = 0; t < tn; ++t) {
            const int4 w4 = *reinterpret_cast<const int4 *>(&Ws[t][ty * 4]);
            const uint32_t vw = *reinterpret_cast<const uint32_t *>(&Vs[t][tx * 4]);
            const int32_t vv[4] = {(int32_t)(int8_t)(vw & 0xff), (int32_t)(int8_t)((vw >> 8) & 0xff),
                                   (int32_t)(int8_t)((vw >> 16) & 0xff), (int32_t)(int8_t)(vw >> 24)};
            const int32_t ww[4] = {w4.x, w4.y, w4.z, w4.w};
#pragma unroll
            for (int r = 0; r < 4; ++r)
#pragma unroll
                for (int c = 0; c < 4; ++c) acc[r][c] += ww[r] * vv[c];
        }
        __syncthreads();
    }
    int32_t *ob = a.out + b * (int64_t)a.Lq * a.d;
#pragma unroll
    for (int r = 0; r < 4; ++r) {
        const int i = i0 + ty * 4 + r, j = j0 + tx * 4;
        if (i < a.Lq && j < a.d)
            *reinterpret_cast<int4 *>(ob + (int64_t)i * a.d + j) =
                make_int4(acc[r][0], acc[r][1], acc[r][2], acc[r][3]);
    }
}

// ---------------------------------------------------------------------------
// bit-shift product on the tensor pipe.  The weight 2^(N - k) (N = 2^bits - 1
// <= 15) is split into lo = 2^(N - k) for N - k < 8 and hi = 2^(N - k - 8) for
// N - k >= 8, both <= 128 and exact in fp16, as are the s8 values; every product
// is an integer below 2^14 in magnitude and each of the two sums stays below
// 2^23 for Lk <= 512, so the fp32 accumulators of two kind::f16 MMAs (lo and hi,
// adjacent TMEM column ranges) hold them exactly, and out = lo + 256 hi.
//
// One CTA per (head, 128 query rows), 8 warps, up to four CTAs per SM.  Per
// round of up to 64 tokens: all threads expand the codes into the fp16 images
// A_lo / A_hi (128 rows x one K atom of 64, K-major, 128-byte swizzle: 16-byte
// chunk c of row r at chunk c ^ (r % 8)), stage the value rows in shared memory
// and transpose them into the B image (d rows = value columns, same layout); one
// thread then issues the MMAs (M = 128, N = d, K = 16 each) and commits to an
// mbarrier that every thread waits on (bounded) before the next round reuses
// the images; the next round's global loads are issued before that wait.  The
// epilogue reads TMEM with 32x32b.x16 loads, converts the exact fp32 sums to
// integers and writes 16 consecutive int32 per thread and piece.
constexpr int kMmaRows = 128;
constexpr int kMmaKC = 64;   // tokens per round: one 64-element K atom
constexpr int kVMax = kMmaKC * 128 / 16 / 256;         // value chunks per thread at d = 128

struct ShiftMmaArgs {
    const uint8_t *code;  // [B][Lq][Lk]
    const int8_t *v;      // [B][Lk][d]
    int32_t *out;         // [B][Lq][d]
    uint64_t code_bytes;  // B * Lq * Lk: no word load starts at or past it
    int Lq, Lk, d;
    uint32_t tab0, tab1;  // high bytes of the fp16 weights, by code & 7 (bytes 0..7)
    // n / m = mulhi(n, ceil(2^32 / m)) for the small n used here
    uint32_t rcp_c;       // m = d / 16 (0 when d == 16: the quotient is n)
    uint32_t rcp_d;       // m = d
    uint32_t tmem_cols;
    uint32_t tile_bytes;  // shared memory for the CTA's rows of codes (min(128, Lq) Lk + 32, rounded up)
    uint32_t *status;
    // fused form: the codes are computed here from int32 logits (Log-Int-Softmax)
    const int32_t *x;     // [B][Lq][Lk] or null
    LisArgs lis;          // its constants (x, code, rows, L unused)
};

__host__ __device__ constexpr uint32_t shift_mma_smem(int d, bool hi, uint32_t tile_bytes)
{
    return 1024u + (hi ? 2u : 1u) * kMmaRows * 128u + (uint32_t)d * 128u + (uint32_t)(kMmaKC * d) + 64u + tile_bytes;
}

// fp32 value of an exact integer with |f| <= 2^22 -> int32 without the conversion pipe.
__device__ __forceinline__ int32_t exact_f2i_small(uint32_t fbits)
{
    return __float_as_int(__fadd_rn(__int_as_float(fbits), 12582912.0f)) - 0x4B400000;
}

// The value rows of one round into registers: up to 2 chunks of 16 bytes per
// thread (zero past Lk).
__device__ __forceinline__ void shift_load_values(const ShiftMmaArgs &a, int tid, int rd, const int8_t *vb,
                                                  uint4 (&vw)[kVMax])
{
    const int d = a.d;
    const int t0 = rd * kMmaKC;
    const int ntok = min(kMmaKC, (a.Lk - t0 + 15) / 16 * 16);
    const int chunks = ntok * d / 16;
#pragma unroll
    for (int u = 0; u < kVMax; ++u) {
        const int it = tid + 256 * u;
        vw[u] = make_uint4(0u, 0u, 0u, 0u);
        if (it < chunks) {
            const int tt = a.rcp_c ? (int)__umulhi((uint32_t)it, a.rcp_c) : it;
            const int cc = (it - tt * (d >> 4)) * 16;
            if (t0 + tt < a.Lk) vw[u] = __ldg(reinterpret_cast<const uint4 *>(vb + (int64_t)(t0 + tt) * d + cc));
        }
    }
}

// Log-Int-Softmax of the CTA's rows straight into the shared code tile (row r
// at r * Lk): warp w takes rows w, w + 8, ...; a row of L <= 256 values is held
// in registers, up to 8 per lane.
__device__ __forceinline__ void lis_rows_to_tile(const ShiftMmaArgs &a, int64_t row0, int rows_here, uint8_t *tile,
                                                 int warp, int lane)
{
    const LisArgs &la = a.lis;
    const int L = a.Lk;
    for (int r = warp; r < rows_here; r += 8) {
        const int32_t *xr = a.x + (row0 + r) * (int64_t)L;
        int32_t xv[8];
        int32_t mx = INT32_MIN;
        // slots past the row (32 j >= L) are skipped by the whole warp
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const int i = lane + 32 * j;
            xv[j] = (32 * j < L && i < L) ? __ldcs(xr + i) : INT32_MIN;
            mx = max(mx, xv[j]);
        }
        mx = __reduce_max_sync(kFull, mx);
        uint64_t ev[8];
        float ef[8];
        uint64_t s = 0;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            if (32 * j >= L) break;
            ev[j] = lis_exp(xv[j], mx, la, ef[j]);
            if (lane + 32 * j < L) s += ev[j];
        }
        s = warp_sum_u64(s);
        const float sf = __ull2float_rn(s);
        uint8_t *tr = tile + r * L;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            if (32 * j >= L) break;  // warp-uniform
            int kh;
            bool nr;
            int k = lis_code_fast(sf, ef[j], la.kmax, kh, nr);
            if (__any_sync(kFull, nr) && nr) k = lis_code_exact(s, ev[j], kh, la.kmax);
            const int i = lane + 32 * j;
            if (i < L) tr[i] = (uint8_t)k;
        }
    }
}

template <bool HI, bool FUSED>
__global__ void __launch_bounds__(256, 4) attn_shift_mma_kernel(const __grid_constant__ ShiftMmaArgs a)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *base = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    uint8_t *A_lo = base;
    uint8_t *A_hi = base + kMmaRows * 128;
    uint8_t *Bs = base + (HI ? 2 : 1) * kMmaRows * 128;
    const int d = a.d;
    const uint32_t batom = (uint32_t)d * 128u;  // bytes of the K atom of B
    uint8_t *raw = Bs + batom;                  // value rows of the round, [token][d]
    uint64_t *bar = reinterpret_cast<uint64_t *>(raw + kMmaKC * d);
    uint64_t *tbar = bar + 1;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bar + 2);
    uint32_t *ok_flag = tmem_slot + 1;
    uint8_t *tile = reinterpret_cast<uint8_t *>(bar) + 64;  // the CTA's rows of codes

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int64_t b = blockIdx.y;
    const int i0 = blockIdx.x * kMmaRows;
    const int rows_here = min(kMmaRows, a.Lq - i0);
    // the CTA's codes are one contiguous range: rows i0 .. i0 + rows_here of head b
    const uint64_t tile_start = (uint64_t)((b * a.Lq + i0) * (int64_t)a.Lk);
    const uint64_t tile_end = tile_start + (uint64_t)rows_here * (uint64_t)a.Lk;
    const uint64_t s0 = tile_start & ~15ull;  // bulk copies start and end on 16-byte boundaries
    const uint64_t e1 = min((tile_end + 15) & ~15ull, a.code_bytes & ~15ull);
    const uint32_t toff = FUSED ? 0u : (uint32_t)(tile_start - s0);
    if (tid == 0) {
        mbar_init(smem_u32(bar), 1);
        mbar_init(smem_u32(tbar), 1);
        fence_mbar_init();
        if (FUSED) {
            mbar_arrive(smem_u32(tbar));
        } else if (e1 > s0) {
            mbar_arrive_expect_tx(smem_u32(tbar), (uint32_t)(e1 - s0));
            bulk_g2s(smem_u32(tile), a.code + s0, (uint32_t)(e1 - s0), smem_u32(tbar));
        } else {
            mbar_arrive(smem_u32(tbar));
        }
    }
    if (warp == 0) {
        tmem_alloc(smem_u32(tmem_slot), a.tmem_cols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t idesc = idesc_f32acc(0, 0, kMmaRows, (uint32_t)d);
    const int8_t *vb = a.v + b * (int64_t)a.Lk * d;
    const int rounds = (a.Lk + kMmaKC - 1) / kMmaKC;
    uint4 vw[kVMax];
    shift_load_values(a, tid, 0, vb, vw);
    bool ok = true;
    {
        // the code tile: bulk copy (one warp polls its barrier), then the bytes past the
        // last whole 16-byte block of the buffer, if this tile reaches them, by plain loads
        if (warp == 0) {
            const bool done = mbar_wait(smem_u32(tbar), 0u, a.status);
            if (lane == 0) *ok_flag = done ? 1u : 0u;
        }
        __syncthreads();
        ok = *reinterpret_cast<volatile uint32_t *>(ok_flag) != 0u;
        if constexpr (FUSED) {
            lis_rows_to_tile(a, b * a.Lq + i0, rows_here, tile, warp, lane);
        } else {
            for (uint64_t x = max(e1, tile_start) + tid; x < tile_end; x += 256) tile[x - s0] = a.code[x];
        }
        __syncthreads();
    }
    for (int rd = 0; rd < rounds && ok; ++rd) {
        const int t0 = rd * kMmaKC;
        const int nks = min(kMmaKC / 16, (a.Lk - t0 + 15) / 16);  // K steps of 16 this round
        const int ntok = nks * 16;                                 // tokens written (zero past Lk)
        const int gpr = ntok / 4;  // 4-token groups per row this round
        const int chunks = ntok * d / 16;
        // rows past Lq get zero weights in the first round and keep them
        const int nrows = rd == 0 ? kMmaRows : rows_here;
        const uint32_t rcp_gpr = (uint32_t)((0x100000000ull + (uint64_t)gpr - 1) / (uint64_t)gpr);
        for (int it = tid; it < nrows * gpr; it += 256) {
            const int row = (int)__umulhi((uint32_t)it, rcp_gpr);  // it / gpr (it < 2^16)
            const int kk = 4 * (it - row * gpr);
            const int t = t0 + kk;
            uint32_t c = 0xFFFFFFFFu;  // >= 2^bits: weight 0
            if (row < rows_here && t < a.Lk) {
                const uint32_t off = toff + (uint32_t)row * (uint32_t)a.Lk + (uint32_t)t;
                const uint32_t *wp = reinterpret_cast<const uint32_t *>(tile + (off & ~3u));
                c = __funnelshift_r(wp[0], wp[1], (off & 3u) * 8u);
                const int nv = a.Lk - t;
                if (nv < 4) c |= 0xFFFFFFFFu << (8 * nv);
            }
            // weight high bytes: the table by code & 7; bit 3 splits lo from hi; codes >= 16 are 0
            const uint32_t x = c & 0x07070707u;
            const uint32_t sel = prmt(x | (x >> 4), 0u, 0x4420u);
            const uint32_t tb = prmt(a.tab0, a.tab1, sel);
            const uint32_t b3 = prmt(c << 4, 0u, 0xBA98u);
            const uint32_t big = prmt(((c & 0xF0F0F0F0u) >> 1) + 0x78787878u, 0u, 0xBA98u);
            const uint32_t off = (uint32_t)(row >> 3) * 1024u + (uint32_t)(row & 7) * 128u +
                                 ((((uint32_t)kk >> 3) ^ (uint32_t)(row & 7)) << 4) + (uint32_t)(kk & 7) * 2u;
            if constexpr (HI) {
                const uint32_t lo = tb & b3 & ~big, hi = tb & ~b3 & ~big;
                *reinterpret_cast<uint2 *>(A_lo + off) = make_uint2(prmt(lo, 0u, 0x1404u), prmt(lo, 0u, 0x3424u));
                *reinterpret_cast<uint2 *>(A_hi + off) = make_uint2(prmt(hi, 0u, 0x1404u), prmt(hi, 0u, 0x3424u));
            } else {
                const uint32_t lo = tb & ~b3 & ~big;
                *reinterpret_cast<uint2 *>(A_lo + off) = make_uint2(prmt(lo, 0u, 0x1404u), prmt(lo, 0u, 0x3424u));
            }
        }
#pragma unroll
        for (int u = 0; u < kVMax; ++u) {
            const int it = tid + 256 * u;
            if (it < chunks) *reinterpret_cast<uint4 *>(raw + it * 16) = vw[u];  // rows of d bytes
        }
        __syncthreads();
        // ---- B: column j, 8 tokens -> one 16-byte chunk of fp16 (1024 + (v + 128) - 1152
        // = v, exactly); lanes 0..7 of a quarter warp take 8 consecutive columns, so
        // its 8 chunks land on distinct banks
        const int groups = ntok / 8;
        for (int it = tid; it < d * groups; it += 256) {
            const int gk = (int)__umulhi((uint32_t)it, a.rcp_d), j = it - gk * d;
            uint32_t bytes[2];
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const uint8_t *src = raw + (gk * 8 + 4 * h) * d + j;
                bytes[h] = prmt(prmt((uint32_t)src[0], (uint32_t)src[d], 0x0040u),
                                prmt((uint32_t)src[2 * d], (uint32_t)src[3 * d], 0x0040u), 0x5410u) ^
                           0x80808080u;
            }
            uint4 o;
            o.x = hsub2_u32(prmt(bytes[0], 0x64646464u, 0x5140u), 0x64806480u);
            o.y = hsub2_u32(prmt(bytes[0], 0x64646464u, 0x7362u), 0x64806480u);
            o.z = hsub2_u32(prmt(bytes[1], 0x64646464u, 0x5140u), 0x64806480u);
            o.w = hsub2_u32(prmt(bytes[1], 0x64646464u, 0x7362u), 0x64806480u);
            const uint32_t off = (uint32_t)(j >> 3) * 1024u + (uint32_t)(j & 7) * 128u +
                                 ((((uint32_t)gk) ^ (uint32_t)(j & 7)) << 4);
            *reinterpret_cast<uint4 *>(Bs + off) = o;
        }
        fence_proxy_async_smem();
        __syncthreads();
        if (tid == 0) {
            tc_fence_after();
            const uint64_t alo = sdesc_sw128(smem_u32(A_lo)), ahi = sdesc_sw128(smem_u32(A_hi));
            const uint64_t bd = sdesc_sw128(smem_u32(Bs));
            for (int ks = 0; ks < nks; ++ks) {
                // descriptor addresses in 16-byte units: 32 bytes (+2) per K step of 16
                const uint64_t aoff = (uint64_t)(ks * 2), boff = aoff;
                const uint32_t acc = (rd > 0 || ks > 0) ? 1u : 0u;
                mma_f16_ss(tmem, alo + aoff, bd + boff, idesc, acc);
                if constexpr (HI) mma_f16_ss(tmem + (uint32_t)d, ahi + aoff, bd + boff, idesc, acc);
            }
            mma_commit(smem_u32(bar));
        }
        __syncwarp();
        // the next round's codes and values travel while the MMAs run; one warp
        // polls the barrier, the others wait at the CTA barrier without issuing
        if (rd + 1 < rounds) shift_load_values(a, tid, rd + 1, vb, vw);
        if (warp == 0) {
            const bool done = mbar_wait(smem_u32(bar), (uint32_t)(rd & 1), a.status);
            if (lane == 0) *ok_flag = done ? 1u : 0u;
        }
        __syncthreads();
        ok = *reinterpret_cast<volatile uint32_t *>(ok_flag) != 0u;
        tc_fence_after();
    }
    if (ok) {
        // ---- epilogue: warp w reads TMEM lanes 32 (w % 4) .. +31 (its rows), pieces of 16 columns
        const int quad = warp & 3, half = warp >> 2;
        const int i = i0 + quad * 32 + lane;
        int32_t *orow = a.out + (b * a.Lq + i) * (int64_t)d;
        const uint32_t trow = tmem + ((uint32_t)(quad * 32) << 16);
        const bool small = a.Lk <= 256;  // |lo|, |hi| <= 2^14 Lk <= 2^22
        for (int p = half; p < d / 16; p += 2) {
            uint32_t lo[16], hi[16];
            tmem_ld16(trow + (uint32_t)(p * 16), lo);
            if constexpr (HI) tmem_ld16(trow + (uint32_t)(d + p * 16), hi);
            tmem_ld_wait();
            int32_t o[16];
#pragma unroll
            for (int q = 0; q < 16; ++q) {
                int32_t vlo = small ? exact_f2i_small(lo[q]) : __float2int_rn(__int_as_float(lo[q]));
                if constexpr (HI) {
                    const int32_t vhi = small ? exact_f2i_small(hi[q]) : __float2int_rn(__int_as_float(hi[q]));
                    vlo = (int32_t)((uint32_t)vlo + ((uint32_t)vhi << 8));
                }
                o[q] = vlo;
            }
            if (i < a.Lq) {
                int4 *dst = reinterpret_cast<int4 *>(orow + p * 16);
#pragma unroll
                for (int q = 0; q < 4; ++q) dst[q] = make_int4(o[4 * q], o[4 * q + 1], o[4 * q + 2], o[4 * q + 3]);
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) tmem_dealloc(tmem, a.tmem_cols);
}

// Constants of the integer exponential from the scale S: fp32 quotients of the
// page's constants, floored.  Returns false when they leave the supported range.
struct LisConsts {
    int64_t x0, b, c;
};

qnn_status lis_constants(float S, LisConsts *k)
{
    if (!(S > 0.0f) || !std::isfinite(S)) return QNN_ERR_INVALID_ARG;
    const double ca = 1.0 / 0.35815147, ba = 0.96963238 / 0.35815147;
    const float S2 = S * S;
    const float fx0 = std::floor((float)(-0.6931) / S);
    const float fb = std::floor((float)ba / S);
    const float fc = std::floor((float)ca / S2);
    if (!std::isfinite(fx0) || !std::isfinite(fb) || !std::isfinite(fc)) return QNN_ERR_OVERFLOW_RISK;
    if (fc >= 2147483648.0f || fb >= 2147483648.0f || fx0 <= -2147483648.0f) return QNN_ERR_OVERFLOW_RISK;
    k->x0 = (int64_t)fx0;
    k->b = (int64_t)fb;
    k->c = (int64_t)fc;
    if (k->x0 >= 0 || k->b <= 0 || k->c <= 0) return QNN_ERR_INVALID_ARG;
    if (-k->x0 >= (1 << 20)) return QNN_ERR_OVERFLOW_RISK;
    return QNN_OK;
}

}  // namespace
}  // namespace qnn

namespace qnn {
namespace {

// Validated Log-Int-Softmax constants for scale S, code width bits and row length L.
qnn_status lis_prepare(float S, int bits, int64_t L, LisArgs &a)
{
    if (L <= 0 || bits < 1 || bits > 5) return QNN_ERR_INVALID_ARG;
    LisConsts k;
    const qnn_status st = lis_constants(S, &k);
    if (st != QNN_OK) return st;
    // s <= L * c_int * 2^30 must stay below 2^64
    if ((uint64_t)L > ((1ull << 34) - 1) / (uint64_t)k.c) return QNN_ERR_OVERFLOW_RISK;
    // z = c - r (b - r) must stay in (0, c] for every remainder r in [0, x0n):
    // r <= b, and the largest r (b - r), at r nearest b / 2, below c
    const int64_t x0n = -k.x0;
    if (30 * x0n >= (1 << 21) || k.b < x0n - 1) return QNN_ERR_INVALID_ARG;
    for (int64_t r : {std::min(x0n - 1, k.b / 2), std::min(x0n - 1, (k.b + 1) / 2), x0n - 1})
        if (r * (k.b - r) >= k.c) return QNN_ERR_INVALID_ARG;
    a = LisArgs{};
    a.L = L;
    a.x0n = (uint32_t)x0n;
    a.ndmax = (uint32_t)(30 * x0n);
    a.b = (int32_t)k.b;
    a.c = (int32_t)k.c;
    // nd <= 30 x0n: with l = floor(log2 x0n) and m = ceil(2^(32 + l) / x0n) < 2^32 the
    // error m x0n - 2^(32+l) < x0n keeps mulhi(nd, m) >> l = floor(nd / x0n) exact
    // (nd x0n < 2^(32 + l)); a power of two 2^l takes m = 2^31, shift l - 1
    int l = 0;
    while ((2ll << l) <= x0n) ++l;
    if (x0n == 1) {
        a.qm = 0;
        a.ql = 0;
    } else if (x0n == (1ll << l)) {
        a.qm = 1u << 31;
        a.ql = (uint32_t)(l - 1);
    } else {
        a.qm = (uint32_t)(((1ull << (32 + l)) + (uint64_t)x0n - 1) / (uint64_t)x0n);
        a.ql = (uint32_t)l;
    }
    a.kmax = 1 << bits;
    return QNN_OK;
}

// Shape checks shared by the shift product and the fused attention.
qnn_status shift_check(int64_t batch, int Lq, int Lk, int d, int bits)
{
    if (batch < 0 || Lq < 0 || Lk <= 0 || d <= 0 || bits < 1 || bits > 4) return QNN_ERR_INVALID_ARG;
    if (d % 16 != 0) return QNN_ERR_UNSUPPORTED;
    if (batch > 65535) return QNN_ERR_UNSUPPORTED;
    // |sum| <= Lk * 128 * 2^(2^bits - 1) must fit int32
    if ((int64_t)Lk * 128 * (1ll << ((1 << bits) - 1)) > (1ll << 31)) return QNN_ERR_OVERFLOW_RISK;
    return QNN_OK;
}

// The tensor-pipe shift product (fused: codes computed from m.x first).
template <bool FUSED>
qnn_status launch_shift_mma(ShiftMmaArgs &m, const uint8_t *code, const int8_t *v, int32_t *out, int64_t batch,
                            int Lq, int Lk, int d, int bits, cudaStream_t s)
{
    // weights split into two fp16 halves when N = 2^bits - 1 >= 8
    const bool hi = bits == 4;
    const int N = (1 << bits) - 1;
    uint8_t tab[8];
    for (int j = 0; j < 8; ++j) {
        const int e = hi ? 7 - j : N - j;  // exponent of the weight for code & 7 == j
        tab[j] = (uint8_t)(e >= 0 ? (e + 15) << 2 : 0);
    }
    m.code = code;
    m.v = v;
    m.out = out;
    m.code_bytes = (uint64_t)batch * (uint64_t)Lq * (uint64_t)Lk;
    m.Lq = Lq;
    m.Lk = Lk;
    m.d = d;
    m.tab0 = (uint32_t)tab[0] | ((uint32_t)tab[1] << 8) | ((uint32_t)tab[2] << 16) | ((uint32_t)tab[3] << 24);
    m.tab1 = (uint32_t)tab[4] | ((uint32_t)tab[5] << 8) | ((uint32_t)tab[6] << 16) | ((uint32_t)tab[7] << 24);
    m.rcp_d = (uint32_t)((0x100000000ull + (uint64_t)d - 1) / (uint64_t)d);
    m.rcp_c = d == 16 ? 0u : (uint32_t)((0x100000000ull + (uint64_t)(d / 16) - 1) / (uint64_t)(d / 16));
    uint32_t cols = 32;
    while (cols < (uint32_t)(hi ? 2 * d : d)) cols *= 2;
    m.tmem_cols = cols;
    m.tile_bytes = ((uint32_t)std::min(Lq, kMmaRows) * (uint32_t)Lk + 32u + 127u) & ~127u;
    m.status = status_word();
    const uint32_t smem = shift_mma_smem(d, hi, m.tile_bytes);
    const dim3 grid((Lq + kMmaRows - 1) / kMmaRows, (unsigned)batch);
    // the largest dynamic shared memory (d = 128, Lk = 512) is set once per kernel and process
    static std::atomic<int> attr_set[2];
    auto kern = hi ? attn_shift_mma_kernel<true, FUSED> : attn_shift_mma_kernel<false, FUSED>;
    if (!attr_set[hi].load(std::memory_order_acquire)) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)shift_mma_smem(128, hi, 128u * 512u + 128u)) != cudaSuccess)
            return QNN_ERR_CUDA;
        attr_set[hi].store(1, std::memory_order_release);
    }
    kern<<<grid, 256, smem, s>>>(m);
    return launch_status();
}

}  // namespace
}  // namespace qnn

extern "C" qnn_status q_log_int_softmax(const int32_t *x, int64_t rows, int64_t L, float S, int bits,
                                        uint8_t *code, qnn_stream_t stream)
{
    using namespace qnn;
    if (rows < 0) return QNN_ERR_INVALID_ARG;
    LisArgs a;
    const qnn_status st = lis_prepare(S, bits, L, a);
    if (st != QNN_OK) return st;
    if (rows == 0) return QNN_OK;
    if (x == nullptr || code == nullptr) return QNN_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(code)) return QNN_ERR_ALIGNMENT;
    a.x = x;
    a.code = code;
    a.rows = rows;
    const int64_t want = (rows + kLisWarps - 1) / kLisWarps;
    cudaStream_t s = (cudaStream_t)stream;
    const int R = L <= 256 ? (int)((L + 31) / 32) : 0;
    // 8 blocks of 8 warps per SM, a grid-stride loop over the rows (measured
    // slightly faster than one wave of the resident blocks)
    const int grid = (int)std::min<int64_t>(want, (int64_t)sm_count() * 8);
    auto launch = [&](auto kern) { kern<<<grid, kLisWarps * 32, 0, s>>>(a); };
#define QNN_LIS(RR)                              \
    case RR:                                     \
        launch(log_int_softmax_kernel<RR>);      \
        break;
    switch (R) {
        QNN_LIS(1)
        QNN_LIS(2)
        QNN_LIS(3)
        QNN_LIS(4)
        QNN_LIS(5)
        QNN_LIS(6)
        QNN_LIS(7)
        QNN_LIS(8)
        QNN_LIS(0)
    }
#undef QNN_LIS
    return launch_status();
}

extern "C" qnn_status q_attn_shift_v(const uint8_t *code, const int8_t *v, int64_t batch, int Lq, int Lk,
                                     int d, int bits, int32_t *out, qnn_stream_t stream)
{
    using namespace qnn;
    qnn_status st = shift_check(batch, Lq, Lk, d, bits);
    if (st != QNN_OK) return st;
    if (batch == 0 || Lq == 0) return QNN_OK;
    if (code == nullptr || v == nullptr || out == nullptr) return QNN_ERR_INVALID_ARG;
    if (!aligned16(code) || !aligned16(v) || !aligned16(out)) return QNN_ERR_ALIGNMENT;
    cudaStream_t s = (cudaStream_t)stream;
    if (d <= 128 && Lk <= 512) {
        ShiftMmaArgs m{};
        return launch_shift_mma<false>(m, code, v, out, batch, Lq, Lk, d, bits, s);
    }
    ShiftArgs a{code, v, out, Lq, Lk, d, 1 << bits};
    const dim3 grid((Lq + kShM - 1) / kShM, (d + kShN - 1) / kShN, (unsigned)batch);
    attn_shift_v_kernel<<<grid, 256, 0, s>>>(a);
    return launch_status();
}

extern "C" qnn_status q_lis_attn_v(const int32_t *x, float S, const int8_t *v, int64_t batch, int Lq, int Lk, int d,
                                   int bits, int32_t *out, qnn_stream_t stream)
{
    using namespace qnn;
    qnn_status st = shift_check(batch, Lq, Lk, d, bits);
    if (st != QNN_OK) return st;
    if (d > 128 || Lk > 256) return QNN_ERR_UNSUPPORTED;
    ShiftMmaArgs m{};
    st = lis_prepare(S, bits, Lk, m.lis);
    if (st != QNN_OK) return st;
    if (batch == 0 || Lq == 0) return QNN_OK;
    if (x == nullptr || v == nullptr || out == nullptr) return QNN_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(v) || !aligned16(out)) return QNN_ERR_ALIGNMENT;
    m.x = x;
    return launch_shift_mma<true>(m, nullptr, v, out, batch, Lq, Lk, d, bits, (cudaStream_t)stream);
}
