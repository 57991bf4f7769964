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
// in exact integers (q from an fp32 quotient estimate with a remainder
// correction).  The row sum s is a u64 warp reduction.  The code is not formed
// from v = round(s / e) per element: for each threshold of log_round (v >= 2,
// 3, 6, 12, ..., 3 * 2^(j-2)) the warp first computes, once per row, the largest
// e whose rounded ratio still reaches it -- E_j, one exact u64 division per lane
// -- and each element's code is then the number of E_j >= e, a binary search
// over the row's E table in shared memory.  That equals log_round(round(s/e))
// exactly, half-to-even ties included.
//
// q_attn_shift_v: out[b][i][j] = sum_t 2^(2^bits - 1 - k[b][i][t]) v[b][t][j]
// over unmasked codes, exact in int32 (the host rejects shapes that could
// overflow).  A 64 x 64 output tile per block, 4 x 4 per thread, the weights
// 2^(N - k) expanded into shared memory once per 64-token chunk.
#include <cuda_runtime.h>
#include <cmath>
#include <cstdint>
#include "qnn_internal.h"

namespace qnn {
namespace {

constexpr unsigned kFull = 0xffffffffu;
constexpr int kLisWarps = 8;

struct LisArgs {
    const int32_t *x;
    uint8_t *code;
    int64_t rows, L;
    int32_t x0n;      // -x0_int (> 0)
    int32_t dmin;     // 30 * x0_int: the clamp of x - max(x)
    int32_t b, c;     // b_int, c_int
    float rcp_x0n;    // fp32 1 / x0n, the quotient estimate
    int kmax;         // 2^bits
};

// Integer exponential of x - mx (mx the row maximum; thr = mx + 30 x0_int).
__device__ __forceinline__ uint64_t lis_exp(int32_t x, int32_t mx, int64_t thr, const LisArgs &a)
{
    // nd = -(x - mx) clamped to 30 |x0_int|; the unsigned difference is exact
    // whenever x >= thr, the only case it is used
    const uint32_t nd = ((int64_t)x < thr) ? (uint32_t)(-a.dmin) : (uint32_t)mx - (uint32_t)x;
    int32_t q = (int32_t)__float2uint_rz(__uint2float_rn(nd) * a.rcp_x0n);
    int32_t r = (int32_t)nd - q * a.x0n;  // nd < 2^20: the estimate is off by one at most
    if (r < 0) {
        --q;
        r += a.x0n;
    } else if (r >= a.x0n) {
        ++q;
        r -= a.x0n;
    }
    // the page's remainder is -r (in (x0_int, 0]): z = (-r)(-r + b) + c
    const int64_t z = (int64_t)a.c - (int64_t)r * (int64_t)(a.b - r);
    return z > 0 ? (uint64_t)z << (30 - q) : 0ull;
}

// E table of one row: lane j-1 computes E_j, the largest e with
// round_half_even(s / e) >= L_j, L_1 = 2 and L_j = 3 * 2^(j-2) (the values of v
// where log_round steps up).  round(s/e) >= L  <=>  2s > (2L-1) e, or equality
// with L even; so E = floor(2s / (2L-1)), minus one when (2L-1) divides 2s and L
// is odd.
__device__ __forceinline__ void lis_table(uint64_t s, int lane, int kmax, uint64_t *E)
{
    if (lane < kmax) {
        const int j = lane + 1;
        const uint64_t Lj = j == 1 ? 2ull : (3ull << (j - 2));
        const uint64_t D = 2 * Lj - 1;
        const uint64_t q1 = s / D;
        const uint64_t r1 = s - q1 * D;
        uint64_t Ej = 2 * q1, r2 = 2 * r1;
        if (r2 >= D) {
            Ej += 1;
            r2 -= D;
        }
        if (r2 == 0 && (Lj & 1)) Ej -= 1;  // s >= 1, so Ej >= 1 here
        E[lane] = Ej;
    }
    __syncwarp();
}

// Code of one exponential: the number of E_j >= e, kmax when masked.
__device__ __forceinline__ uint32_t lis_code(uint64_t e, const uint64_t *E, int kmax)
{
    if (e <= E[kmax - 1]) return (uint32_t)kmax;
    int pos = 0;
    for (int step = kmax >> 1; step; step >>= 1)
        if (E[pos + step - 1] >= e) pos += step;
    return (uint32_t)pos;
}

__device__ __forceinline__ uint64_t warp_sum_u64(uint64_t v)
{
#pragma unroll
    for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(kFull, v, o);
    return v;
}

// R > 0: rows of L <= 32 R held in registers.  R == 0: any L, three passes over
// the row (the later two from cache).
template <int R>
__global__ void __launch_bounds__(kLisWarps * 32) log_int_softmax_kernel(LisArgs a)
{
    __shared__ uint64_t Etab[kLisWarps][32];
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    uint64_t *E = Etab[w];
    const int64_t L = a.L;
    for (int64_t row = (int64_t)blockIdx.x * kLisWarps + w; row < a.rows;
         row += (int64_t)gridDim.x * kLisWarps) {
        const int32_t *xr = a.x + row * L;
        uint8_t *cr = a.code + row * L;
        if constexpr (R > 0) {
            int32_t xv[R];
            int32_t mx = INT32_MIN;
#pragma unroll
            for (int j = 0; j < R; ++j) {
                const int64_t i = lane + 32 * j;
                xv[j] = i < L ? __ldcs(xr + i) : INT32_MIN;
                mx = max(mx, xv[j]);
            }
            mx = __reduce_max_sync(kFull, mx);
            const int64_t thr = (int64_t)mx + a.dmin;
            uint64_t ev[R];
            uint64_t s = 0;
#pragma unroll
            for (int j = 0; j < R; ++j) {
                ev[j] = lis_exp(xv[j], mx, thr, a);
                if (lane + 32 * j < L) s += ev[j];
            }
            s = warp_sum_u64(s);
            lis_table(s, lane, a.kmax, E);
#pragma unroll
            for (int j = 0; j < R; ++j) {
                const int64_t i = lane + 32 * j;
                if (i < L) __stcs(cr + i, (uint8_t)lis_code(ev[j], E, a.kmax));
            }
        } else {
            int32_t mx = INT32_MIN;
            for (int64_t i = lane; i < L; i += 32) mx = max(mx, __ldg(xr + i));
            mx = __reduce_max_sync(kFull, mx);
            const int64_t thr = (int64_t)mx + a.dmin;
            uint64_t s = 0;
            for (int64_t i = lane; i < L; i += 32) s += lis_exp(__ldg(xr + i), mx, thr, a);
            s = warp_sum_u64(s);
            lis_table(s, lane, a.kmax, E);
            for (int64_t i = lane; i < L; i += 32)
                __stcs(cr + i, (uint8_t)lis_code(lis_exp(__ldg(xr + i), mx, thr, a), E, a.kmax));
        }
        __syncwarp();  // E is rewritten for the next row
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

extern "C" qnn_status q_log_int_softmax(const int32_t *x, int64_t rows, int64_t L, float S, int bits,
                                        uint8_t *code, qnn_stream_t stream)
{
    using namespace qnn;
    if (rows < 0 || L <= 0 || bits < 1 || bits > 5) return QNN_ERR_INVALID_ARG;
    LisConsts k;
    const qnn_status st = lis_constants(S, &k);
    if (st != QNN_OK) return st;
    // s <= L * c_int * 2^30 must stay below 2^64
    if ((uint64_t)L > ((1ull << 34) - 1) / (uint64_t)k.c) return QNN_ERR_OVERFLOW_RISK;
    if (rows == 0) return QNN_OK;
    if (x == nullptr || code == nullptr) return QNN_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(code)) return QNN_ERR_ALIGNMENT;
    LisArgs a{};
    a.x = x;
    a.code = code;
    a.rows = rows;
    a.L = L;
    a.x0n = (int32_t)(-k.x0);
    a.dmin = (int32_t)(30 * k.x0);
    a.b = (int32_t)k.b;
    a.c = (int32_t)k.c;
    a.rcp_x0n = 1.0f / (float)a.x0n;
    a.kmax = 1 << bits;
    const int64_t want = (rows + kLisWarps - 1) / kLisWarps;
    const int grid = (int)std::min<int64_t>(want, (int64_t)sm_count() * 8);
    cudaStream_t s = (cudaStream_t)stream;
    if (L <= 32) log_int_softmax_kernel<1><<<grid, kLisWarps * 32, 0, s>>>(a);
    else if (L <= 64) log_int_softmax_kernel<2><<<grid, kLisWarps * 32, 0, s>>>(a);
    else if (L <= 128) log_int_softmax_kernel<4><<<grid, kLisWarps * 32, 0, s>>>(a);
    else if (L <= 256) log_int_softmax_kernel<8><<<grid, kLisWarps * 32, 0, s>>>(a);
    else log_int_softmax_kernel<0><<<grid, kLisWarps * 32, 0, s>>>(a);
    return launch_status();
}

extern "C" qnn_status q_attn_shift_v(const uint8_t *code, const int8_t *v, int64_t batch, int Lq, int Lk,
                                     int d, int bits, int32_t *out, qnn_stream_t stream)
{
    using namespace qnn;
    if (batch < 0 || Lq < 0 || Lk <= 0 || d <= 0 || bits < 1 || bits > 4) return QNN_ERR_INVALID_ARG;
    if (d % 16 != 0) return QNN_ERR_UNSUPPORTED;
    if (batch > 65535) return QNN_ERR_UNSUPPORTED;
    // |sum| <= Lk * 128 * 2^(2^bits - 1) must fit int32
    if ((int64_t)Lk * 128 * (1ll << ((1 << bits) - 1)) > (1ll << 31)) return QNN_ERR_OVERFLOW_RISK;
    if (batch == 0 || Lq == 0) return QNN_OK;
    if (code == nullptr || v == nullptr || out == nullptr) return QNN_ERR_INVALID_ARG;
    if (!aligned16(code) || !aligned16(v) || !aligned16(out)) return QNN_ERR_ALIGNMENT;
    ShiftArgs a{code, v, out, Lq, Lk, d, 1 << bits};
    const dim3 grid((Lq + kShM - 1) / kShM, (d + kShN - 1) / kShN, (unsigned)batch);
    attn_shift_v_kernel<<<grid, 256, 0, (cudaStream_t)stream>>>(a);
    return launch_status();
}
