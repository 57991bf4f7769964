// qnn_mma_kernel.cuh -- the persistent, warp-specialised tcgen05 kernel shared
// by the quantized GEMM and the implicit-GEMM convolutions.
//
// Both compute, for rows r (GEMM rows, or output pixels (n, oh, ow)) and
// columns n (output channels),
//     acc[r][n] = sum_k a(r, k) * B[n][k]            (exact integers)
// followed by the fused epilogue of qnn.h (zero-point term, requant / dequant
// / raw int32).  What differs between the ops is only how a row of the
// activation operand is fetched and re-encoded for the MMA; that is the `Op`
// policy (load / store of one pipeline unit, plus the MMA kind):
//   GemmOp<PTF>  : int8 rows of A [M, K] -> fp16 (kind::f16)
//   ConvU8Op     : im2col of u8 NHWC      -> fp16 (kind::f16)
//   ConvU4Op     : im2col of u4 NHWC      -> e4m3 codes of c / 512 (kind::f8f6f4)
//
//   GemmPackedOp : A already re-encoded (fp16, swizzled) by a pre-pass; the
//                  producer copies it like the weights (no converter warps)
//
// Warp roles (512 threads, one CTA per SM, persistent over 128 x TBN tiles):
//   warps 0-3  : converters -- fetch the activation rows of one pipeline unit
//                (128 rows x one K step) from global memory, one unit ahead,
//                re-encode them and store them into the 128-byte swizzled
//                K-major stage buffer.  Idle for Ops with a prepacked A.
//   warp 4     : TMA producer -- one bulk copy per stage of the prepacked
//                weight tile (already in the swizzled image), and one of the
//                prepacked activation tile for Ops with TMA_A.
//   warp 5     : TMEM owner and MMA issuer -- 4 x tcgen05.mma per stage into
//                one of two TBN-column fp32 TMEM accumulators.
//   warps 8-15 : epilogue -- tcgen05.ld, fp32 -> int32 (exact), optional
//                int32 sums over K chunks, then the fused requant / dequant
//                math and 16-byte stores of 32 consecutive output columns.
// Every mbarrier wait is bounded (qnn_ptx.cuh): on time-out the role sets the
// device status word and winds down instead of hanging.
#pragma once
#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <cstdint>
#include <type_traits>
#include "qnn_gemm_layout.h"
#include "qnn_internal.h"
#include "qnn_ptx.cuh"

namespace qnn {
namespace mk {

using gemm::BM;
using gemm::ROW_BYTES;

constexpr int NUM_THREADS = 512;
constexpr int PRODUCER_WARP = 4;
constexpr int MMA_WARP = 5;
constexpr int EPI_WARP0 = 8;

// Epilogue warps: warps 8-15, plus warps 0-3 when the Op needs no converter
// warps (its A arrives by copy) and the tile has at least three 32-column
// pieces.  Each group of four warps covers the 128 TMEM lanes for its share
// of the pieces (group g: pieces g*P/G .. (g+1)*P/G - 1 of P, G groups).
template <class Op, int TBN>
__host__ __device__ constexpr int epi_warps() { return (Op::TMA_A && TBN >= 128) ? 12 : 8; }
template <class Op, int TBN>
__host__ __device__ constexpr int epi_max_pieces() { return (TBN / 32 + epi_warps<Op, TBN>() / 4 - 1) / (epi_warps<Op, TBN>() / 4); }
constexpr int A_STAGE_BYTES = BM * ROW_BYTES;  // 128-byte rows (every Op but the TMA conv)

struct Params {
    // activation tensor map (implicit-GEMM conv fed by TMA); first, 64-byte aligned
    alignas(64) CUtensorMap tmap;
    // activation operand
    const uint8_t *A;
    int a_u8;                // GEMM: 1 if A holds u8 codes (centred at 128), 0 for s8
    const uint8_t *ptf;      // GEMM: per-K Power-of-Two Factor shifts, or null
    const uint8_t *Ap;       // prepacked activation image [num_m][KT][128 rows][128 B] (TMA_A Ops)
    // convolution geometry (NHWC input, OHWI weights, K order (fh, fw, c))
    int H, W, Cin, OHW, OW, FH, FW, ph, pw, sh, sw;
    uint32_t pad_word;       // input bytes that stand for the padding value z_in
    // TMA conv: output tile = TN images x TH rows x TW columns of pixels; unit = one filter tap
    // x `cpu` input channels (cbn units per tap); zcs: weight column sums, z_cs: their factor
    int Nimg, OH, TW, TH, TN, tiles_x, tiles_y, cpu, cbn;
    const int32_t *zcs;
    int z_cs;
    // weights (prepacked image) and shape of the GEMM view
    const uint8_t *Bp;
    int M, N, K, KT, num_m, num_tiles;
    // exact fp32 chunks: chunk_steps K steps each (host bound); with btrail (the
    // trailer of a prepacked GEMM weight image) the kernel derives the length from
    // the recorded weight magnitudes instead, for activation codes of magnitude at
    // most 128 * 2^a_shift
    int chunk_steps, nchunks;
    const int32_t *btrail;
    int a_shift;
    int amax;                // largest activation magnitude the MMA sees, if not 128 * 2^a_shift
    int ptf_max;             // GEMM with ptf: bound the host was given for every shift byte
    // epilogue
    int mode, relu, z_out, out_bits, out_signed;
    float clip_lo_f, clip_hi_f;  // requant: clip of v before rounding and adding z_out (ReLU folded in)
    const int32_t *zp;
    // weight zero points (Z_w != 0): acc_c += (128 - zw[n]) * rowsum[m], rowsum the
    // per-row sums of the centred activation codes written by the A pre-pass
    const int32_t *zw;
    const int32_t *rowsum;
    const float *row_scale;  // per-row activation scales (dynamic quantization), or null
    const float *Mv;
    const float *Bq;
    const float *D;
    const float *bias;
    const uint8_t *res;
    int res_bits, res_signed, z_res;
    float R;
    float res_c;             // 1.5 * 2^23 + z_res (+ 128 or 8 for signed residual codes)
    void *C;
    int32_t *C32;
    int vec_ok;              // N % 32 == 0: every 32-column piece whole and 16-byte aligned
    // conv layout of the input, the output and the residual (qnn_layout; GEMMs: 0).
    // Output / residual rows m = (n, oh, ow) = n * OHW + pixel.
    int layout;
    uint32_t *status;
};

// Defaults every Op inherits: 4 stages of 128-byte operand rows, and GEMM
// rows in tile order (row r of row block mb is GEMM row mb * 128 + r).
struct OpBase {
    static constexpr int STAGES = 4;
    static constexpr int ROW = 128;
    static constexpr int SUB = 1;            // K steps (operand sub-tiles) per pipeline unit
    static constexpr bool RESB = false;      // weights resident in shared memory for the whole kernel
    static constexpr int B_RES_BYTES = 0;
    static constexpr bool ROTATE_K = true;  // each CTA starts its tiles' K walk at its own offset
    static constexpr bool CACHE_COLS = false;  // epilogue keeps column constants across tiles of one column block
    static constexpr bool LAYOUTS = false;     // outputs / residuals may be in a conv layout (qnn_layout)
    struct PState {};                        // producer-side state of a TMA_A Op
    struct RowInfo {                         // per-thread part of the row mapping
        int r;
    };
    __device__ static RowInfo row_info(const Params &, int r) { return RowInfo{r}; }
    __device__ static int out_row(const Params &, int mb, const RowInfo &ri) { return mb * BM + ri.r; }
    // barriers the Op keeps in its staging area, initialised by thread 0 at kernel start
    __device__ static void init(uint4 *) {}
};

template <class Op, int TBN>
struct __align__(1024) Smem {
    uint8_t a[Op::STAGES][Op::SUB * BM * Op::ROW];
    uint8_t b[Op::STAGES][Op::RESB ? 1024 : Op::SUB * TBN * Op::ROW];
    uint8_t bres[Op::RESB ? Op::B_RES_BYTES : 1024];  // resident weights: [K step][TBN rows][ROW]
    uint4 stg[Op::STG_BYTES / 16];                   // converter staging ring (Op-specific)
    float cols[epi_warps<Op, TBN>()][4 * 32 * epi_max_pieces<Op, TBN>()];  // per epilogue warp: its columns' constants
    uint64_t full[Op::STAGES];   // 4 converter-warp arrivals (none with TMA_A) + the producer's expect_tx
    uint64_t empty[Op::STAGES];
    uint64_t acc_full[2];
    uint64_t acc_empty[2];
    uint64_t mma_done;
    uint64_t bres_full;
    uint64_t plan_ready;         // the chunk plan below has been written
    int32_t plan_steps, plan_count;
    uint32_t tmem_base;
};

template <class Op, int TBN>
constexpr size_t smem_bytes() { return sizeof(Smem<Op, TBN>) + 1024; }

// Walks this CTA's units -- (tile, K step) pairs, tile by tile -- without
// divisions in the steady state.  Each CTA walks K starting at its own offset
// (blockIdx.x mod KT), so CTAs that share a weight block read different slices
// of it at any moment; integer sums do not depend on the order, and a chunk of
// consecutive units still spans at most chunk_steps K steps.
struct UnitCursor {
    int kl;      // position of the unit within its tile, 0 .. KT - 1
    int ks;      // K step the unit covers
    int rot;     // first K step of every tile
    int t;       // tile index
    int mb, nb;  // tile coordinates: row block, column block

    __device__ __forceinline__ void begin(const Params &p, bool rotate = true)
    {
        rot = rotate ? (int)(blockIdx.x % (unsigned)p.KT) : 0;
        t = blockIdx.x;
        kl = 0;
        ks = rot;
        mb = t % p.num_m;
        nb = t / p.num_m;
    }
    __device__ __forceinline__ void next(const Params &p)
    {
        if (++kl == p.KT) {
            kl = 0;
            ks = rot;
            t += gridDim.x;
            mb = t % p.num_m;
            nb = t / p.num_m;
        } else if (++ks == p.KT) {
            ks = 0;
        }
    }
};

// Length (K steps) of the exact accumulation chunks and their number per tile.
// From the weight image's trailer when there is one (the bound certified by the
// prepack for the values actually stored), else the host's bound.  A trailer
// that does not belong to this K is reported as an invalid argument.
struct ChunkPlan {
    int steps, count;
};

__device__ __forceinline__ ChunkPlan chunk_plan(const Params &p, bool report)
{
    int L = p.chunk_steps;
    if (p.btrail) {
        const int32_t magic = __ldg(p.btrail + gemm::TR_MAGIC);
        const int32_t kt = __ldg(p.btrail + gemm::TR_KT);
        if (magic == gemm::TRAILER_MAGIC && kt == p.KT) {
            L = gemm::certified_chunk_steps(__ldg(p.btrail + gemm::TR_STEP_MAX), __ldg(p.btrail + gemm::TR_TOTAL_MAX),
                                            p.amax ? (int64_t)p.amax : (int64_t)128 << p.a_shift, p.KT);
        } else if (report) {
            atomicOr(p.status, kStatusBadArg);
        }
    }
    return ChunkPlan{L, (p.KT + L - 1) / L};
}

// A bounded wait whose outcome is the same on every lane of the warp.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, uint32_t *status)
{
    const bool ok = mbar_wait(bar, parity, status);
    return __all_sync(0xffffffffu, ok);
}

// The same for warps off the MMA issue path, which may be suspended while they wait.
__device__ __forceinline__ bool warp_wait_idle(uint32_t bar, uint32_t parity, uint32_t *status)
{
    const bool ok = mbar_wait_idle(bar, parity, status);
    return __all_sync(0xffffffffu, ok);
}

// ---------------------------------------------------------------- converter
// Converts unit j into its stage.  `ready` says whether the stage's empty
// phase was already seen complete; before the conversion work starts, the
// empty phase of unit j + 1 is probed so that its latency is hidden behind it.
template <class Op, int TBN, int D>
__device__ __forceinline__ bool convert_one(const Params &p, Smem<Op, TBN> &s, typename Op::State &st,
                                            int j, int units, int sub, int rbase,
                                            const typename Op::Unit &u, bool &ready)
{
    constexpr int STAGES = Op::STAGES;
    const int stage = j % STAGES;
    const uint32_t ph = (uint32_t)(j / STAGES) & 1u;
    const bool ok = ready || mbar_wait_idle(smem_u32(&s.empty[stage]), ph ^ 1u, p.status);
    if (!__all_sync(0xffffffffu, ok)) return false;
    const int jn = j + 1;
    const bool probe = mbar_test_wait(smem_u32(&s.empty[jn % STAGES]), ((uint32_t)(jn / STAGES) & 1u) ^ 1u);
    if constexpr (std::is_void<decltype(Op::template store<D>(p, st, s.stg, 0u, j, sub, rbase, u))>::value) {
        Op::template store<D>(p, st, s.stg, smem_u32(&s.a[stage][0]), j, sub, rbase, u);
    } else {
        // Ops whose store waits on its own barriers report a wait that gave up
        if (!__all_sync(0xffffffffu, Op::template store<D>(p, st, s.stg, smem_u32(&s.a[stage][0]), j, sub, rbase, u)))
            return false;
    }
    fence_proxy_async_smem();
    __syncwarp();
    if ((threadIdx.x & 31) == 0) mbar_arrive(smem_u32(&s.full[stage]));
    ready = probe && jn < units;
    return true;
}

// Thread t handles the 16-byte input group (t % 4) of rows (t / 4) + 32 q,
// q = 0..3, of every unit.  The loads of the next D - 1 units are in flight
// while a unit is converted (in registers, or in the Op's staging ring).
template <class Op, int TBN, int D>
__device__ void converter_loop(const Params &p, Smem<Op, TBN> &s, int units)
{
    const int tid = threadIdx.x;
    const int sub = tid & 3;
    const int rbase = tid >> 2;
    typename Op::State st{};
    typename Op::Unit u[D];
    bool ready = false;
#pragma unroll
    for (int d = 0; d < D - 1; ++d) Op::template load<D>(p, st, s.stg, d, d < units, sub, rbase, u[d]);
    for (int j0 = 0; j0 < units; j0 += D) {
#pragma unroll
        for (int d = 0; d < D; ++d) {
            const int j = j0 + d;
            if (j >= units) return;
            const int jn = j + D - 1;
            Op::template load<D>(p, st, s.stg, jn, jn < units, sub, rbase, u[(d + D - 1) % D]);
            if (!convert_one<Op, TBN, D>(p, s, st, j, units, sub, rbase, u[d], ready)) return;
        }
    }
}

// Ops whose in-flight units live in their shared-memory staging ring keep
// only a little per-unit state, so their loop is not unrolled (one copy of the
// converter code keeps the instruction cache warm).
template <class Op, int TBN, int D>
__device__ void converter_loop_rolled(const Params &p, Smem<Op, TBN> &s, int units)
{
    const int tid = threadIdx.x;
    const int sub = tid & 3;
    const int rbase = tid >> 2;
    typename Op::State st{};
    typename Op::Unit u;
    bool ready = false;
    // loads that can give up (Ops waiting on their own barriers) return false then
    auto load = [&](int jj) -> bool {
        if constexpr (std::is_void<decltype(Op::template load<D>(p, st, s.stg, jj, true, sub, rbase, u))>::value) {
            Op::template load<D>(p, st, s.stg, jj, jj < units, sub, rbase, u);
            return true;
        } else {
            return __all_sync(0xffffffffu, Op::template load<D>(p, st, s.stg, jj, jj < units, sub, rbase, u));
        }
    };
#pragma unroll 1
    for (int d = 0; d < D - 1; ++d)
        if (!load(d)) return;
#pragma unroll 1
    for (int j = 0; j < units; ++j) {
        if (!load(j + D - 1)) return;
        if (!convert_one<Op, TBN, D>(p, s, st, j, units, sub, rbase, u, ready)) return;
    }
}

template <class Op, int TBN, bool MULTI>
__device__ void converter_role(const Params &p, Smem<Op, TBN> &s, int units)
{
    if constexpr (Op::REG_RING)
        converter_loop<Op, TBN, MULTI ? Op::DEPTH_MULTI : Op::DEPTH>(p, s, units);
    else
        converter_loop_rolled<Op, TBN, MULTI ? Op::DEPTH_MULTI : Op::DEPTH>(p, s, units);
    // no asynchronous copy of this thread may still be writing when the CTA exits
    asm volatile("cp.async.wait_all;" ::: "memory");
}

// ---------------------------------------------------------------- producer
// The producer and MMA roles run on whole warps: every lane waits on the
// barriers (so the warp never diverges around a wait) and lane 0 issues the
// copies, MMAs and commits.  A wait that times out on any lane stops the role.

template <class Op, int TBN>
__device__ void producer_role(const Params &p, Smem<Op, TBN> &s, int units)
{
    const bool leader = (threadIdx.x & 31) == 0;
    constexpr int STAGES = Op::STAGES;
    constexpr int ROW = Op::ROW;
    constexpr int SUB = Op::SUB;
    const uint32_t b0 = smem_u32(&s.b[0][0]);
    UnitCursor c;
    c.begin(p, Op::ROTATE_K);
    typename Op::PState ps{};
    bool ok = true;
    bool ready = false;
    int j = 0;
    if constexpr (Op::RESB) {
        // the whole (single) weight block, once: K step ks -> bres + ks * TBN * ROW
        if (leader && units > 0) {
            const int steps = p.KT * SUB;
            const uint32_t bar = smem_u32(&s.bres_full);
            mbar_arrive_expect_tx(bar, (uint32_t)(steps * TBN * ROW));
            for (int k = 0; k < steps; ++k)
                bulk_g2s(smem_u32(&s.bres[0]) + k * (TBN * ROW), p.Bp + (int64_t)k * (gemm::BN * ROW), TBN * ROW,
                         bar);
        }
        __syncwarp();
    }
    for (; j < units; ++j, c.next(p)) {
        const int stage = j % STAGES;
        const uint32_t ph = (uint32_t)(j / STAGES) & 1u;
        if (!ready && !warp_wait_idle(smem_u32(&s.empty[stage]), ph ^ 1u, p.status)) {
            ok = false;
            break;
        }
        const int jn = j + 1;
        const bool probe = mbar_test_wait(smem_u32(&s.empty[jn % STAGES]), ((uint32_t)(jn / STAGES) & 1u) ^ 1u);
        if (leader) {
            // columns n0 .. n0 + TBN - 1 live in the 256-row packed block n0 / 256
            const int n0 = c.nb * TBN;
            const uint32_t bar = smem_u32(&s.full[stage]);
            constexpr uint32_t B_BYTES = Op::RESB ? 0u : (uint32_t)(SUB * TBN * ROW);
            if constexpr (Op::TMA_A) {
                mbar_arrive_expect_tx(bar, B_BYTES + SUB * Op::a_bytes(p));
#pragma unroll
                for (int t = 0; t < SUB; ++t)
                    Op::load_a(p, c, ps, t, smem_u32(&s.a[stage][0]) + t * (BM * ROW), bar);
            } else {
                mbar_arrive_expect_tx(bar, B_BYTES);
            }
            if constexpr (!Op::RESB) {
#pragma unroll
                for (int t = 0; t < SUB; ++t) {
                    // columns n0 .. n0 + TBN - 1 of K step ks live in the 256-row packed block n0 / 256
                    const int ks = c.ks * SUB + t;
                    const uint8_t *src = p.Bp + ((int64_t)(n0 / gemm::BN) * p.KT * SUB + ks) * (gemm::BN * ROW) +
                                         (int64_t)(n0 % gemm::BN) * ROW;
                    bulk_g2s(b0 + stage * (SUB * TBN * ROW) + t * (TBN * ROW), src, TBN * ROW, bar);
                }
            }
        }
        ready = __all_sync(0xffffffffu, probe) && jn < units;
    }
    if (!ok) {
        // wind down: let the copies already issued land before the CTA exits
        for (int i = (j > STAGES ? j - STAGES : 0); i < j; ++i) {
            const int stage = i % STAGES;
            const uint32_t ph = (uint32_t)(i / STAGES) & 1u;
            if (!warp_wait(smem_u32(&s.full[stage]), ph, p.status)) break;
        }
    }
}

// ---------------------------------------------------------------- MMA
// The issuing loop is kept as short as possible: it is the one serial
// instruction stream every pipeline unit passes through (one wait, four MMAs,
// one or two commits, counters instead of divisions).
template <class Op, int TBN, bool MULTI>
__device__ void mma_role(const Params &p, Smem<Op, TBN> &s, int my_tiles, uint32_t tmem)
{
    constexpr uint32_t IDESC = idesc_f32acc(0, 0, BM, TBN);  // f16 x f16, or e4m3 x e4m3
    constexpr int STAGES = Op::STAGES;
    constexpr int ROW = Op::ROW;
    constexpr int KSLICES = ROW / 32;  // one MMA per 32-byte K slice of a row
    constexpr int SUB = Op::SUB;
    const bool leader = (threadIdx.x & 31) == 0;
    const int units = my_tiles * p.KT;
    const uint64_t adesc0 = sdesc_sw(smem_u32(&s.a[0][0]), ROW);
    const uint64_t bdesc0 = Op::RESB ? sdesc_sw(smem_u32(&s.bres[0]), ROW) : sdesc_sw(smem_u32(&s.b[0][0]), ROW);
    if constexpr (Op::RESB) {
        if (units > 0 && !warp_wait(smem_u32(&s.bres_full), 0u, p.status)) return;
    }
    // The chunk plan (MULTI) is published in shared memory by warp 6 at kernel
    // start; it is first needed once the first stage has landed, so its global
    // load does not delay the first MMAs.  One chunk per tile: the two TMEM
    // accumulators alternate by tile; several: every chunk goes to accumulator 0
    // and the epilogue keeps the int32 running sums in accumulator 1's columns
    // (for the first unit both choices are accumulator 0, phase 0).
    int chunk_steps = p.KT;
    bool single = true;
    int stage = 0;
    uint32_t sph = 0;  // phase of the current stage's full barrier
    uint32_t u = 0;  // accumulation chunk counter
    int kl = 0;      // unit position within the tile
    int cpos = 0;    // unit position within the accumulation chunk
    for (int j = 0; j < units; ++j) {
        const uint32_t abuf = single ? (u & 1u) : 0u;
        const uint32_t uph = single ? ((u >> 1) & 1u) : (u & 1u);
        const bool first = cpos == 0;
        if (first && !warp_wait(smem_u32(&s.acc_empty[abuf]), uph ^ 1u, p.status)) break;
        if (!warp_wait(smem_u32(&s.full[stage]), sph, p.status)) break;
        tc_fence_after();
        if (MULTI && j == 0) {
            if (!warp_wait(smem_u32(&s.plan_ready), 0u, p.status)) break;
            chunk_steps = s.plan_steps;
            single = s.plan_count == 1;
        }
        const bool last = (cpos == chunk_steps - 1) || (kl == p.KT - 1);
        if (leader) {
            // descriptor start addresses are in 16-byte units: +2 per 32-byte K slice
            const uint64_t ad = adesc0 + (uint64_t)(stage * ((SUB * BM * ROW) >> 4));
            // streamed weights sit in the stage; resident ones are indexed by the K step
            const uint64_t bd = Op::RESB ? bdesc0 + (uint64_t)(kl * SUB * ((TBN * ROW) >> 4))
                                         : bdesc0 + (uint64_t)(stage * ((SUB * TBN * ROW) >> 4));
            const uint32_t d = tmem + abuf * TBN;
#pragma unroll
            for (int t = 0; t < SUB; ++t) {
#pragma unroll
                for (int kk = 0; kk < KSLICES; ++kk) {
                    const uint32_t acc = (first && t == 0 && kk == 0) ? 0u : 1u;
                    const uint64_t at = ad + (uint64_t)(t * ((BM * ROW) >> 4)) + 2 * kk;
                    const uint64_t bt = bd + (uint64_t)(t * ((TBN * ROW) >> 4)) + 2 * kk;
                    if (Op::F8)
                        mma_f8f6f4_ss(d, at, bt, IDESC, acc);
                    else
                        mma_f16_ss(d, at, bt, IDESC, acc);
                }
            }
            mma_commit(smem_u32(&s.empty[stage]));
            if (last) mma_commit(smem_u32(&s.acc_full[abuf]));
        }
        __syncwarp();
        if (++stage == STAGES) {
            stage = 0;
            sph ^= 1u;
        }
        if (last) {
            ++u;
            cpos = 0;
        } else {
            ++cpos;
        }
        if (++kl == p.KT) {
            kl = 0;
            cpos = 0;
        }
    }
    // every MMA issued must have completed before the CTA winds down
    if (leader) mma_commit(smem_u32(&s.mma_done));
    __syncwarp();
    (void)warp_wait(smem_u32(&s.mma_done), 0u, p.status);
}

// ---------------------------------------------------------------- epilogue
__device__ __forceinline__ void st_v4(void *ptr, uint32_t a, uint32_t b, uint32_t c, uint32_t d)
{
    *reinterpret_cast<uint4 *>(ptr) = make_uint4(a, b, c, d);
}

// 32 bytes in one 256-bit store (ptr 32-byte aligned).
__device__ __forceinline__ void st_v8(void *ptr, const uint32_t (&w)[8])
{
    asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(ptr), "r"(w[0]), "r"(w[1]),
                 "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7])
                 : "memory");
}

// Each epilogue warp keeps the per-column constants of its COLS columns in
// shared memory: [0, COLS) M (requant) or D (dequant), [COLS, 2 COLS) Bq or
// bias, [2 COLS, 3 COLS) -zp_term as an fp32 value, [3 COLS, 4 COLS) zp_term
// (as int bits).  The loads of a tile's constants are issued before the warp
// waits for the tile's accumulator and stored to shared memory after it.
template <int COLS>
struct ColumnRegs {
    float a[COLS / 32], b[COLS / 32];
    int32_t z[COLS / 32];
};

template <int COLS>
__device__ __forceinline__ void load_columns(const Params &p, ColumnRegs<COLS> &cr, int nbase, int lane)
{
#pragma unroll
    for (int k = 0; k < COLS / 32; ++k) {
        const int n = nbase + 32 * k + lane;
        const bool in = n < p.N;
        float a = 0.0f, b = 0.0f;
        int32_t z = 0;
        if (in) {
            if (p.mode == QNN_EPI_REQUANT) {
                a = __ldg(p.Mv + n);
                b = __ldg(p.Bq + n);
            } else if (p.mode == QNN_EPI_DEQUANT) {
                a = __ldg(p.D + n);
                b = p.bias ? __ldg(p.bias + n) : 0.0f;
            }
            if (p.zp) z = __ldg(p.zp + n);
            if (p.zcs) z -= p.z_cs * __ldg(p.zcs + n);
        }
        cr.a[k] = a;
        cr.b[k] = b;
        cr.z[k] = z;
    }
}

// Returns whether -zp_term is an fp32 value for every column of the warp
// (always so for |zp_term| <= 2^24): then float(acc) + float(-zp_term) is the
// correctly rounded float(acc - zp_term), the conversion the requant formula
// starts from, without an integer round trip.
template <int COLS>
__device__ __forceinline__ bool store_columns(const ColumnRegs<COLS> &cr, float *cols, int lane, bool &zp_zero)
{
    __syncwarp();
    bool exact = true;
    bool zero = true;
#pragma unroll
    for (int k = 0; k < COLS / 32; ++k) {
        const int32_t z = cr.z[k];
        const int32_t nzi = (int32_t)(0u - (uint32_t)z);
        const float nz = __int2float_rn(nzi);
        exact = exact && z != INT32_MIN && __float2int_rn(nz) == nzi;
        zero = zero && z == 0;
        cols[32 * k + lane] = cr.a[k];
        cols[COLS + 32 * k + lane] = cr.b[k];
        cols[2 * COLS + 32 * k + lane] = nz;
        cols[3 * COLS + 32 * k + lane] = __int_as_float(z);
    }
    __syncwarp();
    zp_zero = __all_sync(0xffffffffu, zero);
    return __all_sync(0xffffffffu, exact);
}

// Element offset (in codes) of output element (row m, column n) in the layout
// of the output and the residual, and the distance between consecutive
// columns: NHWC (and every GEMM) m * N + n; NCHW (image, channel, pixel); NCHW64
// (image, channel block, pixel, channel in block).
// LAY: the op supports conv layouts (conv ops); without it, every tensor is
// [rows, N] row-major and none of the layout code is compiled in (GEMMs).
template <bool LAY>
__device__ __forceinline__ int64_t out_off(const Params &p, int m, int n)
{
    if (!LAY || p.layout == QNN_LAYOUT_NHWC) return (int64_t)m * p.N + n;
    const int img = m / p.OHW;
    const int pix = m - img * p.OHW;
    if (p.layout == QNN_LAYOUT_NCHW) return ((int64_t)img * p.N + n) * p.OHW + pix;
    return (((int64_t)img * (p.N >> 6) + (n >> 6)) * p.OHW + pix) * 64 + (n & 63);
}
template <bool LAY>
__device__ __forceinline__ int64_t out_cstride(const Params &p)
{
    return LAY && p.layout == QNN_LAYOUT_NCHW ? p.OHW : 1;
}

// The residual codes of the 32 columns n0.. of row m (8-bit: 8 words of 4
// codes; 4-bit: 4 words of 8 codes), or zeros without a residual.
template <bool LAY>
__device__ __forceinline__ void load_residual(const Params &p, int m, int n0, uint32_t (&rw)[8])
{
#pragma unroll
    for (int i = 0; i < 8; ++i) rw[i] = 0;
    if (!p.res || m >= p.M || n0 >= p.N) return;
    const int64_t base = out_off<LAY>(p, m, n0);
    if (LAY && p.layout == QNN_LAYOUT_NCHW) {
        // one code per channel plane
        const int64_t cs = p.OHW;
        for (int i = 0; i < 32 && n0 + i < p.N; ++i) {
            const int64_t e = base + (int64_t)i * cs;
            if (p.res_bits == 8)
                rw[i >> 2] |= (uint32_t)p.res[e] << (8 * (i & 3));
            else
                rw[i >> 3] |= (((uint32_t)p.res[e >> 1] >> (4 * (int)(e & 1))) & 15u) << (4 * (i & 7));
        }
        return;
    }
    if (p.res_bits == 8) {
        if (p.vec_ok) {
            const uint4 r0 = ldg_nc_v4(p.res + base), r1 = ldg_nc_v4(p.res + base + 16);
            rw[0] = r0.x; rw[1] = r0.y; rw[2] = r0.z; rw[3] = r0.w;
            rw[4] = r1.x; rw[5] = r1.y; rw[6] = r1.z; rw[7] = r1.w;
        } else {
            for (int i = 0; i < 32 && n0 + i < p.N; ++i)
                rw[i >> 2] |= (uint32_t)p.res[base + i] << (8 * (i & 3));
        }
    } else {
        if (p.vec_ok) {
            const uint4 r0 = ldg_nc_v4(p.res + base / 2);
            rw[0] = r0.x; rw[1] = r0.y; rw[2] = r0.z; rw[3] = r0.w;
        } else {
            for (int i = 0; i < 32 && n0 + i < p.N; i += 2)
                rw[i >> 3] |= (uint32_t)p.res[(base + i) / 2] << (4 * (i & 7));
        }
    }
}

// fp32 1.5 * 2^23: for |x| < 2^22, x + 2^23 * 1.5 lands in [2^23, 2^24) where
// the fp32 spacing is 1, so the sum's bits are 0x4B400000 + x rounded half to
// even (an exact integer x when x is one); byte and nibble fields of those
// bits are the two's-complement low bits of that integer.
constexpr float ROUND_MAGIC = 12582912.0f;
constexpr uint32_t ROUND_MAGIC_BITS = 0x4B400000u;

// Residual term t_n = float(r - z_res) * R + Bq_n for the 32 columns: the code
// r - z_res is rebuilt as an fp32 value from the magic-number bits (exact, as
// |r - z_res| < 2^22), then one fmul and one fadd as in the requant formula.
__device__ __forceinline__ void add_residual(const Params &p, const uint32_t (&rw)[8], float (&t)[32])
{
    if (p.res_bits == 8) {
        const uint32_t flip = p.res_signed ? 0x80808080u : 0u;  // s8 -> offset binary
#pragma unroll
        for (int w = 0; w < 8; ++w) {
            const uint32_t x = rw[w] ^ flip;
#pragma unroll
            for (int b = 0; b < 4; ++b) {
                const float d = __fsub_rn(__uint_as_float(prmt(x, ROUND_MAGIC_BITS, 0x7650u | b)), p.res_c);
                t[4 * w + b] = __fadd_rn(__fmul_rn(d, p.R), t[4 * w + b]);
            }
        }
    } else {
        const uint32_t cx = (p.res_signed ? 8u : 0u) | ROUND_MAGIC_BITS;  // s4 -> offset binary
#pragma unroll
        for (int w = 0; w < 4; ++w) {
#pragma unroll
            for (int b = 0; b < 8; ++b) {
                const float d = __fsub_rn(__uint_as_float(((rw[w] >> (4 * b)) & 15u) ^ cx), p.res_c);
                t[8 * w + b] = __fadd_rn(__fmul_rn(d, p.R), t[8 * w + b]);
            }
        }
    }
}

// Low bytes of four words -> one word (byte k from word k).
__device__ __forceinline__ uint32_t pack_low_bytes(uint32_t c0, uint32_t c1, uint32_t c2, uint32_t c3)
{
    return prmt(prmt(c0, c1, 0x0040u), prmt(c2, c3, 0x0040u), 0x5410u);
}

// Requant / dequant of the 32 consecutive columns n0.. of row m from
// a[k] = float(acc_c) (the correctly rounded fp32 value of the int32 sum minus
// its zero-point term).  ca / cb point at this piece's constants in shared
// memory (warp-uniform broadcast reads); rw holds the piece's residual codes.
// Requant: v = float(acc_c) * M + t (one fmul, one fadd); rounding and the
// clip are done as clamp(v, lo, hi) then a magic-number add, which equals
// clip(rint(v)) for the integer bounds lo = qmin - z_out (or max(0, qmin -
// z_out) with ReLU) and hi = qmax - z_out; z_out is then added to the integer
// -- the fp32 result of the page's formula for every finite v (M, Bq and R
// must be finite).  No conversion instructions are used.
// RS: per-row activation scales -- each column factor becomes fl(rs * factor)
// (instantiated separately so that the common path carries none of it).
// Packed 4-bit NCHW output: neighbouring pixels of a row share a byte, and they
// are rows m, m + 1 of one warp (lanes 2j, 2j + 1; the host requires even output
// widths and even tile widths), so the even lane merges its partner's codes
// and writes the bytes.  Called by every lane; `valid` says whether the lane's
// row exists.
__device__ __forceinline__ void store_nchw_u4(const Params &p, int m, int n0, const uint32_t (&c)[32], bool valid)
{
    uint8_t *C = static_cast<uint8_t *>(p.C);
    const bool even = (threadIdx.x & 1) == 0;
    const int64_t base = valid ? out_off<true>(p, m, n0) : 0;
#pragma unroll
    for (int i = 0; i < 32; ++i) {
        const uint32_t hi = __shfl_down_sync(0xffffffffu, c[i], 1);
        if (even && valid && n0 + i < p.N)
            C[(base + (int64_t)i * p.OHW) >> 1] = (uint8_t)((c[i] & 15u) | ((hi & 15u) << 4));
    }
}

template <bool RS, bool LAY>
__device__ __forceinline__ void epilogue_float_t(const Params &p, int m, int n0, float (&a)[32],
                                                 const float *ca, const float *cb,
                                                 const uint32_t (&rw)[8])
{
    const bool valid = m < p.M && n0 < p.N;
    // NCHW u4 outputs pair up lanes: every lane takes part (warp-uniform test)
    const bool pair = LAY && p.layout == QNN_LAYOUT_NCHW && p.mode == QNN_EPI_REQUANT && p.out_bits == 4;
    if (!valid && !pair) return;
    const bool nchw = LAY && p.layout == QNN_LAYOUT_NCHW;
    const bool vec = p.vec_ok && !nchw;
    const int64_t base = valid ? out_off<LAY>(p, m, n0) : 0;  // element offset of (m, n0)
    const int64_t cs = out_cstride<LAY>(p);
    float rs = 1.0f;
    if constexpr (RS) rs = valid ? __ldg(p.row_scale + m) : 1.0f;
    if (p.mode == QNN_EPI_DEQUANT) {
        float *C = static_cast<float *>(p.C);
        uint32_t y[32];
#pragma unroll
        for (int i = 0; i < 32; i += 4) {
            float4 d = *reinterpret_cast<const float4 *>(ca + i);
            if constexpr (RS) {
                d.x = __fmul_rn(rs, d.x);
                d.y = __fmul_rn(rs, d.y);
                d.z = __fmul_rn(rs, d.z);
                d.w = __fmul_rn(rs, d.w);
            }
            const float4 b = *reinterpret_cast<const float4 *>(cb + i);
            y[i] = __float_as_uint(__fadd_rn(__fmul_rn(a[i], d.x), b.x));
            y[i + 1] = __float_as_uint(__fadd_rn(__fmul_rn(a[i + 1], d.y), b.y));
            y[i + 2] = __float_as_uint(__fadd_rn(__fmul_rn(a[i + 2], d.z), b.z));
            y[i + 3] = __float_as_uint(__fadd_rn(__fmul_rn(a[i + 3], d.w), b.w));
        }
        if (vec) {
#pragma unroll
            for (int i = 0; i < 32; i += 4) st_v4(C + base + i, y[i], y[i + 1], y[i + 2], y[i + 3]);
        } else {
            for (int i = 0; i < 32 && n0 + i < p.N; ++i) C[base + i * cs] = __uint_as_float(y[i]);
        }
        return;
    }
    // REQUANT
    float t[32];
#pragma unroll
    for (int i = 0; i < 32; i += 4) {
        const float4 bq = *reinterpret_cast<const float4 *>(cb + i);
        t[i] = bq.x;
        t[i + 1] = bq.y;
        t[i + 2] = bq.z;
        t[i + 3] = bq.w;
    }
    if (p.res) add_residual(p, rw, t);
    uint8_t *C = static_cast<uint8_t *>(p.C);
    uint32_t c[32];  // low bits: the output codes
#pragma unroll
    for (int i = 0; i < 32; i += 4) {
        const float4 mv = *reinterpret_cast<const float4 *>(ca + i);
        float mm[4] = {mv.x, mv.y, mv.z, mv.w};
        if constexpr (RS) {
#pragma unroll
            for (int k = 0; k < 4; ++k) mm[k] = __fmul_rn(rs, mm[k]);
        }
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            float v = __fadd_rn(__fmul_rn(a[i + k], mm[k]), t[i + k]);
            v = fminf(fmaxf(v, p.clip_lo_f), p.clip_hi_f);
            c[i + k] = __float_as_uint(__fadd_rn(v, ROUND_MAGIC)) + (uint32_t)p.z_out;
        }
    }
    if constexpr (LAY) {
        if (pair) {
            store_nchw_u4(p, m, n0, c, valid);
            return;
        }
        if (nchw) {
            // 8-bit codes, one per channel plane
            for (int i = 0; i < 32 && n0 + i < p.N; ++i) C[base + i * cs] = (uint8_t)c[i];
            return;
        }
    }
    if (p.out_bits == 8) {
        uint32_t ow[8];
#pragma unroll
        for (int w = 0; w < 8; ++w) ow[w] = pack_low_bytes(c[4 * w], c[4 * w + 1], c[4 * w + 2], c[4 * w + 3]);
        if (vec && (reinterpret_cast<uintptr_t>(C) & 31u) == 0) {
            st_v8(C + base, ow);  // the 32 codes of one row in one store: whole 32-byte sectors
        } else if (vec) {
            st_v4(C + base, ow[0], ow[1], ow[2], ow[3]);
            st_v4(C + base + 16, ow[4], ow[5], ow[6], ow[7]);
        } else {
            for (int i = 0; i < 32 && n0 + i < p.N; ++i) C[base + i] = (uint8_t)(ow[i >> 2] >> (8 * (i & 3)));
        }
    } else {
        // codes 2k (low nibble) and 2k + 1 (high nibble) share byte k
        uint32_t ow[4];
#pragma unroll
        for (int w = 0; w < 4; ++w) {
            const uint32_t *q = c + 8 * w;
            const uint32_t ev = pack_low_bytes(q[0], q[2], q[4], q[6]);
            const uint32_t od = pack_low_bytes(q[1], q[3], q[5], q[7]);
            ow[w] = (ev & 0x0F0F0F0Fu) | ((od << 4) & 0xF0F0F0F0u);
        }
        if (vec) {
            st_v4(C + base / 2, ow[0], ow[1], ow[2], ow[3]);
        } else {
            // N is even: a byte holds columns (2i, 2i+1) of this thread's row only
            for (int i = 0; i < 32 && n0 + i < p.N; i += 2)
                C[(base + i) / 2] = (uint8_t)(ow[i >> 3] >> (4 * (i & 7)));
        }
    }
}

template <bool LAY>
__device__ __forceinline__ void epilogue_float_rowscale(const Params &p, int m, int n0, float (&a)[32], const float *ca,
                                                     const float *cb, const uint32_t (&rw)[8])
{
    epilogue_float_t<true, LAY>(p, m, n0, a, ca, cb, rw);
}

template <bool LAY>
__device__ __forceinline__ void epilogue_float(const Params &p, int m, int n0, float (&a)[32], const float *ca,
                                               const float *cb, const uint32_t (&rw)[8])
{
    if (p.row_scale) epilogue_float_rowscale<LAY>(p, m, n0, a, ca, cb, rw);
    else epilogue_float_t<false, LAY>(p, m, n0, a, ca, cb, rw);
}

// The same from int32 sums (multi-chunk K, raw int32 outputs, or zero-point
// terms that are not fp32 values): subtracts zp_term (cz: its int bits), stores
// the raw sums where asked, and converts for the float epilogue.
template <bool LAY>
__device__ __forceinline__ void epilogue_int(const Params &p, int m, int n0, int32_t (&ac)[32],
                                             const float *ca, const float *cb, const float *cz,
                                             const uint32_t (&rw)[8])
{
    const bool valid = m < p.M && n0 < p.N;
    const bool pair = LAY && p.layout == QNN_LAYOUT_NCHW && p.mode == QNN_EPI_REQUANT && p.out_bits == 4;
    if (!valid && !pair) return;
    const bool vec = p.vec_ok && !(LAY && p.layout == QNN_LAYOUT_NCHW);
    const int64_t cs = out_cstride<LAY>(p);
    if (p.zp) {
#pragma unroll
        for (int i = 0; i < 32; i += 4) {
            const float4 z = *reinterpret_cast<const float4 *>(cz + i);
            ac[i] -= __float_as_int(z.x);
            ac[i + 1] -= __float_as_int(z.y);
            ac[i + 2] -= __float_as_int(z.z);
            ac[i + 3] -= __float_as_int(z.w);
        }
    }
    if (p.rowsum) {
        // the weight zero point's term (128 - z_w[n]) * sum_k (a_k - centre), in
        // wrapping 32-bit arithmetic: the final sum fits int32 (host check)
        const uint32_t rs = valid ? (uint32_t)__ldg(p.rowsum + m) : 0u;
#pragma unroll
        for (int i = 0; i < 32; ++i) {
            const int n = n0 + i < p.N ? n0 + i : p.N - 1;
            ac[i] = (int32_t)((uint32_t)ac[i] + (uint32_t)(128 - __ldg(p.zw + n)) * rs);
        }
    }
    const int64_t base = valid ? out_off<LAY>(p, m, n0) : 0;
    if (p.C32 && valid) {
        if (vec) {
#pragma unroll
            for (int i = 0; i < 32; i += 4)
                st_v4(p.C32 + base + i, ac[i], ac[i + 1], ac[i + 2], ac[i + 3]);
        } else {
            for (int i = 0; i < 32 && n0 + i < p.N; ++i) p.C32[base + i * cs] = ac[i];
        }
    }
    if (p.mode == QNN_EPI_S32) {
        if (!valid) return;
        int32_t *C = static_cast<int32_t *>(p.C);
        if (vec) {
#pragma unroll
            for (int i = 0; i < 32; i += 4) st_v4(C + base + i, ac[i], ac[i + 1], ac[i + 2], ac[i + 3]);
        } else {
            for (int i = 0; i < 32 && n0 + i < p.N; ++i) C[base + i * cs] = ac[i];
        }
        return;
    }
    float a[32];
#pragma unroll
    for (int k = 0; k < 32; ++k) a[k] = __int2float_rn(ac[k]);
    epilogue_float<LAY>(p, m, n0, a, ca, cb, rw);
}

// fp32 accumulator value -> exact int32 (the fp32 value times 2^scale_log2 is an integer)
template <int SCALE_LOG2>
__device__ __forceinline__ int32_t acc_to_int(uint32_t bits)
{
    float f = __uint_as_float(bits);
    if (SCALE_LOG2 != 0) f = __fmul_rn(f, (float)(1 << SCALE_LOG2));
    return __float2int_rn(f);
}

// One tile whose K fits one accumulation chunk: the thread's row and its
// warp's columns are converted and stored 32 at a time straight from TMEM
// (the accumulator buffer is released after the last piece is read).
template <class Op, int TBN, int COLS>
__device__ __forceinline__ bool epilogue_stream_tile(const Params &p, Smem<Op, TBN> &s, float *cols,
                                                     const ColumnRegs<COLS> &cr, bool fresh, bool &exact,
                                                     bool &zp_zero, int m,
                                                     int nbase, int npieces, uint32_t taddr0, uint32_t abuf,
                                                     uint32_t u, int lane)
{
    uint32_t rw_next[8];
    load_residual<Op::LAYOUTS>(p, m, nbase, rw_next);
    if (!warp_wait_idle(smem_u32(&s.acc_full[abuf]), (u >> 1) & 1u, p.status)) return false;
    tc_fence_after();
    if (fresh) exact = store_columns<COLS>(cr, cols, lane, zp_zero);
    const bool fast = exact && !p.C32 && p.mode != QNN_EPI_S32 && !p.rowsum && !p.row_scale;
#pragma unroll 1
    for (int jp = 0; jp < npieces; ++jp) {
        uint32_t rw[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) rw[k] = rw_next[k];
        if (jp + 1 < npieces) load_residual<Op::LAYOUTS>(p, m, nbase + (jp + 1) * 32, rw_next);
        uint32_t r[32];
        tmem_ld32(taddr0 + jp * 32, r);
        tmem_ld_wait();
        if (jp == npieces - 1) {
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&s.acc_empty[abuf]));
        }
        if (fast && zp_zero && Op::SCALE_LOG2 == 0 && p.mode == QNN_EPI_REQUANT) {
            // zp_term = 0 in every column (e.g. u8 activations with Z_a = 128): the
            // fp32 sum is the exact integer acc_c, the conversion the formula starts
            // from (a sum of -0 instead of +0 cannot change a requantized code)
            float a[32];
#pragma unroll
            for (int k = 0; k < 32; ++k) a[k] = __uint_as_float(r[k]);
            epilogue_float_t<false, Op::LAYOUTS>(p, m, nbase + jp * 32, a, cols + jp * 32, cols + COLS + jp * 32,
                                                 rw);
        } else if (fast) {
            // the fp32 sum is an exact integer (times 2^-SCALE_LOG2); adding the
            // fp32 -zp_term rounds once, like the int32 -> fp32 conversion
            const float *cn = cols + 2 * COLS + jp * 32;
            float a[32];
#pragma unroll
            for (int k = 0; k < 32; k += 4) {
                const float4 nz = *reinterpret_cast<const float4 *>(cn + k);
                const float z4[4] = {nz.x, nz.y, nz.z, nz.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float f = __uint_as_float(r[k + e]);
                    a[k + e] = Op::SCALE_LOG2 ? __fmaf_rn(f, (float)(1 << Op::SCALE_LOG2), z4[e])
                                              : __fadd_rn(f, z4[e]);
                }
            }
            epilogue_float_t<false, Op::LAYOUTS>(p, m, nbase + jp * 32, a, cols + jp * 32, cols + COLS + jp * 32,
                                                 rw);
        } else {
            int32_t acc[32];
#pragma unroll
            for (int k = 0; k < 32; ++k) acc[k] = acc_to_int<Op::SCALE_LOG2>(r[k]);
            epilogue_int<Op::LAYOUTS>(p, m, nbase + jp * 32, acc, cols + jp * 32, cols + COLS + jp * 32,
                                      cols + 3 * COLS + jp * 32, rw);
        }
    }
    return true;
}

// MULTI == false: one accumulation chunk per tile (epilogue_stream_tile).
// MULTI == true : K is cut into exact chunks (their number is read at run time,
// chunk_plan); each thread keeps int32 sums for its row and its warp's columns
// in registers across the chunks, reading each chunk 16 columns at a time; a
// plan of one chunk takes the streaming path.
template <class Op, int TBN, bool MULTI>
__device__ void epilogue_role(const Params &p, Smem<Op, TBN> &s, int my_tiles, uint32_t tmem)
{
    constexpr int PIECES = epi_max_pieces<Op, TBN>();  // 32-column pieces of a warp (at most)
    constexpr int COLS = PIECES * 32;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int quad = warp & 3;                                    // TMEM lanes 32*quad .. +31
    const int group = warp >= EPI_WARP0 ? (warp - EPI_WARP0) >> 2 : 2;  // warps 8-11, 12-15, 0-3
    constexpr int NG = epi_warps<Op, TBN>() / 4;
    const int p0 = group * (TBN / 32) / NG;                       // first piece of this warp
    const int npieces = (group + 1) * (TBN / 32) / NG - p0;       // 1 .. PIECES
    float *cols = s.cols[warp >= EPI_WARP0 ? warp - EPI_WARP0 : warp + 8];
    uint32_t u = 0;
    const typename Op::RowInfo ri = Op::row_info(p, quad * 32 + lane);
    int nch = 1;
    if constexpr (MULTI) {
        if (!warp_wait_idle(smem_u32(&s.plan_ready), 0u, p.status)) return;
        nch = s.plan_count;
    }
    // the column constants in shared memory serve every tile of the same column
    // block: they are loaded again only when the block changes
    int cur_nbase = -1;
    bool exact = false;
    bool zp_zero = false;
    for (int i = 0; i < my_tiles; ++i) {
        const int t = blockIdx.x + i * gridDim.x;
        const int m = Op::out_row(p, t % p.num_m, ri);
        const int nbase = (t / p.num_m) * TBN + p0 * 32;
        const bool fresh = !Op::CACHE_COLS || nbase != cur_nbase;
        cur_nbase = nbase;
        ColumnRegs<COLS> cr;
        if (fresh) load_columns<COLS>(p, cr, nbase, lane);
        if (nch == 1) {
            const uint32_t abuf = u & 1u;
            const uint32_t taddr = tmem + ((uint32_t)(quad * 32) << 16) + abuf * TBN + p0 * 32;
            if (!epilogue_stream_tile<Op, TBN, COLS>(p, s, cols, cr, fresh, exact, zp_zero, m, nbase, npieces, taddr,
                                                     abuf, u, lane))
                return;
            ++u;
        } else if constexpr (MULTI) {
            // every chunk arrives in accumulator 0; its fp32 sums (exact integers)
            // are added into int32 running sums kept in accumulator 1's columns,
            // then accumulator 0 is released for the next chunk
            const uint32_t lanes = (uint32_t)(quad * 32) << 16;
            const uint32_t fbuf = tmem + lanes + p0 * 32;
            const uint32_t ibuf = tmem + lanes + TBN + p0 * 32;
            for (int c = 0; c < nch; ++c) {
                if (!warp_wait_idle(smem_u32(&s.acc_full[0]), u & 1u, p.status)) return;
                tc_fence_after();
#pragma unroll 1
                for (int q = 0; q < 2 * npieces; ++q) {
                    uint32_t r[16], t[16];
                    tmem_ld16(fbuf + q * 16, r);
                    if (c > 0) tmem_ld16(ibuf + q * 16, t);
                    tmem_ld_wait();
#pragma unroll
                    for (int k = 0; k < 16; ++k) {
                        const int32_t v = acc_to_int<Op::SCALE_LOG2>(r[k]);
                        r[k] = (uint32_t)(c > 0 ? (int32_t)t[k] + v : v);
                    }
                    tmem_st16(ibuf + q * 16, r);
                }
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&s.acc_empty[0]));
                ++u;
            }
            if (fresh) exact = store_columns<COLS>(cr, cols, lane, zp_zero);
#pragma unroll 1
            for (int jp = 0; jp < npieces; ++jp) {
                uint32_t rw[8];
                load_residual<Op::LAYOUTS>(p, m, nbase + jp * 32, rw);
                uint32_t r[32];
                tmem_ld32(ibuf + jp * 32, r);
                tmem_ld_wait();
                int32_t acc[32];
#pragma unroll
                for (int k = 0; k < 32; ++k) acc[k] = (int32_t)r[k];
                epilogue_int<Op::LAYOUTS>(p, m, nbase + jp * 32, acc, cols + jp * 32, cols + COLS + jp * 32,
                                          cols + 3 * COLS + jp * 32, rw);
            }
        }
    }
}

// ---------------------------------------------------------------- kernel
template <class Op, int TBN, bool MULTI>
__global__ void __launch_bounds__(NUM_THREADS, 1) qmma_kernel(const __grid_constant__ Params p)
{
    extern __shared__ uint8_t smem_raw[];
    Smem<Op, TBN> &s = *reinterpret_cast<Smem<Op, TBN> *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int i = 0; i < Op::STAGES; ++i) {
            mbar_init(smem_u32(&s.full[i]), Op::TMA_A ? 1 : 5);
            mbar_init(smem_u32(&s.empty[i]), 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(smem_u32(&s.acc_full[i]), 1);
            mbar_init(smem_u32(&s.acc_empty[i]), epi_warps<Op, TBN>());
        }
        mbar_init(smem_u32(&s.mma_done), 1);
        mbar_init(smem_u32(&s.bres_full), 1);
        mbar_init(smem_u32(&s.plan_ready), 1);
        Op::init(s.stg);
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
    // launched as a programmatic dependent (TMA_A Ops): no thread reads global memory before
    // the preceding kernel on the stream has completed; only the prologue above overlaps it
    if constexpr (Op::TMA_A) grid_dependency_wait();

    const int my_tiles =
        (blockIdx.x < p.num_tiles) ? (p.num_tiles - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;
    const int units = my_tiles * p.KT;

    // Register split per warpgroup (launched with 128 per thread, 65536 in all):
    // converters keep 128, the producer / MMA warpgroup drops to 96 and the
    // epilogue warpgroups take the rest -- 128*128 + 128*96 + 256*144 = 65536;
    // with A arriving by copy, warpgroup 0 is a third epilogue group and the
    // producer / MMA warpgroup drops to 72 (128*72 + 384*144 = 64512) or, for
    // 64-column tiles, warpgroup 0 idles at 24 (128*24 + 128*96 + 256*192 =
    // 64512).
    constexpr bool EPI12 = epi_warps<Op, TBN>() == 12;
    constexpr uint32_t REGS_WG1 = 96;
    constexpr uint32_t REGS_WG1_E12 = 72;
    constexpr uint32_t REGS_EPI = EPI12 ? ((65536u - 128u * REGS_WG1_E12) / 384u) & ~7u
                                        : ((65536u - 128u * (Op::TMA_A ? 24u : 128u) - 128u * REGS_WG1) / 256u) & ~7u;
    constexpr uint32_t REGS_WG0 = EPI12 ? REGS_EPI : (Op::TMA_A ? 24u : 128u);
    static_assert(128u * REGS_WG0 + 128u * (EPI12 ? REGS_WG1_E12 : REGS_WG1) + 256u * REGS_EPI <= 65536u,
                  "register split");
    if (warp < 4) {
        if constexpr (EPI12) {
            regs_inc<REGS_EPI>();
            epilogue_role<Op, TBN, MULTI>(p, s, my_tiles, tmem);
        } else if constexpr (Op::TMA_A) {
            regs_dec<REGS_WG0>();
        } else {
            converter_role<Op, TBN, MULTI>(p, s, units);
        }
    } else if (warp < 8) {
        regs_dec<EPI12 ? REGS_WG1_E12 : REGS_WG1>();
        if (warp == PRODUCER_WARP) producer_role<Op, TBN>(p, s, units);
        if (warp == MMA_WARP) mma_role<Op, TBN, MULTI>(p, s, my_tiles, tmem);
        if (warp == MMA_WARP + 1) {
            if (lane == 0) {
                const ChunkPlan plan = chunk_plan(p, blockIdx.x == 0);
                // a kernel built for one chunk per tile must not be given weights
                // whose sums need more (they would not be exact): reported, not hidden
                if (!MULTI && plan.count > 1 && blockIdx.x == 0) atomicOr(p.status, kStatusBadArg);
                s.plan_steps = plan.steps;
                s.plan_count = plan.count;
                mbar_arrive(smem_u32(&s.plan_ready));  // release: the plan's stores are visible to waiters
            }
            __syncwarp();
            if (Op::TMA_A && blockIdx.x == 0 && p.ptf) {
                // A arrived already multiplied by 2^ptf (the pre-pass): the exact-chunk
                // length rests on every shift byte being at most ptf_max
                bool above = false;
                for (int k = lane; k < p.K; k += 32) above |= __ldg(p.ptf + k) > (uint8_t)p.ptf_max;
                if (__any_sync(0xffffffffu, above) && lane == 0) atomicOr(p.status, kStatusBadArg);
            }
        }
    } else {
        regs_inc<REGS_EPI>();
        epilogue_role<Op, TBN, MULTI>(p, s, my_tiles, tmem);
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == MMA_WARP) tmem_dealloc(tmem, 2 * TBN);
}

template <class Op, int TBN, bool MULTI>
qnn_status launch(Params p, cudaStream_t stream)
{
    static bool attr_set[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return QNN_ERR_CUDA;
    constexpr size_t SMEM = smem_bytes<Op, TBN>();
    static_assert(SMEM <= 232448, "shared memory per block");
    if (!attr_set[dev]) {
        if (cudaFuncSetAttribute(qmma_kernel<Op, TBN, MULTI>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM) != cudaSuccess)
            return QNN_ERR_CUDA;
        attr_set[dev] = true;
    }
    p.num_tiles = p.num_m * ((p.N + TBN - 1) / TBN);
    int grid = qnn::sm_count();
    if (grid > p.num_tiles) grid = p.num_tiles;
    if constexpr (Op::TMA_A) {
        // A comes from the kernel launched just before on the stream (the pre-pass, or
        // whatever wrote the packed image): launched as its programmatic dependent, this
        // kernel's launch and prologue overlap that kernel's tail; every thread waits for
        // it (griddepcontrol.wait) before touching global memory.
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)grid);
        cfg.blockDim = dim3(NUM_THREADS);
        cfg.dynamicSmemBytes = SMEM;
        cfg.stream = stream;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        if (cudaLaunchKernelEx(&cfg, qmma_kernel<Op, TBN, MULTI>, p) != cudaSuccess) {
            (void)cudaGetLastError();
            return QNN_ERR_CUDA;
        }
        return launch_status();
    }
    qmma_kernel<Op, TBN, MULTI><<<grid, NUM_THREADS, SMEM, stream>>>(p);
    return launch_status();
}

// Shared host-side validation of the epilogue descriptor.  out_bits / res_bits
// say how the op stores quantized outputs and residuals.
inline qnn_status setup_epilogue(const qnn_epilogue *e, bool conv, Params &p)
{
    p.mode = e->mode;
    p.relu = e->relu ? 1 : 0;
    p.z_out = e->z_out;
    p.zp = e->zp_term;
    p.Mv = e->M;
    p.Bq = e->Bq;
    p.D = e->D;
    p.bias = e->bias;
    p.row_scale = e->row_scale;
    if (e->row_scale && !aligned16(e->row_scale)) return QNN_ERR_ALIGNMENT;
    switch (e->mode) {
    case QNN_EPI_REQUANT: {
        if (!e->M || !e->Bq) return QNN_ERR_INVALID_ARG;
        const bool ok_dt = conv ? (e->out_dt == QNN_U4 || e->out_dt == QNN_U8 || e->out_dt == QNN_S8)
                                : (e->out_dt == QNN_S8 || e->out_dt == QNN_U8);
        if (!ok_dt) return QNN_ERR_UNSUPPORTED;
        int32_t lo, hi;
        qrange(e->out_dt, 0, &lo, &hi);
        if (e->z_out < lo || e->z_out > hi) return QNN_ERR_INVALID_ARG;
        p.clip_lo_f = (float)(e->relu ? (lo - e->z_out > 0 ? lo - e->z_out : 0) : lo - e->z_out);
        p.clip_hi_f = (float)(hi - e->z_out);
        p.out_bits = (e->out_dt == QNN_U4) ? 4 : 8;
        p.out_signed = (e->out_dt == QNN_S8);
        if (e->residual) {
            const bool ok_r = conv ? (e->res_dt == QNN_U4 || e->res_dt == QNN_U8 || e->res_dt == QNN_S8 ||
                                      e->res_dt == QNN_S4)
                                   : (e->res_dt == QNN_S8 || e->res_dt == QNN_U8);
            if (!ok_r) return QNN_ERR_UNSUPPORTED;
            if (!aligned16(e->residual)) return QNN_ERR_ALIGNMENT;
            p.res = static_cast<const uint8_t *>(e->residual);
            p.res_bits = (e->res_dt == QNN_U4 || e->res_dt == QNN_S4) ? 4 : 8;
            p.res_signed = (e->res_dt == QNN_S8 || e->res_dt == QNN_S4);
            p.z_res = e->z_res;
            p.R = e->R;
            {
                int32_t rlo, rhi;
                qrange(e->res_dt, 0, &rlo, &rhi);
                if (e->z_res < rlo || e->z_res > rhi) return QNN_ERR_INVALID_ARG;
                const int off = p.res_signed ? (p.res_bits == 8 ? 128 : 8) : 0;
                p.res_c = (float)(12582912 + e->z_res + off);
            }
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
    return QNN_OK;
}

}  // namespace mk
}  // namespace qnn
