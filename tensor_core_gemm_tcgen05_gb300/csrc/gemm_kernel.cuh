// Persistent, warp-specialised FP16 GEMM with a fused epilogue for sm_103a (GB300):
//
//     C[M x N] = act(A[M x K] * B[K x N] + bias[N])      FP16 in, FP32 accumulate, FP16 out
//
// The tutorial's tiled tensor-core GEMM ("TileLang: Criando Kernels de GPU ..." on
// noticiai.com.br, section "GEMM com Tensor Cores": tiles of A and B staged global ->
// shared, multiplied on tensor cores, the output tile stored once) and its fused epilogue
// (same page, section "GEMM com epilogo fundido"; "TileLang ..." on pro.edgex.exchange,
// fused-epilogue paragraph: bias, then GELU, applied to the accumulator before the store),
// redesigned for the fifth-generation tensor cores:
//
//  * one CTA per SM, looping over output tiles in a grouped (L2-friendly) raster;
//  * warp 0: TMA producer, fills a STAGES-deep ring of 128-byte-swizzled shared-memory
//    slots (A: BM x 64 K-major; B: 64 x BN as BN/64 boxes of 64 N-columns, MN-major),
//    gated by full/empty mbarriers;
//  * warp 1: allocates Tensor Memory and issues tcgen05.mma (M = BM, N = BN, K = 16) from
//    one thread into one of two FP32 TMEM accumulators, releasing each slot with
//    tcgen05.commit;
//  * warps 2..(1+EPI_WARPS): epilogue. A warp may only read the 32-lane quarter of TMEM
//    given by its warp index mod 4 (= 32 rows of the tile); with 4 epilogue warps each
//    takes all BN columns of its quarter, with 8 each takes half of them. A warp reads its
//    rows with tcgen05.ld, adds the bias, applies the activation in FP32, rounds to FP16
//    and writes 16-byte vectors, masking rows >= M and columns >= N.
//    While it drains accumulator b, the MMA warp already fills accumulator b ^ 1.
//  * stream-K (when there are fewer tiles than SMs): the tile-major sequence of
//    (tile, 64-wide k-block) units is cut into one equal range per CTA, so every SM gets the
//    same share of the MMAs however many tiles there are. A tile cut by range boundaries is
//    summed by the CTA holding its first k-block (its "owner", which reaches that part last
//    in its range): every other CTA with a part of the tile (reached first in its range)
//    writes its FP32 partial accumulator to a workspace slot of its own and raises a ready
//    flag; the owner waits for the flags, pulls each partial into its (by then idle) operand
//    ring with one bulk copy per warp, adds it to the accumulator in Tensor Memory, runs the
//    epilogue and lowers the flags again for the next launch.
// Every mbarrier wait is bounded in time. When a wait runs out the kernel records which
// one in a device error word, tells the other roles to stop, waits (bounded) for its own
// copies and MMAs in flight, frees its Tensor Memory and returns.
#pragma once

#include <cuda.h>
#include <cuda_fp16.h>

#include <cstdint>

#include "ptx.cuh"

namespace gb300 {

// Which wait ran out (the device error word).
enum : uint32_t {
    ERR_PRODUCER_SLOT = 1,
    ERR_MMA_OPERANDS = 2,
    ERR_MMA_ACCUMULATOR = 3,
    ERR_EPILOGUE_ACCUMULATOR = 4,
    ERR_TEARDOWN_DRAIN = 5,
    ERR_STREAMK_PARTIAL = 6,   // a stream-K owner waited too long for another CTA's partial
    ERR_ROW_EXCHANGE = 7,      // a row cluster waited too long for the other CTAs' row statistics
};

// How a launch maps work to CTAs (the kernel's SCHED template argument).
enum : int {
    SCHED_TILES = 0,         // whole tiles, grouped raster, persistent
    SCHED_STREAM_K = 1,      // equal ranges of (tile, k-block) units
    SCHED_SPLIT_K = 3,       // one cluster per tile, CTA r = the r-th of `split` equal k ranges
};

enum : int { EPI_NONE = 0, EPI_GELU = 1, EPI_RELU = 2, EPI_SOFTMAX = 3 };

// Output staging of one epilogue warp: two 32-row x 32-column FP16 boxes (2 KB each,
// 64-byte swizzle) that alternate between being filled and being stored by TMA.
constexpr int EPI_STORE_BOX_BYTES = 32 * 32 * 2;
constexpr int EPI_STORE_WARP_BYTES = 2 * EPI_STORE_BOX_BYTES;
enum : int { DEBUG_WITHHOLD_FIRST_LOAD = 1 };

struct GemmParams {
    int M, N, K;
    int m_blocks, n_blocks, num_tiles, num_kb;
    int group_m;           // m-blocks per raster group
    int group_big = 0;     // the first group_big groups have one m-block more
    int epilogue;          // EPI_*
    const __half *bias;    // N values or nullptr
    __half *C;             // M x N row-major
    uint32_t *err;         // device error word
    uint64_t timeout_ns;   // limit of every wait
    int debug;             // DEBUG_* flags
    // stream-K (one-CTA kernel): 0 = whole tiles per CTA; else the number of
    // (tile, k-block) units, split into gridDim.x equal ranges
    int64_t sk_units = 0;
    float *sk_ws = nullptr;          // [gridDim.x][epilogue warp][chunk][8][32 lanes][4] FP32 partials
    uint32_t *sk_flags = nullptr;    // [gridDim.x][epilogue warps]: 1 = that part is written
    int row_cluster = 0;             // softmax kernel: CTAs per cluster (1, 2, 4 or 8)
    int smx_span = 0;                // softmax kernel: column tiles per CTA of a cluster
    int smx_two_pass = 0;            // softmax kernel: 1 = statistics pass, then output pass
    int split = 0;                   // split-K: CTAs per cluster, each with 1/split of the k-blocks
    int64_t ldc = 0;                 // row stride of C in elements (split-K writes C directly)
    // pair kernel: tiles [0, pair_split_from) are whole work units; each later tile is two
    // units, its left and right N-halves; pair_units = the number of units
    int pair_split_from = 0;
    int pair_units = 0;
};

// BK_: K per stage, 64 or 128 (one or two 128-byte swizzle atoms of A; every stage ends in one
// tcgen05.commit, so longer stages commit half as often). STORE_IN_RING_: the output staging
// boxes overlay the operand ring instead of having their own space; only for launches that
// give each CTA at most one tile (the ring is idle once its accumulator is complete).
// HALF_TAIL_ (with STORE_IN_RING_, whole tiles): the last STAGES k-blocks of a tile are
// multiplied into the left half of the accumulator (N = BN / 2) first, then into the right
// half, so that the epilogue warps of the left columns start while the right half's MMAs run.
template <int BM_, int BN_, int STAGES_, int EPI_WARPS_ = 4, int BK_ = 64, bool STORE_IN_RING_ = false,
          bool HALF_TAIL_ = false>
struct KernelConfig {
    static constexpr int BM = BM_;          // rows of A / C per tile (= UMMA M, = TMEM lanes)
    static constexpr int BN = BN_;          // columns of B / C per tile (= UMMA N)
    static constexpr int BK = BK_;          // K per stage
    static constexpr int UMMA_K = 16;       // K per tcgen05.mma of kind::f16
    static constexpr int STAGES = STAGES_;
    static constexpr bool STORE_IN_RING = STORE_IN_RING_;
    static constexpr bool HALF_TAIL = HALF_TAIL_;
    static constexpr int A_ATOM_BYTES = BM * 64 * 2;   // 64 K-columns of A: one swizzle atom wide
    static constexpr int A_ATOMS = BK / 64;
    static constexpr int A_BYTES = BM * BK * 2;
    static constexpr int B_BOX_N = 64;                 // N per TMA box of B (128 bytes)
    static constexpr int B_BOXES = BN / B_BOX_N;
    static constexpr int B_BOX_BYTES = BK * B_BOX_N * 2;
    static constexpr int B_BYTES = BK * BN * 2;
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
    static constexpr int ACC_BUFS = 2;
    static constexpr int TMEM_COLS = ACC_BUFS * BN;    // FP32 accumulators, one column each
    static constexpr int NUM_EPI_WARPS = EPI_WARPS_;
    static constexpr int EPI_COL_GROUPS = NUM_EPI_WARPS / 4;   // warps sharing a TMEM quarter
    static constexpr int NUM_THREADS = 64 + 32 * NUM_EPI_WARPS;
    // full[s], empty[s], acc_full[b], acc_empty[b], drain, one stream-K partial barrier per
    // epilogue warp, left_half (HALF_TAIL: the left half of the accumulator is complete)
    static constexpr int NUM_BARS = 2 * STAGES + 2 * ACC_BUFS + 1 + NUM_EPI_WARPS + 1;
    // HALF_TAIL: output staging of the epilogue warps of the left columns, in the left halves
    // of the stages' B operands (no MMA reads those once the left half is complete); the
    // other warps stage where STORE_IN_RING puts them, at the start of the ring (A), used
    // only after every MMA is complete
    static constexpr int LEFT_WARPS = NUM_EPI_WARPS / 2;
    static constexpr int LEFT_STAGE_WARPS = (BK * BN) / EPI_STORE_WARP_BYTES;   // B_BYTES / 2 per stage
    // stream-K: one epilogue warp's share of a partial accumulator (32 rows x its columns,
    // FP32), as stored in the workspace and as pulled into the operand ring
    static constexpr int PART_WARP_BYTES = (BN / EPI_COL_GROUPS) * 32 * 4;
    // after the ring: barriers, TMEM address, stop flag; then one BN-wide bias slice per
    // epilogue warp (FP16)
    static constexpr int BIAS_OFFSET = STAGES * STAGE_BYTES + ((NUM_BARS * 8 + 16 + 15) / 16) * 16;
    // then, 1024-aligned, two 32 x 32 FP16 output staging boxes per epilogue warp (or, with
    // STORE_IN_RING, the same boxes at the start of the operand ring)
    static constexpr int BIAS_END = BIAS_OFFSET + NUM_EPI_WARPS * BN * 2;
    static constexpr int STORE_OFFSET = STORE_IN_RING ? 0 : ((BIAS_END + 1023) / 1024) * 1024;
    static constexpr int SMEM_BYTES =
        1024 /* alignment slack */ + (STORE_IN_RING ? BIAS_END : STORE_OFFSET + NUM_EPI_WARPS * EPI_STORE_WARP_BYTES);

    static_assert(BM == 128, "one CTA, M = 128: TMEM lane i holds tile row i");
    static_assert(BN % 64 == 0 && BN >= 64 && BN <= 256, "UMMA N for M = 128");
    static_assert(TMEM_COLS == 128 || TMEM_COLS == 256 || TMEM_COLS == 512, "TMEM alloc size");
    static_assert(NUM_EPI_WARPS == 4 || NUM_EPI_WARPS == 8 || NUM_EPI_WARPS == 16,
                  "one, two or four warps per TMEM lane quarter");
    static_assert((BN / 32) % EPI_COL_GROUPS == 0, "column chunks split evenly between warps");
    static_assert(SMEM_BYTES <= 232448, "exceeds the 227 KB per-CTA shared memory limit");
    static_assert(NUM_EPI_WARPS * PART_WARP_BYTES <= STAGES * STAGE_BYTES, "partials fit the operand ring");
    static_assert(BK == 64 || BK == 128, "one or two swizzle atoms of K per stage");
    static_assert(!STORE_IN_RING || NUM_EPI_WARPS * EPI_STORE_WARP_BYTES <= STAGES * STAGE_BYTES,
                  "output staging fits the operand ring");
    static_assert(!HALF_TAIL || (STORE_IN_RING && EPI_COL_GROUPS % 2 == 0 && (BK * BN) % EPI_STORE_WARP_BYTES == 0 &&
                                 LEFT_WARPS <= STAGES * LEFT_STAGE_WARPS &&
                                 NUM_EPI_WARPS * EPI_STORE_WARP_BYTES <= STAGES * A_BYTES),
                  "half-tail split: whole column groups per half, staging in the left B halves and in A");
};

// UMMA shared-memory descriptor for a 128-byte-swizzled operand tile.
//   bits  0..13 start address >> 4      bits 16..29 leading byte offset >> 4
//   bits 32..45 stride byte offset >> 4 bits 46..48 fixed 0b001
//   bits 49..51 base offset (0: tiles are 1024-byte aligned)   bits 61..63 swizzle (2 = 128 B)
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr, uint32_t lbo_bytes, uint32_t sbo_bytes)
{
    return static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4) |
           (static_cast<uint64_t>((lbo_bytes >> 4) & 0x3FFFu) << 16) |
           (static_cast<uint64_t>((sbo_bytes >> 4) & 0x3FFFu) << 32) | (1ull << 46) | (2ull << 61);
}

// UMMA instruction descriptor, kind::f16: D = FP32, A = B = FP16, A K-major, B MN-major.
//   bits 4..5 D format (1 = F32)   bits 7..9 / 10..12 A / B format (0 = F16)
//   bit 15 A major (0 = K)          bit 16 B major (1 = MN)
//   bits 17..22 N >> 3              bits 24..28 M >> 4
template <int M, int N>
__host__ __device__ constexpr uint32_t idesc_f16_f32()
{
    return (1u << 4) | (0u << 7) | (0u << 10) | (0u << 15) | (1u << 16) |
           (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}

// Grouped raster: tiles are numbered so that consecutive tile indices (which run at the
// same time on neighbouring SMs) sweep `group_m` row-blocks of A against successive
// column-blocks of B, keeping both operand panels hot in L2.
// The first p.group_big groups have group_m + 1 row-blocks, the rest group_m (the last one
// possibly fewer when group_big = 0).
__device__ __forceinline__ void tile_coords(const GemmParams &p, int t, int &mb, int &nb)
{
    const int big_rows = p.group_m + 1;
    const int big_tiles = p.group_big * big_rows * p.n_blocks;
    int first_m, rows, r;
    if (t < big_tiles) {
        const int g = t / (big_rows * p.n_blocks);
        first_m = g * big_rows;
        rows = big_rows;
        r = t - g * big_rows * p.n_blocks;
    } else {
        const int u = t - big_tiles;
        const int per_group = p.group_m * p.n_blocks;
        const int g = u / per_group;
        first_m = p.group_big * big_rows + g * p.group_m;
        rows = min(p.m_blocks - first_m, p.group_m);
        r = u - g * per_group;
    }
    mb = first_m + r % rows;
    nb = r / rows;
}

// First stream-K unit of CTA g (the range of CTA g ends where that of g + 1 begins).
__device__ __forceinline__ int64_t sk_begin(const GemmParams &p, int g)
{
    return static_cast<int64_t>(g) * p.sk_units / static_cast<int64_t>(gridDim.x);
}

// The work of this CTA as segments: k-blocks [k0, k1) of output tile t = (mb, nb).
//  SCHED_TILES: whole tiles blockIdx.x, blockIdx.x + gridDim.x, ... in the grouped raster.
//  SCHED_STREAM_K: the pieces of the tiles that the CTA's unit range covers, in order.
//  SCHED_SPLIT_K: tile clusterid; k-blocks [r * num_kb / split, (r + 1) * num_kb / split) for
//  the CTA of rank r (never empty when num_kb >= split).
template <int SCHED>
struct WorkIter {
    int64_t u = 0, end = 0;
    int t = 0, step = 0, rank = 0;
    __device__ explicit WorkIter(const GemmParams &p)
    {
        if constexpr (SCHED == SCHED_STREAM_K) {
            u = sk_begin(p, static_cast<int>(blockIdx.x));
            end = sk_begin(p, static_cast<int>(blockIdx.x) + 1);
        } else if constexpr (SCHED == SCHED_SPLIT_K) {
            t = static_cast<int>(cluster_id_x());
            rank = static_cast<int>(cluster_ctarank());
        } else {
            t = static_cast<int>(blockIdx.x);
            step = static_cast<int>(gridDim.x);
        }
    }
    __device__ bool next(const GemmParams &p, int &tile, int &mb, int &nb, int &k0, int &k1)
    {
        if constexpr (SCHED == SCHED_STREAM_K) {
            if (u >= end)
                return false;
            tile = static_cast<int>(u / p.num_kb);
            k0 = static_cast<int>(u - static_cast<int64_t>(tile) * p.num_kb);
            k1 = static_cast<int>(min(static_cast<int64_t>(p.num_kb), k0 + (end - u)));
            u += k1 - k0;
            tile_coords(p, tile, mb, nb);
            return true;
        } else if constexpr (SCHED == SCHED_SPLIT_K) {
            if (u != 0 || t >= p.num_tiles)
                return false;
            u = 1;   // one segment
            tile = t;
            tile_coords(p, tile, mb, nb);
            k0 = static_cast<int>(static_cast<int64_t>(rank) * p.num_kb / p.split);
            k1 = static_cast<int>(static_cast<int64_t>(rank + 1) * p.num_kb / p.split);
            return true;
        } else {
            if (t >= p.num_tiles)
                return false;
            tile = t;
            tile_coords(p, tile, mb, nb);
            k0 = 0;
            k1 = p.num_kb;
            t += step;
            return true;
        }
    }
};

struct WaitCtl {
    volatile int *abort;   // shared-memory stop flag
    uint32_t *err;         // device error word
    uint64_t limit_ns;
};

// Wait for phase `parity` of `bar`; give up (and tell everyone) when the limit runs out or
// another role has already given up.
__device__ __forceinline__ bool wait_bounded(uint32_t bar, uint32_t parity, const WaitCtl &w,
                                             uint32_t code)
{
    if (mbar_try_wait(bar, parity))
        return true;
    const uint64_t t0 = global_timer_ns();
    for (;;) {
        if (mbar_try_wait(bar, parity))
            return true;
        if (*w.abort)
            return false;
        if (global_timer_ns() - t0 > w.limit_ns) {
            *w.abort = 1;
            atomicCAS(w.err, 0u, code);
            return false;
        }
    }
}

// Bounded wait for phase `parity` of `bar` by all 32 lanes of a warp together: every lane
// polls (one warp-wide instruction, the same answer in every lane), so the warp stays
// converged and needs no broadcast afterwards; lane 0 records a timeout. Against one lane
// polling and a shuffle to the others: the softmax GEMM 262144 x 256 x 128 40.1 -> 36.8 us,
// the attention forward 64 x 4096 456 -> 422 us.
__device__ __forceinline__ bool wait_warp(uint32_t bar, uint32_t parity, const WaitCtl &w, uint32_t code, int lane)
{
    if (mbar_try_wait(bar, parity))
        return true;
    const uint64_t t0 = global_timer_ns();
    for (;;) {
        if (mbar_try_wait(bar, parity))
            return true;
        if (*w.abort)
            return false;
        if (global_timer_ns() - t0 > w.limit_ns) {
            if (lane == 0) {
                *w.abort = 1;
                atomicCAS(w.err, 0u, code);
            }
            return false;
        }
    }
}

// Teardown wait: only the time limit (used to let in-flight copies and MMAs land).
__device__ __forceinline__ bool wait_until(uint32_t bar, uint32_t parity, uint64_t limit_ns, uint32_t *err)
{
    const uint64_t t0 = global_timer_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (global_timer_ns() - t0 > limit_ns) {
            atomicCAS(err, 0u, static_cast<uint32_t>(ERR_TEARDOWN_DRAIN));
            return false;
        }
    }
    return true;
}

// GELU of two accumulator values at once: GELU(x) = x * Phi(x), with the normal CDF
// Phi(x) = 1 - h for x >= 0 and h for x < 0, where h = erfc(|x| / sqrt(2)) / 2.
// erfc(z), z >= 0, from Abramowitz & Stegun, Handbook of Mathematical Functions, formula
// 7.1.26 (Hastings): erfc(z) = t (a1 + t (a2 + t (a3 + t (a4 + t a5)))) exp(-z^2) with
// t = 1 / (1 + p z), absolute error at most 1.5e-7 (the 1/2 of h is folded into a1..a5).
// Both signs in one expression: with g = x h (0 <= h <= 1/2), GELU(x) = max(x - g, g), since
// g <= x / 2 <= x - g when x >= 0 and x - g = x (1 - h) <= x h = g when x < 0.
// Cost: the reciprocal and the exponential run on the special-function unit; everything else
// is six packed f32x2 instructions per pair plus two max. Extra FP32 instructions in the
// epilogue warps slow the concurrent MMAs of the next tile, so the count matters: this form
// costs about a third of a scalar erff-based one.
__device__ __forceinline__ void gelu_pair(float &x0, float &x1)
{
    constexpr double kL2e = 1.4426950408889634;
    constexpr double kInvSqrt2 = 0.70710678118654752;
    const uint64_t x = f32x2_pack(x0, x1);
    const uint64_t ax = x & 0x7FFFFFFF7FFFFFFFull;   // |x0|, |x1|
    const uint64_t d = f32x2_fma(ax, f32x2_pack(static_cast<float>(0.3275911 * kInvSqrt2),
                                                static_cast<float>(0.3275911 * kInvSqrt2)),
                                 f32x2_pack(1.0f, 1.0f));
    float d0, d1;
    f32x2_unpack(d, d0, d1);
    const uint64_t t = f32x2_pack(rcp_approx(d0), rcp_approx(d1));
    auto splat = [](double c) { return f32x2_pack(static_cast<float>(c), static_cast<float>(c)); };
    uint64_t q = f32x2_fma(splat(0.5 * 1.061405429), t, splat(0.5 * -1.453152027));
    q = f32x2_fma(q, t, splat(0.5 * 1.421413741));
    q = f32x2_fma(q, t, splat(0.5 * -0.284496736));
    q = f32x2_fma(q, t, splat(0.5 * 0.254829592));
    // exp(-z^2) = 2^(-x^2 log2(e) / 2)
    const uint64_t e_arg = f32x2_mul(f32x2_mul(x, splat(-0.5 * kL2e)), x);
    float a0, a1;
    f32x2_unpack(e_arg, a0, a1);
    const uint64_t h = f32x2_mul(t, f32x2_mul(q, f32x2_pack(ex2_approx(a0), ex2_approx(a1))));
    const uint64_t g = f32x2_mul(x, h);
    float g0, g1, r0, r1;
    f32x2_unpack(g, g0, g1);
    f32x2_unpack(f32x2_sub(x, g), r0, r1);
    x0 = fmaxf(r0, g0);
    x1 = fmaxf(r1, g1);
}

// Same as tcgen05.wait::ld, and ties the 32 destination registers of the load it waits
// for to this point, so that no use of them can be scheduled before the wait.
__device__ __forceinline__ void tmem_ld_wait_regs(uint32_t (&r)[32])
{
    asm volatile("tcgen05.wait::ld.sync.aligned;"
                 : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]),
                   "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]),
                   "+r"(r[14]), "+r"(r[15]), "+r"(r[16]), "+r"(r[17]), "+r"(r[18]), "+r"(r[19]),
                   "+r"(r[20]), "+r"(r[21]), "+r"(r[22]), "+r"(r[23]), "+r"(r[24]), "+r"(r[25]),
                   "+r"(r[26]), "+r"(r[27]), "+r"(r[28]), "+r"(r[29]), "+r"(r[30]), "+r"(r[31])
                 :
                 : "memory");
}

// Epilogue of one warp for one tile, step 1 (before the accumulator is ready): lane l
// fetches the bias of tile columns [8l, 8l+8) (columns at or past N read as 0) into
// registers; the load's latency hides behind the wait for the accumulator.
__device__ __forceinline__ uint4 bias_fetch(const GemmParams &p, int n_tile0, int lane)
{
    uint4 bv = make_uint4(0u, 0u, 0u, 0u);
    const int n = n_tile0 + 8 * lane;
    if (p.bias != nullptr && n < p.N)
        bv = __ldg(reinterpret_cast<const uint4 *>(p.bias + n));
    return bv;
}

// One 32-column chunk of one accumulator row per thread: + bias (from this warp's staged
// slice in shared memory), activation in FP32, FP32 -> FP16 (round to nearest even), and
// the 64 bytes of the row into the warp's staging box `box` (32 rows x 64 bytes, laid out
// with the 64-byte swizzle the TMA store expects: 16-byte piece i of row r sits at
// r*64 + (i ^ ((r >> 1) & 3))*16, which also spreads a warp's writes over all banks).
__device__ __forceinline__ void epilogue_math_stage(const GemmParams &p, const uint32_t (&r)[32], const uint4 *sbias,
                                                    uint32_t box, int lane)
{
    float v[32];
#pragma unroll
    for (int j = 0; j < 32; ++j)
        v[j] = __uint_as_float(r[j]);
    if (sbias != nullptr) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uint4 bv = sbias[i];
            const __half2 *bh = reinterpret_cast<const __half2 *>(&bv);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float2 f = __half22float2(bh[e]);
                const uint64_t sum = f32x2_add(f32x2_pack(v[8 * i + 2 * e], v[8 * i + 2 * e + 1]),
                                               f32x2_pack(f.x, f.y));
                f32x2_unpack(sum, v[8 * i + 2 * e], v[8 * i + 2 * e + 1]);
            }
        }
    }
    if (p.epilogue == EPI_GELU) {
#pragma unroll
        for (int j = 0; j < 32; j += 2)
            gelu_pair(v[j], v[j + 1]);
    } else if (p.epilogue == EPI_RELU) {
#pragma unroll
        for (int j = 0; j < 32; ++j)
            v[j] = fmaxf(v[j], 0.0f);
    }
    const uint32_t row_base = box + static_cast<uint32_t>(lane) * 64u;
    const uint32_t sw = static_cast<uint32_t>((lane >> 1) & 3);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        uint4 out;
        __half2 h0 = __floats2half2_rn(v[8 * i + 0], v[8 * i + 1]);
        __half2 h1 = __floats2half2_rn(v[8 * i + 2], v[8 * i + 3]);
        __half2 h2 = __floats2half2_rn(v[8 * i + 4], v[8 * i + 5]);
        __half2 h3 = __floats2half2_rn(v[8 * i + 6], v[8 * i + 7]);
        out.x = *reinterpret_cast<uint32_t *>(&h0);
        out.y = *reinterpret_cast<uint32_t *>(&h1);
        out.z = *reinterpret_cast<uint32_t *>(&h2);
        out.w = *reinterpret_cast<uint32_t *>(&h3);
        st_shared_v4(row_base + ((static_cast<uint32_t>(i) ^ sw) << 4), out);
    }
}

// Bounded wait on a local barrier whose phase is completed by arrivals from the cluster.
__device__ __forceinline__ bool wait_cluster_bounded(uint32_t bar, uint32_t parity, const WaitCtl &w, uint32_t code)
{
    if (mbar_try_wait_cluster(bar, parity))
        return true;
    const uint64_t t0 = global_timer_ns();
    for (;;) {
        if (mbar_try_wait_cluster(bar, parity))
            return true;
        if (*w.abort)
            return false;
        if (global_timer_ns() - t0 > w.limit_ns) {
            *w.abort = 1;
            atomicCAS(w.err, 0u, code);
            return false;
        }
    }
}

// Merge (m, s) into the running (M, S): M = max, S = sum of s * 2^(m - M) (base-2 units).
__device__ __forceinline__ void merge_stats(float &M, float &S, float m, float s)
{
    if (m == -INFINITY)
        return;
    if (m > M) {
        S = S * ex2_approx(M - m) + s;   // M = -inf gives 2^-inf = 0
        M = m;
    } else {
        S += s * ex2_approx(m - M);
    }
}

// Stream-K: a CTA holding a later part of a tile writes its warp's share of the FP32
// accumulator (32 rows, up to CHUNKS chunks of 32 columns starting at TMEM `taddr` /
// output column `n_first`) to its workspace slot. Layout of the warp's share (at `dst`):
// chunk c, then 16-byte piece i (columns 4i..4i+3 of the chunk), then the lane (row), so
// that each store instruction of the warp writes 512 contiguous bytes and the owner can
// fetch the whole share with one bulk copy. Chunks past N and rows past M are skipped, as
// the owner skips them.
template <int CHUNKS>
__device__ __forceinline__ void epilogue_partial_store(const GemmParams &p, uint32_t taddr, float *dst, int n_first,
                                                       int row0, int lane)
{
    const int valid = min(CHUNKS, (p.N - n_first + 31) / 32);
    if (valid <= 0 || row0 >= p.M)
        return;
    uint32_t ra[32], rb[32];
    auto put = [&](const uint32_t(&r)[32], int c) {
        float4 *d = reinterpret_cast<float4 *>(dst) + c * 256 + lane;
#pragma unroll
        for (int i = 0; i < 8; ++i)
            __stcg(d + 32 * i, make_float4(__uint_as_float(r[4 * i]), __uint_as_float(r[4 * i + 1]),
                                           __uint_as_float(r[4 * i + 2]), __uint_as_float(r[4 * i + 3])));
    };
    tmem_ld_32x32b_x32(taddr, ra);
#pragma unroll 1
    for (int c = 0; c < valid; c += 2) {
        tmem_ld_wait_regs(ra);
        if (c + 1 < valid)
            tmem_ld_32x32b_x32(taddr + 32u * (c + 1), rb);
        put(ra, c);
        if (c + 1 < valid) {
            tmem_ld_wait_regs(rb);
            if (c + 2 < valid)
                tmem_ld_32x32b_x32(taddr + 32u * (c + 2), ra);
            put(rb, c + 1);
        }
    }
}

// Stream-K owner: add one contributor's share (already in shared memory at `buf`, laid out
// as epilogue_partial_store wrote it) to this warp's rows of the accumulator in TMEM.
template <int CHUNKS>
__device__ __forceinline__ void fold_partial(uint32_t taddr, uint32_t buf, int valid, int lane)
{
#pragma unroll 1
    for (int c = 0; c < valid; ++c) {
        uint32_t r[32];
        tmem_ld_32x32b_x32(taddr + 32u * c, r);
        float4 q[8];
#pragma unroll
        for (int i = 0; i < 8; ++i)   // consecutive lanes read consecutive 16-byte pieces
            q[i] = ld_shared_f4(buf + static_cast<uint32_t>((c * 256 + 32 * i + lane) * 16));
        tmem_ld_wait_regs(r);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const uint64_t lo = f32x2_add(f32x2_pack(__uint_as_float(r[4 * i]), __uint_as_float(r[4 * i + 1])),
                                          f32x2_pack(q[i].x, q[i].y));
            const uint64_t hi = f32x2_add(f32x2_pack(__uint_as_float(r[4 * i + 2]), __uint_as_float(r[4 * i + 3])),
                                          f32x2_pack(q[i].z, q[i].w));
            float a, b, d, e;
            f32x2_unpack(lo, a, b);
            f32x2_unpack(hi, d, e);
            r[4 * i] = __float_as_uint(a);
            r[4 * i + 1] = __float_as_uint(b);
            r[4 * i + 2] = __float_as_uint(d);
            r[4 * i + 3] = __float_as_uint(e);
        }
        tmem_st_32x32b_x32(taddr + 32u * c, r);
    }
    tmem_st_wait();
}

// Stream-K owner: wait (all lanes of the warp together) until `flag` is 1, bounded like every
// other wait; false if the limit ran out or another role of this CTA gave up.
__device__ __forceinline__ bool wait_flag(const uint32_t *flag, const WaitCtl &w, int lane)
{
    if (__all_sync(0xffffffffu, ld_acquire_gpu_u32(flag) == 1u))
        return true;
    const uint64_t t0 = global_timer_ns();
    for (;;) {
        __nanosleep(64);
        if (__all_sync(0xffffffffu, ld_acquire_gpu_u32(flag) == 1u))
            return true;
        int stop = 0;
        if (lane == 0) {
            if (*w.abort) {
                stop = 1;
            } else if (global_timer_ns() - t0 > w.limit_ns) {
                *w.abort = 1;
                atomicCAS(w.err, 0u, static_cast<uint32_t>(ERR_STREAMK_PARTIAL));
                stop = 1;
            }
        }
        if (__shfl_sync(0xffffffffu, stop, 0))
            return false;
    }
}

// Epilogue of one warp for one tile, step 2 (accumulator ready): up to CHUNKS chunks of 32
// columns starting at TMEM address `taddr` / output column `n_first`, for the 32 output rows
// starting at `row0`. The TMEM load of chunk c+1 is in flight while chunk c is processed;
// each finished 32 x 32 box goes out with one TMA store from the warp's two alternating
// staging boxes (`stage`, toggled through `box_sel`), which clips rows >= M and
// columns >= N. Called by all 32 lanes together (tcgen05.ld is warp-collective).
template <int CHUNKS>
__device__ __forceinline__ void epilogue_tile(const GemmParams &p, uint32_t taddr, int n_first, int row0,
                                              const uint4 *sbias, const CUtensorMap *tmap_c, uint32_t stage,
                                              uint32_t &box_sel, int lane, int n_end = 0x7fffffff)
{
    // columns [n_first, min(N, n_end)) of this warp's rows, 32 per chunk
    const int valid = min(CHUNKS, (min(p.N, n_end) - n_first + 31) / 32);
    if (valid <= 0 || row0 >= p.M)
        return;   // nothing of this warp's part of the tile is inside C
    const bool has_acc = p.num_kb > 0;   // K = 0: the empty sum, no accumulator to read
    uint32_t ra[32], rb[32];
#pragma unroll
    for (int j = 0; j < 32; ++j) {
        ra[j] = 0u;
        rb[j] = 0u;
    }
    auto finish_chunk = [&](const uint32_t(&r)[32], int c) {
        const uint32_t box = stage + box_sel * EPI_STORE_BOX_BYTES;
        if (lane == 0)
            bulk_wait_group_read<1>();   // the store that last used this box has read it
        __syncwarp();
        epilogue_math_stage(p, r, sbias ? sbias + 4 * c : nullptr, box, lane);
        fence_proxy_async_shared();
        __syncwarp();
        if (lane == 0) {
            tma_store_2d(tmap_c, box, n_first + 32 * c, row0, l2_policy_evict_first());
            bulk_commit_group();
        }
        box_sel ^= 1u;
    };
    if (has_acc)
        tmem_ld_32x32b_x32(taddr, ra);
#pragma unroll 1
    for (int c = 0; c < valid; c += 2) {
        if (has_acc) {
            tmem_ld_wait_regs(ra);
            if (c + 1 < valid)
                tmem_ld_32x32b_x32(taddr + 32u * (c + 1), rb);
        }
        finish_chunk(ra, c);
        if (c + 1 < valid) {
            if (has_acc) {
                tmem_ld_wait_regs(rb);
                if (c + 2 < valid)
                    tmem_ld_32x32b_x32(taddr + 32u * (c + 2), ra);
            }
            finish_chunk(rb, c + 1);
        }
    }
}

// Split-K, step 1: an epilogue warp copies its 32 accumulator rows (CHUNKS 32-column chunks
// from chunk c_begin on, TMEM address `taddr` = chunk c_begin) into the CTA's staging area
// (the idle operand ring): FP32 row r at r * BN * 4 bytes, its 16-byte unit u stored at unit
// u ^ (r & 7), so that the eight lanes of a quarter-warp, eight consecutive rows, write eight
// different bank groups.
template <int BN, int CHUNKS>
__device__ __forceinline__ void splitk_stage(uint32_t taddr, uint32_t stage_base, int row, int c_begin)
{
    const uint32_t row_addr = stage_base + static_cast<uint32_t>(row) * (BN * 4);
    const uint32_t sw = static_cast<uint32_t>(row & 7);
#pragma unroll 1
    for (int c = 0; c < CHUNKS; ++c) {
        uint32_t v[32];
        tmem_ld_32x32b_x32(taddr + 32u * static_cast<uint32_t>(c), v);
        tmem_ld_wait_regs(v);
#pragma unroll
        for (int j = 0; j < 8; ++j)
            st_shared_v4(row_addr + (((static_cast<uint32_t>(8 * (c_begin + c) + j)) ^ sw) << 4),
                         make_uint4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]));
    }
}

// Split-K, step 2 (after a cluster barrier: every CTA's partial is staged): the CTA of rank
// `rank` owns rows [rank * R, rank * R + R) of the tile, R = BM / S; epilogue warp w takes R / 4
// of them, and lane l the 16-byte units l and l + 32 (columns 4l..4l+3 and 128+4l..) of each:
// every load instruction of the warp reads 512 contiguous bytes of one staged row (of this
// CTA's or another's, over DSMEM), and every store writes 256 contiguous bytes of C. Rows go
// in four batches of 8 / S each (all S partials of a batch in flight, the next batch's loads
// issued before the current one is added); the S partials are added in rank order, so the
// result does not depend on timing. Then bias, activation, FP16 (rows past M and columns past
// N are skipped; N is a multiple of 8, so a unit is either inside C or past it).
template <int BM, int BN, int WARPS, int S>
__device__ __forceinline__ void splitk_reduce_s(const GemmParams &p, uint32_t stage_base, int mb, int nb, int rank,
                                                int tid)
{
    static_assert(BN == 256 && BM == 128, "two 16-byte units per lane per row");
    constexpr int R = BM / S;
    constexpr int ROWS_W = R / WARPS;             // rows per warp
    constexpr int ROWS_B = 8 / S;                 // rows per batch (16 loads per lane)
    constexpr int BATCHES = ROWS_W / ROWS_B;      // 4 with four warps, 2 with eight
    static_assert(BATCHES >= 1 && ROWS_W % ROWS_B == 0, "whole batches per warp");
    const int w = tid >> 5, lane = tid & 31;
    const int r0 = rank * R + w * ROWS_W;         // first tile row of this warp
    uint32_t src[S];
#pragma unroll
    for (int q = 0; q < S; ++q)
        src[q] = mapa_shared(stage_base, static_cast<uint32_t>(q));
    float4 buf[2][ROWS_B][2][S];
    auto load = [&](int b, float4(&dst)[ROWS_B][2][S]) {
#pragma unroll
        for (int i = 0; i < ROWS_B; ++i) {
            const int r = r0 + b * ROWS_B + i;
            const uint32_t row_off = static_cast<uint32_t>(r) * (BN * 4);
            const uint32_t sw = static_cast<uint32_t>(r & 7);
#pragma unroll
            for (int k = 0; k < 2; ++k) {
                const uint32_t u = static_cast<uint32_t>(k * 32 + lane);
#pragma unroll
                for (int q = 0; q < S; ++q)
                    dst[i][k][q] = ld_shared_cluster_f4(src[q] + row_off + ((u ^ sw) << 4));
            }
        }
    };
    load(0, buf[0]);
#pragma unroll
    for (int b = 0; b < BATCHES; ++b) {
        if (b + 1 < BATCHES)
            load(b + 1, buf[(b + 1) & 1]);
        const float4(&cur)[ROWS_B][2][S] = buf[b & 1];
#pragma unroll
        for (int i = 0; i < ROWS_B; ++i) {
            const int row = mb * BM + r0 + b * ROWS_B + i;
#pragma unroll
            for (int k = 0; k < 2; ++k) {
                float4 a = cur[i][k][0];
#pragma unroll
                for (int q = 1; q < S; ++q) {
                    a.x += cur[i][k][q].x;
                    a.y += cur[i][k][q].y;
                    a.z += cur[i][k][q].z;
                    a.w += cur[i][k][q].w;
                }
                const int col = nb * BN + 4 * (k * 32 + lane);
                if (row >= p.M || col >= p.N)
                    continue;
                float v[4] = {a.x, a.y, a.z, a.w};
                if (p.bias != nullptr) {
                    const uint2 bv = __ldg(reinterpret_cast<const uint2 *>(p.bias + col));
                    const float2 f0 = __half22float2(*reinterpret_cast<const __half2 *>(&bv.x));
                    const float2 f1 = __half22float2(*reinterpret_cast<const __half2 *>(&bv.y));
                    v[0] += f0.x;
                    v[1] += f0.y;
                    v[2] += f1.x;
                    v[3] += f1.y;
                }
                if (p.epilogue == EPI_GELU) {
                    gelu_pair(v[0], v[1]);
                    gelu_pair(v[2], v[3]);
                } else if (p.epilogue == EPI_RELU) {
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        v[e] = fmaxf(v[e], 0.0f);
                }
                __half2 h0 = __floats2half2_rn(v[0], v[1]), h1 = __floats2half2_rn(v[2], v[3]);
                *reinterpret_cast<uint2 *>(p.C + static_cast<int64_t>(row) * p.ldc + col) =
                    make_uint2(*reinterpret_cast<uint32_t *>(&h0), *reinterpret_cast<uint32_t *>(&h1));
            }
        }
    }
}

template <int BM, int BN, int WARPS>
__device__ __forceinline__ void splitk_reduce(const GemmParams &p, uint32_t stage_base, int mb, int nb, int rank,
                                              int tid)
{
    if (p.split == 8)
        splitk_reduce_s<BM, BN, WARPS, 8>(p, stage_base, mb, nb, rank, tid);
    else if (p.split == 4)
        splitk_reduce_s<BM, BN, WARPS, 4>(p, stage_base, mb, nb, rank, tid);
    else
        splitk_reduce_s<BM, BN, WARPS, 2>(p, stage_base, mb, nb, rank, tid);
}

// SCHED: SCHED_TILES (whole tiles per CTA), SCHED_STREAM_K (p.sk_units > 0, workspace and
// flags set) or SCHED_SPLIT_K (launched in clusters of p.split CTAs). Epilogues NONE, GELU
// and RELU (the softmax epilogue has a kernel of its own).
template <class Cfg, int SCHED = SCHED_TILES>
__global__ void __launch_bounds__(Cfg::NUM_THREADS, 1)
    gemm_tcgen05_kernel(const __grid_constant__ CUtensorMap tmap_a, const __grid_constant__ CUtensorMap tmap_b,
                        const __grid_constant__ CUtensorMap tmap_c, const GemmParams p)
{
    constexpr int BM = Cfg::BM, BN = Cfg::BN, BK = Cfg::BK, STAGES = Cfg::STAGES;
    constexpr uint32_t IDESC = idesc_f16_f32<BM, BN>();
    constexpr uint32_t IDESC_HALF = idesc_f16_f32<BM, BN / 2>();
    static_assert(!Cfg::HALF_TAIL || SCHED == SCHED_TILES, "the half tail is for whole-tile epilogues");

    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;   // swizzled tiles need 1024-byte alignment
    uint8_t *sp = smem_raw + (base - raw);
    const uint32_t sA = base;
    const uint32_t sB = base + STAGES * Cfg::A_BYTES;
    uint64_t *bars = reinterpret_cast<uint64_t *>(sp + STAGES * Cfg::STAGE_BYTES);
    const uint32_t bar0 = smem_u32(bars);
    // barrier k lives at bar0 + 8k: full[s], empty[s], acc_full[b], acc_empty[b], drain,
    // part[epilogue warp]
    const uint32_t full0 = bar0, empty0 = bar0 + 8u * STAGES;
    const uint32_t accf0 = bar0 + 16u * STAGES, acce0 = accf0 + 8u * Cfg::ACC_BUFS;
    const uint32_t drain = acce0 + 8u * Cfg::ACC_BUFS, part0 = drain + 8u;
    const uint32_t left_half = part0 + 8u * Cfg::NUM_EPI_WARPS;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + Cfg::NUM_BARS);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    uint4 *bias_stage = reinterpret_cast<uint4 *>(sp + Cfg::BIAS_OFFSET);
    const uint32_t store_stage = base + Cfg::STORE_OFFSET;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(full0 + 8u * s, 1);
            mbar_init(empty0 + 8u * s, 1);
        }
        for (int b = 0; b < Cfg::ACC_BUFS; ++b) {
            mbar_init(accf0 + 8u * b, 1);
            mbar_init(acce0 + 8u * b, Cfg::NUM_EPI_WARPS);
        }
        mbar_init(drain, 1);
        for (int w = 0; w < Cfg::NUM_EPI_WARPS; ++w)
            mbar_init(part0 + 8u * w, 1);
        mbar_init(left_half, 1);
        *abort_flag = 0;
        fence_mbar_init();
        if (p.num_kb > 0) {
            tma_prefetch_desc(&tmap_a);
            tma_prefetch_desc(&tmap_b);
        }
        tma_prefetch_desc(&tmap_c);
    }
    if (warp == 1) {
        tmem_alloc<1>(smem_u32(tmem_slot), Cfg::TMEM_COLS);
        tmem_relinquish<1>();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem_base = *tmem_slot;
    // Everything above (barrier set-up, Tensor Memory allocation, descriptor prefetch) may
    // overlap the previous kernel in the stream; no global memory is touched before this.
    grid_dependency_wait();
    grid_dependents_launch();
    const WaitCtl wc{abort_flag, p.err, p.timeout_ns};

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0, issued = 0, issued_parity = 0;
            bool ok = true, withhold = (p.debug & DEBUG_WITHHOLD_FIRST_LOAD) != 0;
            WorkIter<SCHED> work(p);
            int t, mb, nb, k0, k1;
            while (ok && work.next(p, t, mb, nb, k0, k1)) {
                for (int kb = k0; kb < k1; ++kb) {
                    if (!wait_bounded(empty0 + 8u * stage, phase ^ 1u, wc, ERR_PRODUCER_SLOT)) {
                        ok = false;
                        break;
                    }
                    if (withhold) {
                        withhold = false;   // test hook: this slot's operands never arrive
                    } else {
                        const uint32_t fb = full0 + 8u * stage;
                        mbar_arrive_expect_tx(fb, Cfg::STAGE_BYTES);
#pragma unroll
                        for (int a = 0; a < Cfg::A_ATOMS; ++a)
                            tma_load_2d(sA + stage * Cfg::A_BYTES + a * Cfg::A_ATOM_BYTES, &tmap_a, fb,
                                        kb * BK + 64 * a, mb * BM);
#pragma unroll
                        for (int j = 0; j < Cfg::B_BOXES; ++j)
                            tma_load_2d(sB + stage * Cfg::B_BYTES + j * Cfg::B_BOX_BYTES, &tmap_b, fb,
                                        nb * BN + j * Cfg::B_BOX_N, kb * BK);
                        issued |= 1u << stage;
                        issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
                    }
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            if (!ok) {   // let every copy this thread started land before the CTA exits
                for (int s = 0; s < STAGES; ++s)
                    if (issued & (1u << s))
                        wait_until(full0 + 8u * s, (issued_parity >> s) & 1u, p.timeout_ns, p.err);
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            // Shared-memory descriptors of stage 0's A and B; every other step is a constant
            // offset in the start-address field (16-byte units; addresses stay below 256 KB, so
            // the 14-bit field never carries). A, K-major: the next 16 K-values are 32 bytes
            // further along each 128-byte swizzled row, 8-row groups 1024 bytes apart, the
            // second 64 K-values (BK = 128) one atom further. B, MN-major: 16 K-rows are 2048
            // bytes further, 8-row K groups 1024 bytes apart (SBO), 64-column N atoms one box
            // apart (LBO).
            const uint64_t a_desc0 = sw128_desc(sA, 16, 1024), b_desc0 = sw128_desc(sB, Cfg::B_BOX_BYTES, 1024);
            int stage = 0, acc = 0;
            uint32_t phase = 0, acc_phase = 0;
            bool ok = true;
            WorkIter<SCHED> work(p);
            int t, mb, nb, k0, k1;
            while (ok && work.next(p, t, mb, nb, k0, k1)) {
                if (!wait_bounded(acce0 + 8u * acc, acc_phase ^ 1u, wc, ERR_MMA_ACCUMULATOR)) {
                    ok = false;
                    break;
                }
                tc_fence_after_sync();
                const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN);
                // k-blocks [tail, k1) go into the left half only, and stay in the ring for the
                // right half below (HALF_TAIL; otherwise tail = k1)
                const int tail = Cfg::HALF_TAIL ? max(k0, k1 - STAGES) : k1;
                int tail_stage = stage;
                for (int kb = k0; kb < k1; ++kb) {
                    if (!wait_bounded(full0 + 8u * stage, phase, wc, ERR_MMA_OPERANDS)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after_sync();
                    const uint64_t a_st = a_desc0 + static_cast<uint64_t>(stage * (Cfg::A_BYTES >> 4));
                    const uint64_t b_st = b_desc0 + static_cast<uint64_t>(stage * (Cfg::B_BYTES >> 4));
                    if (Cfg::HALF_TAIL && kb >= tail) {
                        if (kb == tail)
                            tail_stage = stage;
#pragma unroll
                        for (int kk = 0; kk < BK / Cfg::UMMA_K; ++kk)
                            umma_f16<1>(d_tmem,
                                        a_st + static_cast<uint64_t>((kk >> 2) * (Cfg::A_ATOM_BYTES >> 4) + 2 * (kk & 3)),
                                        b_st + static_cast<uint64_t>(128 * kk), IDESC_HALF, (kb != k0 || kk != 0) ? 1u : 0u);
                    } else {
#pragma unroll
                        for (int kk = 0; kk < BK / Cfg::UMMA_K; ++kk)
                            umma_f16<1>(d_tmem,
                                        a_st + static_cast<uint64_t>((kk >> 2) * (Cfg::A_ATOM_BYTES >> 4) + 2 * (kk & 3)),
                                        b_st + static_cast<uint64_t>(128 * kk), IDESC, (kb != k0 || kk != 0) ? 1u : 0u);
                        umma_commit(empty0 + 8u * stage);   // slot free once these MMAs have read it
                    }
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok)
                    break;
                if constexpr (Cfg::HALF_TAIL) {
                    umma_commit(left_half);   // columns [0, BN / 2) complete (also when K = 0)
                    // the right half of the tail k-blocks: B from its second half of N atoms. The
                    // tail's slots are not released: each CTA has one tile, no load waits for them.
                    int st = tail_stage;
                    for (int kb = tail; kb < k1; ++kb) {
                        const uint64_t a_st = a_desc0 + static_cast<uint64_t>(st * (Cfg::A_BYTES >> 4));
                        const uint64_t b_st =
                            b_desc0 + static_cast<uint64_t>(st * (Cfg::B_BYTES >> 4) + ((Cfg::B_BYTES / 2) >> 4));
#pragma unroll
                        for (int kk = 0; kk < BK / Cfg::UMMA_K; ++kk)
                            umma_f16<1>(d_tmem + static_cast<uint32_t>(BN / 2),
                                        a_st + static_cast<uint64_t>((kk >> 2) * (Cfg::A_ATOM_BYTES >> 4) + 2 * (kk & 3)),
                                        b_st + static_cast<uint64_t>(128 * kk), IDESC_HALF, (kb != k0 || kk != 0) ? 1u : 0u);
                        if (++st == STAGES)
                            st = 0;
                    }
                }
                umma_commit(accf0 + 8u * acc);          // accumulator complete
                if (++acc == Cfg::ACC_BUFS) {
                    acc = 0;
                    acc_phase ^= 1u;
                }
            }
            if (!ok) {   // let every MMA this thread issued finish before TMEM is freed
                umma_commit(drain);
                wait_until(drain, 0, p.timeout_ns, p.err);
            }
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ epilogue warps
        const int quarter = warp & 3;                 // TMEM lanes this warp may access
        const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
        constexpr int CHUNKS = BN / 32 / Cfg::EPI_COL_GROUPS;   // 32-column chunks per warp
        const int c_begin = ((warp - 2) >> 2) * CHUNKS;
        uint4 *my_bias = bias_stage + (warp - 2) * (BN / 8);   // this warp's BN-wide bias slice
        // HALF_TAIL: the warps of columns [0, BN / 2) read the accumulator once its left half is
        // complete and stage their output in the stages' left B halves (4 KB per warp)
        const bool left = Cfg::HALF_TAIL && c_begin * 32 < BN / 2;
        const uint32_t my_stage =
            left ? sB + static_cast<uint32_t>(((warp - 2) / Cfg::LEFT_STAGE_WARPS) * Cfg::B_BYTES +
                                              ((warp - 2) % Cfg::LEFT_STAGE_WARPS) * EPI_STORE_WARP_BYTES)
                 : store_stage + static_cast<uint32_t>(warp - 2) * EPI_STORE_WARP_BYTES;
        uint32_t box_sel = 0;
        int acc = 0;
        uint32_t acc_phase = 0, left_phase = 0;
        const int ew = warp - 2;   // this warp's stream-K flag and partial-barrier index
        // floats per workspace slot, and the offset of this warp's share in a slot
        constexpr int64_t SLOT = static_cast<int64_t>(BM) * BN;
        const int64_t my_share = static_cast<int64_t>(ew) * (Cfg::PART_WARP_BYTES / 4);
        uint32_t part_phase = 0;
        if constexpr (SCHED == SCHED_SPLIT_K) {
            // this CTA's partial sum of its tile into the staging area; the cluster reduces
            // the partials after the barrier below
            static_assert(BM * BN * 4 <= Cfg::STAGES * Cfg::STAGE_BYTES, "the staged partial fits the operand ring");
            WorkIter<SCHED> work(p);
            int t, mb, nb, k0, k1;
            if (work.next(p, t, mb, nb, k0, k1)) {
                int ok = 1;
                if (lane == 0)
                    ok = wait_bounded(accf0, 0u, wc, ERR_EPILOGUE_ACCUMULATOR) ? 1 : 0;
                if (__shfl_sync(0xffffffffu, ok, 0)) {
                    tc_fence_after_sync();
                    splitk_stage<BN, CHUNKS>(tmem_base + lane_base + static_cast<uint32_t>(c_begin * 32), sA,
                                             quarter * 32 + lane, c_begin);
                }
            }
        } else {
            WorkIter<SCHED> work(p);
            int t, mb, nb, k0, k1;
            while (work.next(p, t, mb, nb, k0, k1)) {
                const uint4 bv = bias_fetch(p, nb * BN, lane);
                // all lanes poll (see wait_warp): fewer issue slots taken from the producer and
                // MMA threads than one lane spinning (2048^3 at the power limit: 19.4 -> 18.6 us)
                int ok = wait_warp(left ? left_half : accf0 + 8u * acc, left ? left_phase : acc_phase, wc,
                                   ERR_EPILOGUE_ACCUMULATOR, lane) ? 1 : 0;
                left_phase ^= 1u;
                if (!ok)
                    break;
                tc_fence_after_sync();
                const uint32_t tacc = tmem_base + lane_base + static_cast<uint32_t>(acc * BN + c_begin * 32);
                const int n_first = nb * BN + c_begin * 32, row0 = mb * BM + quarter * 32;
                if (SCHED == SCHED_STREAM_K && k0 > 0) {
                    // a later part of a cut tile: hand the partial sum to the tile's owner
                    epilogue_partial_store<CHUNKS>(p, tacc, p.sk_ws + static_cast<int64_t>(blockIdx.x) * SLOT + my_share,
                                                   n_first, row0, lane);
                    __threadfence();
                    __syncwarp();
                    if (lane == 0)
                        st_release_gpu_u32(p.sk_flags + blockIdx.x * Cfg::NUM_EPI_WARPS + ew, 1u);
                } else {
                    int n_parts = 0;
                    if (SCHED == SCHED_STREAM_K && k1 < p.num_kb) {
                        // Owner of a cut tile: the CTAs whose ranges begin inside it hold the rest.
                        // This is the last part of this CTA's range, so its MMAs are complete and
                        // the operand ring is idle: each warp pulls a contributor's share into its
                        // own piece of the ring and adds it to its rows in TMEM.
                        const int64_t tile_end = static_cast<int64_t>(t + 1) * p.num_kb;
                        const int g0 = static_cast<int>(blockIdx.x);
                        while (g0 + n_parts + 1 < static_cast<int>(gridDim.x) && sk_begin(p, g0 + n_parts + 1) < tile_end)
                            ++n_parts;
                        const int valid = min(CHUNKS, (p.N - n_first + 31) / 32);
                        const bool inside = valid > 0 && row0 < p.M;
                        const uint32_t buf = sA + static_cast<uint32_t>(ew * Cfg::PART_WARP_BYTES);
                        for (int j = 1; ok && j <= n_parts; ++j) {
                            ok = wait_flag(p.sk_flags + (g0 + j) * Cfg::NUM_EPI_WARPS + ew, wc, lane) ? 1 : 0;
                            if (!ok || !inside)
                                continue;
                            if (lane == 0) {
                                fence_proxy_async_global();   // acquired data, read next by the copy engine
                                mbar_arrive_expect_tx(part0 + 8u * ew, Cfg::PART_WARP_BYTES);
                                bulk_load_g2s(buf, p.sk_ws + static_cast<int64_t>(g0 + j) * SLOT + my_share,
                                              Cfg::PART_WARP_BYTES, part0 + 8u * ew);
                                ok = wait_bounded(part0 + 8u * ew, part_phase, wc, ERR_STREAMK_PARTIAL) ? 1 : 0;
                            }
                            part_phase ^= 1u;
                            ok = __shfl_sync(0xffffffffu, ok, 0);
                            if (ok)
                                fold_partial<CHUNKS>(tacc, buf, valid, lane);
                        }
                        if (!ok)
                            break;
                    }
                    if (p.bias != nullptr) {
                        my_bias[lane] = bv;
                        __syncwarp();
                    }
                    epilogue_tile<CHUNKS>(p, tacc, n_first, row0, p.bias != nullptr ? my_bias + c_begin * 4 : nullptr,
                                          &tmap_c, my_stage, box_sel, lane);
                    if (n_parts > 0 && lane == 0) {   // consumed: lower the flags for the next launch
                        for (int j = 1; j <= n_parts; ++j)
                            p.sk_flags[(static_cast<int>(blockIdx.x) + j) * Cfg::NUM_EPI_WARPS + ew] = 0u;
                    }
                }
                tc_fence_before_sync();
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(acce0 + 8u * acc);   // this warp's rows of the accumulator are read
                if (++acc == Cfg::ACC_BUFS) {
                    acc = 0;
                    acc_phase ^= 1u;
                }
            }
        }
        if (lane == 0)
            bulk_wait_group<0>();   // every output box of this warp has reached global memory
        __syncwarp();
    }

    if constexpr (SCHED == SCHED_SPLIT_K) {
        // every thread of every CTA of the cluster, on every path (also after a timeout)
        cluster_sync();   // all partials are staged
        if (warp >= 2) {
            WorkIter<SCHED> work(p);
            int t, mb, nb, k0, k1;
            if (work.next(p, t, mb, nb, k0, k1) && *abort_flag == 0)
                splitk_reduce<BM, BN, Cfg::NUM_EPI_WARPS>(p, sA, mb, nb, static_cast<int>(cluster_ctarank()),
                                                          static_cast<int>(threadIdx.x) - 64);
        }
        cluster_sync();   // no CTA leaves while another may still read its partial
    }
    tc_fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after_sync();
        tmem_dealloc<1>(tmem_base, Cfg::TMEM_COLS);
    }
}

}  // namespace gb300
