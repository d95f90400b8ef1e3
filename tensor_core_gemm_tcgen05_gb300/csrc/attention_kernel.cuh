// FlashAttention forward for sm_103a (GB300), head dimension 128, FP16 in and out:
//
//     O[h][i][:] = sum_j softmax_j(scale * Q[h][i][:] . K[h][j][:]) V[h][j][:]   (j <= i if causal)
//
// The tutorial's fused attention ("TileLang ..." on pro.edgex.exchange, FlashAttention
// paragraph: query, key and value tiles processed without writing the full score matrix to
// global memory, online softmax with running maxima, normalising sums and rescaling factors,
// tensor-core tile products; "TileLang: Criando Kernels de GPU ..." on noticiai.com.br,
// section "Softmax por linha e FlashAttention": Q K^T and P V on tensor cores, max subtracted
// per block; "Designing High-Performance GPU Kernels with TileLang" on spaxe.top: causal and
// non-causal). Built on the same fifth-generation tensor-core machinery as the GEMM:
//
//  * one CTA per (head, block of 256 queries) = two query tiles A and B of 128 rows; heads in
//    groups of eight, within a group the blocks with the most keys (causal) first;
//  * warp 0: TMA producer. Both Q tiles once (K-major, two 128-byte-swizzled atoms of 64 head
//    dims each), then K and V blocks of 128 keys through a two-stage ring; 3-D tensor maps
//    [head][row][dim] so that rows past the sequence read as zero;
//  * warp 1: MMA issuer. S_t = Q_t K_j^T (M = N = 128, K = 128, both operands K-major from
//    shared memory) into tile t's TMEM score columns; O_t += P_t V_j with P_t read from Tensor
//    Memory (written by the softmax over the first half of the score columns, FP16 pairs)
//    and V MN-major from shared memory, in two halves: keys 0..63 as soon as the softmax has
//    written their P, keys 64..127 once all of P is written. Issue order per key block j:
//    P_A V_j, S_A for block j + 1, P_B V_j, S_B for block j + 1, so that the tensor cores work
//    on one tile while the other tile's softmax runs;
//  * warps 2..5 (tile A) and 6..9 (tile B): online softmax, one query row per thread (its
//    TMEM lane). Per block: the row maximum of the scores; when it exceeds the running
//    maximum by more than kRescaleThreshold, the row of O is rescaled in TMEM (after the
//    previous P V product); p = 2^(s * scale * log2(e) - m) written as FP16 over the scores
//    (the A operand of P V), summed into the running denominator l. At the end: O / l.
// Every mbarrier wait is bounded in time, as in the GEMM kernels.
#pragma once

#include <type_traits>

#include "gemm_kernel.cuh"

namespace gb300 {

// A row's running maximum is raised (and its row of O rescaled) only when a block's maximum
// exceeds it by more than this many base-2 units; otherwise probabilities are taken against
// the old maximum and stay below 2^8, well inside FP16 and FP32.
constexpr float kRescaleThreshold = 8.0f;

// Heads per group in the order of the work items (see the kernel): at most this many,
// the groups of a launch made equal in size.
constexpr int kAttnHeadGroup = 8;
constexpr int kAttnHeadGroupCausal = 16;

struct AttnParams {
    int H;              // heads (batch x heads)
    int Sq, Sk;         // query and key lengths
    int q_blocks;       // ceil(Sq / 256): CTAs per head
    int causal;
    float scale_log2;   // scale * log2(e): scores are kept in base-2 units
    uint32_t *err;
    uint64_t timeout_ns;
};

struct AttnConfig {
    static constexpr int D = 128;         // head dimension
    static constexpr int BQ = 128;        // queries per tile (= TMEM lanes)
    static constexpr int TILES = 2;       // query tiles per CTA
    static constexpr int BKV = 128;       // keys per block
    static constexpr int ATOM_BYTES = 128 * 128;   // 128 rows x 64 FP16 (one 128-byte swizzle row each)
    static constexpr int TILE_BYTES = 2 * ATOM_BYTES;  // 128 x 128 FP16
    static constexpr int KV_STAGES = 2;
    // shared memory: Q_A Q_B | K[0] V[0] | K[1] V[1] | barriers
    static constexpr int Q_OFF = 0;
    static constexpr int KV_OFF = TILES * TILE_BYTES;
    static constexpr int BAR_OFF = KV_OFF + KV_STAGES * 2 * TILE_BYTES;
    // barriers: q_full, kv_full[2], kv_empty[2], s_full[2], p_full[2], pv_done[2], drain,
    // p_half[2] (the first 64 keys' P written)
    static constexpr int NUM_BARS = 1 + 2 * KV_STAGES + 4 * TILES + 1;
    static constexpr int SMEM_BYTES = 1024 + BAR_OFF + NUM_BARS * 8 + 16;
    static constexpr int NUM_THREADS = 64 + TILES * 128;
    // TMEM: S_A | S_B | O_A | O_B, 128 columns each; P_t over the first 64 columns of S_t
    static constexpr int TMEM_COLS = 512;
    static constexpr int S_COL = 0, O_COL = 256;
    static_assert(SMEM_BYTES <= 232448, "exceeds the 227 KB per-CTA shared memory limit");
};

// Instruction descriptor, kind::f16, FP32 accumulate, FP16 operands, M = N = 128, A K-major.
// b_mn_major: B is MN-major (V, head dims contiguous) instead of K-major (K, keys' dims
// contiguous).
template <bool B_MN_MAJOR>
__host__ __device__ constexpr uint32_t idesc_attn()
{
    return (1u << 4) | (B_MN_MAJOR ? (1u << 16) : 0u) | (static_cast<uint32_t>(128 >> 3) << 17) |
           (static_cast<uint32_t>(128 >> 4) << 24);
}

// Descriptor of 16-wide K step kk of a K-major 128 x 128 tile stored as two 128-byte-swizzled
// atoms of 64 K columns (atom = kk / 4; 32 bytes further along the swizzled row per step).
__device__ __forceinline__ uint64_t kmajor_step_desc(uint32_t tile, int kk)
{
    return sw128_desc(tile + static_cast<uint32_t>(kk >> 2) * AttnConfig::ATOM_BYTES +
                          static_cast<uint32_t>(kk & 3) * 32u,
                      16, 1024);
}

// Descriptor of 16-key step kk of V (keys x head dims, head dims contiguous = MN-major):
// two atoms of 64 head dims 16 KB apart (LBO), 8-key groups 1 KB apart (SBO), 16 keys =
// 2048 bytes per step.
__device__ __forceinline__ uint64_t v_step_desc(uint32_t tile, int kk)
{
    return sw128_desc(tile + static_cast<uint32_t>(kk) * 2048u, AttnConfig::ATOM_BYTES, 1024);
}

// Reads the four 32-column chunks of a 128-column TMEM row range starting at `addr` and
// hands each to fn(chunk registers, chunk index); the load of chunk c+1 is in flight while
// chunk c is processed. Warp-collective.
template <class Fn>
__device__ __forceinline__ void two_buffered_chunks(uint32_t addr, uint32_t (&va)[32], uint32_t (&vb)[32], Fn &&fn)
{
    tmem_ld_32x32b_x32(addr, va);
    tmem_ld_wait_regs(va);
    tmem_ld_32x32b_x32(addr + 32u, vb);
    fn(va, 0);
    tmem_ld_wait_regs(vb);
    tmem_ld_32x32b_x32(addr + 64u, va);
    fn(vb, 1);
    tmem_ld_wait_regs(va);
    tmem_ld_32x32b_x32(addr + 96u, vb);
    fn(va, 2);
    tmem_ld_wait_regs(vb);
    fn(vb, 3);
}

// Online softmax of one warp of tile t's softmax group: each thread owns query row r of the
// tile (TMEM lane r). Per key block j: (1) read the 128 scores of the row and take their
// maximum in base-2 units (keys past the sequence, or after the query when causal, are left
// out); (2) if the maximum grew by more than kRescaleThreshold for some row of the warp, wait
// for the previous P V product of this tile and rescale the warp's rows of O by
// 2^(m_old - m_new); (3) read the scores again and write p = 2^(s - m_new) as FP16 pairs over
// the first 64 score columns (chunk c of 32 keys to columns 16c..16c+15: each lies in score
// columns that were already read), summing p into the running denominator l. At the end the
// row of O is divided by l and stored.
//
// `o_stage`: the tile's Q buffer in shared memory, free once its last S product has
// completed, where the rows of O are staged for the TMA store (`tmap_o`).
// The completion of the tile's P V product of block b: with `pv_per_stage` false, phase b of
// the barrier `pv_done`; with it true (tile B), phase b / 2 of barrier b mod 2 of the pair at
// `pv_done` (the key/value ring's empty barriers, which tile B's P V products complete).
__device__ __forceinline__ void attention_softmax_warp(const AttnParams &p, uint32_t tmem, int tile, uint32_t s_full,
                                                       uint32_t p_half, uint32_t p_full, uint32_t pv_done,
                                                       const WaitCtl &wc, int warp, int lane, int q0, int h, int n_kv,
                                                       uint32_t o_stage, const CUtensorMap *tmap_o, bool pv_per_stage)
{
    auto wait_pv = [&](int b) -> bool {
        const uint32_t ub = static_cast<uint32_t>(b);
        return pv_per_stage ? wait_warp(pv_done + 8u * (ub & 1u), (ub >> 1) & 1u, wc, ERR_EPILOGUE_ACCUMULATOR, lane)
                            : wait_warp(pv_done, ub & 1u, wc, ERR_EPILOGUE_ACCUMULATOR, lane);
    };
    using Cfg = AttnConfig;
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;
    const int qi = q0 + r;
    const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t s_addr = tmem + lane_base + static_cast<uint32_t>(Cfg::S_COL + tile * Cfg::BQ);
    const uint32_t o_addr = tmem + lane_base + static_cast<uint32_t>(Cfg::O_COL + tile * Cfg::D);
    const int kmax = p.causal ? min(p.Sk - 1, qi) : p.Sk - 1;   // last key this row sees
    const float sl2 = p.scale_log2;
    float m = -INFINITY, l = 0.0f;
    uint32_t va[32], vb[32];
    for (int j = 0; j < n_kv; ++j) {
        if (!wait_warp(s_full, static_cast<uint32_t>(j) & 1u, wc, ERR_EPILOGUE_ACCUMULATOR, lane))
            return;
        tc_fence_after_sync();
        const int k0 = j * Cfg::BKV;
        // The block's work is compiled twice: without any masking when no key of the block is
        // masked for any row of the warp (every block but the last, or the diagonal one when
        // causal), and with the per-key mask otherwise. The choice is warp-uniform: the body
        // holds warp-collective Tensor Memory loads and stores.
        const bool all_full = __all_sync(0xffffffffu, k0 + Cfg::BKV - 1 <= kmax);
        auto block = [&](auto full_tag) -> bool {
            constexpr bool full = decltype(full_tag)::value;
            // Block maximum of scale * s (base-2 units). On unmasked blocks: the maximum (minimum
            // for a negative scale) of the raw scores in four independent three-input chains,
            // scaled once.
            float mb = -INFINITY;
            float r0 = sl2 >= 0.0f ? -INFINITY : INFINITY, r1 = r0, r2 = r0, r3 = r0;
            auto max_chunk = [&](const uint32_t(&x)[32], int c) {
                if constexpr (full) {
                    if (sl2 >= 0.0f) {
    #pragma unroll
                        for (int e = 0; e < 32; e += 8) {
                            r0 = fmax3(r0, __uint_as_float(x[e]), __uint_as_float(x[e + 1]));
                            r1 = fmax3(r1, __uint_as_float(x[e + 2]), __uint_as_float(x[e + 3]));
                            r2 = fmax3(r2, __uint_as_float(x[e + 4]), __uint_as_float(x[e + 5]));
                            r3 = fmax3(r3, __uint_as_float(x[e + 6]), __uint_as_float(x[e + 7]));
                        }
                    } else {
    #pragma unroll
                        for (int e = 0; e < 32; e += 8) {
                            r0 = fmin3(r0, __uint_as_float(x[e]), __uint_as_float(x[e + 1]));
                            r1 = fmin3(r1, __uint_as_float(x[e + 2]), __uint_as_float(x[e + 3]));
                            r2 = fmin3(r2, __uint_as_float(x[e + 4]), __uint_as_float(x[e + 5]));
                            r3 = fmin3(r3, __uint_as_float(x[e + 6]), __uint_as_float(x[e + 7]));
                        }
                    }
                } else {
    #pragma unroll
                    for (int e = 0; e < 32; ++e)
                        if (k0 + 32 * c + e <= kmax)
                            mb = fmaxf(mb, __uint_as_float(x[e]) * sl2);
                }
            };
            two_buffered_chunks(s_addr, va, vb, max_chunk);
            if constexpr (full)
                mb = (sl2 >= 0.0f ? fmax3(fmaxf(r0, r1), r2, r3) : fmin3(fminf(r0, r1), r2, r3)) * sl2;
            // keep the old maximum unless this block's exceeds it by more than the threshold
            const bool raise = mb > m + kRescaleThreshold || m == -INFINITY;
            const float m_new = raise ? mb : m;
            const float m_use = m_new == -INFINITY ? 0.0f : m_new;
            const float alpha = raise ? ex2_approx(m - m_use) : 1.0f;   // 0 on the first block (m = -inf)
            if (j > 0 && __any_sync(0xffffffffu, alpha != 1.0f)) {
                if (!wait_pv(j - 1))   // P_t V of block j - 1 done
                    return false;
                tc_fence_after_sync();
    #pragma unroll 1
                for (int c = 0; c < 4; ++c) {
                    tmem_ld_32x32b_x32(o_addr + 32u * c, va);
                    tmem_ld_wait_regs(va);
    #pragma unroll
                    for (int e = 0; e < 32; e += 2) {
                        float a, b;
                        f32x2_unpack(f32x2_mul(f32x2_pack(__uint_as_float(va[e]), __uint_as_float(va[e + 1])),
                                               f32x2_pack(alpha, alpha)),
                                     a, b);
                        va[e] = __float_as_uint(a);
                        va[e + 1] = __float_as_uint(b);
                    }
                    tmem_st_32x32b_x32(o_addr + 32u * c, va);
                }
                tmem_st_wait();
            }
            // four independent packed partial sums
            uint64_t sum2[4] = {f32x2_pack(0.0f, 0.0f), f32x2_pack(0.0f, 0.0f), f32x2_pack(0.0f, 0.0f),
                                f32x2_pack(0.0f, 0.0f)};
            const uint64_t scale2 = f32x2_pack(sl2, sl2), neg_m2 = f32x2_pack(-m_use, -m_use);
            auto p_chunk = [&](const uint32_t(&x)[32], int c) {
                uint32_t pk[16];
    #pragma unroll
                for (int i = 0; i < 16; ++i) {
                    float t0, t1;
                    f32x2_unpack(f32x2_fma(f32x2_pack(__uint_as_float(x[2 * i]), __uint_as_float(x[2 * i + 1])), scale2,
                                           neg_m2),
                                 t0, t1);
                    float p0 = ex2_approx(t0), p1 = ex2_approx(t1);
                    if constexpr (!full) {
                        const int k = k0 + 32 * c + 2 * i;
                        p0 = k <= kmax ? p0 : 0.0f;
                        p1 = k + 1 <= kmax ? p1 : 0.0f;
                    }
                    sum2[i & 3] = f32x2_add(sum2[i & 3], f32x2_pack(p0, p1));
                    __half2 hh = __floats2half2_rn(p0, p1);
                    pk[i] = *reinterpret_cast<uint32_t *>(&hh);
                }
                tmem_st_32x32b_x16(s_addr + 16u * static_cast<uint32_t>(c), pk);   // P over read scores
            };
            // P of keys 0..63 first, announced on p_half so that P V can start on them while keys
            // 64..127 are computed
            tmem_ld_32x32b_x32(s_addr, va);
            tmem_ld_wait_regs(va);
            tmem_ld_32x32b_x32(s_addr + 32u, vb);
            p_chunk(va, 0);
            tmem_ld_wait_regs(vb);
            tmem_ld_32x32b_x32(s_addr + 64u, va);
            p_chunk(vb, 1);
            tmem_st_wait();
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(p_half);
            tmem_ld_wait_regs(va);
            tmem_ld_32x32b_x32(s_addr + 96u, vb);
            p_chunk(va, 2);
            tmem_ld_wait_regs(vb);
            p_chunk(vb, 3);
            float s0, s1;
            f32x2_unpack(f32x2_add(f32x2_add(sum2[0], sum2[1]), f32x2_add(sum2[2], sum2[3])), s0, s1);
            l = l * alpha + (s0 + s1);
            m = m_new;
            tmem_st_wait();
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(p_full);   // P_t written (and O_t rescaled): the MMA warp may multiply
            return true;
        };
        if (!(all_full ? block(std::true_type{}) : block(std::false_type{})))
            return;
    }
    if (n_kv == 0)
        return;
    if (!wait_pv(n_kv - 1))
        return;
    tc_fence_after_sync();
    const float inv = l > 0.0f ? 1.0f / l : 0.0f;
    // The warp's 32 rows of O / l, rounded to FP16, staged as two 64-column boxes of 32 rows
    // (128-byte swizzle: 16-byte piece k of row r at piece k ^ (r mod 8)), then written by two
    // TMA stores, which clip rows past the sequence. The last S product of the tile, which
    // read the buffer, completed before pv_done's last phase.
    const uint32_t row_base = o_stage + static_cast<uint32_t>(quarter) * 4096u + static_cast<uint32_t>(lane) * 128u;
#pragma unroll 1
    for (int c = 0; c < 4; ++c) {
        tmem_ld_32x32b_x32(o_addr + 32u * c, va);
        tmem_ld_wait_regs(va);
        const uint32_t row = row_base + static_cast<uint32_t>(c >> 1) * Cfg::ATOM_BYTES;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            uint32_t pk[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                __half2 hh = __floats2half2_rn(__uint_as_float(va[8 * i + 2 * e]) * inv,
                                               __uint_as_float(va[8 * i + 2 * e + 1]) * inv);
                pk[e] = *reinterpret_cast<uint32_t *>(&hh);
            }
            const uint32_t piece = static_cast<uint32_t>(((c & 1) * 4 + i) ^ (lane & 7));
            st_shared_v4(row + piece * 16u, make_uint4(pk[0], pk[1], pk[2], pk[3]));
        }
    }
    fence_proxy_async_shared();
    __syncwarp();
    const int row0 = q0 + quarter * 32;
    if (lane == 0 && row0 < p.Sq) {
        for (int a = 0; a < 2; ++a)
            tma_store_3d(tmap_o, o_stage + static_cast<uint32_t>(a) * Cfg::ATOM_BYTES + static_cast<uint32_t>(quarter) * 4096u,
                         64 * a, row0, h);
        bulk_commit_group();
        bulk_wait_group<0>();   // the stores have read shared memory and written O before the CTA ends
    }
    __syncwarp();
}

__global__ void __launch_bounds__(AttnConfig::NUM_THREADS, 1)
    attention_fwd_kernel(const __grid_constant__ CUtensorMap tmap_q, const __grid_constant__ CUtensorMap tmap_k,
                         const __grid_constant__ CUtensorMap tmap_v, const __grid_constant__ CUtensorMap tmap_o,
                         const AttnParams p)
{
    using Cfg = AttnConfig;
    constexpr uint32_t ATOM = Cfg::ATOM_BYTES, TILE = Cfg::TILE_BYTES;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *sp = smem_raw + (base - raw);
    const uint32_t sQ = base + Cfg::Q_OFF, sKV = base + Cfg::KV_OFF;
    // barrier k lives at bar0 + 8k: q_full, kv_full[2], kv_empty[2], s_full[2], p_full[2],
    // pv_done[2], drain (index [t] = query tile)
    const uint32_t q_full = base + Cfg::BAR_OFF;
    const uint32_t kv_full0 = q_full + 8u, kv_empty0 = kv_full0 + 8u * Cfg::KV_STAGES;
    const uint32_t s_full0 = kv_empty0 + 8u * Cfg::KV_STAGES, p_full0 = s_full0 + 8u * Cfg::TILES;
    const uint32_t pv_done0 = p_full0 + 8u * Cfg::TILES, drain = pv_done0 + 8u * Cfg::TILES;
    const uint32_t p_half0 = drain + 8u;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sp + Cfg::BAR_OFF + Cfg::NUM_BARS * 8);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    // work item: query block qb (256 queries, two tiles) of head h. Heads are taken in groups
    // of at most 8 (16 when causal), all groups of a launch the same size up to one head;
    // within a group the blocks with the most keys (causal) go first, heads fastest. The CTAs
    // in flight then share the keys and values of a few heads in L2 (64 x 4096 full: +8 %
    // against all heads at once) and, when causal, the long items still start before the
    // short ones; larger groups when causal keep the last group's long items from starting
    // late (64 x 4096 causal: +1.4 % with 16 against 8; a last group of 4 heads behind five
    // of 12: -11 %).
    const int g_max = p.causal ? kAttnHeadGroupCausal : kAttnHeadGroup;
    const int n_grp = (p.H + g_max - 1) / g_max;
    const int g_size = (p.H + n_grp - 1) / n_grp;   // heads per group (the last may have fewer)
    const int grp = static_cast<int>(blockIdx.x) / (g_size * p.q_blocks);
    const int r = static_cast<int>(blockIdx.x) % (g_size * p.q_blocks);
    const int heads_in_grp = min(g_size, p.H - grp * g_size);
    const int qb = p.q_blocks - 1 - r / heads_in_grp;
    const int h = grp * g_size + r % heads_in_grp;
    const int q0 = qb * Cfg::TILES * Cfg::BQ;
    const int k_end = p.causal ? min(p.Sk, q0 + Cfg::TILES * Cfg::BQ) : p.Sk;   // keys any row may see
    const int n_kv = (k_end + Cfg::BKV - 1) / Cfg::BKV;
    // key blocks of tile t (causal: tile A's rows see no key past q0 + 127, so the block of
    // keys q0 + 128 .. q0 + 255 is left out for it)
    int n_t[Cfg::TILES];
#pragma unroll
    for (int t = 0; t < Cfg::TILES; ++t)
        n_t[t] = p.causal ? min(n_kv, (min(p.Sk, q0 + (t + 1) * Cfg::BQ) + Cfg::BKV - 1) / Cfg::BKV) : n_kv;

    if (threadIdx.x == 0) {
        mbar_init(q_full, 1);
        for (int s = 0; s < Cfg::KV_STAGES; ++s) {
            mbar_init(kv_full0 + 8u * s, 1);
            mbar_init(kv_empty0 + 8u * s, 1);
        }
        for (int t = 0; t < Cfg::TILES; ++t) {
            mbar_init(s_full0 + 8u * t, 1);
            mbar_init(p_full0 + 8u * t, 4);   // the four softmax warps of tile t
            mbar_init(pv_done0 + 8u * t, 1);
            mbar_init(p_half0 + 8u * t, 4);
        }
        mbar_init(drain, 1);
        *abort_flag = 0;
        fence_mbar_init();
        tma_prefetch_desc(&tmap_o);
        // Q and the first key/value block go out before the Tensor Memory allocation and the
        // block barrier, so that their latency overlaps the rest of the set-up (the barriers
        // are initialised and fenced above; the wait orders the reads after the previous grid)
        grid_dependency_wait();
        mbar_arrive_expect_tx(q_full, Cfg::TILES * TILE);
        for (int t = 0; t < Cfg::TILES; ++t) {
            tma_load_3d(sQ + t * TILE, &tmap_q, q_full, 0, q0 + t * Cfg::BQ, h);
            tma_load_3d(sQ + t * TILE + ATOM, &tmap_q, q_full, 64, q0 + t * Cfg::BQ, h);
        }
        if (n_kv > 0) {
            const uint32_t fb = kv_full0, sK = sKV, sV = sKV + TILE;
            mbar_arrive_expect_tx(fb, 2 * TILE);
            tma_load_3d(sK, &tmap_k, fb, 0, 0, h);
            tma_load_3d(sK + ATOM, &tmap_k, fb, 64, 0, h);
            tma_load_3d(sV, &tmap_v, fb, 0, 0, h);
            tma_load_3d(sV + ATOM, &tmap_v, fb, 64, 0, h);
        }
    }
    if (warp == 1) {
        tmem_alloc<1>(smem_u32(tmem_slot), Cfg::TMEM_COLS);
        tmem_relinquish<1>();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = *tmem_slot;
    grid_dependency_wait();   // nothing above touched global memory
    grid_dependents_launch();
    const WaitCtl wc{abort_flag, p.err, p.timeout_ns};

    if (warp == 0) {
        // ---------------------------------------------------------------- TMA producer
        if (lane == 0) {
            // Q and key/value block 0 were issued during the set-up (stage 0, phase 0)
            bool ok = true;
            uint32_t issued = n_kv > 0 ? 1u : 0u, issued_parity = 0;
            for (int j = 1; j < n_kv; ++j) {
                const int s = j & 1;
                const uint32_t ph = static_cast<uint32_t>(j >> 1) & 1u;
                if (!wait_bounded(kv_empty0 + 8u * s, ph ^ 1u, wc, ERR_PRODUCER_SLOT)) {
                    ok = false;
                    break;
                }
                const uint32_t fb = kv_full0 + 8u * s;
                const uint32_t sK = sKV + static_cast<uint32_t>(s) * 2u * TILE, sV = sK + TILE;
                mbar_arrive_expect_tx(fb, 2 * TILE);
                tma_load_3d(sK, &tmap_k, fb, 0, j * Cfg::BKV, h);
                tma_load_3d(sK + ATOM, &tmap_k, fb, 64, j * Cfg::BKV, h);
                tma_load_3d(sV, &tmap_v, fb, 0, j * Cfg::BKV, h);
                tma_load_3d(sV + ATOM, &tmap_v, fb, 64, j * Cfg::BKV, h);
                issued |= 1u << s;
                issued_parity = (issued_parity & ~(1u << s)) | (ph << s);
            }
            if (!ok) {   // let every copy this thread started land before the CTA exits
                wait_until(q_full, 0, p.timeout_ns, p.err);
                for (int s = 0; s < Cfg::KV_STAGES; ++s)
                    if (issued & (1u << s))
                        wait_until(kv_full0 + 8u * s, (issued_parity >> s) & 1u, p.timeout_ns, p.err);
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ---------------------------------------------------------------- MMA issuer
        if (lane == 0) {
            constexpr uint32_t ID_QK = idesc_attn<false>(), ID_PV = idesc_attn<true>();
            bool ok = wait_bounded(q_full, 0, wc, ERR_MMA_OPERANDS);
            // S_t = Q_t K_j^T into tile t's score columns
            const uint64_t q_desc0 = kmajor_step_desc(sQ, 0), k_desc0 = kmajor_step_desc(sKV, 0),
                           v_desc0 = v_step_desc(sKV + TILE, 0);
            auto issue_qk = [&](int t, int j) {
                const uint64_t qd = q_desc0 + static_cast<uint64_t>(t * (TILE >> 4));
                const uint64_t kd = k_desc0 + static_cast<uint64_t>((j & 1) * (2 * TILE >> 4));
                const uint32_t d = tmem + static_cast<uint32_t>(Cfg::S_COL + t * Cfg::BQ);
#pragma unroll
                for (int kk = 0; kk < Cfg::D / 16; ++kk) {
                    const uint64_t off = static_cast<uint64_t>(((kk >> 2) * Cfg::ATOM_BYTES + (kk & 3) * 32) >> 4);
                    umma_f16<1>(d, qd + off, kd + off, ID_QK, kk != 0 ? 1u : 0u);
                }
                umma_commit(s_full0 + 8u * t);
            };
            // O_t += P_t V_j, P_t from TMEM (8 columns per 16 keys)
            // (keys 0..63 as soon as their P is written, keys 64..127 once all of it is)
            auto issue_pv = [&](int t, int j) -> bool {
                const uint64_t vd = v_desc0 + static_cast<uint64_t>((j & 1) * (2 * TILE >> 4));
                const uint32_t d = tmem + static_cast<uint32_t>(Cfg::O_COL + t * Cfg::D);
                const uint32_t a = tmem + static_cast<uint32_t>(Cfg::S_COL + t * Cfg::BQ);
                for (int part = 0; part < 2; ++part) {
                    const uint32_t bar = (part == 0 ? p_half0 : p_full0) + 8u * t;
                    if (!wait_bounded(bar, static_cast<uint32_t>(j) & 1u, wc, ERR_MMA_OPERANDS))
                        return false;
                    tc_fence_after_sync();
#pragma unroll
                    for (int kk = 4 * part; kk < 4 * part + 4; ++kk)
                        umma_f16_tmem_a(d, a + 8u * static_cast<uint32_t>(kk), vd + static_cast<uint64_t>(kk * (2048 >> 4)), ID_PV,
                                        (j | kk) != 0 ? 1u : 0u);
                }
                // Tile A's product completes pv_done[0]; tile B's is followed at once by the
                // commit that frees the key/value stage, whose completion serves for it too (one
                // commit fewer per block: each holds the tensor pipe for about 40 cycles).
                if (t == 0)
                    umma_commit(pv_done0);
                return true;
            };
            // the next S_t overwrites P_t: only once this tile's P V product has finished
            auto next_qk = [&](int t, int j) -> bool {
                const uint32_t uj = static_cast<uint32_t>(j);
                if (!(t == 0 ? wait_bounded(pv_done0, uj & 1u, wc, ERR_MMA_ACCUMULATOR)
                             : wait_bounded(kv_empty0 + 8u * (uj & 1u), (uj >> 1) & 1u, wc, ERR_MMA_ACCUMULATOR)))
                    return false;
                tc_fence_after_sync();
                issue_qk(t, j + 1);
                return true;
            };
            if (ok && n_kv > 0) {
                ok = wait_bounded(kv_full0, 0, wc, ERR_MMA_OPERANDS);
                if (ok) {
                    tc_fence_after_sync();
                    issue_qk(0, 0);
                    issue_qk(1, 0);
                }
            }
            // block j of tile t exists for j < n_t[t] (n_t[0] <= n_t[1] = n_kv)
            for (int j = 0; ok && j < n_kv; ++j) {
                if (j < n_t[0] && !issue_pv(0, j)) {
                    ok = false;
                    break;
                }
                if (j + 1 < n_kv) {
                    const int s = (j + 1) & 1;
                    if (!wait_bounded(kv_full0 + 8u * s, static_cast<uint32_t>((j + 1) >> 1) & 1u, wc, ERR_MMA_OPERANDS) ||
                        (j + 1 < n_t[0] && !next_qk(0, j))) {
                        ok = false;
                        break;
                    }
                }
                if (!issue_pv(1, j)) {
                    ok = false;
                    break;
                }
                umma_commit(kv_empty0 + 8u * (j & 1));   // K_j and V_j consumed by both tiles
                if (j + 1 < n_t[1] && !next_qk(1, j)) {
                    ok = false;
                    break;
                }
            }
            if (!ok) {
                umma_commit(drain);
                wait_until(drain, 0, p.timeout_ns, p.err);
            }
        }
        __syncwarp();
    } else {
        // ---------------------------------------------------------------- online softmax
        const int t = (warp - 2) >> 2;   // warps 2..5: tile A, 6..9: tile B
        attention_softmax_warp(p, tmem, t, s_full0 + 8u * t, p_half0 + 8u * t, p_full0 + 8u * t,
                               t == 0 ? pv_done0 : kv_empty0, wc, warp, lane, q0 + t * Cfg::BQ, h,
                               t == 0 ? n_t[0] : n_t[1], sQ + t * TILE, &tmap_o, t != 0);
    }

    tc_fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after_sync();
        tmem_dealloc<1>(tmem, Cfg::TMEM_COLS);
    }
}

}  // namespace gb300
