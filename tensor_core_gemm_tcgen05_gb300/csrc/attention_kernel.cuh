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
//  * one CTA per (head, block of 128 queries); the blocks with the most keys (causal) start
//    first;
//  * warp 0: TMA producer. Q once (two 128-byte-swizzled K-major atoms of 64 head dims), then
//    K and V blocks of 128 keys through a two-stage ring; 3-D tensor maps [head][row][dim] so
//    rows past the sequence read as zero;
//  * warp 1: MMA issuer. S_j = Q K_j^T (M = N = 128, K = 128, both operands K-major) into one
//    of two TMEM score buffers, so that S_{j+1} is computed while the softmax of block j
//    runs; then O += P_j V_j (P K-major from shared memory, V MN-major) into a TMEM FP32
//    accumulator;
//  * warps 2..5: online softmax. Each thread owns one query row (its TMEM lane). Per block it
//    reads its 128 scores from TMEM, takes the row maximum, rescales the row of O in TMEM by
//    exp(m_old - m_new) when the maximum grew, writes p = exp(s - m_new) as FP16 into the
//    shared-memory P tile (the K-major 128-byte-swizzled layout the MMA reads) and keeps the
//    running sum l; at the end it writes O / l.
// Every mbarrier wait is bounded in time, as in the GEMM kernels.
#pragma once

#include "gemm_kernel.cuh"

namespace gb300 {

// 2^x with the MUFU.EX2 instruction (flushes denormal results to zero, which only affects
// probabilities below 2^-126, far under FP16's smallest value).
__device__ __forceinline__ float fast_exp2(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// A row's running maximum is raised (and its row of O rescaled) only when a block's maximum
// exceeds it by more than this many base-2 units; otherwise probabilities are taken against
// the old maximum and stay below 2^8, well inside FP16 and FP32.
constexpr float kRescaleThreshold = 8.0f;

struct AttnParams {
    int H;              // heads (batch x heads)
    int Sq, Sk;         // query and key lengths
    int q_blocks;       // ceil(Sq / 128)
    int causal;
    float scale_log2;   // scale * log2(e): scores are kept in base-2 units
    __half *O;          // [H][Sq][128]
    uint32_t *err;
    uint64_t timeout_ns;
};

struct AttnConfig {
    static constexpr int D = 128;         // head dimension
    static constexpr int BQ = 128;        // queries per CTA (= TMEM lanes)
    static constexpr int BKV = 128;       // keys per block
    static constexpr int ATOM_BYTES = 128 * 128;   // 128 rows x 64 FP16 (one 128-byte swizzle row each)
    static constexpr int TILE_BYTES = 2 * ATOM_BYTES;  // 128 x 128 FP16
    static constexpr int KV_STAGES = 2;
    // shared memory: Q | K[0] V[0] | K[1] V[1] | P | barriers
    static constexpr int Q_OFF = 0;
    static constexpr int KV_OFF = TILE_BYTES;
    static constexpr int P_OFF = KV_OFF + KV_STAGES * 2 * TILE_BYTES;
    static constexpr int BAR_OFF = P_OFF + TILE_BYTES;
    // barriers: q_full, kv_full[2], kv_empty[2], s_full[2], s_empty[2], p_full, pv_done, drain
    static constexpr int NUM_BARS = 1 + 2 * KV_STAGES + 2 * 2 + 3;
    static constexpr int SMEM_BYTES = 1024 + BAR_OFF + NUM_BARS * 8 + 16;
    static constexpr int NUM_THREADS = 192;
    static constexpr int TMEM_COLS = 512;   // S0 | S1 | O (128 columns each)
    static constexpr int S_COL = 0, O_COL = 256;
    static_assert(SMEM_BYTES <= 232448, "exceeds the 227 KB per-CTA shared memory limit");
};

// Instruction descriptor, kind::f16, FP32 accumulate, FP16 operands, M = N = 128.
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

// Online softmax of one epilogue warp (warps 2..5): each thread owns query row r of the
// block (TMEM lane r). Per key block j: (1) read the 128 scores of the row and take their
// maximum (base-2 units; keys past the sequence, or after the query when causal, are left
// out); (2) once the previous P V product has finished, rescale the row of O in TMEM by
// 2^(m_old - m_new) if the maximum grew by more than kRescaleThreshold (skipped when no row
// of the warp needs it); (3) read
// the scores again and write p = 2^(s - m_new) as FP16 into the P tile, K-major with the
// 128-byte swizzle (16-byte piece c of row r at atom (c / 8), r * 128 + ((c % 8) ^ (r % 8)) * 16),
// summing p into the running denominator l. At the end the row of O is divided by l.
__device__ __forceinline__ void attention_softmax_warp(const AttnParams &p, uint32_t tmem, uint32_t sP,
                                                       uint32_t s_full0, uint32_t s_empty0, uint32_t p_full,
                                                       uint32_t pv_done, const WaitCtl &wc, int warp, int lane,
                                                       int q0, int h, int n_kv)
{
    using Cfg = AttnConfig;
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;
    const int qi = q0 + r;
    const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t o_addr = tmem + lane_base + Cfg::O_COL;
    const int kmax = p.causal ? min(p.Sk - 1, qi) : p.Sk - 1;   // last key this row sees
    float m = -INFINITY, l = 0.0f;
    uint32_t v[32], va[32], vb[32];
    for (int j = 0; j < n_kv; ++j) {
        const int b = j & 1;
        int w = 1;
        if (lane == 0)
            w = wait_bounded(s_full0 + 8u * b, static_cast<uint32_t>(j >> 1) & 1u, wc, ERR_EPILOGUE_ACCUMULATOR) ? 1 : 0;
        if (!__shfl_sync(0xffffffffu, w, 0))
            return;
        tc_fence_after_sync();
        const uint32_t s_addr = tmem + lane_base + Cfg::S_COL + static_cast<uint32_t>(b) * 128u;
        const int k0 = j * Cfg::BKV;
        float mb = -INFINITY;
        auto max_chunk = [&](const uint32_t(&x)[32], int c) {
#pragma unroll
            for (int e = 0; e < 32; ++e) {
                const float t = __uint_as_float(x[e]) * p.scale_log2;
                mb = (k0 + 32 * c + e <= kmax) ? fmaxf(mb, t) : mb;
            }
        };
        two_buffered_chunks(s_addr, va, vb, max_chunk);
        // keep the old maximum unless this block's exceeds it by more than the threshold
        const bool raise = mb > m + kRescaleThreshold || m == -INFINITY;
        const float m_new = raise ? mb : m;
        const float m_use = m_new == -INFINITY ? 0.0f : m_new;
        const float alpha = raise ? fast_exp2(m - m_use) : 1.0f;   // 0 on the first block (m = -inf)
        if (j > 0) {
            if (lane == 0)
                w = wait_bounded(pv_done, static_cast<uint32_t>(j - 1) & 1u, wc, ERR_EPILOGUE_ACCUMULATOR) ? 1 : 0;
            if (!__shfl_sync(0xffffffffu, w, 0))
                return;
            tc_fence_after_sync();
            if (__any_sync(0xffffffffu, alpha != 1.0f)) {
#pragma unroll 1
                for (int c = 0; c < 4; ++c) {
                    tmem_ld_32x32b_x32(o_addr + 32u * c, v);
                    tmem_ld_wait_regs(v);
#pragma unroll
                    for (int e = 0; e < 32; ++e)
                        v[e] = __float_as_uint(__uint_as_float(v[e]) * alpha);
                    tmem_st_32x32b_x32(o_addr + 32u * c, v);
                    tmem_st_wait();
                }
            }
        }
        float sum = 0.0f;
        auto p_chunk = [&](const uint32_t(&x)[32], int c) {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                uint32_t pk[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int idx = 8 * i + 2 * e;
                    const int k = k0 + 32 * c + idx;
                    const float p0 = k <= kmax ? fast_exp2(fmaf(__uint_as_float(x[idx]), p.scale_log2, -m_use)) : 0.0f;
                    const float p1 =
                        k + 1 <= kmax ? fast_exp2(fmaf(__uint_as_float(x[idx + 1]), p.scale_log2, -m_use)) : 0.0f;
                    sum += p0 + p1;
                    __half2 hh = __floats2half2_rn(p0, p1);
                    pk[e] = *reinterpret_cast<uint32_t *>(&hh);
                }
                const int kc = 4 * c + i;   // 16-byte piece of the row: keys 8kc .. 8kc+7
                const uint32_t addr = sP + static_cast<uint32_t>(kc >> 3) * Cfg::ATOM_BYTES +
                                      static_cast<uint32_t>(r) * 128u +
                                      ((static_cast<uint32_t>(kc & 7) ^ static_cast<uint32_t>(r & 7)) << 4);
                st_shared_v4(addr, make_uint4(pk[0], pk[1], pk[2], pk[3]));
            }
        };
        two_buffered_chunks(s_addr, va, vb, p_chunk);
        l = l * alpha + sum;
        m = m_new;
        fence_proxy_async_shared();   // P is read by the tensor cores (async proxy)
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) {
            mbar_arrive(s_empty0 + 8u * b);   // score buffer b may be overwritten
            mbar_arrive(p_full);              // P tile ready, O rescaled
        }
    }
    if (n_kv == 0)
        return;
    int w = 1;
    if (lane == 0)
        w = wait_bounded(pv_done, static_cast<uint32_t>(n_kv - 1) & 1u, wc, ERR_EPILOGUE_ACCUMULATOR) ? 1 : 0;
    if (!__shfl_sync(0xffffffffu, w, 0))
        return;
    tc_fence_after_sync();
    const float inv = l > 0.0f ? 1.0f / l : 0.0f;
    __half *orow = p.O + (static_cast<int64_t>(h) * p.Sq + qi) * Cfg::D;
#pragma unroll 1
    for (int c = 0; c < 4; ++c) {
        tmem_ld_32x32b_x32(o_addr + 32u * c, v);
        tmem_ld_wait_regs(v);
        if (qi < p.Sq) {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                uint32_t pk[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    __half2 hh = __floats2half2_rn(__uint_as_float(v[8 * i + 2 * e]) * inv,
                                                   __uint_as_float(v[8 * i + 2 * e + 1]) * inv);
                    pk[e] = *reinterpret_cast<uint32_t *>(&hh);
                }
                *reinterpret_cast<uint4 *>(orow + 32 * c + 8 * i) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
            }
        }
    }
}

__global__ void __launch_bounds__(AttnConfig::NUM_THREADS, 1)
    attention_fwd_kernel(const __grid_constant__ CUtensorMap tmap_q, const __grid_constant__ CUtensorMap tmap_k,
                         const __grid_constant__ CUtensorMap tmap_v, const AttnParams p)
{
    using Cfg = AttnConfig;
    constexpr uint32_t ATOM = Cfg::ATOM_BYTES, TILE = Cfg::TILE_BYTES;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *sp = smem_raw + (base - raw);
    const uint32_t sQ = base + Cfg::Q_OFF, sKV = base + Cfg::KV_OFF, sP = base + Cfg::P_OFF;
    const uint32_t q_full = base + Cfg::BAR_OFF;
    const uint32_t kv_full0 = q_full + 8u, kv_empty0 = kv_full0 + 8u * Cfg::KV_STAGES;
    const uint32_t s_full0 = kv_empty0 + 8u * Cfg::KV_STAGES, s_empty0 = s_full0 + 16u;
    const uint32_t p_full = s_empty0 + 16u, pv_done = p_full + 8u, drain = pv_done + 8u;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sp + Cfg::BAR_OFF + Cfg::NUM_BARS * 8);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    // work item: query block qb of head h; the blocks with the most keys go first
    const int qb = p.q_blocks - 1 - static_cast<int>(blockIdx.x / static_cast<unsigned>(p.H));
    const int h = static_cast<int>(blockIdx.x % static_cast<unsigned>(p.H));
    const int q0 = qb * Cfg::BQ;
    const int k_end = p.causal ? min(p.Sk, q0 + Cfg::BQ) : p.Sk;   // keys any row of the block may see
    const int n_kv = (k_end + Cfg::BKV - 1) / Cfg::BKV;

    if (threadIdx.x == 0) {
        mbar_init(q_full, 1);
        for (int s = 0; s < Cfg::KV_STAGES; ++s) {
            mbar_init(kv_full0 + 8u * s, 1);
            mbar_init(kv_empty0 + 8u * s, 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(s_full0 + 8u * b, 1);
            mbar_init(s_empty0 + 8u * b, 4);
        }
        mbar_init(p_full, 4);
        mbar_init(pv_done, 1);
        mbar_init(drain, 1);
        *abort_flag = 0;
        fence_mbar_init();
        tma_prefetch_desc(&tmap_q);
        tma_prefetch_desc(&tmap_k);
        tma_prefetch_desc(&tmap_v);
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
            mbar_arrive_expect_tx(q_full, TILE);
            tma_load_3d(sQ, &tmap_q, q_full, 0, q0, h);
            tma_load_3d(sQ + ATOM, &tmap_q, q_full, 64, q0, h);
            bool ok = true;
            uint32_t issued = 0, issued_parity = 0;
            for (int j = 0; j < n_kv; ++j) {
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
            // S_j = Q K_j^T into score buffer j % 2
            auto issue_qk = [&](int j) -> bool {
                const int s = j & 1;
                const uint32_t ph = static_cast<uint32_t>(j >> 1) & 1u;
                if (!wait_bounded(kv_full0 + 8u * s, ph, wc, ERR_MMA_OPERANDS))
                    return false;
                if (!wait_bounded(s_empty0 + 8u * s, ph ^ 1u, wc, ERR_MMA_ACCUMULATOR))
                    return false;
                tc_fence_after_sync();
                const uint32_t sK = sKV + static_cast<uint32_t>(s) * 2u * TILE;
                const uint32_t d = tmem + Cfg::S_COL + static_cast<uint32_t>(s) * 128u;
#pragma unroll
                for (int kk = 0; kk < Cfg::D / 16; ++kk)
                    umma_f16<1>(d, kmajor_step_desc(sQ, kk), kmajor_step_desc(sK, kk), ID_QK, kk != 0 ? 1u : 0u);
                umma_commit(s_full0 + 8u * s);
                return true;
            };
            if (ok && n_kv > 0)
                ok = issue_qk(0);
            for (int j = 0; ok && j < n_kv; ++j) {
                if (j + 1 < n_kv && !issue_qk(j + 1)) {   // the next scores overlap this softmax
                    ok = false;
                    break;
                }
                if (!wait_bounded(p_full, static_cast<uint32_t>(j) & 1u, wc, ERR_MMA_OPERANDS)) {
                    ok = false;
                    break;
                }
                tc_fence_after_sync();
                const uint32_t sV = sKV + static_cast<uint32_t>(j & 1) * 2u * TILE + TILE;
#pragma unroll
                for (int kk = 0; kk < Cfg::BKV / 16; ++kk)
                    umma_f16<1>(tmem + Cfg::O_COL, kmajor_step_desc(sP, kk), v_step_desc(sV, kk), ID_PV,
                                (j | kk) != 0 ? 1u : 0u);
                umma_commit(pv_done);                   // O updated, P tile free
                umma_commit(kv_empty0 + 8u * (j & 1));  // K_j and V_j consumed
            }
            if (!ok) {
                umma_commit(drain);
                wait_until(drain, 0, p.timeout_ns, p.err);
            }
        }
        __syncwarp();
    } else {
        // ---------------------------------------------------------------- online softmax
        attention_softmax_warp(p, tmem, sP, s_full0, s_empty0, p_full, pv_done, wc, warp, lane, q0, h, n_kv);
    }

    tc_fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after_sync();
        tmem_dealloc<1>(tmem, Cfg::TMEM_COLS);
    }
}

}  // namespace gb300
