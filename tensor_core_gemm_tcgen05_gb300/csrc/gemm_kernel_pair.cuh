// CTA-pair variant of the GEMM kernel (tcgen05 cta_group::2), for problems with enough
// output tiles to fill the GPU.
//
// A cluster of two CTAs on neighbouring SMs computes one 256 x BN output tile:
//  * CTA r (r = 0, 1) stages its own half of the operands in its own shared memory: rows
//    [r*128, r*128+128) of the A tile and columns [r*BN/2, (r+1)*BN/2) of the B tile, with
//    the same TMA boxes and 128-byte swizzle as the one-CTA kernel. Nothing is multicast:
//    each CTA reads its halves from global memory itself.
//  * One thread of CTA 0 issues tcgen05.mma.cta_group::2 with M = 256: the tensor cores of
//    both SMs read both CTAs' shared memory, and each CTA's Tensor Memory receives the
//    128 x BN accumulator of its own rows. Per SM this halves the B bytes moved per MMA
//    compared with a 128 x BN tile on one SM, which is what keeps the tensor pipe fed.
//  * Both producers count their bytes on CTA 0's "full" barrier; CTA 0's commits arrive on
//    the "empty" and "accumulator full" barriers of both CTAs (multicast); both CTAs'
//    epilogue warps arrive on CTA 0's "accumulator empty" barrier.
//  * Each CTA's epilogue warps drain their own Tensor Memory exactly as in the one-CTA
//    kernel (epilogue_tile), overlapping the next tile's MMAs (two accumulators).
// Waits are bounded as in the one-CTA kernel; a CTA that gives up also raises the stop
// flag of its peer, and both CTAs meet at a cluster barrier before Tensor Memory is freed.
//
// Work units: pair p takes units p, p + P, p + 2P, ... (P pairs). When the tiles leave a last
// round that at most half of the pairs would work on, the host splits each tile of that round
// into its left and right N-halves (256 x BN/2, UMMA N = BN/2, one B box per CTA), so that
// the round takes half as long and no reduction is needed.
#pragma once

#include "gemm_kernel.cuh"

namespace gb300 {

// STORE_IN_RING_: the output staging boxes overlay the operand ring (launches that give each
// pair at most one work unit: the ring is idle once the accumulator is complete).
template <int BN_, int STAGES_, int EPI_WARPS_ = 4, int BK_ = 64, bool STORE_IN_RING_ = false>
struct PairConfig {
    static constexpr int CTA_BM = 128;     // rows per CTA (= TMEM lanes)
    static constexpr int BM = 256;         // rows per pair tile (= UMMA M)
    static constexpr int BN = BN_;         // columns per tile (= UMMA N)
    static constexpr int CTA_BN = BN / 2;  // B columns staged by each CTA
    // K per ring stage: one or two 64-wide 128-byte swizzle atoms of A (16 KB each per CTA).
    // The MMA thread commits the stage's empty barrier once per stage, and each commit holds
    // the tensor pipe for about 40 cycles, so wider stages issue fewer of them.
    static constexpr int BK = BK_;
    static constexpr int A_ATOM_BYTES = CTA_BM * 64 * 2;
    static constexpr int A_ATOMS = BK / 64;
    static constexpr int UMMA_K = 16;
    static constexpr int STAGES = STAGES_;
    static constexpr bool STORE_IN_RING = STORE_IN_RING_;
    static constexpr int A_BYTES = CTA_BM * BK * 2;
    static constexpr int B_BOX_N = 64;
    static constexpr int B_BOXES = CTA_BN / B_BOX_N;
    static constexpr int B_BOX_BYTES = BK * B_BOX_N * 2;
    static constexpr int B_BYTES = BK * CTA_BN * 2;
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;   // per CTA
    static constexpr int ACC_BUFS = 2;
    static constexpr int TMEM_COLS = ACC_BUFS * BN;
    static constexpr int NUM_EPI_WARPS = EPI_WARPS_;
    static constexpr int EPI_COL_GROUPS = NUM_EPI_WARPS / 4;
    static constexpr int NUM_THREADS = 64 + 32 * NUM_EPI_WARPS;
    static constexpr int NUM_BARS = 2 * STAGES + 2 * ACC_BUFS + 1;
    static constexpr int BIAS_OFFSET = STAGES * STAGE_BYTES + ((NUM_BARS * 8 + 16 + 15) / 16) * 16;
    static constexpr int BIAS_END = BIAS_OFFSET + NUM_EPI_WARPS * BN * 2;
    static constexpr int STORE_OFFSET = STORE_IN_RING ? 0 : ((BIAS_END + 1023) / 1024) * 1024;
    static constexpr int SMEM_BYTES =
        1024 + (STORE_IN_RING ? BIAS_END : STORE_OFFSET + NUM_EPI_WARPS * EPI_STORE_WARP_BYTES);

    static_assert(BN % 128 == 0 && BN >= 128 && BN <= 256, "UMMA N for M = 256, two 64-column boxes per CTA");
    static_assert(BK == 64 || BK == 128, "one or two A atoms per stage; B boxes BK rows tall");
    static_assert(TMEM_COLS == 256 || TMEM_COLS == 512, "TMEM alloc size");
    static_assert(NUM_EPI_WARPS == 4 || NUM_EPI_WARPS == 8 || NUM_EPI_WARPS == 16,
                  "one, two or four warps per TMEM lane quarter");
    static_assert(!STORE_IN_RING || NUM_EPI_WARPS * EPI_STORE_WARP_BYTES <= STAGES * STAGE_BYTES,
                  "output staging fits the operand ring");
    static_assert((BN / 32) % EPI_COL_GROUPS == 0, "column chunks split evenly between warps");
    static_assert(SMEM_BYTES <= 232448, "exceeds the 227 KB per-CTA shared memory limit");
};

// Work unit u: its tile t and which part of it (0: whole, 1: left half, 2: right half).
__device__ __forceinline__ void pair_unit(const GemmParams &p, int u, int &t, int &half)
{
    const int f = p.pair_split_from;
    if (u < f) {
        t = u;
        half = 0;
    } else {
        t = f + ((u - f) >> 1);
        half = 1 + ((u - f) & 1);
    }
}

__device__ __forceinline__ void st_shared_cluster_u32(uint32_t addr, uint32_t v)
{
    asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}

struct PairWaitCtl {
    volatile int *abort;     // this CTA's stop flag
    uint32_t peer_abort;     // the peer's stop flag (shared::cluster address)
    uint32_t *err;
    uint64_t limit_ns;
};

// Bounded wait with cluster-scope acquire (phases may be completed by the peer CTA).
__device__ __forceinline__ bool pair_wait(uint32_t bar, uint32_t parity, const PairWaitCtl &w, uint32_t code)
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
            st_shared_cluster_u32(w.peer_abort, 1u);
            atomicCAS(w.err, 0u, code);
            return false;
        }
    }
}

// The same wait by all 32 lanes of a warp together (see wait_warp): for the epilogue warps,
// which spend most of a tile waiting for the next accumulator. A converged warp polling costs
// fewer issue slots (and less power) than one lane spinning through a branch and a shuffle:
// 8192^3 at the power limit 718 -> 702 us, the MLP problem + bias + GELU 732 -> 722 us.
__device__ __forceinline__ bool pair_wait_warp(uint32_t bar, uint32_t parity, const PairWaitCtl &w, uint32_t code,
                                               int lane)
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
            if (lane == 0) {
                *w.abort = 1;
                st_shared_cluster_u32(w.peer_abort, 1u);
                atomicCAS(w.err, 0u, code);
            }
            return false;
        }
    }
}

template <class Cfg>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(Cfg::NUM_THREADS, 1)
    gemm_tcgen05_pair_kernel(const __grid_constant__ CUtensorMap tmap_a, const __grid_constant__ CUtensorMap tmap_b,
                             const __grid_constant__ CUtensorMap tmap_c, const GemmParams p)
{
    constexpr int BM = Cfg::BM, BN = Cfg::BN, BK = Cfg::BK, STAGES = Cfg::STAGES;
    constexpr uint32_t IDESC = idesc_f16_f32<BM, BN>();
    constexpr uint32_t IDESC_HALF = idesc_f16_f32<BM, BN / 2>();
    static_assert(Cfg::B_BOXES % 2 == 0, "a half tile takes half of each CTA's B boxes");

    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *sp = smem_raw + (base - raw);
    const uint32_t sA = base;
    const uint32_t sB = base + STAGES * Cfg::A_BYTES;
    uint64_t *bars = reinterpret_cast<uint64_t *>(sp + STAGES * Cfg::STAGE_BYTES);
    const uint32_t bar0 = smem_u32(bars);
    const uint32_t full0 = bar0, empty0 = bar0 + 8u * STAGES;
    const uint32_t accf0 = bar0 + 16u * STAGES, acce0 = accf0 + 8u * Cfg::ACC_BUFS;
    const uint32_t drain = acce0 + 8u * Cfg::ACC_BUFS;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + Cfg::NUM_BARS);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    uint4 *bias_stage = reinterpret_cast<uint4 *>(sp + Cfg::BIAS_OFFSET);
    const uint32_t store_stage = base + Cfg::STORE_OFFSET;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();
    const bool leader = rank == 0;
    const int cluster_id = static_cast<int>(blockIdx.x >> 1);
    const int num_clusters = static_cast<int>(gridDim.x >> 1);
    const int num_units = p.pair_units;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(full0 + 8u * s, 1);
            mbar_init(empty0 + 8u * s, 1);
        }
        for (int b = 0; b < Cfg::ACC_BUFS; ++b) {
            mbar_init(accf0 + 8u * b, 1);
            mbar_init(acce0 + 8u * b, 2 * Cfg::NUM_EPI_WARPS);
        }
        mbar_init(drain, 1);
        *abort_flag = 0;
        fence_mbar_init();
        if (p.num_kb > 0) {
            tma_prefetch_desc(&tmap_a);
            tma_prefetch_desc(&tmap_b);
        }
        tma_prefetch_desc(&tmap_c);
    }
    __syncwarp();
    cluster_sync();   // both CTAs' barriers exist before any remote arrive or TMA byte count
    if (warp == 1) {
        tmem_alloc<2>(smem_u32(tmem_slot), Cfg::TMEM_COLS);   // one warp of each CTA, together
        tmem_relinquish<2>();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem_base = *tmem_slot;
    // Everything above (barrier set-up, Tensor Memory allocation, descriptor prefetch) may
    // overlap the previous kernel in the stream; no global memory is touched before this.
    grid_dependency_wait();
    grid_dependents_launch();
    const uint32_t full0_leader = mapa_shared(full0, 0);
    const uint32_t acce0_leader = mapa_shared(acce0, 0);
    const PairWaitCtl wc{abort_flag, mapa_shared(smem_u32(const_cast<int *>(abort_flag)), rank ^ 1u), p.err,
                         p.timeout_ns};

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer (both CTAs)
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0, issued = 0, issued_parity = 0;
            bool ok = true, withhold = leader && (p.debug & DEBUG_WITHHOLD_FIRST_LOAD) != 0;
            for (int u = cluster_id; ok && u < num_units; u += num_clusters) {
                int t, half, mb, nb;
                pair_unit(p, u, t, half);
                tile_coords(p, t, mb, nb);
                // this CTA's B columns: its BN/2 of a whole tile, its BN/4 of a half
                const int b_boxes = half ? Cfg::B_BOXES / 2 : Cfg::B_BOXES;
                const int b_col0 = nb * BN + (half == 2 ? BN / 2 : 0) + static_cast<int>(rank) * b_boxes * Cfg::B_BOX_N;
                const uint32_t tx = 2u * static_cast<uint32_t>(Cfg::A_BYTES + b_boxes * Cfg::B_BOX_BYTES);
                for (int kb = 0; kb < p.num_kb; ++kb) {
                    if (!pair_wait(empty0 + 8u * stage, phase ^ 1u, wc, ERR_PRODUCER_SLOT)) {
                        ok = false;
                        break;
                    }
                    if (withhold) {
                        withhold = false;   // test hook: this slot's operands never arrive
                    } else {
                        const uint32_t fb = full0_leader + 8u * stage;
                        if (leader)   // CTA 0's barrier counts the bytes of both CTAs
                            mbar_arrive_expect_tx(full0 + 8u * stage, tx);
#pragma unroll
                        for (int a = 0; a < Cfg::A_ATOMS; ++a)
                            tma_load_2d_pair(sA + stage * Cfg::A_BYTES + a * Cfg::A_ATOM_BYTES, &tmap_a, fb,
                                             kb * BK + 64 * a, mb * BM + static_cast<int>(rank) * Cfg::CTA_BM);
                        for (int j = 0; j < b_boxes; ++j)
                            tma_load_2d_pair(sB + stage * Cfg::B_BYTES + j * Cfg::B_BOX_BYTES, &tmap_b, fb,
                                             b_col0 + j * Cfg::B_BOX_N, kb * BK);
                        issued |= 1u << stage;
                        issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
                    }
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            if (!ok) {
                if (leader) {   // the full barriers see both CTAs' copies land
                    for (int s = 0; s < STAGES; ++s)
                        if (issued & (1u << s))
                            wait_until(full0 + 8u * s, (issued_parity >> s) & 1u, p.timeout_ns, p.err);
                } else {        // copies land within microseconds; give them a fixed margin
                    const uint64_t t0 = global_timer_ns();
                    while (global_timer_ns() - t0 < 200000ull) {
                    }
                }
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer (CTA 0 only)
        if (leader && lane == 0) {
            // descriptors of stage 0's A and B; steps are constant offsets in the start-address
            // field (A: 32 bytes per 16 K-values within a 64-wide atom, the next atom 16 KB on;
            // B: 2048 bytes per 16 K-rows; one stage apart)
            const uint64_t a_desc0 = sw128_desc(sA, 16, 1024), b_desc0 = sw128_desc(sB, Cfg::B_BOX_BYTES, 1024);
            int stage = 0, acc = 0;
            uint32_t phase = 0, acc_phase = 0;
            bool ok = true;
            for (int u = cluster_id; ok && u < num_units; u += num_clusters) {
                int t, half;
                pair_unit(p, u, t, half);
                const uint32_t idesc = half ? IDESC_HALF : IDESC;   // N = BN/2: one B box per CTA
                if (!pair_wait(acce0 + 8u * acc, acc_phase ^ 1u, wc, ERR_MMA_ACCUMULATOR)) {
                    ok = false;
                    break;
                }
                tc_fence_after_sync();
                const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN);
                for (int kb = 0; kb < p.num_kb; ++kb) {
                    if (!pair_wait(full0 + 8u * stage, phase, wc, ERR_MMA_OPERANDS)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after_sync();
                    const uint64_t a_st = a_desc0 + static_cast<uint64_t>(stage * (Cfg::A_BYTES >> 4));
                    const uint64_t b_st = b_desc0 + static_cast<uint64_t>(stage * (Cfg::B_BYTES >> 4));
#pragma unroll
                    for (int kk = 0; kk < BK / Cfg::UMMA_K; ++kk)
                        umma_f16<2>(d_tmem,
                                    a_st + static_cast<uint64_t>((kk >> 2) * (Cfg::A_ATOM_BYTES >> 4) + 2 * (kk & 3)),
                                    b_st + static_cast<uint64_t>(128 * kk), idesc, (kb | kk) != 0 ? 1u : 0u);
                    umma_commit_pair(empty0 + 8u * stage, 0x3);   // both CTAs' slots are free
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok)
                    break;
                umma_commit_pair(accf0 + 8u * acc, 0x3);          // both CTAs' accumulators done
                if (++acc == Cfg::ACC_BUFS) {
                    acc = 0;
                    acc_phase ^= 1u;
                }
            }
            if (!ok) {
                umma_commit_pair(drain, 0x1);
                wait_until(drain, 0, p.timeout_ns, p.err);
            }
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ epilogue warps (both CTAs)
        const int quarter = warp & 3;
        const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
        constexpr int CHUNKS = BN / 32 / Cfg::EPI_COL_GROUPS;
        const int c_begin = ((warp - 2) >> 2) * CHUNKS;
        uint4 *my_bias = bias_stage + (warp - 2) * (BN / 8);
        const uint32_t my_stage = store_stage + static_cast<uint32_t>(warp - 2) * EPI_STORE_WARP_BYTES;
        uint32_t box_sel = 0;
        int acc = 0;
        uint32_t acc_phase = 0;
        for (int u = cluster_id; u < num_units; u += num_clusters) {
            int t, half, mb, nb;
            pair_unit(p, u, t, half);
            tile_coords(p, t, mb, nb);
            // the unit's first column and width (a half tile's accumulator is columns [0, BN/2))
            const int n0 = nb * BN + (half == 2 ? BN / 2 : 0);
            const int n_end = n0 + (half ? BN / 2 : BN);
            const uint4 bv = bias_fetch(p, n0, lane);
            if (!pair_wait_warp(accf0 + 8u * acc, acc_phase, wc, ERR_EPILOGUE_ACCUMULATOR, lane))
                break;
            tc_fence_after_sync();
            if (p.bias != nullptr) {
                my_bias[lane] = bv;
                __syncwarp();
            }
            epilogue_tile<CHUNKS>(p, tmem_base + lane_base + static_cast<uint32_t>(acc * BN + c_begin * 32),
                                  n0 + c_begin * 32, mb * BM + static_cast<int>(rank) * Cfg::CTA_BM + quarter * 32,
                                  p.bias != nullptr ? my_bias + c_begin * 4 : nullptr, &tmap_c, my_stage, box_sel,
                                  lane, n_end);
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0)
                mbar_arrive_cluster(acce0_leader + 8u * acc);   // CTA 0's MMA may reuse it
            if (++acc == Cfg::ACC_BUFS) {
                acc = 0;
                acc_phase ^= 1u;
            }
        }
        if (lane == 0)
            bulk_wait_group<0>();   // every output box of this warp has reached global memory
        __syncwarp();
    }

    tc_fence_before_sync();
    __syncthreads();
    cluster_sync();   // the pair's MMAs and remote arrivals are over before TMEM is freed
    if (warp == 1) {
        tc_fence_after_sync();
        tmem_dealloc<2>(tmem_base, Cfg::TMEM_COLS);
    }
}

}  // namespace gb300
