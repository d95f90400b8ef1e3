// GEMM with a row-softmax epilogue for sm_103a (GB300):
//
//     C[r][:] = softmax over the row of (A[M x K] * B[K x N] + bias[N])     FP16 in and out
//
// "Designing High-Performance GPU Kernels with TileLang" (spaxe.top), fused-softmax
// paragraph: the row-wise softmax is applied to the GEMM result inside the kernel, and no
// intermediate (logits, row statistics) is written to global memory. The logits stay in
// FP32 (Tensor Memory, then registers); C is written once.
//
// Same operand path as the GEMM kernel (TMA producer warp, 128-byte-swizzled ring, one MMA
// thread issuing tcgen05.mma into two 128 x 256 FP32 accumulators in TMEM), with sixteen
// epilogue warps: four per TMEM lane quarter, each owning 64 of a tile's 256 columns for its
// 32 rows (one row per thread). A thread reads its 64 logits from TMEM with one pair of
// loads, releases the accumulator, and works on registers only.
//
// Work: a thread-block cluster of CS CTAs owns a 128-row block at a time (row blocks
// clusterid, clusterid + clusters, ...); CTA r owns the column tiles [r*span, (r+1)*span).
//  * One tile per row (N <= 256, CS = 1): the tile's row maximum and sum of exponentials are
//    merged over the four column groups through shared memory, and each thread scales the
//    exponentials it already holds: one exponential per element.
//  * Wider rows: each CTA sweeps its tiles twice. Pass 1 keeps a running (maximum, sum of
//    2^(x - maximum)) per row and thread (the online form of the row statistics); the
//    statistics are merged over the column groups, then over the cluster's CTAs through
//    distributed shared memory, once per row block. Pass 2 recomputes each tile's logits
//    (the tensor cores' cost is small next to the epilogue's when K is small) and writes
//    exp(x - max) / sum. No width limit: only row statistics cross CTAs.
//
// Every wait is bounded in time (the error word records which one ran out); the column-group
// merge uses mbarriers, not bar.sync, so that a warp that gives up cannot strand the others.
#pragma once

#include "gemm_kernel.cuh"

namespace gb300 {

template <int STAGES_>
struct SoftmaxConfig {
    static constexpr int BM = 128, BN = 256, BK = 64, UMMA_K = 16;
    static constexpr int STAGES = STAGES_;
    static constexpr int A_BYTES = BM * BK * 2;
    static constexpr int B_BOX_N = 64;
    static constexpr int B_BOXES = BN / B_BOX_N;
    static constexpr int B_BOX_BYTES = BK * B_BOX_N * 2;
    static constexpr int B_BYTES = BK * BN * 2;
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
    static constexpr int ACC_BUFS = 2;
    static constexpr int TMEM_COLS = ACC_BUFS * BN;
    static constexpr int NUM_EPI_WARPS = 16;
    static constexpr int GROUPS = 4;                    // epilogue warps per TMEM lane quarter
    static constexpr int WARP_COLS = BN / GROUPS;       // 64 columns per epilogue warp
    static constexpr int NUM_THREADS = 64 + 32 * NUM_EPI_WARPS;
    // full[s], empty[s], acc_full[b], acc_empty[b], drain, group[4 quarters],
    // stats_ready[2], stats_read[2]
    static constexpr int NUM_BARS = 2 * STAGES + 2 * ACC_BUFS + 1 + 4 + 4;
    // after the ring: barriers, TMEM address, stop flag; then each epilogue warp's 64 bias
    // values (FP16, 128 bytes)
    static constexpr int BIAS_OFFSET = STAGES * STAGE_BYTES + ((NUM_BARS * 8 + 16 + 15) / 16) * 16;
    // then, 1024-aligned, one 32 x 64 FP16 output staging box per epilogue warp (128-byte
    // swizzle; C's tensor map has 64 x 32 boxes)
    static constexpr int STORE_BOX_BYTES = 32 * WARP_COLS * 2;
    static constexpr int STORE_OFFSET = ((BIAS_OFFSET + NUM_EPI_WARPS * WARP_COLS * 2 + 1023) / 1024) * 1024;
    // then the column-group statistics: [2 buffers][4 quarters][4 groups][32 lanes] (max, sum)
    static constexpr int GROUP_OFFSET = STORE_OFFSET + NUM_EPI_WARPS * STORE_BOX_BYTES;
    // then the cluster statistics of this CTA: [2 buffers][128 rows] (max, sum)
    static constexpr int CLUSTER_OFFSET = GROUP_OFFSET + 2 * 4 * GROUPS * 32 * 8;
    static constexpr int SMEM_BYTES = 1024 /* alignment slack */ + CLUSTER_OFFSET + 2 * BM * 8;

    static_assert(WARP_COLS == 64, "two 32-column chunks per epilogue warp, 128-byte output rows");
    static_assert(STORE_BOX_BYTES % 1024 == 0, "128-byte-swizzled boxes start 1024-byte aligned");
    static_assert(SMEM_BYTES <= 232448, "exceeds the 227 KB per-CTA shared memory limit");
};

// Both 32-register halves of a 64-column TMEM read are ready after tmem_ld_wait_regs on the
// first (the wait covers every earlier load); this ties the second half's registers to that
// point as well (no instruction).
__device__ __forceinline__ void regs_after_wait(uint32_t (&r)[32])
{
    asm volatile(""
                 : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]),
                   "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]),
                   "+r"(r[14]), "+r"(r[15]), "+r"(r[16]), "+r"(r[17]), "+r"(r[18]), "+r"(r[19]),
                   "+r"(r[20]), "+r"(r[21]), "+r"(r[22]), "+r"(r[23]), "+r"(r[24]), "+r"(r[25]),
                   "+r"(r[26]), "+r"(r[27]), "+r"(r[28]), "+r"(r[29]), "+r"(r[30]), "+r"(r[31])
                 :
                 : "memory");
}

// Maximum of 32 values.
__device__ __forceinline__ float max32(const float *v)
{
    float q[4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
        q[i] = fmax3(v[8 * i], v[8 * i + 1], v[8 * i + 2]);
#pragma unroll
    for (int i = 0; i < 4; ++i)
        q[i] = fmax3(q[i], v[8 * i + 3], v[8 * i + 4]);
#pragma unroll
    for (int i = 0; i < 4; ++i)
        q[i] = fmax3(q[i], v[8 * i + 5], v[8 * i + 6]);
#pragma unroll
    for (int i = 0; i < 4; ++i)
        q[i] = fmaxf(q[i], v[8 * i + 7]);
    return fmaxf(fmax3(q[0], q[1], q[2]), q[3]);
}

// 32 logits of this thread, x = acc + bias (FP32); columns at or past N are -inf (they
// contribute 2^-inf = 0). `sbias`: the 32 bias values of these columns as four 16-byte
// vectors (or nullptr).
__device__ __forceinline__ void logits(const uint32_t (&r)[32], const uint4 *sbias, int n_first, int N, float *v)
{
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
                const int j = 8 * i + 2 * e;
                const float2 f = __half22float2(bh[e]);
                f32x2_unpack(f32x2_add(f32x2_pack(v[j], v[j + 1]), f32x2_pack(f.x, f.y)), v[j], v[j + 1]);
            }
        }
    }
    if (n_first + 32 > N) {
#pragma unroll
        for (int j = 0; j < 32; ++j)
            if (n_first + j >= N)
                v[j] = -INFINITY;
    }
}

constexpr float kSmxLog2e = 1.4426950408889634f;

// v = 2^(v * log2(e) + off) in place for 32 values (one packed FMA per pair, then the
// exponentials), returning their sum (two packed partial sums).
__device__ __forceinline__ float exp2_fma_sum(float *v, float off)
{
    const uint64_t l2e = f32x2_pack(kSmxLog2e, kSmxLog2e), o = f32x2_pack(off, off);
    uint64_t sa = f32x2_pack(0.0f, 0.0f), sb = sa;
#pragma unroll
    for (int j = 0; j < 32; j += 2) {
        float d0, d1;
        f32x2_unpack(f32x2_fma(f32x2_pack(v[j], v[j + 1]), l2e, o), d0, d1);
        v[j] = ex2_approx(d0);
        v[j + 1] = ex2_approx(d1);
        if ((j & 2) == 0)
            sa = f32x2_add(sa, f32x2_pack(v[j], v[j + 1]));
        else
            sb = f32x2_add(sb, f32x2_pack(v[j], v[j + 1]));
    }
    float s0, s1;
    f32x2_unpack(f32x2_add(sa, sb), s0, s1);
    return s0 + s1;
}

// v = 2^(v * log2(e) + off) in place for 32 values, no sum.
__device__ __forceinline__ void exp2_fma(float *v, float off)
{
    const uint64_t l2e = f32x2_pack(kSmxLog2e, kSmxLog2e), o = f32x2_pack(off, off);
#pragma unroll
    for (int j = 0; j < 32; j += 2) {
        float d0, d1;
        f32x2_unpack(f32x2_fma(f32x2_pack(v[j], v[j + 1]), l2e, o), d0, d1);
        v[j] = ex2_approx(d0);
        v[j + 1] = ex2_approx(d1);
    }
}

// Merge N (maximum, sum) pairs in base-2 units, in index order, without branches: M is the
// largest maximum, S = sum of s_i 2^(m_i - M). A pair with m = -inf has s = 0 and adds 0.
template <int N>
__device__ __forceinline__ void merge_pairs(const float2 (&o)[N], float &m, float &s)
{
    float M = o[0].x;
#pragma unroll
    for (int i = 1; i < N; ++i)
        M = fmaxf(M, o[i].x);
    const float Ms = M == -INFINITY ? 0.0f : M;   // (no pair with a finite maximum)
    float S = 0.0f;
#pragma unroll
    for (int i = 0; i < N; ++i)
        S = fmaf(o[i].y, ex2_approx(o[i].x - Ms), S);
    m = M;
    s = S;
}

// Scale 32 FP32 values (SCALE) or take them as they are, round to FP16 and write them as half
// `h` (columns 32h..32h+31) of this thread's row of the warp's 32 x 64 staging box (128-byte
// rows, 128-byte swizzle: 16-byte piece i of row r at r*128 + (i ^ (r & 7))*16, which also
// spreads each quarter-warp's writes over all banks).
template <bool SCALE>
__device__ __forceinline__ void stage_row(const float *v, float scale, uint32_t box, int h, int lane)
{
    const uint64_t sc = f32x2_pack(scale, scale);
    const uint32_t row_base = box + static_cast<uint32_t>(lane) * 128u;
    const uint32_t sw = static_cast<uint32_t>(lane & 7);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        uint32_t w[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int j = 8 * i + 2 * e;
            float a = v[j], b = v[j + 1];
            if constexpr (SCALE)
                f32x2_unpack(f32x2_mul(f32x2_pack(a, b), sc), a, b);
            __half2 hv = __floats2half2_rn(a, b);
            w[e] = *reinterpret_cast<uint32_t *>(&hv);
        }
        st_shared_v4(row_base + (((static_cast<uint32_t>(4 * h + i)) ^ sw) << 4), make_uint4(w[0], w[1], w[2], w[3]));
    }
}

// Before the warp refills its staging box: the stores that last used them have read them.
__device__ __forceinline__ void staging_free(int lane)
{
    if (lane == 0)
        bulk_wait_group_read<0>();
    __syncwarp();
}

// Send the warp's staged 32 x 64 box with one TMA store to columns n_first.., rows row0..
// (the store clips rows >= M and columns >= N).
__device__ __forceinline__ void store_box(uint32_t stage, const CUtensorMap *tmap_c, int n_first, int row0, int lane)
{
    fence_proxy_async_shared();
    __syncwarp();
    if (lane == 0) {
        tma_store_2d(tmap_c, stage, n_first, row0, l2_policy_evict_first());
        bulk_commit_group();
    }
}

// Merge a row's (max, sum) over the four column-group warps of a lane quarter: each writes
// its pair, arrives on the quarter's mbarrier (count 4) and waits for the phase; then every
// warp merges the four pairs in group order, so all four get the same result bit for bit.
// Slots are double-buffered by merge count; a warp cannot reach merge i + 2 before all four
// have passed merge i + 1, hence finished reading merge i. False if the wait ran out.
__device__ __forceinline__ bool group_merge(uint32_t slots, uint32_t bar, uint32_t count, int quarter, int group,
                                            int lane, float &m, float &s, const WaitCtl &wc)
{
    const uint32_t buf = count & 1u;
    const uint32_t base = slots + ((buf * 4u + static_cast<uint32_t>(quarter)) * 4u * 32u) * 8u;
    st_shared_f2(base + (static_cast<uint32_t>(group) * 32u + static_cast<uint32_t>(lane)) * 8u, m, s);
    __syncwarp();
    if (lane == 0)
        mbar_arrive(bar);   // release: the pairs above
    if (!wait_warp(bar, count & 1u, wc, ERR_ROW_EXCHANGE, lane))
        return false;
    float2 o[4];
#pragma unroll
    for (int g = 0; g < 4; ++g)
        o[g] = ld_shared_f2(base + (static_cast<uint32_t>(g) * 32u + static_cast<uint32_t>(lane)) * 8u);
    merge_pairs<4>(o, m, s);
    return true;
}

// Merge the CTA's row statistics with those of the other CTAs of the cluster (cs > 1):
// the group-0 warp of each lane quarter writes its rows' pairs to this CTA's buffer `buf`
// and arrives on every CTA's stats_ready[buf] (lane r on CTA r); every epilogue warp of
// every CTA waits for its own stats_ready[buf], reads all CTAs' pairs for its row over
// distributed shared memory, merges them in rank order (the same result everywhere) and
// arrives on every CTA's stats_read[buf]. A buffer is rewritten (two row blocks later) only
// after every reader has arrived. False if a wait ran out.
__device__ __forceinline__ bool cluster_merge(uint32_t stats, uint32_t ready0, uint32_t read0, uint32_t unit, int cs,
                                              int group, int row, int lane, float &m, float &s, const WaitCtl &wc)
{
    const uint32_t buf = unit & 1u, use = unit >> 1;
    const uint32_t slot = stats + (buf * 128u + static_cast<uint32_t>(row)) * 8u;
    int ok = 1;
    if (group == 0) {
        if (use > 0 && lane == 0)   // every reader is done with what this buffer held before
            ok = wait_cluster_bounded(read0 + 8u * buf, (use - 1u) & 1u, wc, ERR_ROW_EXCHANGE) ? 1 : 0;
        if (!__shfl_sync(0xffffffffu, ok, 0))
            return false;
        st_shared_f2(slot, m, s);
        __syncwarp();
        if (lane < cs)   // release: the pairs above
            mbar_arrive_cluster(mapa_shared(ready0 + 8u * buf, static_cast<uint32_t>(lane)));
    }
    if (lane == 0)
        ok = wait_cluster_bounded(ready0 + 8u * buf, use & 1u, wc, ERR_ROW_EXCHANGE) ? 1 : 0;
    if (!__shfl_sync(0xffffffffu, ok, 0))
        return false;
    float2 v[8];   // cs <= 8; ranks past cs read as (-inf, 0)
#pragma unroll
    for (int r = 0; r < 8; ++r)
        v[r] = r < cs ? ld_shared_cluster_f2(mapa_shared(slot, static_cast<uint32_t>(r))) : make_float2(-INFINITY, 0.0f);
    merge_pairs<8>(v, m, s);
    __syncwarp();
    if (lane < cs)   // release: the reads above
        mbar_arrive_cluster(mapa_shared(read0 + 8u * buf, static_cast<uint32_t>(lane)));
    return true;
}

// The CTA's tiles: row blocks clusterid, clusterid + clusters, ...; per row block, PASSES
// sweeps over the column tiles [rank * span, min((rank + 1) * span, n_blocks)).
struct SoftmaxWork {
    int rb, rb_step, j0, j1, passes;
    __device__ explicit SoftmaxWork(const GemmParams &p)
    {
        rb = static_cast<int>(cluster_id_x());
        rb_step = static_cast<int>(cluster_count_x());
        j0 = static_cast<int>(cluster_ctarank()) * p.smx_span;
        j1 = min(j0 + p.smx_span, p.n_blocks);
        passes = p.smx_two_pass ? 2 : 1;
    }
};

// Launched in clusters of p.row_cluster CTAs (1 allowed); p.n_blocks = ceil(N / 256),
// p.smx_span column tiles per CTA. TWO_PASS = p.smx_two_pass: false only for N <= 256 with
// one CTA per row block (a template argument, so that each form is compiled for its own
// register needs).
template <class Cfg, bool TWO_PASS>
__global__ void __launch_bounds__(Cfg::NUM_THREADS, 1)
    gemm_softmax_kernel(const __grid_constant__ CUtensorMap tmap_a, const __grid_constant__ CUtensorMap tmap_b,
                        const __grid_constant__ CUtensorMap tmap_c, const GemmParams p)
{
    constexpr int BM = Cfg::BM, BN = Cfg::BN, BK = Cfg::BK, STAGES = Cfg::STAGES;
    constexpr uint32_t IDESC = idesc_f16_f32<BM, BN>();

    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;   // swizzled tiles need 1024-byte alignment
    uint8_t *sp = smem_raw + (base - raw);
    const uint32_t sA = base;
    const uint32_t sB = base + STAGES * Cfg::A_BYTES;
    uint64_t *bars = reinterpret_cast<uint64_t *>(sp + STAGES * Cfg::STAGE_BYTES);
    const uint32_t bar0 = smem_u32(bars);
    const uint32_t full0 = bar0, empty0 = bar0 + 8u * STAGES;
    const uint32_t accf0 = bar0 + 16u * STAGES, acce0 = accf0 + 8u * Cfg::ACC_BUFS;
    const uint32_t drain = acce0 + 8u * Cfg::ACC_BUFS, group0 = drain + 8u;
    const uint32_t ready0 = group0 + 32u, read0 = ready0 + 16u;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + Cfg::NUM_BARS);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    uint4 *bias_stage = reinterpret_cast<uint4 *>(sp + Cfg::BIAS_OFFSET);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int cs = p.row_cluster;

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
        for (int q = 0; q < 4; ++q)
            mbar_init(group0 + 8u * q, Cfg::GROUPS);
        for (int b = 0; b < 2; ++b) {
            mbar_init(ready0 + 8u * b, static_cast<uint32_t>(cs * 4));   // group-0 warps of every CTA
            mbar_init(read0 + 8u * b, static_cast<uint32_t>(cs * Cfg::NUM_EPI_WARPS));
        }
        *abort_flag = 0;
        fence_mbar_init();
        if (p.num_kb > 0) {
            tma_prefetch_desc(&tmap_a);
            tma_prefetch_desc(&tmap_b);
        }
        tma_prefetch_desc(&tmap_c);
    }
    __syncwarp();
    cluster_sync();   // every CTA's barriers exist before any remote arrival
    if (warp == 1) {
        tmem_alloc<1>(smem_u32(tmem_slot), Cfg::TMEM_COLS);
        tmem_relinquish<1>();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem_base = *tmem_slot;
    // Everything above may overlap the previous kernel in the stream; no global memory is
    // touched before this.
    grid_dependency_wait();
    grid_dependents_launch();
    const WaitCtl wc{abort_flag, p.err, p.timeout_ns};
    const SoftmaxWork work(p);

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0, issued = 0, issued_parity = 0;
            bool ok = true, withhold = (p.debug & DEBUG_WITHHOLD_FIRST_LOAD) != 0;
            for (int rb = work.rb; ok && rb < p.m_blocks; rb += work.rb_step)
                for (int pass = 0; ok && pass < work.passes; ++pass)
                    for (int j = work.j0; ok && j < work.j1; ++j)
                        for (int kb = 0; kb < p.num_kb; ++kb) {
                            if (!wait_bounded(empty0 + 8u * stage, phase ^ 1u, wc, ERR_PRODUCER_SLOT)) {
                                ok = false;
                                break;
                            }
                            if (withhold) {
                                withhold = false;   // test hook: this slot's operands never arrive
                            } else {
                                const uint32_t fb = full0 + 8u * stage;
                                mbar_arrive_expect_tx(fb, Cfg::STAGE_BYTES);
                                tma_load_2d(sA + stage * Cfg::A_BYTES, &tmap_a, fb, kb * BK, rb * BM);
#pragma unroll
                                for (int i = 0; i < Cfg::B_BOXES; ++i)
                                    tma_load_2d(sB + stage * Cfg::B_BYTES + i * Cfg::B_BOX_BYTES, &tmap_b, fb,
                                                j * BN + i * Cfg::B_BOX_N, kb * BK);
                                issued |= 1u << stage;
                                issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
                            }
                            if (++stage == STAGES) {
                                stage = 0;
                                phase ^= 1u;
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
            int stage = 0, acc = 0;
            uint32_t phase = 0, acc_phase = 0;
            bool ok = true;
            for (int rb = work.rb; ok && rb < p.m_blocks; rb += work.rb_step)
                for (int pass = 0; ok && pass < work.passes; ++pass)
                    for (int j = work.j0; ok && j < work.j1; ++j) {
                        if (!wait_bounded(acce0 + 8u * acc, acc_phase ^ 1u, wc, ERR_MMA_ACCUMULATOR)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after_sync();
                        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN);
                        for (int kb = 0; kb < p.num_kb; ++kb) {
                            if (!wait_bounded(full0 + 8u * stage, phase, wc, ERR_MMA_OPERANDS)) {
                                ok = false;
                                break;
                            }
                            tc_fence_after_sync();
                            const uint32_t a0 = sA + stage * Cfg::A_BYTES;
                            const uint32_t b0 = sB + stage * Cfg::B_BYTES;
#pragma unroll
                            for (int kk = 0; kk < BK / Cfg::UMMA_K; ++kk) {
                                const uint64_t adesc = sw128_desc(a0 + kk * 32, 16, 1024);
                                const uint64_t bdesc = sw128_desc(b0 + kk * 2048, Cfg::B_BOX_BYTES, 1024);
                                umma_f16<1>(d_tmem, adesc, bdesc, IDESC, (kb | kk) != 0 ? 1u : 0u);
                            }
                            umma_commit(empty0 + 8u * stage);
                            if (++stage == STAGES) {
                                stage = 0;
                                phase ^= 1u;
                            }
                        }
                        if (!ok)
                            break;
                        umma_commit(accf0 + 8u * acc);   // accumulator complete
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
        const int ew = warp - 2;
        const int quarter = warp & 3;              // TMEM lanes this warp may access
        const int group = ew >> 2;                 // its 64 columns of each tile
        const int row = quarter * 32 + lane;       // this thread's row of the tile
        const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
        uint4 *my_bias = bias_stage + ew * (Cfg::WARP_COLS / 8);
        const uint32_t my_stage = base + Cfg::STORE_OFFSET + static_cast<uint32_t>(ew) * Cfg::STORE_BOX_BYTES;
        const uint32_t group_slots = base + Cfg::GROUP_OFFSET;
        const uint32_t my_group_bar = group0 + 8u * static_cast<uint32_t>(quarter);
        const bool has_acc = p.num_kb > 0;   // K = 0: the empty sum, no accumulator to read
        int acc = 0;
        uint32_t acc_phase = 0, merges = 0, unit = 0;
        bool ok = true;

        // Wait for the next accumulator and stage its bias slice (this warp's 64 columns) in
        // shared memory; then read its halves (load) and hand it back to the MMA warp (release).
        auto acquire = [&](int j) -> bool {
            const int n_first = j * BN + group * Cfg::WARP_COLS;
            uint4 bv = make_uint4(0u, 0u, 0u, 0u);
            if (p.bias != nullptr && lane < 8 && n_first + 8 * lane < p.N)
                bv = __ldg(reinterpret_cast<const uint4 *>(p.bias + n_first + 8 * lane));
            if (!wait_warp(accf0 + 8u * acc, acc_phase, wc, ERR_EPILOGUE_ACCUMULATOR, lane))
                return false;
            tc_fence_after_sync();
            if (p.bias != nullptr) {
                if (lane < 8)
                    my_bias[lane] = bv;
                __syncwarp();
            }
            return true;
        };
        auto load = [&](int h, uint32_t (&r)[32]) {
            if (has_acc) {
                tmem_ld_32x32b_x32(tmem_base + lane_base +
                                       static_cast<uint32_t>(acc * BN + group * Cfg::WARP_COLS + 32 * h),
                                   r);
                tmem_ld_wait_regs(r);
            } else {
#pragma unroll
                for (int i = 0; i < 32; ++i)
                    r[i] = 0u;
            }
        };
        auto release = [&]() {
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(acce0 + 8u * acc);   // this warp's part of the accumulator is read
            if (++acc == Cfg::ACC_BUFS) {
                acc = 0;
                acc_phase ^= 1u;
            }
        };

        for (int rb = work.rb; ok && rb < p.m_blocks; rb += work.rb_step, ++unit) {
            const int row0 = rb * BM + quarter * 32;
            const uint4 *sbias = p.bias != nullptr ? my_bias : nullptr;
            if constexpr (!TWO_PASS) {
                // one tile spans the row: all 64 values stay in registers
                if (!acquire(0)) {
                    ok = false;
                    break;
                }
                const int n_first = group * Cfg::WARP_COLS;
                float v[64];
                {
                    uint32_t r0[32], r1[32];
                    if (has_acc) {
                        const uint32_t t = tmem_base + lane_base + static_cast<uint32_t>(acc * BN + n_first);
                        tmem_ld_32x32b_x32(t, r0);
                        tmem_ld_32x32b_x32(t + 32u, r1);
                        tmem_ld_wait_regs(r0);
                        regs_after_wait(r1);
                    } else {
#pragma unroll
                        for (int i = 0; i < 32; ++i) {
                            r0[i] = 0u;
                            r1[i] = 0u;
                        }
                    }
                    release();
                    logits(r0, sbias, n_first, p.N, v);
                    logits(r1, sbias ? sbias + 4 : nullptr, n_first + 32, p.N, v + 32);
                }
                // statistics in base-2 units: mg = this warp's maximum times log2(e)
                const float mg = fmaxf(max32(v), max32(v + 32)) * kSmxLog2e;
                float m = mg, s = 0.0f;
                if (mg != -INFINITY)   // (a warp whose columns all lie past N has nothing to add)
                    s = exp2_fma_sum(v, -mg) + exp2_fma_sum(v + 32, -mg);
                if (!group_merge(group_slots, my_group_bar, merges++, quarter, group, lane, m, s, wc)) {
                    ok = false;
                    break;
                }
                // m is the row maximum, s the row's sum of 2^(x log2(e) - m); v holds 2^(x log2(e) - mg)
                const float scale = mg != -INFINITY ? ex2_approx(mg - m) * rcp_approx(s) : 0.0f;
                staging_free(lane);
                stage_row<true>(v, scale, my_stage, 0, lane);
                stage_row<true>(v + 32, scale, my_stage, 1, lane);
                store_box(my_stage, &tmap_c, n_first, row0, lane);
            } else {
                // pass 1: running row statistics over this CTA's tiles, 32 columns at a time
                float m = -INFINITY, s = 0.0f;
                for (int j = work.j0; j < work.j1; ++j) {
                    if (!acquire(j)) {
                        ok = false;
                        break;
                    }
#pragma unroll 1
                    for (int h = 0; h < 2; ++h) {
                        uint32_t r[32];
                        load(h, r);
                        if (h == 1)
                            release();
                        float v[32];
                        logits(r, sbias ? sbias + 4 * h : nullptr, j * BN + group * Cfg::WARP_COLS + 32 * h, p.N, v);
                        const float mn = fmaxf(m, max32(v) * kSmxLog2e);   // base-2 units
                        if (mn != -INFINITY) {
                            const float sh = exp2_fma_sum(v, -mn);
                            s = s * ex2_approx(m - mn) + sh;   // m = -inf gives 2^-inf = 0
                            m = mn;
                        }
                    }
                }
                if (!ok)
                    break;
                if (!group_merge(group_slots, my_group_bar, merges++, quarter, group, lane, m, s, wc)) {
                    ok = false;
                    break;
                }
                if (cs > 1 && !cluster_merge(base + Cfg::CLUSTER_OFFSET, ready0, read0, unit, cs, group, row, lane, m, s,
                                             wc)) {
                    ok = false;
                    break;
                }
                // pass 2: exp(x - max) / sum = 2^(x log2(e) - m - log2(s)) from the recomputed logits
                const float off = -m - lg2_approx(s);
                for (int j = work.j0; j < work.j1; ++j) {
                    if (!acquire(j)) {
                        ok = false;
                        break;
                    }
                    const int n_first = j * BN + group * Cfg::WARP_COLS;
                    staging_free(lane);
#pragma unroll 1
                    for (int h = 0; h < 2; ++h) {
                        uint32_t r[32];
                        load(h, r);
                        if (h == 1)
                            release();
                        float v[32];
                        logits(r, sbias ? sbias + 4 * h : nullptr, n_first + 32 * h, p.N, v);
                        exp2_fma(v, off);
                        stage_row<false>(v, 1.0f, my_stage, h, lane);
                    }
                    store_box(my_stage, &tmap_c, n_first, row0, lane);
                }
            }
        }
        if (lane == 0)
            bulk_wait_group<0>();   // every output box of this warp has reached global memory
        __syncwarp();
    }

    tc_fence_before_sync();
    __syncthreads();
    cluster_sync();   // no CTA leaves while another may still read its statistics
    if (warp == 1) {
        tc_fence_after_sync();
        tmem_dealloc<1>(tmem_base, Cfg::TMEM_COLS);
    }
}

}  // namespace gb300
