// Host side of the C ABI declared in include/gemm.h: argument checks, tensor-map encoding
// and the launch of the persistent tcgen05 GEMM kernel (gemm_kernel.cuh).
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <cstdio>
#include <cstring>
#include <new>

#include "gemm.h"
#include "gemm_kernel.cuh"
#include "gemm_kernel_pair.cuh"
#include "softmax_gemm_kernel.cuh"
#include "softmax_kernel.cuh"
#include "attention_kernel.cuh"
#include "clock_probe.cuh"

namespace {

#ifndef GB300_EPI_WARPS
#define GB300_EPI_WARPS 4
#endif
using Cfg = gb300::KernelConfig<128, 256, 4, GB300_EPI_WARPS>;
#ifndef GB300_PAIR_STAGES
#define GB300_PAIR_STAGES 3
#endif
#ifndef GB300_PAIR_BK
#define GB300_PAIR_BK 128
#endif
using PairCfg = gb300::PairConfig<256, GB300_PAIR_STAGES, GB300_EPI_WARPS, GB300_PAIR_BK>;
// One work unit per pair (all tiles in one wave): sixteen epilogue warps, output staging in
// the idle ring.
using Pair1WCfg = gb300::PairConfig<256, GB300_PAIR_STAGES, 16, GB300_PAIR_BK, true>;
#ifndef GB300_PAIR1W
#define GB300_PAIR1W 1
#endif
// The same 128 x 256 tiles with sixteen epilogue warps (four per TMEM lane quarter, 64
// columns each, 96 registers): the whole-tile kernel when all tiles fit one wave, where every
// CTA's epilogue is an exposed tail that more warps shorten (2048^3 + bias + GELU, same box: 4
// warps 18.6 us, 8 warps 18.0, 16 warps 17.3; plain 15.6, 15.0, 15.0). Each CTA has one tile,
// so its output staging overlays the idle operand ring, which leaves room for a fourth stage
// (2048^3 14.7 -> 13.9 us, 2048 x 2048 x 8192 55.5 -> 46.1, 1024 x 4096 x 4096 + bias + GELU
// 27.5 -> 24.8); two 128-wide stages in the same space were 3-9 % slower than three 64-wide.
// The last four k-blocks go into the left half of the accumulator first (HALF_TAIL), so that
// half's epilogue warps start during the right half's MMAs: 0.1-4 % on one-wave shapes (the
// right half's N = 128 MMAs use the whole shared-memory bandwidth, which the overlapped
// epilogue's staging also needs; giving every warp a chunk of each half was no better).
using Cfg16 = gb300::KernelConfig<128, 256, 4, 16, 64, true, true>;
// The softmax epilogue's kernel: 128 x 256 tiles, 3-stage ring, sixteen epilogue warps.
using SoftCfg = gb300::SoftmaxConfig<3>;
// Split-K runs on an instance with eight epilogue warps (two per TMEM lane quarter, each with
// half of the columns): twice the warps to stage the partial and to read the other CTAs'
// partials over DSMEM (measured 2-5 % faster than four on 5 of 6 few-tile shapes). Its
// epilogue writes C with plain stores, so the (unused) output staging overlays the ring, and
// the ring has four stages (192 KB; it holds the 128 KB partial): 256 x 4096 x 8192 23.2 ->
// 21.3 us, 2048 x 1024 x 8192 + bias + GELU 34.4 -> 32.3 against three.
using SplitCfg = gb300::KernelConfig<128, 256, 4, 8, 64, true>;
#ifndef GB300_GROUP_PANEL_MB
#define GB300_GROUP_PANEL_MB 32
#endif
// Raster group size: as many row blocks as keep the group's panel of A (rows x K) within
// this many bytes, so that the panel stays in L2 while the group sweeps all of B's column
// blocks; B then streams from DRAM once per group (at least kMinGroup row blocks).
constexpr int64_t kGroupPanelBytes = static_cast<int64_t>(GB300_GROUP_PANEL_MB) << 20;
constexpr int kMinGroup = 4;

int raster_group(int m_blocks, int rows_per_block, int K)
{
    const int64_t panel = static_cast<int64_t>(rows_per_block) * (K > 0 ? K : 1) * 2;
    const int64_t g = kGroupPanelBytes / panel;
    return static_cast<int>(std::max<int64_t>(kMinGroup, std::min<int64_t>(m_blocks, g)));
}

#ifndef GB300_BALANCED_GROUPS
#define GB300_BALANCED_GROUPS 1
#endif
// Raster groups of about equal size: the group count is m_blocks / target rounded to the
// nearest integer (at least one), the row-blocks spread evenly (the first `big` groups one
// larger). A last group of a few row-blocks would stream all of B again for them (M = 8200
// with 256-row blocks and 16-block groups: 16 + 16 + 1; here 17 + 16).
void raster_groups(int m_blocks, int rows_per_block, int K, int &group_m, int &big)
{
    const int g = raster_group(m_blocks, rows_per_block, K);
    big = 0;
    group_m = g;
    if (!GB300_BALANCED_GROUPS || m_blocks <= 0)
        return;
    const int count = std::max(1, (2 * m_blocks + g) / (2 * g));
    group_m = m_blocks / count;
    big = m_blocks % count;
}
constexpr uint64_t kDefaultTimeoutNs = 2000000000ull;
constexpr int64_t kSoftmaxMaxCtas = int64_t(1) << 20;   // row softmax grid cap (CTAs loop past it)
constexpr int kSoftmaxClusterMax = 8;   // softmax: clusters of 1, 2, 4 or 8 CTAs per row block
// gemm_run_host splits C into at most this many bands (column bands: also two row halves of
// A when A is at least kHostChunkMinBytes) whose uploads, GEMMs and downloads overlap;
// outputs smaller than kHostChunkMinBytes are not split.
constexpr int kHostChunksMax = 8;
constexpr size_t kHostChunkMinBytes = size_t(32) << 20;
constexpr uint64_t kMinTimeoutNs = 1000000ull;
// Stream-K (one-CTA kernel): each CTA gets at least this many (tile, k-block) units, and
// stream-K is taken only when it runs at least twice as many CTAs as there are tiles. The
// hand-off of a cut tile (partials written, pulled in by the owner, added in TMEM) costs a
// few microseconds on the critical path; measured on GB300, it pays off for 32 tiles of
// 128 x 256 x 8192 (39.8 -> 28.0 us) but not for 128 tiles on 152 SMs (2048^3: 15.3 us
// whole tiles, 23 us stream-K).
constexpr int64_t kStreamKMinUnits = 16;
constexpr int kSplitKMinBlocks = 8;   // split-K: k-blocks per CTA at least
#ifndef GB300_PAIR_LONG_K
#define GB300_PAIR_LONG_K 8192
#endif
constexpr int kPairLongK = GB300_PAIR_LONG_K;   // pairs for a one-wave problem from this K on
constexpr int kStreamKMinSpread = 2;

}  // namespace

struct gemm_ctx {
    int device = -1;
    int num_sms = 0;
    PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
    bool pair1w_ok = false;   // the one-wave pair instance runs as many clusters at once
    uint32_t *d_err = nullptr;
    uint64_t timeout_ns = kDefaultTimeoutNs;
    int debug = 0;
    int last_cuda_error = 0;
    int max_clusters = 0;   // co-resident CTA pairs of the pair kernel (0: pair kernel unusable)
    // stream-K workspace: one FP32 128 x 256 partial accumulator per SM, and per SM one
    // ready flag per epilogue warp (zero between launches)
    float *sk_ws = nullptr;
    uint32_t *sk_flags = nullptr;
    // softmax kernel: co-resident clusters of cs = 1, 2, 4, 8 CTAs (0: that size cannot be
    // scheduled; cs = 1 must be possible for the softmax epilogue to be offered at all)
    int softmax_clusters[kSoftmaxClusterMax + 1] = {};
    // split-K: co-resident clusters of 2, 4 and 8 CTAs of the split-K instance, per size
    int split_clusters[9] = {};
    // gemm_run_host: device staging buffers, two copy streams and the events that order
    // the chunked pipeline (created on first use)
    void *stage = nullptr;
    size_t stage_bytes = 0;
    cudaStream_t copy_in = nullptr, copy_out = nullptr;
    cudaEvent_t ev_start = nullptr, ev_done = nullptr;
    cudaEvent_t ev_in[2 * kHostChunksMax] = {}, ev_mm[2 * kHostChunksMax] = {};
};

namespace {

// Make `device` current for the lifetime of the guard, then restore the caller's device.
class DeviceGuard {
  public:
    explicit DeviceGuard(int device)
    {
        if (cudaGetDevice(&prev_) != cudaSuccess) {
            cudaGetLastError();
            prev_ = -1;
        }
        if (prev_ != device)
            cudaSetDevice(device);
    }
    ~DeviceGuard()
    {
        int cur = -1;
        if (prev_ >= 0 && cudaGetDevice(&cur) == cudaSuccess && cur != prev_)
            cudaSetDevice(prev_);
    }

  private:
    int prev_ = -1;
};

int cuda_fail(gemm_ctx *ctx, cudaError_t e, int code)
{
    if (ctx)
        ctx->last_cuda_error = static_cast<int>(e);
    cudaGetLastError();   // clear the sticky-free error state
    return code;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// True when p is device (or managed) memory that `device` can address directly.
bool on_device(const void *p, int device)
{
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    if (a.type == cudaMemoryTypeManaged)
        return true;
    return a.type == cudaMemoryTypeDevice && a.device == device;
}

bool overlaps(const void *a, size_t na, const void *b, size_t nb)
{
    if (!a || !b || na == 0 || nb == 0)
        return false;
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
    return a0 < b0 + nb && b0 < a0 + na;
}

// Size and epilogue rules (no pointers): GEMM_OK also for the empty problems M = 0 or N = 0.
int check_shape(const gemm_ctx *ctx, int64_t M, int64_t N, int64_t K, int epilogue)
{
    if (!ctx)
        return GEMM_ERR_ARG;
    if (M < 0 || N < 0 || K < 0 || M > INT32_MAX || N > INT32_MAX || K > INT32_MAX)
        return GEMM_ERR_ARG;
    if (epilogue < GEMM_EPI_NONE || epilogue > GEMM_EPI_SOFTMAX)
        return GEMM_ERR_ARG;
    if (M == 0 || N == 0)
        return GEMM_OK;
    if (epilogue == GEMM_EPI_SOFTMAX && ctx->softmax_clusters[1] == 0)
        return GEMM_ERR_ARG;   // the device cannot run the softmax kernel
    if (N % 8 != 0 || K % 8 != 0)
        return GEMM_ERR_ALIGN;
    return GEMM_OK;
}

// Shape/pointer rules shared by gemm_run and gemm_run_host (everything but memory kind).
int check_args(gemm_ctx *ctx, int64_t M, int64_t N, int64_t K, const void *A, const void *B,
               const void *bias, void *C, int epilogue)
{
    int rc = check_shape(ctx, M, N, K, epilogue);
    if (rc != GEMM_OK || M == 0 || N == 0)
        return rc;
    if (!C || (K > 0 && (!A || !B)))
        return GEMM_ERR_ARG;
    if (!aligned16(C) || (K > 0 && (!aligned16(A) || !aligned16(B))) || (bias && !aligned16(bias)))
        return GEMM_ERR_ALIGN;
    const size_t cb = static_cast<size_t>(M) * N * 2;
    if (overlaps(C, cb, A, static_cast<size_t>(M) * K * 2) ||
        overlaps(C, cb, B, static_cast<size_t>(K) * N * 2) || overlaps(C, cb, bias, static_cast<size_t>(N) * 2))
        return GEMM_ERR_ARG;
    return GEMM_OK;
}

// 2-D FP16 tensor map over a row-major [outer x inner] matrix with boxes of
// box_inner x box_outer elements (swizzled as given); loads read out-of-range elements as
// zero, stores skip them.
bool encode_2d(gemm_ctx *ctx, CUtensorMap *map, const void *ptr, uint64_t inner, uint64_t outer,
               uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_128B,
               uint64_t ld = 0 /* row stride in elements; 0: tightly packed */)
{
    const cuuint64_t dims[2] = {inner, outer};
    const cuuint64_t strides[1] = {(ld ? ld : inner) * 2};
    const cuuint32_t box[2] = {box_inner, box_outer};
    const cuuint32_t estr[2] = {1, 1};
    const CUresult r = ctx->encode(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void *>(ptr), dims,
                                   strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
                                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// Launch with programmatic stream serialisation: the kernel may be scheduled while the
// previous kernel in the stream is finishing and overlaps its own set-up with that tail;
// it waits (griddepcontrol.wait) before touching global memory.
void launch_pdl(void (*kernel)(CUtensorMap, CUtensorMap, CUtensorMap, gb300::GemmParams), int grid, int threads,
                int smem, cudaStream_t stream, const CUtensorMap &ta, const CUtensorMap &tb, const CUtensorMap &tc,
                const gb300::GemmParams &p)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
    cfg.blockDim = dim3(static_cast<unsigned>(threads), 1, 1);
    cfg.dynamicSmemBytes = static_cast<size_t>(smem);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaLaunchKernelEx(&cfg, kernel, ta, tb, tc, p);
}

// The same with a cluster of `cluster` CTAs along x (grid a multiple of it).
void launch_pdl_cluster(void (*kernel)(CUtensorMap, CUtensorMap, CUtensorMap, gb300::GemmParams), int grid,
                        int cluster, int threads, int smem, cudaStream_t stream, const CUtensorMap &ta,
                        const CUtensorMap &tb, const CUtensorMap &tc, const gb300::GemmParams &p)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
    cfg.blockDim = dim3(static_cast<unsigned>(threads), 1, 1);
    cfg.dynamicSmemBytes = static_cast<size_t>(smem);
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = static_cast<unsigned>(cluster);
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    cudaLaunchKernelEx(&cfg, kernel, ta, tb, tc, p);
}

// The kernel instance gemm_run launches for a problem, with its grid and the schedule fields
// of its parameters. make_plan decides; launch runs the plan; gemm_describe reports it.
enum PlanKind : int {
    PLAN_PAIR, PLAN_PAIR1W, PLAN_TILES, PLAN_TILES16, PLAN_STREAMK, PLAN_SPLITK, PLAN_ROWCLUSTER, PLAN_ROWCLUSTER2
};

struct Plan {
    PlanKind kind = PLAN_TILES;
    int grid = 0;      // CTAs launched
    int cluster = 1;   // CTAs per thread-block cluster (1: no cluster attribute)
    int m_blocks = 0, n_blocks = 0, num_tiles = 0, group_m = 1, group_big = 0;
    int split = 0, row_cluster = 0, smx_span = 0, smx_two_pass = 0;
    int64_t sk_units = 0;
    int pair_split_from = 0, pair_units = 0;   // pair kernel: tiles kept whole, work units
};

const char *plan_kernel_name(PlanKind k)
{
    switch (k) {
    case PLAN_PAIR: return "gemm_tcgen05_pair_kernel<PairConfig<256,3,4,128>>";
    case PLAN_PAIR1W: return "gemm_tcgen05_pair_kernel<PairConfig<256,3,16,128,true>>";
    case PLAN_TILES: return "gemm_tcgen05_kernel<KernelConfig<128,256,4,4>,SCHED_TILES>";
    case PLAN_TILES16: return "gemm_tcgen05_kernel<KernelConfig<128,256,4,16,64,true,true>,SCHED_TILES>";
    case PLAN_STREAMK: return "gemm_tcgen05_kernel<KernelConfig<128,256,4,4>,SCHED_STREAM_K>";
    case PLAN_SPLITK: return "gemm_tcgen05_kernel<KernelConfig<128,256,4,8,64,true>,SCHED_SPLIT_K>";
    case PLAN_ROWCLUSTER: return "gemm_softmax_kernel<SoftmaxConfig<3>,false>";
    case PLAN_ROWCLUSTER2: return "gemm_softmax_kernel<SoftmaxConfig<3>,true>";
    }
    return "unknown";
}

// Choose the kernel instance and grid for an M x N x K problem (sizes already checked,
// M, N > 0).
Plan make_plan(const gemm_ctx *ctx, int M, int N, int K, int epilogue)
{
    Plan pl;
    const int num_kb = (K + Cfg::BK - 1) / Cfg::BK;
    if (epilogue == GEMM_EPI_SOFTMAX) {
        static_assert(SoftCfg::BM == Cfg::BM && SoftCfg::BN == Cfg::BN && SoftCfg::BK == Cfg::BK &&
                          SoftCfg::B_BOX_N == Cfg::B_BOX_N,
                      "same tensor-map boxes as the GEMM kernel");
        pl.kind = PLAN_ROWCLUSTER;
        pl.m_blocks = (M + SoftCfg::BM - 1) / SoftCfg::BM;
        pl.n_blocks = (N + SoftCfg::BN - 1) / SoftCfg::BN;
        pl.num_tiles = pl.m_blocks * pl.n_blocks;
        pl.group_m = 1;
        int cs = 1, span = 1;
        if (pl.n_blocks > 1) {
            // Two passes over each CTA's span of column tiles. Cluster size: the one that
            // minimises the tile epilogues of the busiest CTA, rounds x (2 x span + 1 for the
            // statistics exchange when cs > 1), with the co-resident clusters of that size;
            // ties go to the smaller cluster.
            int64_t best = INT64_MAX;
            for (int c = 1; c <= kSoftmaxClusterMax; c *= 2) {
                const int conc = std::min(pl.m_blocks, ctx->softmax_clusters[c]);
                if (conc <= 0)
                    continue;
                const int sp = (pl.n_blocks + c - 1) / c;
                const int64_t rounds = (pl.m_blocks + conc - 1) / conc;
                const int64_t cost = rounds * (2 * sp + (c > 1 ? 1 : 0));
                if (cost < best) {
                    best = cost;
                    cs = c;
                    span = sp;
                }
            }
        }
        pl.row_cluster = cs;
        pl.smx_span = span;
        pl.smx_two_pass = pl.n_blocks > 1 ? 1 : 0;
        if (pl.smx_two_pass)
            pl.kind = PLAN_ROWCLUSTER2;
        pl.cluster = cs;
        pl.grid = std::min(pl.m_blocks, ctx->softmax_clusters[cs]) * cs;
        return pl;
    }
    // 256 x 256 tiles on CTA pairs when there are enough of them to give every pair at
    // least one; otherwise 128 x 256 tiles on single SMs (twice as many tiles to spread).
    // Also pairs for a long K when at least three quarters of the pairs get a tile and the
    // single-SM tiles would fit one wave: each pair's SM moves 64 operand bytes per clock of
    // tensor work from L2 against 96 for a single SM's 128 x 256 tile (on 128 SMs about all
    // that L2 delivers at once), which outweighs the pair's dearer start and 4-warp epilogue
    // once K >= 8192 (64 pair tiles: 2048 x 2048 x 8192 +1.6 %, x 16384 +7.1 %, 4096 x 1024
    // x 8192 +5.2 %; at K = 6144 -3.7 %).
    const int pair_tiles = ((M + PairCfg::BM - 1) / PairCfg::BM) * ((N + PairCfg::BN - 1) / PairCfg::BN);
    const int one_tiles = ((M + Cfg::BM - 1) / Cfg::BM) * ((N + Cfg::BN - 1) / Cfg::BN);
    bool pair = ctx->max_clusters > 0 &&
                (pair_tiles >= ctx->max_clusters || (K >= kPairLongK && 4 * pair_tiles >= 3 * ctx->max_clusters &&
                                                     one_tiles <= ctx->num_sms));
    if (ctx->debug & (GEMM_DEBUG_FORCE_SINGLE | GEMM_DEBUG_FORCE_SPLITK))
        pair = false;
    if ((ctx->debug & GEMM_DEBUG_FORCE_PAIR) && ctx->max_clusters > 0)
        pair = true;
    if (pair) {
        pl.kind = PLAN_PAIR;
        pl.m_blocks = (M + PairCfg::BM - 1) / PairCfg::BM;
        pl.n_blocks = (N + PairCfg::BN - 1) / PairCfg::BN;
        pl.num_tiles = pl.m_blocks * pl.n_blocks;
        raster_groups(pl.m_blocks, PairCfg::BM, K, pl.group_m, pl.group_big);
        pl.cluster = 2;
        pl.grid = 2 * std::min(pl.num_tiles, ctx->max_clusters);
        // A last round of tiles that at most half of the pairs would work on (8192^3: 1024
        // tiles on 76 pairs leave 36) runs as twice as many N-halves, one per pair: that
        // round takes half as long.
        const int pairs = pl.grid / 2;
        const int last = pl.num_tiles % pairs;
        pl.pair_split_from = (last > 0 && 2 * last <= pairs) ? pl.num_tiles - last : pl.num_tiles;
        pl.pair_units = pl.pair_split_from + 2 * (pl.num_tiles - pl.pair_split_from);
        // one unit per pair: the sixteen-warp instance, its output staged in the idle ring
        if (GB300_PAIR1W && pl.pair_units <= pairs && ctx->pair1w_ok)
            pl.kind = PLAN_PAIR1W;
        return pl;
    }
    pl.m_blocks = (M + Cfg::BM - 1) / Cfg::BM;
    pl.n_blocks = (N + Cfg::BN - 1) / Cfg::BN;
    pl.num_tiles = pl.m_blocks * pl.n_blocks;
    raster_groups(pl.m_blocks, Cfg::BM, K, pl.group_m, pl.group_big);
    pl.grid = std::min(pl.num_tiles, ctx->num_sms);
    // Split-K when the tiles leave most SMs idle: a cluster of S CTAs per tile, each with
    // 1/S of the k-blocks (at least kSplitKMinBlocks of them), the partials summed over
    // DSMEM; S = 8, 4 or 2, the largest whose clusters all run at once.
    const int64_t units = static_cast<int64_t>(pl.num_tiles) * num_kb;
    int split = 0;
    if (units > 0 && !(ctx->debug & GEMM_DEBUG_FORCE_STREAMK)) {
        for (int cs = 8; cs >= 2 && !split; cs /= 2) {
            if (ctx->split_clusters[cs] <= 0 || num_kb < cs)
                continue;
            if (ctx->debug & GEMM_DEBUG_FORCE_SPLITK)
                split = cs;   // any tile count (several waves) and any k-blocks >= cs
            else if (static_cast<int64_t>(pl.num_tiles) * cs <= ctx->num_sms &&
                     pl.num_tiles <= ctx->split_clusters[cs] && num_kb >= kSplitKMinBlocks * cs)
                split = cs;
        }
    }
    if (split > 0) {
        pl.kind = PLAN_SPLITK;
        pl.split = split;
        pl.cluster = split;
        pl.grid = pl.num_tiles * split;
        return pl;
    }
    // Otherwise stream-K when the tiles leave most SMs idle: the (tile, k-block) units are
    // split evenly over up to every SM.
    if (units > 0) {
        int g_sk = 0;
        if (ctx->debug & GEMM_DEBUG_FORCE_STREAMK)
            g_sk = static_cast<int>(std::min<int64_t>(ctx->num_sms, units));
        else if (static_cast<int64_t>(pl.num_tiles) * kStreamKMinSpread <= ctx->num_sms)
            g_sk = static_cast<int>(std::min<int64_t>(ctx->num_sms, units / kStreamKMinUnits));
        if (g_sk >= kStreamKMinSpread * pl.num_tiles || ((ctx->debug & GEMM_DEBUG_FORCE_STREAMK) && g_sk > 0)) {
            pl.kind = PLAN_STREAMK;
            pl.sk_units = units;
            pl.grid = g_sk;
            return pl;
        }
    }
    // one wave: sixteen epilogue warps
    pl.kind = pl.num_tiles <= ctx->num_sms ? PLAN_TILES16 : PLAN_TILES;
    return pl;
}

// ldb / ldc: row strides of B and C in elements (0: N, tightly packed); A is always packed.
// gemm_run_host uses them to run column bands of a larger B and C.
int launch(gemm_ctx *ctx, int M, int N, int K, const void *A, const void *B, const void *bias, void *C,
           int epilogue, cudaStream_t stream, int64_t ldb = 0, int64_t ldc = 0)
{
    CUtensorMap ta, tb, tc;
    std::memset(&ta, 0, sizeof(ta));
    std::memset(&tb, 0, sizeof(tb));
    const Plan pl = make_plan(ctx, M, N, K, epilogue);
    // K per ring stage of the chosen kernel: A goes in 64-wide boxes either way, B in boxes
    // of that many rows
    const int bk = (pl.kind == PLAN_PAIR || pl.kind == PLAN_PAIR1W) ? PairCfg::BK
                   : pl.kind == PLAN_TILES16                      ? Cfg16::BK
                                                                  : Cfg::BK;
    static_assert(Pair1WCfg::BK == PairCfg::BK, "one B box height for both pair instances");
    // Pair1WCfg stages its output in the operand ring: one unit per pair at most
    if (pl.kind == PLAN_PAIR1W && pl.grid < 2 * pl.pair_units)
        return GEMM_ERR_ARG;
    // Cfg16 stages its output in the operand ring: one tile per CTA at most
    if (pl.kind == PLAN_TILES16 && pl.grid < pl.num_tiles)
        return GEMM_ERR_ARG;
    if (K > 0) {
        if (!encode_2d(ctx, &ta, A, static_cast<uint64_t>(K), static_cast<uint64_t>(M), Cfg::BK, Cfg::BM) ||
            !encode_2d(ctx, &tb, B, static_cast<uint64_t>(N), static_cast<uint64_t>(K), Cfg::B_BOX_N,
                       static_cast<uint32_t>(bk), CU_TENSOR_MAP_SWIZZLE_128B, static_cast<uint64_t>(ldb)))
            return GEMM_ERR_LAUNCH;
    }
    // C is written by TMA in 32 x 32 boxes staged with the 64-byte swizzle; the softmax
    // kernel writes 32-row x 64-column boxes staged with the 128-byte swizzle
    const bool smx = pl.kind == PLAN_ROWCLUSTER || pl.kind == PLAN_ROWCLUSTER2;
    if (!encode_2d(ctx, &tc, C, static_cast<uint64_t>(N), static_cast<uint64_t>(M), smx ? 64 : 32, 32,
                   smx ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B, static_cast<uint64_t>(ldc)))
        return GEMM_ERR_LAUNCH;
    gb300::GemmParams p;
    p.M = M;
    p.N = N;
    p.K = K;
    p.num_kb = (K + bk - 1) / bk;
    p.epilogue = epilogue;
    p.bias = static_cast<const __half *>(bias);
    p.C = static_cast<__half *>(C);
    p.ldc = ldc > 0 ? ldc : N;
    p.err = ctx->d_err;
    p.timeout_ns = ctx->timeout_ns;
    p.debug = ctx->debug & GEMM_DEBUG_WITHHOLD_FIRST_LOAD;
    p.m_blocks = pl.m_blocks;
    p.n_blocks = pl.n_blocks;
    p.num_tiles = pl.num_tiles;
    p.group_m = pl.group_m;
    p.group_big = pl.group_big;
    p.split = pl.split;
    p.row_cluster = pl.row_cluster;
    p.smx_span = pl.smx_span;
    p.smx_two_pass = pl.smx_two_pass;
    p.pair_split_from = pl.pair_split_from;
    p.pair_units = pl.pair_units;
    if (pl.kind == PLAN_STREAMK) {
        p.sk_units = pl.sk_units;
        p.sk_ws = ctx->sk_ws;
        p.sk_flags = ctx->sk_flags;
    }
    switch (pl.kind) {
    case PLAN_ROWCLUSTER:
    case PLAN_ROWCLUSTER2:
        if (pl.smx_two_pass)
            launch_pdl_cluster(gb300::gemm_softmax_kernel<SoftCfg, true>, pl.grid, pl.cluster, SoftCfg::NUM_THREADS,
                               SoftCfg::SMEM_BYTES, stream, ta, tb, tc, p);
        else
            launch_pdl_cluster(gb300::gemm_softmax_kernel<SoftCfg, false>, pl.grid, pl.cluster, SoftCfg::NUM_THREADS,
                               SoftCfg::SMEM_BYTES, stream, ta, tb, tc, p);
        break;
    case PLAN_PAIR:
        launch_pdl(gb300::gemm_tcgen05_pair_kernel<PairCfg>, pl.grid, PairCfg::NUM_THREADS, PairCfg::SMEM_BYTES,
                   stream, ta, tb, tc, p);
        break;
    case PLAN_PAIR1W:
        launch_pdl(gb300::gemm_tcgen05_pair_kernel<Pair1WCfg>, pl.grid, Pair1WCfg::NUM_THREADS,
                   Pair1WCfg::SMEM_BYTES, stream, ta, tb, tc, p);
        break;
    case PLAN_SPLITK:
        launch_pdl_cluster(gb300::gemm_tcgen05_kernel<SplitCfg, gb300::SCHED_SPLIT_K>, pl.grid, pl.cluster,
                           SplitCfg::NUM_THREADS, SplitCfg::SMEM_BYTES, stream, ta, tb, tc, p);
        break;
    case PLAN_STREAMK:
        launch_pdl(gb300::gemm_tcgen05_kernel<Cfg, gb300::SCHED_STREAM_K>, pl.grid, Cfg::NUM_THREADS,
                   Cfg::SMEM_BYTES, stream, ta, tb, tc, p);
        break;
    case PLAN_TILES16:
        launch_pdl(gb300::gemm_tcgen05_kernel<Cfg16, gb300::SCHED_TILES>, pl.grid, Cfg16::NUM_THREADS,
                   Cfg16::SMEM_BYTES, stream, ta, tb, tc, p);
        break;
    case PLAN_TILES:
        launch_pdl(gb300::gemm_tcgen05_kernel<Cfg, gb300::SCHED_TILES>, pl.grid, Cfg::NUM_THREADS, Cfg::SMEM_BYTES,
                   stream, ta, tb, tc, p);
        break;
    }
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess)
        return cuda_fail(ctx, e, GEMM_ERR_LAUNCH);
    return GEMM_OK;
}

// Row softmax with the rows in registers: G threads per row, V 16-byte vectors per thread,
// register budget for MIN_CTAS CTAs per SM. One CTA per row group (the hardware balances
// them); past kSoftmaxMaxCtas CTAs the kernel's CTAs loop over the remaining rows.
template <int G, int V, int MIN_CTAS>
void launch_softmax_regs(int64_t rows, int cols, const __half *x, __half *y, cudaStream_t st)
{
    constexpr int BLOCK = G < 256 ? 256 : G;
    constexpr int GROUPS = BLOCK / G;
    const unsigned grid = static_cast<unsigned>(std::min<int64_t>((rows + GROUPS - 1) / GROUPS, kSoftmaxMaxCtas));
    gb300::row_softmax_regs_kernel<G, V, MIN_CTAS><<<grid, BLOCK, 0, st>>>(x, y, rows, cols);
}

}  // namespace

extern "C" {

int gemm_create(gemm_ctx **out, int device)
{
    if (!out)
        return GEMM_ERR_ARG;
    *out = nullptr;
    int count = 0;
    if (cudaGetDeviceCount(&count) != cudaSuccess) {
        cudaGetLastError();
        return GEMM_ERR_DEVICE;
    }
    if (device < 0 || device >= count)
        return GEMM_ERR_DEVICE;
    int major = 0, minor = 0, sms = 0, smem_optin = 0;
    cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, device);
    cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, device);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device);
    cudaDeviceGetAttribute(&smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, device);
    if (major != 10 || minor != 3 || sms <= 0 || smem_optin < Cfg::SMEM_BYTES)
        return GEMM_ERR_DEVICE;

    gemm_ctx *ctx = new (std::nothrow) gemm_ctx();
    if (!ctx)
        return GEMM_ERR_NOMEM;
    ctx->device = device;
    ctx->num_sms = sms;
    DeviceGuard guard(device);
    cudaError_t e = cudaFuncSetAttribute(gb300::gemm_tcgen05_kernel<Cfg, gb300::SCHED_TILES>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::SMEM_BYTES);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(gb300::gemm_tcgen05_kernel<Cfg, gb300::SCHED_STREAM_K>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::SMEM_BYTES);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(gb300::gemm_tcgen05_kernel<Cfg16, gb300::SCHED_TILES>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg16::SMEM_BYTES);
    if (e != cudaSuccess) {
        delete ctx;
        return cuda_fail(nullptr, e, GEMM_ERR_DEVICE);
    }
    e = cudaFuncSetAttribute(gb300::attention_fwd_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             gb300::AttnConfig::SMEM_BYTES);
    if (e != cudaSuccess) {
        delete ctx;
        return cuda_fail(nullptr, e, GEMM_ERR_DEVICE);
    }
    // The clock sampler shares an SM with the kernels it watches: with the default
    // preference a CTA without shared memory may configure its SM for a small shared-memory
    // carve-out, and no CTA needing 200+ KB can join that SM until it exits (a persistent
    // GEMM then waits for it). Ask for the largest carve-out, the configuration the GEMM
    // kernels use.
    e = cudaFuncSetAttribute(gb300::clock_probe_kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                             cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess) {
        delete ctx;
        return cuda_fail(nullptr, e, GEMM_ERR_DEVICE);
    }
    // The pair kernel is used only if the device can co-schedule its clusters.
    if (cudaFuncSetAttribute(gb300::gemm_tcgen05_pair_kernel<PairCfg>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             PairCfg::SMEM_BYTES) == cudaSuccess) {
        cudaLaunchConfig_t lc = {};
        lc.gridDim = dim3(2 * (sms / 2), 1, 1);
        lc.blockDim = dim3(PairCfg::NUM_THREADS, 1, 1);
        lc.dynamicSmemBytes = PairCfg::SMEM_BYTES;
        int clusters = 0;
        if (cudaOccupancyMaxActiveClusters(&clusters, gb300::gemm_tcgen05_pair_kernel<PairCfg>, &lc) == cudaSuccess)
            ctx->max_clusters = clusters;
        // the one-wave instance: as many clusters at once, or it is not used
        lc.blockDim = dim3(Pair1WCfg::NUM_THREADS, 1, 1);
        lc.dynamicSmemBytes = Pair1WCfg::SMEM_BYTES;
        clusters = 0;
        if (cudaFuncSetAttribute(gb300::gemm_tcgen05_pair_kernel<Pair1WCfg>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, Pair1WCfg::SMEM_BYTES) == cudaSuccess &&
            cudaOccupancyMaxActiveClusters(&clusters, gb300::gemm_tcgen05_pair_kernel<Pair1WCfg>, &lc) == cudaSuccess)
            ctx->pair1w_ok = clusters >= ctx->max_clusters;
    }
    cudaGetLastError();
    // Split-K clusters: how many clusters of 2, 4 and 8 CTAs fit at once (0: that size is not
    // used).
    {
        auto *sk = gb300::gemm_tcgen05_kernel<SplitCfg, gb300::SCHED_SPLIT_K>;
        if (cudaFuncSetAttribute(sk, cudaFuncAttributeMaxDynamicSharedMemorySize, SplitCfg::SMEM_BYTES) == cudaSuccess) {
            for (int cs = 2; cs <= 8; cs *= 2) {
                cudaLaunchConfig_t lc = {};
                lc.gridDim = dim3(static_cast<unsigned>(cs * (sms / cs)), 1, 1);
                lc.blockDim = dim3(SplitCfg::NUM_THREADS, 1, 1);
                lc.dynamicSmemBytes = SplitCfg::SMEM_BYTES;
                cudaLaunchAttribute a[1];
                a[0].id = cudaLaunchAttributeClusterDimension;
                a[0].val.clusterDim.x = static_cast<unsigned>(cs);
                a[0].val.clusterDim.y = 1;
                a[0].val.clusterDim.z = 1;
                lc.attrs = a;
                lc.numAttrs = 1;
                int n = 0;
                if (cudaOccupancyMaxActiveClusters(&n, sk, &lc) == cudaSuccess)
                    ctx->split_clusters[cs] = n;
            }
        }
        cudaGetLastError();
    }
    // Softmax kernel: how many clusters of 1, 2, 4 and 8 CTAs fit at once (a size that
    // cannot be scheduled stays 0 and is not used).
    {
        auto *sk = gb300::gemm_softmax_kernel<SoftCfg, true>;   // same resources as <SoftCfg, false>
        if (cudaFuncSetAttribute(gb300::gemm_softmax_kernel<SoftCfg, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 SoftCfg::SMEM_BYTES) == cudaSuccess &&
            cudaFuncSetAttribute(sk, cudaFuncAttributeMaxDynamicSharedMemorySize, SoftCfg::SMEM_BYTES) == cudaSuccess) {
            for (int cs = 1; cs <= kSoftmaxClusterMax; cs *= 2) {
                cudaLaunchConfig_t lc = {};
                lc.gridDim = dim3(static_cast<unsigned>(cs * (sms / cs)), 1, 1);
                lc.blockDim = dim3(SoftCfg::NUM_THREADS, 1, 1);
                lc.dynamicSmemBytes = SoftCfg::SMEM_BYTES;
                cudaLaunchAttribute a[1];
                a[0].id = cudaLaunchAttributeClusterDimension;
                a[0].val.clusterDim.x = static_cast<unsigned>(cs);
                a[0].val.clusterDim.y = 1;
                a[0].val.clusterDim.z = 1;
                lc.attrs = a;
                lc.numAttrs = 1;
                int n = 0;
                if (cudaOccupancyMaxActiveClusters(&n, sk, &lc) == cudaSuccess)
                    ctx->softmax_clusters[cs] = n;
            }
        }
        cudaGetLastError();
    }
    void *fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
    if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !fn) {
        delete ctx;
        return cuda_fail(nullptr, e, GEMM_ERR_DEVICE);
    }
    ctx->encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    const size_t ws_bytes = static_cast<size_t>(sms) * Cfg::BM * Cfg::BN * sizeof(float);
    const size_t flag_bytes = static_cast<size_t>(sms) * Cfg::NUM_EPI_WARPS * sizeof(uint32_t);
    e = cudaMalloc(&ctx->d_err, sizeof(uint32_t));
    if (e == cudaSuccess)
        e = cudaMemset(ctx->d_err, 0, sizeof(uint32_t));
    if (e == cudaSuccess)
        e = cudaMalloc(&ctx->sk_ws, ws_bytes);
    if (e == cudaSuccess)
        e = cudaMalloc(&ctx->sk_flags, flag_bytes);
    if (e == cudaSuccess)
        e = cudaMemset(ctx->sk_flags, 0, flag_bytes);
    if (e != cudaSuccess) {
        if (ctx->d_err)
            cudaFree(ctx->d_err);
        if (ctx->sk_ws)
            cudaFree(ctx->sk_ws);
        if (ctx->sk_flags)
            cudaFree(ctx->sk_flags);
        delete ctx;
        return cuda_fail(nullptr, e, GEMM_ERR_NOMEM);
    }
    *out = ctx;
    return GEMM_OK;
}

int gemm_run(gemm_ctx *ctx, int64_t M, int64_t N, int64_t K, const void *A, const void *B, const void *bias,
             void *C, int epilogue, void *stream)
{
    int rc = check_args(ctx, M, N, K, A, B, bias, C, epilogue);
    if (rc != GEMM_OK || M == 0 || N == 0)
        return rc;
    if (!on_device(C, ctx->device) || (K > 0 && (!on_device(A, ctx->device) || !on_device(B, ctx->device))) ||
        (bias && !on_device(bias, ctx->device)))
        return GEMM_ERR_DEVICE;
    DeviceGuard guard(ctx->device);
    return launch(ctx, static_cast<int>(M), static_cast<int>(N), static_cast<int>(K), A, B, bias, C, epilogue,
                  static_cast<cudaStream_t>(stream));
}

int gemm_run_host(gemm_ctx *ctx, int64_t M, int64_t N, int64_t K, const void *A, const void *B,
                  const void *bias, void *C, int epilogue, void *stream)
{
    int rc = check_args(ctx, M, N, K, A, B, bias, C, epilogue);
    if (rc != GEMM_OK || M == 0 || N == 0)
        return rc;
    auto round256 = [](size_t x) { return (x + 255) & ~static_cast<size_t>(255); };
    const size_t a_b = static_cast<size_t>(M) * K * 2, b_b = static_cast<size_t>(K) * N * 2;
    const size_t bias_b = bias ? static_cast<size_t>(N) * 2 : 0, c_b = static_cast<size_t>(M) * N * 2;
    const size_t need = round256(a_b) + round256(b_b) + round256(bias_b) + round256(c_b);
    DeviceGuard guard(ctx->device);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e;
    if (!ctx->copy_in) {   // first call: the pipeline's streams and events
        e = cudaStreamCreateWithFlags(&ctx->copy_in, cudaStreamNonBlocking);
        if (e == cudaSuccess)
            e = cudaStreamCreateWithFlags(&ctx->copy_out, cudaStreamNonBlocking);
        if (e == cudaSuccess)
            e = cudaEventCreateWithFlags(&ctx->ev_start, cudaEventDisableTiming);
        if (e == cudaSuccess)
            e = cudaEventCreateWithFlags(&ctx->ev_done, cudaEventDisableTiming);
        for (int i = 0; i < 2 * kHostChunksMax && e == cudaSuccess; ++i) {
            e = cudaEventCreateWithFlags(&ctx->ev_in[i], cudaEventDisableTiming);
            if (e == cudaSuccess)
                e = cudaEventCreateWithFlags(&ctx->ev_mm[i], cudaEventDisableTiming);
        }
        if (e != cudaSuccess)
            return cuda_fail(ctx, e, GEMM_ERR_NOMEM);
    }
    if (need > ctx->stage_bytes) {
        if (ctx->stage) {
            cudaStreamSynchronize(s);
            cudaFree(ctx->stage);
            ctx->stage = nullptr;
            ctx->stage_bytes = 0;
        }
        e = cudaMalloc(&ctx->stage, need);
        if (e != cudaSuccess) {
            ctx->stage = nullptr;
            return cuda_fail(ctx, e, GEMM_ERR_NOMEM);
        }
        ctx->stage_bytes = need;
    }
    char *base = static_cast<char *>(ctx->stage);
    char *dA = base, *dB = base + round256(a_b);
    char *dbias = bias ? base + round256(a_b) + round256(b_b) : nullptr;
    char *dC = base + round256(a_b) + round256(b_b) + round256(bias_b);

    if ((e = cudaEventRecord(ctx->ev_start, s)) != cudaSuccess ||
        (e = cudaStreamWaitEvent(ctx->copy_in, ctx->ev_start, 0)) != cudaSuccess ||
        (e = cudaStreamWaitEvent(ctx->copy_out, ctx->ev_start, 0)) != cudaSuccess)
        return cuda_fail(ctx, e, GEMM_ERR_LAUNCH);
    if (bias_b && (e = cudaMemcpyAsync(dbias, bias, bias_b, cudaMemcpyHostToDevice, s)) != cudaSuccess)
        return cuda_fail(ctx, e, GEMM_ERR_LAUNCH);
    // The output is produced in bands whose upload, GEMM and download overlap (copy_in, s,
    // copy_out). The operand every band needs goes first, whole; the other one is cut into
    // bands. Cutting C into column bands sends all of A first, cutting it into row bands
    // all of B: whichever is smaller goes first, so the first band starts sooner. (The
    // softmax epilogue needs whole rows, so it always uses row bands.)
    // 4 bands; 8 from 256 MiB of output on (MLP 8200 x 16384: 2.195 -> 2.168 ms per call, the
    // host link being the bound either way; 2 bands: 2.407 ms)
    const int parts = c_b < kHostChunkMinBytes ? 1 : (c_b >= 8 * kHostChunkMinBytes ? kHostChunksMax : 4);
    const bool by_cols = parts > 1 && a_b < b_b && epilogue != GEMM_EPI_SOFTMAX;
    if (by_cols) {
        int64_t cols = (N + parts - 1) / parts;
        cols = (cols + 255) / 256 * 256;   // whole 256-column tiles
        const int bands = static_cast<int>((N + cols - 1) / cols);
        // A large A is also cut in two row halves (the first of whole 256-row tiles), so that
        // the first GEMM needs half of A and one band of B, not all of A, before the first
        // download can start. Uploads go once each, in the order the GEMMs need them: A_0,
        // B_0, A_1, B_1, B_2, ...; GEMM (i, j) waits for A_i and B_j.
        int64_t rows_h = M;
        if (a_b >= kHostChunkMinBytes) {
            const int64_t h = (M / 2 + 255) / 256 * 256;
            if (h < M)
                rows_h = h;
        }
        const int halves = rows_h < M ? 2 : 1;
        const size_t pitch = static_cast<size_t>(N) * 2;
        cudaEvent_t *ev_a = ctx->ev_in, *ev_b = ctx->ev_in + 2;   // after A_i, after B_j
        auto upload_a = [&](int i) -> cudaError_t {
            const int64_t r0 = i * rows_h, mi = std::min<int64_t>(rows_h, M - r0);
            const size_t off = static_cast<size_t>(r0) * K * 2, len = static_cast<size_t>(mi) * K * 2;
            cudaError_t err = len ? cudaMemcpyAsync(dA + off, static_cast<const char *>(A) + off, len,
                                                    cudaMemcpyHostToDevice, ctx->copy_in)
                                  : cudaSuccess;
            return err == cudaSuccess ? cudaEventRecord(ev_a[i], ctx->copy_in) : err;
        };
        auto upload_b = [&](int j) -> cudaError_t {
            const int64_t c0 = j * cols, nj = std::min<int64_t>(cols, N - c0);
            const size_t off = static_cast<size_t>(c0) * 2;
            cudaError_t err = K > 0 ? cudaMemcpy2DAsync(dB + off, pitch, static_cast<const char *>(B) + off, pitch,
                                                        static_cast<size_t>(nj) * 2, static_cast<size_t>(K),
                                                        cudaMemcpyHostToDevice, ctx->copy_in)
                                    : cudaSuccess;
            return err == cudaSuccess ? cudaEventRecord(ev_b[j], ctx->copy_in) : err;
        };
        if ((e = upload_a(0)) != cudaSuccess || (e = upload_b(0)) != cudaSuccess ||
            (halves == 2 && (e = upload_a(1)) != cudaSuccess))
            return cuda_fail(ctx, e, GEMM_ERR_LAUNCH);
        for (int j = 1; j < bands; ++j)
            if ((e = upload_b(j)) != cudaSuccess)
                return cuda_fail(ctx, e, GEMM_ERR_LAUNCH);
        int k = 0;
        for (int j = 0; j < bands; ++j) {
            const int64_t c0 = j * cols, nj = std::min<int64_t>(cols, N - c0);
            const size_t off = static_cast<size_t>(c0) * 2, width = static_cast<size_t>(nj) * 2;
            for (int i = 0; i < halves; ++i, ++k) {
                const int64_t r0 = i * rows_h, mi = std::min<int64_t>(rows_h, M - r0);
                const size_t a_off = static_cast<size_t>(r0) * K * 2, c_off = static_cast<size_t>(r0) * pitch + off;
                if ((e = cudaStreamWaitEvent(s, ev_a[i], 0)) != cudaSuccess ||
                    (e = cudaStreamWaitEvent(s, ev_b[j], 0)) != cudaSuccess)
                    return cuda_fail(ctx, e, GEMM_ERR_LAUNCH);
                rc = launch(ctx, static_cast<int>(mi), static_cast<int>(nj), static_cast<int>(K),
                            K ? dA + a_off : nullptr, K ? dB + off : nullptr, dbias ? dbias + off : nullptr,
                            dC + c_off, epilogue, s, N, N);
                if (rc != GEMM_OK)
                    return rc;
                if ((e = cudaEventRecord(ctx->ev_mm[k], s)) != cudaSuccess ||
                    (e = cudaStreamWaitEvent(ctx->copy_out, ctx->ev_mm[k], 0)) != cudaSuccess)
                    return cuda_fail(ctx, e, GEMM_ERR_LAUNCH);
                if ((e = cudaMemcpy2DAsync(static_cast<char *>(C) + c_off, pitch, dC + c_off, pitch, width,
                                           static_cast<size_t>(mi), cudaMemcpyDeviceToHost, ctx->copy_out)) !=
                    cudaSuccess)
                    return cuda_fail(ctx, e, GEMM_ERR_LAUNCH);
            }
        }
    } else {
        int64_t rows = (M + parts - 1) / parts;
        rows = (rows + 255) / 256 * 256;   // whole 256-row tiles
        const int chunks = static_cast<int>((M + rows - 1) / rows);
        if (b_b && (e = cudaMemcpyAsync(dB, B, b_b, cudaMemcpyHostToDevice, s)) != cudaSuccess)
            return cuda_fail(ctx, e, GEMM_ERR_LAUNCH);
        for (int i = 0; i < chunks; ++i) {
            const int64_t r0 = i * rows, mi = std::min<int64_t>(rows, M - r0);
            const size_t a_off = static_cast<size_t>(r0) * K * 2, c_off = static_cast<size_t>(r0) * N * 2;
            const size_t a_len = static_cast<size_t>(mi) * K * 2, c_len = static_cast<size_t>(mi) * N * 2;
            if (a_len && (e = cudaMemcpyAsync(dA + a_off, static_cast<const char *>(A) + a_off, a_len,
                                              cudaMemcpyHostToDevice, ctx->copy_in)) != cudaSuccess)
                return cuda_fail(ctx, e, GEMM_ERR_LAUNCH);
            if ((e = cudaEventRecord(ctx->ev_in[i], ctx->copy_in)) != cudaSuccess ||
                (e = cudaStreamWaitEvent(s, ctx->ev_in[i], 0)) != cudaSuccess)
                return cuda_fail(ctx, e, GEMM_ERR_LAUNCH);
            rc = launch(ctx, static_cast<int>(mi), static_cast<int>(N), static_cast<int>(K), K ? dA + a_off : nullptr,
                        K ? dB : nullptr, dbias, dC + c_off, epilogue, s);
            if (rc != GEMM_OK)
                return rc;
            if ((e = cudaEventRecord(ctx->ev_mm[i], s)) != cudaSuccess ||
                (e = cudaStreamWaitEvent(ctx->copy_out, ctx->ev_mm[i], 0)) != cudaSuccess)
                return cuda_fail(ctx, e, GEMM_ERR_LAUNCH);
            if ((e = cudaMemcpyAsync(static_cast<char *>(C) + c_off, dC + c_off, c_len, cudaMemcpyDeviceToHost,
                                     ctx->copy_out)) != cudaSuccess)
                return cuda_fail(ctx, e, GEMM_ERR_LAUNCH);
        }
    }
    if ((e = cudaEventRecord(ctx->ev_done, ctx->copy_out)) != cudaSuccess ||
        (e = cudaStreamWaitEvent(s, ctx->ev_done, 0)) != cudaSuccess ||
        (e = cudaStreamSynchronize(s)) != cudaSuccess)
        return cuda_fail(ctx, e, GEMM_ERR_LAUNCH);
    return gemm_last_device_error(ctx, nullptr);
}

int gemm_last_device_error(gemm_ctx *ctx, uint32_t *detail)
{
    if (!ctx)
        return GEMM_ERR_ARG;
    DeviceGuard guard(ctx->device);
    uint32_t w = 0;
    cudaError_t e = cudaMemcpy(&w, ctx->d_err, sizeof(w), cudaMemcpyDeviceToHost);
    if (e == cudaSuccess && w != 0)
        e = cudaMemset(ctx->d_err, 0, sizeof(uint32_t));
    // a kernel that gave up may have left stream-K ready flags raised: lower them all
    if (e == cudaSuccess && w != 0)
        e = cudaMemset(ctx->sk_flags, 0, static_cast<size_t>(ctx->num_sms) * Cfg::NUM_EPI_WARPS * sizeof(uint32_t));
    if (e != cudaSuccess)
        return cuda_fail(ctx, e, GEMM_ERR_LAUNCH);
    if (detail)
        *detail = w;
    return w ? GEMM_ERR_TIMEOUT : GEMM_OK;
}

int gemm_last_cuda_error(gemm_ctx *ctx) { return ctx ? ctx->last_cuda_error : 0; }

int gemm_destroy(gemm_ctx *ctx)
{
    if (!ctx)
        return GEMM_OK;
    {
        DeviceGuard guard(ctx->device);
        if (ctx->d_err)
            cudaFree(ctx->d_err);
        if (ctx->sk_ws)
            cudaFree(ctx->sk_ws);
        if (ctx->sk_flags)
            cudaFree(ctx->sk_flags);
        if (ctx->stage)
            cudaFree(ctx->stage);
        for (int i = 0; i < 2 * kHostChunksMax; ++i) {
            if (ctx->ev_in[i])
                cudaEventDestroy(ctx->ev_in[i]);
            if (ctx->ev_mm[i])
                cudaEventDestroy(ctx->ev_mm[i]);
        }
        if (ctx->ev_start)
            cudaEventDestroy(ctx->ev_start);
        if (ctx->ev_done)
            cudaEventDestroy(ctx->ev_done);
        if (ctx->copy_in)
            cudaStreamDestroy(ctx->copy_in);
        if (ctx->copy_out)
            cudaStreamDestroy(ctx->copy_out);
        cudaGetLastError();
    }
    delete ctx;
    return GEMM_OK;
}

const char *gemm_status_string(int status)
{
    switch (status) {
    case GEMM_OK: return "GEMM_OK";
    case GEMM_ERR_ARG: return "GEMM_ERR_ARG: invalid argument";
    case GEMM_ERR_ALIGN: return "GEMM_ERR_ALIGN: pointer not 16-byte aligned or N, K not multiples of 8";
    case GEMM_ERR_DEVICE: return "GEMM_ERR_DEVICE: device missing, not sm_103, or buffer not on the device";
    case GEMM_ERR_LAUNCH: return "GEMM_ERR_LAUNCH: a CUDA call failed";
    case GEMM_ERR_TIMEOUT: return "GEMM_ERR_TIMEOUT: an in-kernel wait ran out";
    case GEMM_ERR_NOMEM: return "GEMM_ERR_NOMEM: allocation failed";
    default: return "unknown gemm status";
    }
}

int gemm_num_sms(gemm_ctx *ctx) { return ctx ? ctx->num_sms : 0; }

int gemm_describe(gemm_ctx *ctx, int64_t M, int64_t N, int64_t K, int epilogue, char *buf, int64_t len)
{
    if (!buf || len <= 0)
        return GEMM_ERR_ARG;
    buf[0] = '\0';
    const int rc = check_shape(ctx, M, N, K, epilogue);
    if (rc != GEMM_OK)
        return rc;
    if (M == 0 || N == 0) {
        std::snprintf(buf, static_cast<size_t>(len), "none (empty problem, nothing is launched)");
        return GEMM_OK;
    }
    const Plan pl = make_plan(ctx, static_cast<int>(M), static_cast<int>(N), static_cast<int>(K), epilogue);
    const int n = std::snprintf(buf, static_cast<size_t>(len), "%s grid=%d cluster=%d tiles=%d",
                                plan_kernel_name(pl.kind), pl.grid, pl.cluster, pl.num_tiles);
    if (pl.kind == PLAN_PAIR && pl.pair_units > pl.num_tiles && n > 0 && n < len)
        std::snprintf(buf + n, static_cast<size_t>(len - n), " (last %d split in N-halves)",
                      pl.num_tiles - pl.pair_split_from);
    return GEMM_OK;
}

int gemm_num_pairs(gemm_ctx *ctx) { return ctx ? ctx->max_clusters : 0; }

int gemm_clock_trace(gemm_ctx *ctx, uint64_t *trace, int max_samples, uint64_t interval_ns, uint64_t duration_ns,
                     void *stream)
{
    if (!ctx || !trace || max_samples < 1 || max_samples > (1 << 20) || interval_ns < 1000u ||
        interval_ns > 10000000u || duration_ns > 10000000000ull)
        return GEMM_ERR_ARG;
    if (!aligned16(trace))
        return GEMM_ERR_ALIGN;
    if (!on_device(trace, ctx->device))
        return GEMM_ERR_DEVICE;
    DeviceGuard guard(ctx->device);
    gb300::clock_probe_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(trace, max_samples, interval_ns,
                                                                               duration_ns);
    const cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? GEMM_OK : cuda_fail(ctx, e, GEMM_ERR_LAUNCH);
}

int gemm_attention_fwd(gemm_ctx *ctx, int64_t heads, int64_t seq_q, int64_t seq_k, int64_t head_dim, const void *Q,
                       const void *K, const void *V, void *O, float scale, int causal, void *stream)
{
    using Cfg = gb300::AttnConfig;
    if (!ctx || heads < 0 || seq_q < 0 || seq_k < 0 || heads > INT32_MAX || seq_q > INT32_MAX || seq_k > INT32_MAX)
        return GEMM_ERR_ARG;
    if (head_dim != Cfg::D || (causal != 0 && causal != 1) || !(scale == scale))
        return GEMM_ERR_ARG;
    if (heads == 0 || seq_q == 0)
        return GEMM_OK;
    if (seq_k == 0 || !Q || !K || !V || !O)
        return GEMM_ERR_ARG;
    if (!aligned16(Q) || !aligned16(K) || !aligned16(V) || !aligned16(O))
        return GEMM_ERR_ALIGN;
    const size_t qb = static_cast<size_t>(heads) * seq_q * Cfg::D * 2, kb = static_cast<size_t>(heads) * seq_k * Cfg::D * 2;
    if (overlaps(O, qb, Q, qb) || overlaps(O, qb, K, kb) || overlaps(O, qb, V, kb))
        return GEMM_ERR_ARG;
    const int64_t q_blocks = (seq_q + Cfg::TILES * Cfg::BQ - 1) / (Cfg::TILES * Cfg::BQ);
    if (heads * q_blocks > INT32_MAX)
        return GEMM_ERR_ARG;
    if (!on_device(Q, ctx->device) || !on_device(K, ctx->device) || !on_device(V, ctx->device) ||
        !on_device(O, ctx->device))
        return GEMM_ERR_DEVICE;
    DeviceGuard guard(ctx->device);
    // [head][row][dim] views, boxes of 64 dims (one 128-byte swizzle row) x box_rows rows:
    // 128 query rows (a query tile), 128 key rows (a key block)
    auto encode_3d = [&](CUtensorMap *map, const void *ptr, int64_t rows, uint32_t box_rows) {
        const cuuint64_t dims[3] = {static_cast<cuuint64_t>(Cfg::D), static_cast<cuuint64_t>(rows),
                                    static_cast<cuuint64_t>(heads)};
        const cuuint64_t strides[2] = {static_cast<cuuint64_t>(Cfg::D) * 2, static_cast<cuuint64_t>(rows) * Cfg::D * 2};
        const cuuint32_t box[3] = {64, box_rows, 1};
        const cuuint32_t estr[3] = {1, 1, 1};
        return ctx->encode(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, const_cast<void *>(ptr), dims, strides, box, estr,
                           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
    };
    // O: stores of 32 rows (one softmax warp's share of a query tile)
    CUtensorMap tq, tk, tv, to;
    if (!encode_3d(&tq, Q, seq_q, Cfg::BQ) || !encode_3d(&tk, K, seq_k, Cfg::BKV) ||
        !encode_3d(&tv, V, seq_k, Cfg::BKV) || !encode_3d(&to, O, seq_q, 32))
        return GEMM_ERR_LAUNCH;
    gb300::AttnParams p;
    p.H = static_cast<int>(heads);
    p.Sq = static_cast<int>(seq_q);
    p.Sk = static_cast<int>(seq_k);
    p.q_blocks = static_cast<int>(q_blocks);
    p.causal = causal;
    p.scale_log2 = scale * 1.4426950408889634f;
    p.err = ctx->d_err;
    p.timeout_ns = ctx->timeout_ns;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(heads * q_blocks), 1, 1);
    cfg.blockDim = dim3(Cfg::NUM_THREADS, 1, 1);
    cfg.dynamicSmemBytes = Cfg::SMEM_BYTES;
    cfg.stream = static_cast<cudaStream_t>(stream);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaLaunchKernelEx(&cfg, gb300::attention_fwd_kernel, tq, tk, tv, to, p);
    const cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? GEMM_OK : cuda_fail(ctx, e, GEMM_ERR_LAUNCH);
}


int gemm_row_softmax(gemm_ctx *ctx, int64_t rows, int64_t cols, const void *X, void *Y, void *stream)
{
    if (!ctx || rows < 0 || cols < 0 || cols > INT32_MAX)
        return GEMM_ERR_ARG;
    if (rows == 0 || cols == 0)
        return GEMM_OK;
    if (!X || !Y)
        return GEMM_ERR_ARG;
    if (cols % 8 != 0 || !aligned16(X) || !aligned16(Y))
        return GEMM_ERR_ALIGN;
    const size_t bytes = static_cast<size_t>(rows) * static_cast<size_t>(cols) * 2;
    if (X != Y && overlaps(X, bytes, Y, bytes))   // in place is fine, partial overlap is not
        return GEMM_ERR_ARG;
    if (!on_device(X, ctx->device) || !on_device(Y, ctx->device))
        return GEMM_ERR_DEVICE;
    DeviceGuard guard(ctx->device);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const int c = static_cast<int>(cols);
    const __half *x = static_cast<const __half *>(X);
    __half *y = static_cast<__half *>(Y);
    // Rows held in registers (see launch_softmax_regs): a warp per row up to 2048 columns, a
    // 256-thread CTA per row up to 16384. Where it measured faster, the CTAs per SM are as
    // many as the registers allow without spilling (3 at 8 vectors per thread: 80 registers;
    // 5 at 4 with a CTA per row: 48), since the bytes in flight per SM are what keep HBM busy
    // (three rows of 16384 per SM instead of two: 88 -> 79 us at 8192 rows). Longer rows go
    // to the streaming kernel (faster than 16 vectors per thread at one CTA per SM: the row's
    // loads and arithmetic cannot overlap).
    if (cols <= 256)
        launch_softmax_regs<32, 1, 8>(rows, c, x, y, st);
    else if (cols <= 512)
        launch_softmax_regs<32, 2, 8>(rows, c, x, y, st);
    else if (cols <= 1024)
        launch_softmax_regs<32, 4, 4>(rows, c, x, y, st);
    else if (cols <= 2048)
        launch_softmax_regs<32, 8, 3>(rows, c, x, y, st);
    else if (cols <= 4096)
        launch_softmax_regs<256, 2, 8>(rows, c, x, y, st);
    else if (cols <= 8192)
        launch_softmax_regs<256, 4, 5>(rows, c, x, y, st);
    else if (cols <= 16384)
        launch_softmax_regs<256, 8, 3>(rows, c, x, y, st);
    else {   // longer rows: streamed (read once up to 32768 columns)
        const int64_t blocks = std::min<int64_t>(rows, static_cast<int64_t>(ctx->num_sms) * 8);
        gb300::row_softmax_kernel<256><<<static_cast<unsigned>(blocks), 256, 0, st>>>(x, y, rows, c);
    }
    const cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? GEMM_OK : cuda_fail(ctx, e, GEMM_ERR_LAUNCH);
}

int gemm_set_timeout_ns(gemm_ctx *ctx, uint64_t ns)
{
    if (!ctx)
        return GEMM_ERR_ARG;
    ctx->timeout_ns = std::max(ns, kMinTimeoutNs);
    return GEMM_OK;
}

int gemm_set_debug(gemm_ctx *ctx, int flags)
{
    if (!ctx || (flags & ~(GEMM_DEBUG_WITHHOLD_FIRST_LOAD | GEMM_DEBUG_FORCE_SINGLE | GEMM_DEBUG_FORCE_PAIR |
                           GEMM_DEBUG_FORCE_STREAMK | GEMM_DEBUG_FORCE_SPLITK)))
        return GEMM_ERR_ARG;
    ctx->debug = flags;
    return GEMM_OK;
}

}  // extern "C"
