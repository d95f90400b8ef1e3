// Row-wise softmax, FP16 in and out, FP32 arithmetic, for sm_103a:
//
//     Y[r][j] = exp(X[r][j] - m_r) / sum_k exp(X[r][k] - m_r),   m_r = max_k X[r][k]
//
// The tutorial's row softmax ("TileLang: Criando Kernels de GPU ..." on noticiai.com.br,
// section "Softmax por linha e FlashAttention": per row the maximum, the subtraction, the
// exponential and the normalisation; "TileLang ..." on pro.edgex.exchange: max and sum
// reductions kept in registers). The work is bound by HBM bandwidth (one read and one write
// of every element), so the kernels are built for bandwidth, not tensor cores. A group of G
// threads (one warp, or a 256-thread CTA for long rows) owns a row.
//  * Rows of up to 16384 columns (row_softmax_regs_kernel): each thread loads its V 16-byte
//    vectors of the row at once (all loads in flight together, which is what keeps HBM busy)
//    and keeps them in registers; the maximum is taken on the FP16 values (exact), then the
//    sum of exp(x - m), then the outputs, all from the registers: X is read once.
//  * Longer rows (row_softmax_kernel): pass 1 reads the row once with 16-byte loads, keeping
//    per thread a running maximum m and a sum s of exp(x - m) that is rescaled whenever m
//    grows (the "online" form), and each thread's first 16 vectors in registers and shared
//    memory; pass 2 writes exp(x - m) * (1 / s) from those and reads only the rest of the
//    row again (rows of up to 32768 columns are read once).
// The (m, s) statistics of a group are merged with warp shuffles (and shared memory across
// the warps of a CTA).
#pragma once

#include <cuda_fp16.h>

#include <cstdint>

#include "ptx.cuh"

namespace gb300 {

constexpr float kLog2e = 1.4426950408889634f;

// Merge two (max, sum of exp(x - max)) pairs.
__device__ __forceinline__ void softmax_merge(float &m, float &s, float m2, float s2)
{
    const float mn = fmaxf(m, m2);
    if (mn == -INFINITY)   // both empty
        return;
    s = s * exp2f((m - mn) * kLog2e) + s2 * exp2f((m2 - mn) * kLog2e);
    m = mn;
}

// FP16 pairs as 32-bit words (bit casts, no memory).
__device__ __forceinline__ __half2 u32_as_half2(uint32_t u)
{
    return __halves2half2(__ushort_as_half(static_cast<unsigned short>(u & 0xFFFFu)),
                          __ushort_as_half(static_cast<unsigned short>(u >> 16)));
}
__device__ __forceinline__ uint32_t half2_as_u32(__half2 h)
{
    return static_cast<uint32_t>(__half_as_ushort(__low2half(h))) |
           (static_cast<uint32_t>(__half_as_ushort(__high2half(h))) << 16);
}

// Maximum of the 8 FP16 values of a vector, in FP16 (exact).
__device__ __forceinline__ __half2 hmax_vec(__half2 acc, const uint4 &q)
{
    return __hmax2(__hmax2(acc, __hmax2(u32_as_half2(q.x), u32_as_half2(q.y))),
                   __hmax2(u32_as_half2(q.z), u32_as_half2(q.w)));
}

// Sum of exp(x - m) over the two values of a pair (mb = m * log2 e). ex2.approx (MUFU;
// results below 2^-126 flush to 0, far under the smallest FP16 output).
__device__ __forceinline__ float exp_pair_sum(uint32_t u, float mb)
{
    const float2 p = __half22float2(u32_as_half2(u));
    return ex2_approx(fmaf(p.x, kLog2e, -mb)) + ex2_approx(fmaf(p.y, kLog2e, -mb));
}

// exp(x - m) / s of the two values of a pair, rounded to FP16.
__device__ __forceinline__ uint32_t softmax_pair(uint32_t u, float mb, float inv)
{
    const float2 p = __half22float2(u32_as_half2(u));
    return half2_as_u32(__floats2half2_rn(ex2_approx(fmaf(p.x, kLog2e, -mb)) * inv,
                                          ex2_approx(fmaf(p.y, kLog2e, -mb)) * inv));
}

// Block-wide reduction of one value per warp through shared memory: `op` merges.
template <int WARPS, class Op>
__device__ __forceinline__ float block_reduce(float v, float *red, int warp, int lane, Op op)
{
    __syncthreads();   // the previous use of red is over
    if (lane == 0)
        red[warp] = v;
    __syncthreads();
    float r = red[0];
#pragma unroll
    for (int w = 1; w < WARPS; ++w)
        r = op(r, red[w]);
    return r;
}

// G threads per row (a warp, or a whole CTA of 256 to 1024 threads), V 16-byte vectors per
// thread: rows of up to G * V * 8 columns, held in registers. The vectors past the row's end
// read as -inf (they add 0). A CTA has max(G, 256) threads (8 rows per CTA when G = 32);
// MIN_CTAS: CTAs per SM the register budget is sized for.
template <int G, int V, int MIN_CTAS>
__global__ void __launch_bounds__(G < 256 ? 256 : G, MIN_CTAS)
    row_softmax_regs_kernel(const __half *__restrict__ X, __half *__restrict__ Y, int64_t rows, int cols)
{
    static_assert(G == 32 || G == 256 || G == 512 || G == 1024, "a warp or the whole block per row");
    constexpr int BLOCK = G < 256 ? 256 : G;
    constexpr int GROUPS = BLOCK / G;
    __shared__ float red[BLOCK / 32];
    const int group = threadIdx.x / G;
    const int t = threadIdx.x % G;
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int vecs = cols / 8;
    const uint4 neg = make_uint4(0xFC00FC00u, 0xFC00FC00u, 0xFC00FC00u, 0xFC00FC00u);   // -inf

    // G > 32: every thread of the block takes the same rows (the block reductions need them all)
    for (int64_t r = static_cast<int64_t>(blockIdx.x) * GROUPS + group; r < rows;
         r += static_cast<int64_t>(gridDim.x) * GROUPS) {
        const uint4 *xr = reinterpret_cast<const uint4 *>(X + r * cols);
        uint4 q[V];
#pragma unroll
        for (int i = 0; i < V; ++i)
            q[i] = t + i * G < vecs ? __ldcs(xr + t + i * G) : neg;
        __half2 hm = u32_as_half2(0xFC00FC00u);
#pragma unroll
        for (int i = 0; i < V; ++i)
            hm = hmax_vec(hm, q[i]);
        float m = fmaxf(__low2float(hm), __high2float(hm));
#pragma unroll
        for (int off = 16; off > 0; off >>= 1)
            m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
        if constexpr (G > 32)
            m = block_reduce<G / 32>(m, red, warp, lane, [](float a, float b) { return fmaxf(a, b); });
        const float mb = m * kLog2e;

        float s = 0.0f;
#pragma unroll
        for (int i = 0; i < V; ++i)
            s += (exp_pair_sum(q[i].x, mb) + exp_pair_sum(q[i].y, mb)) +
                 (exp_pair_sum(q[i].z, mb) + exp_pair_sum(q[i].w, mb));
#pragma unroll
        for (int off = 16; off > 0; off >>= 1)
            s += __shfl_xor_sync(0xffffffffu, s, off);
        if constexpr (G > 32)
            s = block_reduce<G / 32>(s, red, warp, lane, [](float a, float b) { return a + b; });
        const float inv = 1.0f / s;

        uint4 *yr = reinterpret_cast<uint4 *>(Y + r * cols);
#pragma unroll
        for (int i = 0; i < V; ++i) {
            if (t + i * G < vecs)
                __stcs(yr + t + i * G, make_uint4(softmax_pair(q[i].x, mb, inv), softmax_pair(q[i].y, mb, inv),
                                                  softmax_pair(q[i].z, mb, inv), softmax_pair(q[i].w, mb, inv)));
        }
    }
}

// Running (max, sum of exp(x - max)) of a row piece, updated with N more 16-byte vectors
// (vectors past the row's end are -inf and add nothing): the vectors' maximum in FP16
// (exact), the old sum rescaled once. Nothing changes while every value so far is -inf.
template <int N>
__device__ __forceinline__ void online_update(float &m, float &s, const uint4 (&q)[N])
{
    __half2 hm = u32_as_half2(0xFC00FC00u);
#pragma unroll
    for (int i = 0; i < N; ++i)
        hm = hmax_vec(hm, q[i]);
    const float mn = fmaxf(m, fmaxf(__low2float(hm), __high2float(hm)));
    if (mn == -INFINITY)
        return;
    const float mb = mn * kLog2e;
    float add = 0.0f;
#pragma unroll
    for (int i = 0; i < N; ++i)
        add += (exp_pair_sum(q[i].x, mb) + exp_pair_sum(q[i].y, mb)) +
               (exp_pair_sum(q[i].z, mb) + exp_pair_sum(q[i].w, mb));
    s = s * ex2_approx((m - mn) * kLog2e) + add;   // m = -inf at first: the product is 0
    m = mn;
}

// Rows longer than row_softmax_regs_kernel takes (above 16384 columns): a 256-thread CTA per
// row, walked by a persistent grid. Pass 1 reads the row once, keeping each thread's first
// RV vectors in registers and its next SV in shared memory ([i][thread]: each thread reads
// back only what it wrote, so no barrier), and updates a running (max, rescaled sum); the
// CTA's statistics are merged with warp shuffles and shared memory; pass 2 writes exp(x - m)
// / s from registers, then from shared memory, and re-reads only the part of the row past
// (RV + SV) * 256 vectors (rows of up to 32768 columns are read once).
template <int G>
__global__ void __launch_bounds__(256) row_softmax_kernel(const __half *__restrict__ X, __half *__restrict__ Y,
                                                          int64_t rows, int cols)
{
    static_assert(G == 256, "the whole block per row");
    constexpr int RV = 8, SV = 8;
    __shared__ uint4 cache[SV][G];
    __shared__ float red_m[8], red_s[8];
    const int t = threadIdx.x;
    const int lane = t & 31;
    const int vecs = cols / 8;                 // 16-byte vectors per row
    const uint4 neg = make_uint4(0xFC00FC00u, 0xFC00FC00u, 0xFC00FC00u, 0xFC00FC00u);   // -inf

    for (int64_t r = blockIdx.x; r < rows; r += gridDim.x) {
        const uint4 *xr = reinterpret_cast<const uint4 *>(X + r * cols);
        uint4 *yr = reinterpret_cast<uint4 *>(Y + r * cols);

        // pass 1
        float m = -INFINITY, s = 0.0f;
        uint4 q[RV];
#pragma unroll
        for (int i = 0; i < RV; ++i)
            q[i] = t + i * G < vecs ? __ldcs(xr + t + i * G) : neg;
        {
            uint4 c[SV];
#pragma unroll
            for (int i = 0; i < SV; ++i)
                c[i] = t + (RV + i) * G < vecs ? __ldcs(xr + t + (RV + i) * G) : neg;
            online_update<RV>(m, s, q);
#pragma unroll
            for (int i = 0; i < SV; ++i)
                cache[i][t] = c[i];
            online_update<SV>(m, s, c);
        }
        for (int v = t + (RV + SV) * G; v < vecs; v += G) {
            const uint4 c[1] = {__ldg(xr + v)};   // read again in pass 2: keep it in L2
            online_update<1>(m, s, c);
        }
        // merge within the warp, then across the warps of the block
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            const float m2 = __shfl_xor_sync(0xffffffffu, m, off);
            const float s2 = __shfl_xor_sync(0xffffffffu, s, off);
            softmax_merge(m, s, m2, s2);
        }
        __syncthreads();   // the previous row's reads of red_* are done
        if (lane == 0) {
            red_m[t >> 5] = m;
            red_s[t >> 5] = s;
        }
        __syncthreads();
        m = red_m[0];
        s = red_s[0];
#pragma unroll
        for (int w = 1; w < G / 32; ++w)
            softmax_merge(m, s, red_m[w], red_s[w]);
        const float inv = 1.0f / s;
        const float mb = m * kLog2e;

        // pass 2: exp(x - m) / s
        auto out = [&](const uint4 &x) {
            return make_uint4(softmax_pair(x.x, mb, inv), softmax_pair(x.y, mb, inv), softmax_pair(x.z, mb, inv),
                              softmax_pair(x.w, mb, inv));
        };
#pragma unroll
        for (int i = 0; i < RV; ++i)
            if (t + i * G < vecs)
                __stcs(yr + t + i * G, out(q[i]));
#pragma unroll
        for (int i = 0; i < SV; ++i)
            if (t + (RV + i) * G < vecs)
                __stcs(yr + t + (RV + i) * G, out(cache[i][t]));
        for (int v = t + (RV + SV) * G; v < vecs; v += G)
            __stcs(yr + v, out(__ldg(xr + v)));
    }
}

}  // namespace gb300
