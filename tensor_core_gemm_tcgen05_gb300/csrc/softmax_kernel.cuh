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
//  * Longer rows (row_softmax_kernel): pass 1 streams the row with 16-byte loads and keeps,
//    per thread, a running maximum m and a sum s of exp(x - m) that is rescaled whenever m
//    grows (the "online" form, so the row is read once for both statistics); pass 2 reads
//    the row again and writes exp(x - m) * (1 / s) with 16-byte stores.
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

template <int G>   // threads per row: 32 (one warp) or a multiple of 32 up to the block size
__global__ void __launch_bounds__(256) row_softmax_kernel(const __half *__restrict__ X, __half *__restrict__ Y,
                                                          int64_t rows, int cols)
{
    static_assert(G == 32 || G == 256, "a warp or the whole block per row");
    constexpr int GROUPS = 256 / G;            // rows in flight per block
    __shared__ float red_m[8], red_s[8];
    const int group = threadIdx.x / G;
    const int t = threadIdx.x % G;             // thread within the row group
    const int lane = threadIdx.x & 31;
    const int vecs = cols / 8;                 // 16-byte vectors per row

    for (int64_t r = static_cast<int64_t>(blockIdx.x) * GROUPS + group; r < rows;
         r += static_cast<int64_t>(gridDim.x) * GROUPS) {
        const uint4 *xr = reinterpret_cast<const uint4 *>(X + r * cols);
        uint4 *yr = reinterpret_cast<uint4 *>(Y + r * cols);

        // pass 1: running max and rescaled sum of exponentials
        float m = -INFINITY, s = 0.0f;
        for (int v = t; v < vecs; v += G) {
            const uint4 q = __ldg(xr + v);
            const __half2 *h = reinterpret_cast<const __half2 *>(&q);
            float f[8];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float2 p = __half22float2(h[e]);
                f[2 * e] = p.x;
                f[2 * e + 1] = p.y;
            }
            float vm = f[0];
#pragma unroll
            for (int e = 1; e < 8; ++e)
                vm = fmaxf(vm, f[e]);
            const float mn = fmaxf(m, vm);
            if (mn == -INFINITY)
                continue;   // everything so far is -inf: nothing to add yet
            float add = 0.0f;
#pragma unroll
            for (int e = 0; e < 8; ++e)
                add += exp2f((f[e] - mn) * kLog2e);
            s = s * exp2f((m - mn) * kLog2e) + add;   // m = -inf at first: exp2f(-inf) = 0
            m = mn;
        }
        // merge within the warp
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            const float m2 = __shfl_xor_sync(0xffffffffu, m, off);
            const float s2 = __shfl_xor_sync(0xffffffffu, s, off);
            softmax_merge(m, s, m2, s2);
        }
        if constexpr (G > 32) {   // merge across the warps of the block
            const int warp = threadIdx.x >> 5;
            __syncthreads();      // the previous row's reads of red_* are done
            if (lane == 0) {
                red_m[warp] = m;
                red_s[warp] = s;
            }
            __syncthreads();
            m = red_m[0];
            s = red_s[0];
#pragma unroll
            for (int w = 1; w < G / 32; ++w)
                softmax_merge(m, s, red_m[w], red_s[w]);
        }
        const float inv = 1.0f / s;
        const float mb = m * kLog2e;

        // pass 2: write exp(x - m) / s
        for (int v = t; v < vecs; v += G) {
            const uint4 q = __ldg(xr + v);
            const __half2 *h = reinterpret_cast<const __half2 *>(&q);
            uint4 out;
            uint32_t *o = reinterpret_cast<uint32_t *>(&out);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float2 p = __half22float2(h[e]);
                const float a = exp2f(fmaf(p.x, kLog2e, -mb)) * inv;
                const float b = exp2f(fmaf(p.y, kLog2e, -mb)) * inv;
                __half2 hh = __floats2half2_rn(a, b);
                o[e] = *reinterpret_cast<uint32_t *>(&hh);
            }
            __stcs(yr + v, out);
        }
    }
}

}  // namespace gb300
