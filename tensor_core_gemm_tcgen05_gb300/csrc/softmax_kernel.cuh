// Row-wise softmax, FP16 in and out, FP32 arithmetic, for sm_103a:
//
//     Y[r][j] = exp(X[r][j] - m_r) / sum_k exp(X[r][k] - m_r),   m_r = max_k X[r][k]
//
// The tutorial's row softmax ("TileLang: Criando Kernels de GPU ..." on noticiai.com.br,
// section "Softmax por linha e FlashAttention": per row the maximum, the subtraction, the
// exponential and the normalisation; "TileLang ..." on pro.edgex.exchange: max and sum
// reductions kept in registers). The work is bound by HBM bandwidth (one read and one write
// of every element), so the kernel is built for bandwidth, not tensor cores:
//  * a group of G threads (one warp, or a 256-thread CTA for long rows) owns a row; rows are
//    walked by a persistent grid;
//  * pass 1 streams the row with 16-byte loads and keeps, per thread, a running maximum m
//    and a sum s of exp(x - m) that is rescaled whenever m grows (the "online" form, so the
//    row is read once for both statistics); the (m, s) pairs of the group are merged with
//    warp shuffles (and shared memory across warps);
//  * pass 2 reads the row again (it was just read, so from L2/L1) and writes
//    exp(x - m) * (1 / s) with 16-byte stores.
#pragma once

#include <cuda_fp16.h>

#include <cstdint>

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
