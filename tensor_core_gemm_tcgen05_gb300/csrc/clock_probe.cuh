// Measurement aid: the SM clock as the hardware counts it while other kernels run.
//
// One thread samples the SM cycle counter (clock64) and the global nanosecond timer at fixed
// intervals and writes the pairs to global memory; between samples it sleeps. Launched on a
// stream of its own, it shares an SM with the kernel being timed (one warp slot, no shared
// memory), and the cycles per nanosecond between consecutive samples are the SM clock that
// kernel ran at, at a resolution that power-sensor polling from the host does not reach.
#pragma once

#include <cstdint>

#include "ptx.cuh"

namespace gb300 {

__device__ __forceinline__ uint64_t sm_clock64()
{
    uint64_t c;
    asm volatile("mov.u64 %0, %%clock64;" : "=l"(c));
    return c;
}

// trace[2i] = global timer (ns), trace[2i + 1] = clock64, for i < max_samples, one sample
// every interval_ns until duration_ns has passed. Every loop is bounded: each wait ends at
// the next sample time, and there are at most max_samples of them.
__global__ void clock_probe_kernel(uint64_t *trace, int max_samples, uint64_t interval_ns, uint64_t duration_ns)
{
    if (threadIdx.x != 0 || blockIdx.x != 0)
        return;
    const uint64_t t0 = global_timer_ns();
    uint64_t next = t0;
    for (int i = 0; i < max_samples; ++i) {
        uint64_t t = global_timer_ns();
        while (t < next) {
            const uint64_t left = next - t;
            __nanosleep(static_cast<unsigned>(left < 20000u ? left : 20000u));
            t = global_timer_ns();
        }
        const uint64_t c = sm_clock64();
        trace[2 * i] = t;
        trace[2 * i + 1] = c;
        if (t - t0 >= duration_ns)
            break;
        next += interval_ns;
    }
}

}  // namespace gb300
