// Bounded grid barrier of the cooperative routing kernels of libep_gb300
// (internal, not part of the C ABI).  Every block of a launch arrives once and
// waits until every block has arrived, or gives up after kBarrierNs.
#pragma once

#include <cstdint>

#include "ep_device.cuh"

namespace ep {

constexpr uint64_t kBarrierNs = 500000000ull;   // 0.5 s

__device__ __forceinline__ void st_release_u64(unsigned long long *p, unsigned long long v)
{
    asm volatile("st.release.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

__device__ __forceinline__ unsigned long long ld_acquire_u64(const unsigned long long *p)
{
    unsigned long long v;
    asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}

// Grid barrier of the cooperative routing kernels.  A launch's tag mixes the
// host's per-call tag with a launch counter kept in the workspace header, so
// that replays of one captured launch (a CUDA graph repeats the host tag)
// still get a tag that no flag left by an earlier launch holds; the workspace
// needs no initialisation.  Block 0 advances the counter after its wait: by
// then every block has arrived, and a block reads the counter before it
// arrives.
struct GridBarrier {
    unsigned long long *flags;    // [gridDim]
    unsigned long long *epoch;    // launch counter (workspace header)
    unsigned long long host_tag;  // different for every host call
};

// Thread 0 only: this launch's tag and the counter value it was made from.
__device__ __forceinline__ unsigned long long barrier_tag(const GridBarrier &g, unsigned long long *e_out)
{
    const unsigned long long e = *reinterpret_cast<const volatile unsigned long long *>(g.epoch);
    *e_out = e;
    const unsigned long long tag = g.host_tag ^ (e * 0x9e3779b97f4a7c15ull);
    return tag != 0 ? tag : 1;
}

// Thread 0 only, after a __syncthreads that follows every write the other
// blocks will read.
__device__ __forceinline__ void barrier_arrive(const GridBarrier &g, unsigned long long tag)
{
    // st.release orders before the flag every write of this thread and, via
    // the preceding __syncthreads, of the whole block (release is cumulative)
    st_release_u64(&g.flags[blockIdx.x], tag);
}

// Whole block: waits (bounded) for every block's flag; false for the whole
// block if one did not arrive in time.  *s_fail is a shared word cleared
// before the block's first __syncthreads.
__device__ __forceinline__ bool barrier_wait(const GridBarrier &g, unsigned long long tag, unsigned long long e, int *s_fail)
{
    // spin with acquire loads (each pairs with the release of the block's
    // barrier_arrive), then __syncthreads carries the ordering to the rest of
    // the block.  Measured on an otherwise empty cooperative launch of 128
    // blocks: 6.6 us with acquire polling, about 11 us with relaxed polling
    // followed by an acquire fence.
    bool ok = true;
    for (int i = threadIdx.x; i < (int)gridDim.x && ok; i += blockDim.x) {
        if (ld_acquire_u64(&g.flags[i]) == tag)
            continue;
        const uint64_t t0 = global_timer_ns();
        while (ld_acquire_u64(&g.flags[i]) != tag)
            if (global_timer_ns() - t0 > kBarrierNs) {
                ok = false;
                break;
            }
    }
    if (!ok)
        *s_fail = 1;
    __syncthreads();
    if (blockIdx.x == 0 && threadIdx.x == 0)
        *reinterpret_cast<volatile unsigned long long *>(g.epoch) = e + 1;
    return *s_fail == 0;
}

}  // namespace ep
