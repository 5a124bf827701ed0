// Device helpers of the expert-batched slot computations of libep_gb300
// (internal, not part of the C ABI): vLLM BatchedPrepareAndFinalize.prepare
// gives each local expert's tokens slots 0, 1, ... in token order.
#pragma once

#include <cstdint>

#include "ep_device.cuh"
#include "ep_internal.h"

namespace ep {

// Per-rank (or per-expert) totals over nb blocks' partial counts part[bb * P + p]
// and the sum over the blocks before block b, accumulated into the shared
// s_tot / s_before (zeroed by the caller) by slices of the block's threads.
__device__ __forceinline__ void block_rank_sums(const int32_t *__restrict__ part, int nb, int P, int b,
                                                int32_t *s_tot, int32_t *s_before)
{
    const int nsl = blockDim.x / P;
    const int p = threadIdx.x % P, sl = threadIdx.x / P;
    if (sl >= nsl)
        return;
    int tot = 0, bef = 0;
    for (int bb0 = sl; bb0 < nb; bb0 += nsl * 8) {
        int v[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int bb = bb0 + u * nsl;
            v[u] = bb < nb ? part[(int64_t)bb * P + p] : 0;
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            tot += v[u];
            bef += (bb0 + u * nsl < b) ? v[u] : 0;
        }
    }
    if (tot != 0)
        atomicAdd(&s_tot[p], tot);
    if (bef != 0)
        atomicAdd(&s_before[p], bef);
}

// Block 0's per-expert totals: kept count, aligned tokens_per_expert, drops.
__device__ __forceinline__ int finish_expert_count(const SlotLimits &L, int e, int tot, int32_t *tokens_per_expert)
{
    const int kept = min(tot, L.cap);
    tokens_per_expert[e] = min((kept + L.align - 1) / L.align * L.align, L.M);
    if (L.dropped != nullptr)
        L.dropped[e] = tot - kept;
    if (L.kept != nullptr)
        L.kept[e] = kept;
    return tot > L.cap && !L.silent ? EP_ERR_CAPACITY : 0;
}

// Transpose of the warp's 32 x 32 bit matrix (row l = lane l's word): lane e
// gets the word whose bit l is bit e of lane l's word.  Recursive block
// transpose, halving the block size each step (16, 8, 4, 2, 1).
__device__ __forceinline__ uint32_t warp_transpose32(uint32_t x, int lane)
{
    uint32_t m = 0x0000ffffu;
#pragma unroll
    for (int j = 16; j > 0; j >>= 1, m ^= m << j) {
        const uint32_t y = __shfl_xor_sync(kFull, x, j);
        x = (lane & j) ? (((y >> j) & m) | (x & ~m)) : ((x & m) | ((y & m) << j));
    }
    return x;
}

}  // namespace ep
