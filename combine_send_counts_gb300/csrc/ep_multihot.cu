// Top-k indices to a multihot routing map and dense probabilities:
// NeMo AutoModel token_dispatcher, _DeepepManager._indices_to_multihot and
// _HybridEPManager._indices_to_multihot.
//
//   routing_map[t,e] = 1 iff some slot k of token t names expert e;
//   probs[t,e]       = sum over those slots of topk_probs[t,k], fp32 from
//                      +0.0f in ascending k (one slot: its probability).
//
// HBM-bound output writes (T*E bytes + 4*T*E bytes) from a small input (12*T*K
// bytes).  One warp per token: lanes k < K load slot k's id and probability in
// one coalesced load, the warp broadcasts them by shuffle, and lane l owns the
// 8 experts [8l, 8l+8) of each 256-expert window, accumulating in registers
// and writing one 8-byte map store and two 16-byte probability stores, so
// the warp's stores cover 256 contiguous bytes of map and 1 KB of probs.
#include "ep_device.cuh"
#include "ep_internal.h"

namespace ep {
namespace {

constexpr int kMultihotThreads = 256;
constexpr int kMultihotWarps = kMultihotThreads / 32;

template <bool VEC>
__global__ void __launch_bounds__(kMultihotThreads)
multihot_kernel(const int64_t *__restrict__ idx, const float *__restrict__ p, int64_t T, int K, int E,
                uint8_t *__restrict__ routing_map, float *__restrict__ probs, int32_t *err)
{
    const int lane = threadIdx.x & 31;
    const int64_t t = (int64_t)blockIdx.x * kMultihotWarps + (threadIdx.x >> 5);
    if (t >= T)
        return;   // whole warp
    int64_t my_id = -1;
    float my_p = 0.0f;
    if (lane < K) {
        my_id = idx[t * K + lane];
        if (probs != nullptr)   // topk_probs may be NULL for a map-only call
            my_p = p[t * K + lane];
    }
    const bool bad = lane < K && (my_id < -1 || my_id >= E);
    if (bad)
        my_id = -1;   // ignored slot
    if (__any_sync(kFull, bad) && lane == 0)
        raise(err, EP_ERR_INVALID_EXPERT);
    for (int w0 = 0; w0 < E; w0 += 256) {
        const int e0 = w0 + 8 * lane;
        float acc[8];
#pragma unroll
        for (int j = 0; j < 8; ++j)
            acc[j] = 0.0f;
        uint32_t hit = 0;
        for (int k = 0; k < K; ++k) {   // ascending k: the sum order
            const int64_t id = __shfl_sync(kFull, my_id, k);
            const float pk = __shfl_sync(kFull, my_p, k);
            const int64_t j = id - e0;
            if (id >= 0 && j >= 0 && j < 8) {
#pragma unroll
                for (int jj = 0; jj < 8; ++jj)   // static register index
                    if (jj == j)
                        acc[jj] = __fadd_rn(acc[jj], pk);
                hit |= 1u << j;
            }
        }
        if (e0 >= E)
            continue;
        if (VEC) {
            uint32_t lo = 0, hi = 0;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                lo |= ((hit >> j) & 1u) << (8 * j);
                hi |= ((hit >> (j + 4)) & 1u) << (8 * j);
            }
            if (routing_map != nullptr)
                *reinterpret_cast<uint2 *>(routing_map + t * E + e0) = make_uint2(lo, hi);
            if (probs != nullptr) {
                float4 *dst = reinterpret_cast<float4 *>(probs + t * E + e0);
                dst[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
                dst[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
            }
        } else {
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                if (e0 + j >= E)
                    break;
                if (routing_map != nullptr)
                    routing_map[t * E + e0 + j] = (uint8_t)((hit >> j) & 1u);
                if (probs != nullptr)
                    probs[t * E + e0 + j] = acc[j];
            }
        }
    }
}

}  // namespace
}  // namespace ep

using namespace ep;

extern "C" int ep_indices_to_multihot(const int64_t *topk_idx, const float *topk_probs, int64_t T, int K, int E,
                                      uint8_t *routing_map, float *probs, int32_t *err, ep_stream_t stream_)
{
    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
    if (T < 0 || K < 1 || K > EP_MAX_TOPK || E < 1 || E > EP_MAX_EXPERTS)
        return EP_ERR_INVALID_ARG;
    if (T == 0)
        return EP_OK;
    if (topk_idx == nullptr || (routing_map == nullptr && probs == nullptr) || (probs != nullptr && topk_probs == nullptr))
        return EP_ERR_INVALID_ARG;
    if ((int64_t)T * E >= ((int64_t)1 << 40))
        return EP_ERR_UNSUPPORTED;
    const int64_t blocks = ceil_div(T, kMultihotWarps);
    const bool vec = E % 8 == 0 && (routing_map == nullptr || aligned(routing_map, 8)) &&
                     (probs == nullptr || aligned(probs, 16));
    if (vec)
        multihot_kernel<true><<<blocks, kMultihotThreads, 0, stream>>>(topk_idx, topk_probs, T, K, E, routing_map,
                                                                       probs, err);
    else
        multihot_kernel<false><<<blocks, kMultihotThreads, 0, stream>>>(topk_idx, topk_probs, T, K, E, routing_map,
                                                                        probs, err);
    return launch_status();
}
