// Top-k indices to a multihot routing map and dense probabilities:
// NeMo AutoModel token_dispatcher, _DeepepManager._indices_to_multihot and
// _HybridEPManager._indices_to_multihot.
//
//   routing_map[t,e] = 1 iff some slot k of token t names expert e;
//   probs[t,e]       = sum over those slots of topk_probs[t,k], fp32 from
//                      +0.0f in ascending k (one slot: its probability).
//
// HBM-bound output writes (T*E bytes + 4*T*E bytes) from a small input (12*T*K
// bytes).  One warp per token at a time (a grid of one resident wave, warps
// looping over tokens).  Lanes k < K hold slot k; __match_any_sync
// groups the lanes naming the same expert and the lowest lane of each group
// sums the group's probabilities in ascending slot order (the order of the
// definition).  Per 256-expert window the warp zeroes a shared-memory row,
// the group leaders place their sums and hit flags, and each lane writes its 8
// experts with one 8-byte map store and two 16-byte probability stores, so a
// warp's stores cover 256 contiguous map bytes and 1 KB of probabilities.
#include <algorithm>
#include <atomic>

#include "ep_device.cuh"
#include "ep_internal.h"

namespace ep {
namespace {

constexpr int kMultihotThreads = 256;
constexpr int kMultihotWarps = kMultihotThreads / 32;
constexpr int kWindow = 256;   // experts per pass: 8 per lane

template <bool VEC>
__global__ void __launch_bounds__(kMultihotThreads)
multihot_kernel(const int64_t *__restrict__ idx, const float *__restrict__ p, int64_t T, int K, int E,
                uint8_t *__restrict__ routing_map, float *__restrict__ probs, int32_t *err)
{
    __shared__ __align__(16) float s_p[kMultihotWarps][kWindow];
    __shared__ __align__(16) uint8_t s_h[kMultihotWarps][kWindow];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t nw = (int64_t)gridDim.x * kMultihotWarps;
    int64_t t = (int64_t)blockIdx.x * kMultihotWarps + warp;
    // a token's slots: lane k < K holds slot k (id -1 = masked or ignored)
    auto load = [&](int64_t tt, int &id, float &pk, bool &bad) {
        id = -1;
        pk = 0.0f;
        bad = false;
        if (tt < T && lane < K) {
            const int64_t v = idx[tt * K + lane];
            bad = v < -1 || v >= E;
            id = bad ? -1 : (int)v;   // an invalid slot is ignored
            if (probs != nullptr)     // topk_probs may be NULL for a map-only call
                pk = p[tt * K + lane];
        }
    };
    int id, id_n;
    float pk, pk_n;
    bool bad, bad_n;
    load(t, id, pk, bad);
    float *sp = s_p[warp];
    uint8_t *sh = s_h[warp];
    for (; t < T; t += nw) {
        load(t + nw, id_n, pk_n, bad_n);   // the warp's next token, if any, loads while this one is written
        if (__any_sync(kFull, bad) && lane == 0)
            raise(err, EP_ERR_INVALID_EXPERT);
        const unsigned peers = __match_any_sync(kFull, id);
        const bool leader = id >= 0 && (peers & lanemask_lt()) == 0;
        float sum = 0.0f;   // the group's probabilities, ascending slot order from +0.0f
        if (id >= 0)
            for (unsigned m = peers; m != 0; m &= m - 1)
                sum = __fadd_rn(sum, __shfl_sync(peers, pk, __ffs(m) - 1));
        for (int w0 = 0; w0 < E; w0 += kWindow) {
            reinterpret_cast<float4 *>(sp)[2 * lane] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
            reinterpret_cast<float4 *>(sp)[2 * lane + 1] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
            reinterpret_cast<uint2 *>(sh)[lane] = make_uint2(0u, 0u);
            __syncwarp();
            if (leader && id >= w0 && id < w0 + kWindow) {
                sp[id - w0] = sum;
                sh[id - w0] = 1;
            }
            __syncwarp();
            const int e0 = w0 + 8 * lane;
            if (e0 < E) {
                const float4 a = reinterpret_cast<const float4 *>(sp)[2 * lane];
                const float4 b = reinterpret_cast<const float4 *>(sp)[2 * lane + 1];
                const uint2 h = reinterpret_cast<const uint2 *>(sh)[lane];
                if (VEC) {
                    if (routing_map != nullptr)
                        *reinterpret_cast<uint2 *>(routing_map + t * E + e0) = h;
                    if (probs != nullptr) {
                        float4 *dst = reinterpret_cast<float4 *>(probs + t * E + e0);
                        dst[0] = a;
                        dst[1] = b;
                    }
                } else {
                    const float pv[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        if (e0 + j >= E)
                            break;
                        if (routing_map != nullptr)
                            routing_map[t * E + e0 + j] = sh[8 * lane + j];
                        if (probs != nullptr)
                            probs[t * E + e0 + j] = pv[j];
                    }
                }
            }
            __syncwarp();   // the window is read before the next pass zeroes it
        }
        id = id_n;
        pk = pk_n;
        bad = bad_n;
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
    const bool vec = E % 8 == 0 && (routing_map == nullptr || aligned(routing_map, 8)) &&
                     (probs == nullptr || aligned(probs, 16));
    // at most one wave of resident blocks, each warp looping over tokens with
    // the next token's slots loaded ahead: on 32 K tokens this beat one warp
    // per token (16.3 -> 14.3 us; the same at 16 K tokens), since short-lived
    // blocks pay their scheduling in every wave
    static PerDevice resident[2];   // blocks per SM, [vec]
    const int dev = current_device();
    int per_sm = resident[vec ? 1 : 0].get(dev);
    if (per_sm < 0) {
        int n = 0;
        const cudaError_t e = vec ? cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, multihot_kernel<true>,
                                                                                 kMultihotThreads, 0)
                                  : cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, multihot_kernel<false>,
                                                                                 kMultihotThreads, 0);
        if (e != cudaSuccess) {
            cudaGetLastError();
            n = 4;
        }
        per_sm = std::max(n, 1);
        resident[vec ? 1 : 0].put(dev, per_sm);
    }
    const int64_t blocks = std::min<int64_t>(ceil_div(T, kMultihotWarps), (int64_t)per_sm * device_sm_count());
    if (vec)
        multihot_kernel<true><<<blocks, kMultihotThreads, 0, stream>>>(topk_idx, topk_probs, T, K, E, routing_map,
                                                                       probs, err);
    else
        multihot_kernel<false><<<blocks, kMultihotThreads, 0, stream>>>(topk_idx, topk_probs, T, K, E, routing_map,
                                                                        probs, err);
    return launch_status();
}
