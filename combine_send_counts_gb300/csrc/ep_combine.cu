// Combine kernels of libep_gb300:
//   ep_combine          -- axolotl integrations.expert_parallel.torch_dispatch,
//                          combine; NeMo uccl_ep.buffer, Buffer.combine
//                          (an unweighted sum)
//   ep_batched_combine  -- vLLM BatchedPrepareAndFinalize.finalize; NeMo
//                          uccl_ep.buffer, Buffer.low_latency_combine (reduce
//                          weighted)
//
// Both read, for every output token, its source rows in a fixed order and
// accumulate them in fp32.  The work is HBM-bound and its rows are scattered,
// so the kernel keeps many row loads in flight with the TMA engine rather
// than with registers:
//
//   * three persistent CTAs per SM, each with its own ring; items are (token,
//     column chunk) pairs, claimed from a shared counter (or dealt round-robin),
//     a few at a time and one at a time near the end;
//   * warp 0 is the producer: it resolves the source lists of 32 items at a
//     time, publishes each item's descriptor (token, chunk, source count,
//     weights) in a small queue and issues one 1-D bulk copy
//     (cp.async.bulk, global -> shared) per source row chunk into a ring of
//     B shared-memory buffers, each tracked by a "full" mbarrier (transaction
//     bytes) and an "empty" mbarrier (consumer warps' release);
//   * warps 1..8 are consumers: they take the items in the same order, wait
//     for each source buffer, accumulate it into fp32 registers (16 bytes of
//     the row per thread and pass), release the buffer and write the output
//     chunk once with 16-byte streaming stores.
//
// Every wait is bounded (EP_ERR_TIMEOUT after a second); a CTA that gives up
// waits, again with a bound, for its own copies in flight before it exits.
#include <algorithm>
#include <atomic>
#include <type_traits>

#include "ep_device.cuh"
#include "ep_internal.h"
#include "ep_rows.cuh"

namespace ep {

constexpr int kConsumerWarps = 8;
constexpr int kConsumers = kConsumerWarps * 32;
constexpr int kGatherThreads = 32 + kConsumers;
constexpr int kQueue = 16;          // descriptor slots: how far the producer may run ahead in items
constexpr int kVMax = 4;            // 16-byte vectors per consumer thread per chunk
constexpr int kMaxChunkCols = kConsumers * kVMax * 8;   // 8192 bf16 columns = 16 KB per buffer
constexpr int kMaxBuffers = 64;
constexpr size_t kSmemBudget = 72 * 1024;    // three CTAs per SM
constexpr uint64_t kWaitNs = 1000000000ull;       // 1 s
constexpr uint64_t kDrainNs = 50000000ull;        // 50 ms per buffer when draining after a timeout
constexpr int kSendTaper = 4;      // claims per CTA left when the send layout's claims shrink to one item
constexpr int kBatchedTaper = 2;   // the same on the batched layout

struct Desc {
    int64_t t;
    int32_t c;
    int32_t nsrc;       // -1 ends the sequence
    float w[kMaxList];
};

struct GatherGeom {
    int H;          // columns per row
    int CH;         // columns per chunk (multiple of 8)
    int nchunk;     // chunks per row
    int B;          // ring buffers, a power of two
    int logB;       // log2(B): buffer of use u is u & (B-1), its phase parity (u >> logB) & 1
    int RB;         // bytes per ring buffer (multiple of 128)
    int lpi;        // lanes of the producer warp per item (8, 16 or 32)
    int cb;         // items per claim (32 / lpi)
    int taper;      // claims from the counter shrink to one item once at most this many items remain (0: never)
};

__host__ __device__ inline size_t gather_smem_bytes(const GatherGeom &g)
{
    return (size_t)g.B * g.RB                       // ring
           + sizeof(uint64_t) * (2 * g.B + 2 * kQueue)   // mbarriers
           + sizeof(int64_t) * g.B                   // last armed use per buffer
           + sizeof(Desc) * kQueue;                  // descriptor queue
}

// counter: NULL for a static round-robin of claims over the CTAs, or a
// device word set to 0 before the launch, from which the producers claim
// their next items (balances skewed source counts).
template <class Rows, bool WEIGHTED, bool OUT_F32>
__global__ void __launch_bounds__(kGatherThreads, 3)   // three CTAs per SM: at most 75 registers
gather_tma_kernel(const uint8_t *__restrict__ y, int64_t T, GatherGeom g, Rows rows, int64_t n_rows,
                  int err_bits, void *__restrict__ out, unsigned int *counter, int32_t *err)
{
    extern __shared__ __align__(128) uint8_t smem[];
    const int D = rows.len();
    uint8_t *ring = smem;
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + (size_t)g.B * g.RB);
    uint64_t *empty = full + g.B;
    uint64_t *qfull = empty + g.B;
    uint64_t *qempty = qfull + kQueue;
    int64_t *last_use = reinterpret_cast<int64_t *>(qempty + kQueue);
    Desc *desc = reinterpret_cast<Desc *>(last_use + g.B);
    __shared__ int s_abort;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int b = 0; b < g.B; ++b) {
            mbar_init(&full[b], 1);
            mbar_init(&empty[b], kConsumerWarps);
            last_use[b] = -1;
        }
        for (int q = 0; q < kQueue; ++q) {
            mbar_init(&qfull[q], 1);
            mbar_init(&qempty[q], kConsumerWarps);
        }
        s_abort = 0;
        fence_mbar_init();
    }
    __syncthreads();

    volatile int *abort_flag = &s_abort;
    const int n_items = (int)(T * g.nchunk);   // < 2^31, checked on the host
    int bad = 0;

    if (warp == 0) {
        // ---------------------------------------------------------- producer
        // Lane l serves item l / lpi of a claim and source slots j0 = l % lpi
        // and j0 + 32 (lists longer than 32).
        const int my_i = lane / g.lpi, j0 = lane % g.lpi, j1 = j0 + 32;
        const unsigned item_lanes = (g.lpi == 32 ? kFull : ((1u << g.lpi) - 1u)) << (my_i * g.lpi);
        uint32_t static_k = 0;
        // A claim is `count` consecutive items from `base`.  From the shared
        // counter a CTA takes g.cb items at a time until it sees at most
        // g.taper items left, then one at a time, so that the CTAs run out of
        // work at nearly the same time.
        // A claim is issued one loop iteration before its value is needed
        // (claim_issue: lane 0's atomic, or the static index), and taken with
        // claim_take, so that the producer does not wait for the atomic's
        // round trip on every claim.
        int seen = 0;   // the counter's value at this CTA's last claim taken
        auto claim_issue = [&](int &count) -> int {
            count = g.cb;
            if (counter == nullptr)
                return (int)((blockIdx.x + (static_k++) * gridDim.x) * (uint32_t)g.cb);
            if (n_items - seen <= g.taper)
                count = 1;
            int raw = 0;
            if (lane == 0)
                raw = (int)atomicAdd(counter, (unsigned)count);
            return raw;
        };
        auto claim_take = [&](int raw) -> int {
            if (counter == nullptr)
                return raw;
            const int c = __shfl_sync(kFull, raw, 0);
            seen = c;
            return c;
        };
        auto load = [&](int base, int count, typename Rows::Raw &r0, typename Rows::Raw &r1, bool &v0, bool &v1) {
            const int item = base + my_i;
            v0 = false;
            v1 = false;
            if (my_i < count && item < n_items) {
                const int64_t t = g.nchunk == 1 ? item : item / g.nchunk;
                v0 = j0 < D;
                v1 = j1 < D;
                if (v0)
                    r0 = rows.load(t, j0);
                if (v1)
                    r1 = rows.load(t, j1);
            }
        };

        uint32_t use = 0;  // buffer uses armed so far (warp-uniform)
        uint32_t k = 0;    // descriptors published so far
        typename Rows::Raw rc0{}, rc1{}, rn0{}, rn1{};
        bool vc0, vc1, vn0, vn1;
        int n_cur, n_nxt, n_aft;
        int c_cur = claim_take(claim_issue(n_cur));
        int c_nxt = claim_take(claim_issue(n_nxt));
        int raw_aft = claim_issue(n_aft);   // in flight during the first iteration
        load(c_cur, n_cur, rc0, rc1, vc0, vc1);
        while (c_cur < n_items && !*abort_flag) {
            load(c_nxt, n_nxt, rn0, rn1, vn0, vn1);   // used by the next claim
            bool ok = true;
            int32_t r0 = -1, r1 = -1;
            if (vc0) {
                r0 = rows.decode(rc0);
                if (r0 >= n_rows) {
                    bad = err_bits;
                    r0 = -1;
                }
            }
            if (vc1) {
                r1 = rows.decode(rc1);
                if (r1 >= n_rows) {
                    bad = err_bits;
                    r1 = -1;
                }
            }
            const float w0 = WEIGHTED && vc0 ? rows.weight(rc0) : 1.0f;
            const float w1 = WEIGHTED && vc1 ? rows.weight(rc1) : 1.0f;
            const unsigned bal0 = __ballot_sync(kFull, r0 >= 0);
            const unsigned bal1 = __ballot_sync(kFull, r1 >= 0);
            for (int i = 0; i < n_cur && ok; ++i) {
                const int item = c_cur + i;
                if (item >= n_items)
                    break;
                const unsigned m = (g.lpi == 32 ? kFull : ((1u << g.lpi) - 1u)) << (i * g.lpi);
                const int n0 = __popc(bal0 & m), nsrc = n0 + __popc(bal1 & m);
                const bool mine = item_lanes == m;
                const int q = (int)(k % kQueue);
                if (lane == 0 && k >= kQueue)
                    ok = mbar_wait(&qempty[q], ((k / kQueue) - 1) & 1, kWaitNs);
                ok = __all_sync(kFull, ok);
                if (!ok)
                    break;
                const int chunk = g.nchunk == 1 ? 0 : item % g.nchunk;
                if (lane == 0) {
                    desc[q].t = g.nchunk == 1 ? item : item / g.nchunk;
                    desc[q].c = chunk;
                    desc[q].nsrc = nsrc;
                }
                const int o0 = __popc(bal0 & m & lanemask_lt());
                const int o1 = n0 + __popc(bal1 & m & lanemask_lt());
                if (WEIGHTED && mine) {
                    if (r0 >= 0)
                        desc[q].w[o0] = w0;
                    if (r1 >= 0)
                        desc[q].w[o1] = w1;
                }
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(&qfull[q]);
                ++k;
                const int col0 = chunk * g.CH;
                const uint32_t bytes = (uint32_t)min(g.CH, g.H - col0) * 2u;
                // Sources are issued in rounds of B ordinals: within a round
                // every buffer appears once, and a lane waits on a buffer only
                // after the buffer's previous use has been armed (an earlier
                // round or item).  Waiting earlier could match a parity two
                // phases back and re-arm a buffer still in use.
                for (int round = 0; (round << g.logB) < nsrc; ++round) {
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const int32_t r = h == 0 ? r0 : r1;
                        const int o = h == 0 ? o0 : o1;
                        if (!mine || r < 0 || (o >> g.logB) != round)
                            continue;
                        const uint32_t u = use + o;
                        const int b = (int)(u & (g.B - 1));
                        if (u >= (uint32_t)g.B && !mbar_wait(&empty[b], ((u >> g.logB) - 1) & 1, kWaitNs)) {
                            ok = false;
                            continue;
                        }
                        mbar_arrive_expect_tx(&full[b], bytes);
                        bulk_g2s(ring + (size_t)b * g.RB, y + ((int64_t)r * g.H + col0) * 2, bytes, &full[b]);
                        last_use[b] = u;
                    }
                    __syncwarp();
                }
                use += nsrc;
                ok = __all_sync(kFull, ok);
            }
            if (!ok) {
                bad |= EP_ERR_TIMEOUT;
                *abort_flag = 1;
                break;
            }
            c_cur = c_nxt;
            c_nxt = claim_take(raw_aft);
            n_cur = n_nxt;
            n_nxt = n_aft;
            raw_aft = claim_issue(n_aft);
            rc0 = rn0;
            rc1 = rn1;
            vc0 = vn0;
            vc1 = vn1;
        }
        // end of the sequence for the consumers
        if (!*abort_flag) {
            const int q = (int)(k % kQueue);
            bool ok = true;
            if (lane == 0 && k >= kQueue)
                ok = mbar_wait(&qempty[q], ((k / kQueue) - 1) & 1, kWaitNs);
            if (lane == 0 && ok) {
                desc[q].nsrc = -1;
                mbar_arrive(&qfull[q]);
            }
            if (!__all_sync(kFull, ok)) {
                bad |= EP_ERR_TIMEOUT;
                *abort_flag = 1;
            }
        }
    } else {
        // --------------------------------------------------------- consumers
        const int ct = threadIdx.x - 32;
        uint32_t use = 0, k = 0;
        while (true) {
            const int q = (int)(k % kQueue);
            if (*abort_flag || !mbar_wait(&qfull[q], (k / kQueue) & 1, kWaitNs)) {
                bad |= *abort_flag ? 0 : EP_ERR_TIMEOUT;
                *abort_flag = 1;
                break;
            }
            const int nsrc = desc[q].nsrc;
            if (nsrc < 0)
                break;
            const int64_t t = desc[q].t;
            const int col0 = desc[q].c * g.CH;
            const int nv = min(g.CH, g.H - col0) / 8;
            float acc[kVMax][8];
#pragma unroll
            for (int v = 0; v < kVMax; ++v)
#pragma unroll
                for (int e = 0; e < 8; ++e)
                    acc[v][e] = 0.0f;
            bool ok = true;
            for (int o = 0; o < nsrc; ++o) {
                const uint32_t u = use + o;
                const int b = (int)(u & (g.B - 1));
                if (!mbar_wait(&full[b], (u >> g.logB) & 1, kWaitNs)) {
                    ok = false;
                    break;
                }
                const float wj = WEIGHTED ? desc[q].w[o] : 1.0f;
                const uint4 *src = reinterpret_cast<const uint4 *>(ring + (size_t)b * g.RB);
#pragma unroll
                for (int v = 0; v < kVMax; ++v) {
                    const int i = ct + v * kConsumers;
                    if (i < nv) {
                        const uint4 x = src[i];
                        const float f[8] = {bf16_lo(x.x), bf16_hi(x.x), bf16_lo(x.y), bf16_hi(x.y),
                                            bf16_lo(x.z), bf16_hi(x.z), bf16_lo(x.w), bf16_hi(x.w)};
#pragma unroll
                        for (int e = 0; e < 8; ++e)
                            acc[v][e] = WEIGHTED ? __fmaf_rn(wj, f[e], acc[v][e]) : __fadd_rn(acc[v][e], f[e]);
                    }
                }
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(&empty[b]);
            }
            if (!ok) {
                bad |= EP_ERR_TIMEOUT;
                *abort_flag = 1;
                break;
            }
            use += nsrc;
#pragma unroll
            for (int v = 0; v < kVMax; ++v) {
                const int i = ct + v * kConsumers;
                if (i >= nv)
                    continue;
                const int64_t e0 = t * g.H + col0 + (int64_t)i * 8;   // first element of this vector
                if (OUT_F32) {
                    float4 *o4 = reinterpret_cast<float4 *>(static_cast<float *>(out) + e0);
                    o4[0] = make_float4(acc[v][0], acc[v][1], acc[v][2], acc[v][3]);
                    o4[1] = make_float4(acc[v][4], acc[v][5], acc[v][6], acc[v][7]);
                } else {
                    uint4 o;
                    o.x = pack_bf16x2(acc[v][0], acc[v][1]);
                    o.y = pack_bf16x2(acc[v][2], acc[v][3]);
                    o.z = pack_bf16x2(acc[v][4], acc[v][5]);
                    o.w = pack_bf16x2(acc[v][6], acc[v][7]);
                    st_stream(reinterpret_cast<uint4 *>(static_cast<uint16_t *>(out) + e0), o);
                }
            }
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&qempty[q]);
            ++k;
        }
    }

    __syncthreads();
    if (*abort_flag && threadIdx.x == 0) {
        // copies this CTA armed may still be landing in its shared memory:
        // wait for the last use of every buffer before the CTA exits
        for (int b = 0; b < g.B; ++b)
            if (last_use[b] >= 0)
                (void)mbar_wait(&full[b], (uint32_t)(last_use[b] >> g.logB) & 1, kDrainNs);
    }
    raise(err, bad);
}

// ------------------------------------------------------------ launch policy --
static GatherGeom gather_geometry(int H, int D)
{
    GatherGeom g;
    g.H = H;
    g.nchunk = (int)ceil_div(H, kMaxChunkCols);
    g.CH = (int)align_up((size_t)ceil_div(H, g.nchunk), 8);
    g.RB = (int)align_up((size_t)g.CH * 2, 128);
    g.lpi = D <= 8 ? 8 : D <= 16 ? 16 : 32;
    g.cb = 32 / g.lpi;
    g.taper = 0;
    g.B = 0;
    g.logB = 0;
    const size_t fixed = gather_smem_bytes(g);
    const size_t fit = std::min<size_t>(kMaxBuffers, (kSmemBudget - fixed) / (g.RB + 2 * sizeof(uint64_t) + sizeof(int64_t)));
    while ((size_t)(2 << g.logB) <= fit)
        ++g.logB;
    g.B = 1 << g.logB;
    return g;
}

template <class Rows, bool WEIGHTED, bool OUT_F32>
static int launch_gather_tma(const void *y, int64_t T, int H, const Rows &rows, int64_t n_rows, int err_bits,
                             void *out, void *ws, size_t ws_bytes, int32_t *err, cudaStream_t stream)
{
    const int D = rows.len();
    GatherGeom g = gather_geometry(H, D);
    const size_t smem = gather_smem_bytes(g);
    auto kernel = gather_tma_kernel<Rows, WEIGHTED, OUT_F32>;
    static PerDevice smem_set;   // per instantiation and device; raising the limit is idempotent
    const int dev = current_device();
    if ((int)smem > smem_set.get(dev)) {
        if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess) {
            cudaGetLastError();
            return EP_ERR_CUDA;
        }
        smem_set.put(dev, (int)smem);
    }
    const int64_t items = T * g.nchunk;
    if (items >= ((int64_t)1 << 30))
        return EP_ERR_UNSUPPORTED;
    const int grid = (int)std::min<int64_t>(ceil_div(items, g.cb), 3 * device_sm_count());
    if (grid == 0)
        return EP_OK;
    // One-item claims for the last few claims' worth per CTA (thresholds
    // measured: on the send layout, about three 14 KB sources per token, 4
    // claims took the large combine from 141.1 to 138.4 us, 2 and 3 were
    // slower; on the batched layout, about two 8 KB sources per token, 2
    // claims took it from 35.5 to 33.9 us, 4 and 6 were slower).
    g.taper = (std::is_same<Rows, BatchedRows>::value ? kBatchedTaper : kSendTaper) * grid * g.cb;
    unsigned int *counter = nullptr;
    if (ws != nullptr && ws_bytes >= EP_COMBINE_WS_BYTES) {
        counter = static_cast<unsigned int *>(ws);
        if (cudaMemsetAsync(counter, 0, sizeof(unsigned int), stream) != cudaSuccess) {
            cudaGetLastError();
            return EP_ERR_CUDA;
        }
    }
    gather_tma_kernel<Rows, WEIGHTED, OUT_F32><<<grid, kGatherThreads, smem, stream>>>(
        static_cast<const uint8_t *>(y), T, g, rows, n_rows, err_bits, out, counter, err);
    return launch_status();
}

static bool row_shape_ok(int64_t T, int H)
{
    return T >= 0 && H >= 8 && H % 8 == 0 && T < ((int64_t)1 << 31);
}

}  // namespace ep

// ================================================================ C ABI ====
using namespace ep;

extern "C" int ep_combine(const void *y, int64_t T, int H, const int32_t *token_pos, int P,
                          int64_t num_send, void *out, int out_dtype, void *ws, size_t ws_bytes, int32_t *err,
                          ep_stream_t stream_)
{
    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
    if (!row_shape_ok(T, H) || P < 1 || P > EP_MAX_RANKS || num_send < 0 || num_send >= ((int64_t)1 << 31))
        return EP_ERR_INVALID_ARG;
    if (out_dtype != 0 && out_dtype != 1)
        return EP_ERR_UNSUPPORTED;
    if (T > 0 && (token_pos == nullptr || out == nullptr || !aligned(out, 16)))
        return EP_ERR_INVALID_ARG;
    if (num_send > 0 && (y == nullptr || !aligned(y, 16)))
        return EP_ERR_INVALID_ARG;
    if (T == 0)
        return EP_OK;
    const SendRows rows{token_pos, P};
    if (out_dtype == 1)
        return launch_gather_tma<SendRows, false, true>(y, T, H, rows, num_send, EP_ERR_COUNT_MISMATCH, out, ws,
                                                        ws_bytes, err, stream);
    return launch_gather_tma<SendRows, false, false>(y, T, H, rows, num_send, EP_ERR_COUNT_MISMATCH, out, ws,
                                                     ws_bytes, err, stream);
}

extern "C" int ep_batched_combine(const void *y, const int64_t *topk_idx, const float *topk_weights,
                                  const int32_t *slot, int64_t T, int K, int H, int E_local, int rank,
                                  int max_num_tokens, void *out, void *ws, size_t ws_bytes, int32_t *err,
                                  ep_stream_t stream_)
{
    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
    if (!row_shape_ok(T, H) || K < 1 || K > EP_MAX_TOPK || E_local < 1 || rank < 0 || max_num_tokens < 0)
        return EP_ERR_INVALID_ARG;
    if ((int64_t)E_local * max_num_tokens >= ((int64_t)1 << 31))
        return EP_ERR_UNSUPPORTED;
    if (T > 0 && (topk_idx == nullptr || topk_weights == nullptr || slot == nullptr || out == nullptr ||
                  !aligned(out, 16)))
        return EP_ERR_INVALID_ARG;
    if ((int64_t)E_local * max_num_tokens > 0 && (y == nullptr || !aligned(y, 16)))
        return EP_ERR_INVALID_ARG;
    if (T == 0)
        return EP_OK;
    const BatchedRows rows{topk_idx, slot, topk_weights, K, (int64_t)rank * E_local, E_local, max_num_tokens, false};
    return launch_gather_tma<BatchedRows, true, false>(y, T, H, rows, (int64_t)E_local * max_num_tokens,
                                                       EP_ERR_CAPACITY, out, ws, ws_bytes, err, stream);
}
