// Chunked forward driver of libep_gb300 (host code only):
// axolotl integrations.expert_parallel.torch_dispatch, dispatch_chunked_forward
// and chunk_bounds.  The tokens are split into contiguous chunks; the split
// counts of every chunk come from ONE count launch and ONE device-to-host
// copy; then each chunk runs layout -> dispatch -> the caller's local kernel
// -> combine into the chunk's rows of the output.
//
// The pages overlap chunk i+1's all-to-alls with chunk i's expert compute.
// On one GPU there is no exchange to hide; ep_dispatch_chunked_forward runs
// the chunks in order on the caller's stream, and
// ep_dispatch_chunked_forward_nosync (below) drops the host round trip and
// overlaps chunk i+1's routing and dispatch with chunk i's expert kernel and
// combine on a second stream.
#include <cstring>

#include "ep_internal.h"

extern "C" int ep_local_expert_fp8_callback(void *user, int chunk, int64_t n_rows, int K, int H,
                                            const void *recv_x, const float *recv_scale,
                                            const int64_t *send_idx, const float *send_w, void *local_out,
                                            int32_t *err, ep_stream_t stream)
{
    (void)user;
    (void)chunk;
    return ep_local_expert_fp8(static_cast<const uint8_t *>(recv_x), recv_scale, send_idx, send_w, n_rows, K, H,
                               local_out, err, stream);
}

extern "C" int ep_dispatch_chunked_forward(const void *x, const int64_t *topk_idx, const float *topk_weights,
                                           int64_t T, int K, int H, int P, int E_local, int chunks, int fp8,
                                           ep_local_kernel_fn local_kernel, void *user, void *out,
                                           const ep_chunk_buffers *b, int32_t *h_counts, int32_t *err,
                                           ep_stream_t stream)
{
    using namespace ep;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (b == nullptr || local_kernel == nullptr || h_counts == nullptr || chunks < 1 || chunks > EP_MAX_CHUNKS)
        return EP_ERR_INVALID_ARG;
    if (T < 0 || H < 8 || H % 8 != 0 || K < 1 || P < 1)
        return EP_ERR_INVALID_ARG;
    if (fp8 && (H % 128 != 0 || b->recv_scale == nullptr))
        return fp8 && H % 128 != 0 ? EP_ERR_UNSUPPORTED : EP_ERR_INVALID_ARG;
    if (T > 0 && (x == nullptr || out == nullptr))
        return EP_ERR_INVALID_ARG;

    int64_t bounds[EP_MAX_CHUNKS + 1];
    int rc = ep_chunk_bounds(T, chunks, bounds);
    if (rc != EP_OK)
        return rc;
    // one count pass for all chunks
    rc = ep_compute_send_counts(topk_idx, T, K, P, E_local, bounds, chunks, b->dest, b->is_in_rank, b->send_counts,
                                b->rank_offsets, nullptr, b->ws, b->ws_bytes, err, stream);
    if (rc != EP_OK)
        return rc;
    // one device-to-host copy of every chunk's counts
    if (cudaMemcpyAsync(h_counts, b->send_counts, sizeof(int32_t) * (size_t)chunks * P, cudaMemcpyDeviceToHost,
                        s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess) {
        cudaGetLastError();
        return EP_ERR_CUDA;
    }

    for (int c = 0; c < chunks; ++c) {
        const int64_t s0 = bounds[c], len = bounds[c + 1] - bounds[c];
        int64_t n = 0;
        for (int p = 0; p < P; ++p)
            n += h_counts[(size_t)c * P + p];
        if (n > b->max_rows)
            return EP_ERR_CAPACITY;
        const int64_t *idx_c = topk_idx + s0 * K;
        int32_t *tp_c = b->token_pos + s0 * P;
        rc = ep_build_send_layout(idx_c, topk_weights + s0 * K, b->dest + s0 * K, b->is_in_rank + s0 * P, len, K, P,
                                  E_local, n, b->send_token_idx, b->send_rank, b->send_idx, b->send_w, tp_c, b->ws,
                                  b->ws_bytes, err, stream);
        if (rc != EP_OK)
            return rc;
        rc = ep_dispatch(static_cast<const char *>(x) + (size_t)s0 * H * 2, len, H, tp_c, P, n, b->recv_x,
                         fp8 ? b->recv_scale : nullptr, fp8, err, stream);
        if (rc != EP_OK)
            return rc;
        rc = local_kernel(user, c, n, K, H, b->recv_x, fp8 ? b->recv_scale : nullptr, b->send_idx, b->send_w,
                          b->local_out, err, stream);
        if (rc != EP_OK)
            return rc;
        rc = ep_combine(b->local_out, len, H, tp_c, P, n, static_cast<char *>(out) + (size_t)s0 * H * 2, 0,
                        b->combine_ws, b->combine_ws != nullptr ? EP_COMBINE_WS_BYTES : 0, err, stream);
        if (rc != EP_OK)
            return rc;
    }
    return EP_OK;
}

// ------------------------------------------------------ no-sync, pipelined --
// The chunked forward with worst-case row buffers: nothing waits on the host.
// Routing and dispatch of every chunk run on the producer stream, the local
// kernel and combine on the consumer stream; with two row sets, chunk c+1's
// producer work overlaps chunk c's consumer work.  Event `ready` hands a set
// from producer to consumer, `freed[s]` hands set s back.

extern "C" int ep_local_expert_fp8_dev_callback(void *user, int chunk, int64_t max_rows, const int32_t *n_rows,
                                                int K, int H, const void *recv_x, const float *recv_scale,
                                                const int64_t *send_idx, const float *send_w, void *local_out,
                                                int32_t *err, ep_stream_t stream)
{
    (void)user;
    (void)chunk;
    (void)err;
    if (n_rows == nullptr)
        return EP_ERR_INVALID_ARG;
    return ep::launch_local_expert_fp8(static_cast<const uint8_t *>(recv_x), recv_scale, send_idx, send_w, max_rows,
                                       n_rows, K, H, local_out, reinterpret_cast<cudaStream_t>(stream));
}

namespace {

// Events of one pipelined call; destroyed when the call returns (the driver
// releases an event whose recorded work is still pending once it completes).
struct PipelineEvents {
    cudaEvent_t fork = nullptr, ready = nullptr, freed[2] = {nullptr, nullptr};
    bool ok = true;

    explicit PipelineEvents(bool two)
    {
        if (!two)
            return;
        ok = cudaEventCreateWithFlags(&fork, cudaEventDisableTiming) == cudaSuccess &&
             cudaEventCreateWithFlags(&ready, cudaEventDisableTiming) == cudaSuccess &&
             cudaEventCreateWithFlags(&freed[0], cudaEventDisableTiming) == cudaSuccess &&
             cudaEventCreateWithFlags(&freed[1], cudaEventDisableTiming) == cudaSuccess;
    }
    ~PipelineEvents()
    {
        for (cudaEvent_t e : {fork, ready, freed[0], freed[1]})
            if (e != nullptr)
                cudaEventDestroy(e);
    }
};

// `dst` waits for the work enqueued so far on `src`.
int order_after(cudaEvent_t ev, cudaStream_t src, cudaStream_t dst)
{
    if (cudaEventRecord(ev, src) != cudaSuccess || cudaStreamWaitEvent(dst, ev, 0) != cudaSuccess) {
        cudaGetLastError();
        return EP_ERR_CUDA;
    }
    return EP_OK;
}

}  // namespace

extern "C" int ep_dispatch_chunked_forward_nosync(const void *x, const int64_t *topk_idx, const float *topk_weights,
                                                  int64_t T, int K, int H, int P, int E_local, int chunks, int fp8,
                                                  ep_local_kernel_dev_fn local_kernel, void *user, void *out,
                                                  const ep_pipeline_buffers *b, int32_t *err, ep_stream_t stream,
                                                  ep_stream_t aux_stream)
{
    using namespace ep;
    if (b == nullptr || local_kernel == nullptr || chunks < 1 || chunks > EP_MAX_CHUNKS)
        return EP_ERR_INVALID_ARG;
    if (b->n_sets != 1 && b->n_sets != 2)
        return EP_ERR_INVALID_ARG;
    const bool two = b->n_sets == 2;
    if (two && (aux_stream == nullptr || aux_stream == stream))
        return EP_ERR_INVALID_ARG;
    if (T < 0 || H < 8 || H % 8 != 0 || K < 1 || P < 1 || b->max_rows < 0)
        return EP_ERR_INVALID_ARG;
    if (fp8 && H % 128 != 0)
        return EP_ERR_UNSUPPORTED;
    for (int i = 0; i < b->n_sets; ++i)
        if (fp8 && b->sets[i].recv_scale == nullptr)
            return EP_ERR_INVALID_ARG;
    if (T > 0 && (x == nullptr || out == nullptr))
        return EP_ERR_INVALID_ARG;
    if (b->ws_bytes < ep_workspace_size(T, K, P, E_local, chunks))
        return EP_ERR_INVALID_ARG;

    int64_t bounds[EP_MAX_CHUNKS + 1];
    int rc = ep_chunk_bounds(T, chunks, bounds);
    if (rc != EP_OK)
        return rc;
    cudaStream_t cons = reinterpret_cast<cudaStream_t>(stream);
    cudaStream_t prod = two ? reinterpret_cast<cudaStream_t>(aux_stream) : cons;
    ep_stream_t prod_s = two ? aux_stream : stream;
    PipelineEvents ev(two);
    if (!ev.ok)
        return EP_ERR_CUDA;
    if (two && (rc = order_after(ev.fork, cons, prod)) != EP_OK)   // producer starts after earlier work
        return rc;

    const int64_t W = b->max_rows;
    for (int c = 0; c < chunks; ++c) {
        const int64_t s0 = bounds[c], len = bounds[c + 1] - bounds[c];
        const int set = two ? (c & 1) : 0;
        const ep_row_set &r = b->sets[set];
        int32_t *tp_c = b->token_pos + s0 * P;
        int32_t *off_c = b->rank_offsets + (size_t)c * (P + 1);
        // producer: the set's previous consumer (chunk c-2) must be done with it
        if (two && c >= 2 && cudaStreamWaitEvent(prod, ev.freed[set], 0) != cudaSuccess) {
            cudaGetLastError();
            return EP_ERR_CUDA;
        }
        rc = ep_route_nosync(topk_idx + s0 * K, topk_weights + s0 * K, len, K, P, E_local, W, b->dest + s0 * K,
                             b->is_in_rank + s0 * P, b->send_counts + (size_t)c * P, off_c, nullptr,
                             r.send_token_idx, r.send_rank, r.send_idx, r.send_w, tp_c, b->ws, b->ws_bytes, err,
                             prod_s);
        if (rc != EP_OK)
            return rc;
        // the route just enqueued on the producer stream writes nothing the
        // dispatch reads before its dependency wait
        rc = dispatch_rows(static_cast<const char *>(x) + (size_t)s0 * H * 2, len, H, tp_c, P, W, r.recv_x,
                           fp8 ? r.recv_scale : nullptr, fp8, err, prod, true);
        if (rc != EP_OK)
            return rc;
        if (two && (rc = order_after(ev.ready, prod, cons)) != EP_OK)
            return rc;
        // consumer
        rc = local_kernel(user, c, W, off_c + P, K, H, r.recv_x, fp8 ? r.recv_scale : nullptr, r.send_idx, r.send_w,
                          r.local_out, err, stream);
        if (rc != EP_OK)
            return rc;
        rc = ep_combine(r.local_out, len, H, tp_c, P, W, static_cast<char *>(out) + (size_t)s0 * H * 2, 0,
                        b->combine_ws, b->combine_ws != nullptr ? EP_COMBINE_WS_BYTES : 0, err, stream);
        if (rc != EP_OK)
            return rc;
        if (two && cudaEventRecord(ev.freed[set], cons) != cudaSuccess) {
            cudaGetLastError();
            return EP_ERR_CUDA;
        }
    }
    return EP_OK;
}

// ----------------------------------------------- route + dispatch, no sync --
// ep_route_nosync followed by ep_dispatch into the worst-case rows, with the
// dispatch launched as a programmatic dependent of the routing kernel: its
// blocks start loading their input rows while the routing kernel finishes.
extern "C" int ep_dispatch_nosync(const void *x, const int64_t *topk_idx, const float *topk_weights, int64_t T,
                                  int K, int H, int P, int E_local, int64_t num_worst_rows, int fp8, int32_t *dest,
                                  uint8_t *is_in_rank, int32_t *send_counts, int32_t *rank_offsets,
                                  int32_t *tokens_per_expert, int32_t *send_token_idx, int32_t *send_rank,
                                  int64_t *send_idx, float *send_w, int32_t *token_pos, void *recv_x,
                                  float *recv_scale, void *ws, size_t ws_bytes, int32_t *err, ep_stream_t stream)
{
    if (fp8 != 0 && fp8 != 1)
        return EP_ERR_UNSUPPORTED;
    if (fp8 && H % 128 != 0)
        return EP_ERR_UNSUPPORTED;
    if (H < 8 || H % 8 != 0 || (T > 0 && (x == nullptr || !ep::aligned(x, 16))) ||
        (num_worst_rows > 0 && (recv_x == nullptr || (fp8 && recv_scale == nullptr))))
        return EP_ERR_INVALID_ARG;
    int rc = ep_route_nosync(topk_idx, topk_weights, T, K, P, E_local, num_worst_rows, dest, is_in_rank, send_counts,
                             rank_offsets, tokens_per_expert, send_token_idx, send_rank, send_idx, send_w, token_pos,
                             ws, ws_bytes, err, stream);
    if (rc != EP_OK)
        return rc;
    return ep::dispatch_rows(x, T, H, token_pos, P, num_worst_rows, recv_x, fp8 ? recv_scale : nullptr, fp8, err,
                             reinterpret_cast<cudaStream_t>(stream), true);
}
