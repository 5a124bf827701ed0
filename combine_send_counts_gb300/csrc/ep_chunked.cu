// Chunked forward driver of libep_gb300 (host code only):
// axolotl integrations.expert_parallel.torch_dispatch, dispatch_chunked_forward
// and chunk_bounds.  The tokens are split into contiguous chunks; the split
// counts of every chunk come from ONE count launch and ONE device-to-host
// copy; then each chunk runs layout -> dispatch -> the caller's local kernel
// -> combine into the chunk's rows of the output.
//
// The pages overlap chunk i+1's all-to-alls with chunk i's expert compute.
// On one GPU there is no exchange to hide, so the chunks run in order on the
// caller's stream.
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
