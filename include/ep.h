/*
 * ep.h -- C ABI of the GB300 (sm_103a) MoE top-k token dispatch / combine
 * library (libep_gb300.so).
 *
 * The P destination ranks of expert parallelism are logical partitions of one
 * GPU's HBM: rank p's receive buffer is the segment [rank_offsets[p],
 * rank_offsets[p+1]) of one rank-major send buffer, so "sending" is the layout
 * write itself and no collective runs.
 *
 * Citations name the page and the section that define each operation:
 *   [AX] axolotl docs, integrations.expert_parallel.torch_dispatch
 *   [UB] NeMo AutoModel docs, nemo_automodel.components.moe.uccl_ep.buffer
 *   [VB] vLLM docs, vllm.model_executor.layers.fused_moe.prepare_finalize
 *   [ND] NeMo AutoModel docs, nemo_automodel.components.moe.megatron.token_dispatcher
 *
 * Conventions shared by every call
 *   - Pointers are DEVICE pointers unless their name starts with h_ (host).
 *     The caller owns every buffer; the library allocates nothing and keeps no
 *     state between calls (the "handle" of [AX] TorchEPHandle is token_pos +
 *     send_counts for the send layout, slot + tokens_per_expert for the
 *     expert-batched layout).
 *   - Every call is asynchronous on `stream` (a cudaStream_t; NULL is the
 *     legacy default stream) and never synchronises the host.
 *   - The return value is a status detected on the host (argument checks,
 *     launch failures): EP_OK, or one EP_ERR_* bit.  On a non-OK return
 *     nothing was launched by the failing step.
 *   - Errors found on the device are OR-ed into *err (a device int32 the
 *     caller zeroes and reads after synchronising; may be NULL).  A kernel that
 *     finds a bad element skips it and never writes out of bounds.
 *   - Matrices are row-major and contiguous.  Row matrices of hidden
 *     vectors (bf16 or fp8 rows: x, y, recv_x, b_x, out and their fp8 forms)
 *     must start 16-byte aligned and H must be a multiple of 8 (the calls
 *     return EP_ERR_INVALID_ARG otherwise); workspaces have their own rule
 *     below.  Every other array (ids, weights, counts, layouts, flags, scales,
 *     multihot outputs) needs only its element type's natural alignment:
 *     wider stores are used only where a pointer allows them.
 *   - Token, row and count indices are int32 (T * min(K,P) < 2^31); expert ids
 *     are int64 with -1 meaning "unrouted" ([AX] dispatch, [UB]
 *     get_dispatch_layout).
 *   - Limits: 1 <= K <= 32, 1 <= P <= 64, P * E_local <= 8192, chunks <= 64.
 */
#ifndef EP_GB300_H
#define EP_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t. */
typedef struct CUstream_st *ep_stream_t;

enum ep_status {
    EP_OK = 0,
    EP_ERR_INVALID_ARG = 1,     /* host: null pointer, bad size, misalignment, small workspace */
    EP_ERR_INVALID_EXPERT = 2,  /* device: a topk id outside [-1, P*E_local); slot treated as unrouted */
    EP_ERR_COUNT_MISMATCH = 4,  /* device: num_send differs from the routed count, or a row index
                                   outside [0, num_send), or dest / is_in_rank disagree */
    EP_ERR_CAPACITY = 8,        /* device: an expert received more than max_num_tokens tokens */
    EP_ERR_UNSUPPORTED = 16,    /* host: a mode outside the limits (e.g. fp8 with H % 128 != 0) */
    EP_ERR_CUDA = 32,           /* host: a CUDA launch failed */
    EP_ERR_TIMEOUT = 64         /* device: a bounded wait gave up */
};

#define EP_MAX_TOPK 32
#define EP_MAX_RANKS 64
#define EP_MAX_EXPERTS 8192
#define EP_MAX_CHUNKS 64
#define EP_COMBINE_WS_BYTES 16   /* optional scratch of ep_combine / ep_batched_combine */

/* Human-readable name of a status value (a single bit, or EP_OK). */
const char *ep_status_str(int status);

/* Bytes of device workspace that every workspace-taking call below needs for
 * these sizes (chunks <= 1 means one chunk).  The workspace must start
 * 256-byte aligned; its contents need not be initialised and are scratch,
 * except that its first 256 bytes count the launches of the single-launch
 * (cooperative) routing kernels: keep them between calls that share the
 * workspace, captured or not.  Calls whose kernels overlap on the GPU must not
 * share a workspace. */
size_t ep_workspace_size(int64_t T, int K, int P, int E_local, int chunks);

/* [AX] chunk_bounds (host only): `chunks` contiguous [start, end) token
 * ranges, h_bounds[i] .. h_bounds[i+1]; every chunk has floor(T / chunks)
 * tokens and the last takes the remainder, so leading chunks are empty when
 * T < chunks.  h_bounds has chunks + 1 entries. */
int ep_chunk_bounds(int64_t T, int chunks, int64_t *h_bounds);

/* [AX] compute_send_counts, [UB] Buffer.get_dispatch_layout.
 *   topk_idx [T,K] int64: global expert ids, -1 = unrouted.
 *   Expert e is owned by rank e / E_local.
 * Outputs:
 *   dest [T,K] int32: owning rank per slot, -1 where unrouted (or invalid).
 *   is_in_rank [T,P] uint8: 1 iff some slot of token t is owned by rank p.
 *   send_counts [C,P] int32, C = max(chunks,1): tokens of chunk c sent to p.
 *   rank_offsets [C,P+1] int32 or NULL: exclusive prefix of send_counts per
 *     chunk (rank p's segment of chunk c is [off[c,p], off[c,p+1]) ).
 *   tokens_per_expert [P*E_local] int32 or NULL: over all T tokens, the
 *     number of tokens naming expert e in at least one slot.
 * Chunks: with chunks > 1, h_chunk_bounds (host, chunks+1 entries,
 * non-decreasing from 0 to T, e.g. from ep_chunk_bounds) splits the tokens,
 * and all chunks' counts come from this one call ([AX]
 * dispatch_chunked_forward: one count pass, one device-to-host copy).
 * Device errors: EP_ERR_INVALID_EXPERT. */
int ep_compute_send_counts(const int64_t *topk_idx, int64_t T, int K, int P, int E_local,
                           const int64_t *h_chunk_bounds, int chunks,
                           int32_t *dest, uint8_t *is_in_rank, int32_t *send_counts,
                           int32_t *rank_offsets, int32_t *tokens_per_expert,
                           void *ws, size_t ws_bytes, int32_t *err, ep_stream_t stream);

/* [AX] build_send_layout (DeepEP layout contract of the [AX] module
 * description): rank-major, token-ascending send order.  For each rank p in
 * ascending order and each token t in ascending order with is_in_rank[t,p],
 * one row n of the send buffer:
 *   send_token_idx[n] = t, send_rank[n] = p, token_pos[t,p] = n,
 *   send_idx[n,k] = topk_idx[t,k] - p*E_local if dest[t,k] == p, else -1,
 *   send_w[n,k]   = topk_weights[t,k]          if dest[t,k] == p, else +0.0f.
 * token_pos [T,P] int32 is -1 where t is not sent to p; it is the handle that
 * ep_dispatch and ep_combine take.
 *   topk_weights [T,K] fp32; dest, is_in_rank from ep_compute_send_counts.
 *   num_send: host value, the number of rows the caller allocated for
 *     send_token_idx [N], send_rank [N], send_idx [N,K] int64, send_w [N,K]
 *     fp32.  It must equal sum(is_in_rank) (passing it from the host avoids
 *     a device sync, [AX] build_send_layout); a different device count sets
 *     EP_ERR_COUNT_MISMATCH and rows at or past num_send are not written
 *     (with T == 0 a non-zero num_send is returned as EP_ERR_COUNT_MISMATCH).
 * Device errors: EP_ERR_COUNT_MISMATCH. */
int ep_build_send_layout(const int64_t *topk_idx, const float *topk_weights,
                         const int32_t *dest, const uint8_t *is_in_rank,
                         int64_t T, int K, int P, int E_local, int64_t num_send,
                         int32_t *send_token_idx, int32_t *send_rank, int64_t *send_idx,
                         float *send_w, int32_t *token_pos,
                         void *ws, size_t ws_bytes, int32_t *err, ep_stream_t stream);

/* [AX] compute_send_counts followed by build_send_layout, without the host
 * round trip: the [UB] Buffer.dispatch "num_worst_tokens" mode, where the
 * receive buffers are sized for the worst case so that no CPU sync is needed
 * and the call can be enqueued back to back (or captured in a CUDA graph).
 * Computes the outputs of both calls for one chunk:
 *   dest, is_in_rank, send_counts [P], rank_offsets [P+1] (rank_offsets[P] =
 *   N, the number of rows the layout uses), tokens_per_expert [P*E_local] or
 *   NULL, and the send layout rows send_token_idx, send_rank, send_idx,
 *   send_w and token_pos exactly as ep_build_send_layout defines them.
 *   num_worst_rows: rows allocated in the send buffers (T * min(K, P) always
 *     suffices).  Rows N .. num_worst_rows-1 are left untouched; pass
 *     num_worst_rows as num_send to ep_dispatch / ep_combine.  If N exceeds it,
 *     EP_ERR_CAPACITY is set and rows past it are not written (token_pos -1).
 * One cooperative launch when its blocks fit on the GPU at once, else two
 * launches; ws as for ep_compute_send_counts with chunks = 1.  The call may be
 * captured in a CUDA graph: every replay recomputes all outputs from the
 * current contents of topk_idx and topk_weights.
 * Device errors: EP_ERR_INVALID_EXPERT, EP_ERR_CAPACITY, EP_ERR_COUNT_MISMATCH,
 * EP_ERR_TIMEOUT (the single launch's blocks did not all arrive within 0.5 s;
 * the outputs are then undefined). */
int ep_route_nosync(const int64_t *topk_idx, const float *topk_weights, int64_t T, int K, int P,
                    int E_local, int64_t num_worst_rows,
                    int32_t *dest, uint8_t *is_in_rank, int32_t *send_counts, int32_t *rank_offsets,
                    int32_t *tokens_per_expert,
                    int32_t *send_token_idx, int32_t *send_rank, int64_t *send_idx, float *send_w,
                    int32_t *token_pos, void *ws, size_t ws_bytes, int32_t *err, ep_stream_t stream);

/* ep_route_nosync with the receive alignment of [UB] Buffer.dispatch
 * (expert_alignment) applied to the send layout: every rank's segment starts
 * at a multiple of `alignment` rows, i.e. rank_offsets is the exclusive scan
 * of round_up(send_counts[p], alignment) (send_counts stays the true count).
 * Rank p's rows keep the order of ep_build_send_layout from rank_offsets[p];
 * the rows after them up to rank_offsets[p+1] are pad rows carrying no token:
 * send_token_idx -1, send_rank p, send_idx -1, send_w +0 (so a local kernel
 * over whole segments adds nothing for them; ep_dispatch does not write their
 * recv_x rows).  token_pos points at the rows in this padded layout, so
 * ep_dispatch / ep_combine work unchanged.  tokens_per_expert, if requested,
 * is rounded up to a multiple of `alignment`.
 *   num_worst_rows: T * min(K, P) + P * (alignment - 1) always suffices.
 *   alignment >= 1 (1 is ep_route_nosync).
 * Errors as ep_route_nosync. */
int ep_route_nosync_aligned(const int64_t *topk_idx, const float *topk_weights, int64_t T, int K, int P,
                            int E_local, int64_t num_worst_rows, int alignment,
                            int32_t *dest, uint8_t *is_in_rank, int32_t *send_counts, int32_t *rank_offsets,
                            int32_t *tokens_per_expert,
                            int32_t *send_token_idx, int32_t *send_rank, int64_t *send_idx, float *send_w,
                            int32_t *token_pos, void *ws, size_t ws_bytes, int32_t *err, ep_stream_t stream);

/* [AX] dispatch on the collective-free local path, [UB] Buffer.dispatch
 * payloads: recv_x[n] = x[t] for every (t, p) with n = token_pos[t,p] >= 0.
 * Each source row is read once and written to each of its rows.
 *   x [T,H] bf16.  token_pos [T,P] from ep_build_send_layout.
 *   fp8 == 0: recv_x [num_send,H] bf16 (bit copy); recv_scale must be NULL.
 *   fp8 == 1: recv_x [num_send,H] fp8 e4m3 and recv_scale [num_send,H/128]
 *     fp32, quantised per token in 1x128 groups: a = max(max|x|, 1e-4),
 *     q = e4m3_rn_satfinite(x * (448/a)), scale = a/448 (fp32, round to
 *     nearest even); every row sent for a token carries the same bytes.
 *     NaN elements do not enter the maximum; a group holding +-inf has
 *     scale +inf and reciprocal +0 (finite elements give +-0 codes,
 *     infinities and NaNs NaN codes).  Needs H % 128 == 0.
 * Device errors: EP_ERR_COUNT_MISMATCH (a token_pos entry >= num_send). */
int ep_dispatch(const void *x, int64_t T, int H, const int32_t *token_pos, int P,
                int64_t num_send, void *recv_x, float *recv_scale, int fp8,
                int32_t *err, ep_stream_t stream);

/* [UB] Buffer.dispatch in num_worst_tokens mode on the collective-free path:
 * ep_route_nosync (all its outputs, rows sized num_worst_rows) followed by
 * ep_dispatch of x into recv_x (bf16, or fp8 codes + scales when fp8 = 1),
 * in one call.  The dispatch is launched as a programmatic dependent of the
 * routing kernel, so its blocks load their input rows while routing
 * finishes; x must therefore be complete before the call (it is read by the
 * dispatch before the routing kernel ends, never written by it).  Arguments
 * and errors as the two calls; recv_scale is used only with fp8 = 1. */
int ep_dispatch_nosync(const void *x, const int64_t *topk_idx, const float *topk_weights, int64_t T, int K,
                       int H, int P, int E_local, int64_t num_worst_rows, int fp8,
                       int32_t *dest, uint8_t *is_in_rank, int32_t *send_counts, int32_t *rank_offsets,
                       int32_t *tokens_per_expert, int32_t *send_token_idx, int32_t *send_rank,
                       int64_t *send_idx, float *send_w, int32_t *token_pos, void *recv_x, float *recv_scale,
                       void *ws, size_t ws_bytes, int32_t *err, ep_stream_t stream);

/* [AX] combine, [UB] Buffer.combine (an unweighted sum): the local
 * expert kernel has already weighted and summed over K, so
 *   out[t] = sum over p ascending with token_pos[t,p] >= 0 of y[token_pos[t,p]]
 * accumulated in fp32 from +0.0f and rounded once; tokens sent nowhere give
 * +0 ([AX] dispatch: unrouted tokens combine to zero).
 *   y [num_send,H] bf16.  out [T,H]: bf16 (out_dtype 0) or fp32 (out_dtype 1).
 *   ws: optional device scratch of at least EP_COMBINE_WS_BYTES bytes (any
 *     contents; 16-byte aligned), or NULL.  With it the SMs take work from a
 *     shared counter that the call first clears with one cudaMemsetAsync, which
 *     balances skewed source counts; with NULL the work is dealt round-robin.
 *     Results are identical either way.  Calls that overlap on the GPU must not
 *     share a ws.
 * Device errors: EP_ERR_COUNT_MISMATCH (a token_pos entry >= num_send). */
int ep_combine(const void *y, int64_t T, int H, const int32_t *token_pos, int P,
               int64_t num_send, void *out, int out_dtype, void *ws, size_t ws_bytes,
               int32_t *err, ep_stream_t stream);

/* [VB] BatchedPrepareAndFinalize.prepare, unquantised branch: the
 * expert-batched layout [E_local, max_num_tokens, H].  Local experts are
 * [rank*E_local, (rank+1)*E_local).  For local expert e_l, the tokens naming
 * it in some slot, in ascending token order, take slots 0, 1, ...:
 *   b_x[e_l, s] = x[t],  slot[t,k] = s for every k naming e_l,
 *   tokens_per_expert[e_l] = number of such tokens (clipped to M).
 * slot [T,K] int32 is -1 for slots naming non-local experts; it is the handle
 * of ep_batched_combine.  Rows at or past tokens_per_expert[e_l] are left
 * untouched unless zero_pad != 0 (then zero-filled, as the page's zero
 * allocation does).  A token past max_num_tokens is dropped (slot -1, row not
 * written) and sets EP_ERR_CAPACITY.
 *   x [T,H] bf16, topk_idx [T,K] int64, E = total experts (E % E_local == 0),
 *   tokens_per_expert [E_local] int32.
 *   ws: ep_workspace_size(T, K, E / E_local, E_local, 1) bytes, 256-byte
 *     aligned.  With E_local <= 64 the slots take one launch (one
 *     thread-block cluster up to 32768 tokens, else a cooperative launch).
 * Device errors: EP_ERR_INVALID_EXPERT, EP_ERR_CAPACITY, EP_ERR_TIMEOUT. */
int ep_batched_prepare(const void *x, const int64_t *topk_idx, int64_t T, int K, int H,
                       int E, int E_local, int rank, int max_num_tokens,
                       void *b_x, int32_t *tokens_per_expert, int32_t *slot, int zero_pad,
                       void *ws, size_t ws_bytes, int32_t *err, ep_stream_t stream);

/* Scale layouts of ep_batched_prepare_fp8 ([UB] Buffer.low_latency_dispatch
 * returns the scales of the expert-batched fp8 payload with the last two
 * dimensions column-major; [VB] prepare's batched scale shape is row-major).
 * G = H/128 groups per row, M = max_num_tokens, (e, s, g) = local expert,
 * slot, group. */
#define EP_SCALE_ROW_F32 0    /* fp32 [E_local, M, G] row-major: (e,s,g) at (e*M + s)*G + g */
#define EP_SCALE_COL_F32 1    /* fp32 [E_local, M, G], last two dims column-major: (e,s,g) at (e*G + g)*M + s */
#define EP_SCALE_COL_UE8M0 2  /* int32 [E_local, M, G/4], last two dims column-major: int (e,s,j) at
                               * (e*(G/4) + j)*M + s; its byte i (least significant first) is the
                               * UE8M0 code of group 4j+i.  Needs round_scale = 1 and H % 512 == 0. */

/* [VB] BatchedPrepareAndFinalize.prepare, quantised branch, with the fp8
 * payload of [UB] Buffer.low_latency_dispatch (use_fp8, round_scale,
 * use_ue8m0): the slots, tokens_per_expert, capacity rule and slot handle of
 * ep_batched_prepare, with rows of e4m3 codes b_q [E_local, M, H] and group
 * scales b_scale in scale_fmt.  Each token is quantised once in 1x128 groups
 * and every slot it takes carries the same bytes; with a = max(max|x|, 1e-4):
 *   round_scale = 0: q = e4m3_rn_satfinite(x * (448/a)), scale = a/448 (fp32,
 *     round to nearest even), exactly as ep_dispatch with fp8 = 1;
 *   round_scale = 1: scale = the smallest power of two >= a/448 (the fp32
 *     quotient), q = e4m3_rn_satfinite(x / scale) (exact division); its UE8M0
 *     code is log2(scale) + 127.
 *   Non-finite inputs, both forms: NaN elements do not enter the maximum; a
 *   group holding +-inf has scale +inf, reciprocal +0 and UE8M0 code 255.
 * zero_pad != 0 zero-fills the codes and scale entries of slots at or past
 * tokens_per_expert (the page's zero-initialised outputs); otherwise they are
 * left untouched.  b_q 16-byte aligned, b_scale 4-byte aligned; ws as for
 * ep_batched_prepare.
 * Host errors: EP_ERR_UNSUPPORTED (H % 128 != 0; UE8M0 without round_scale or
 * with H % 512 != 0), EP_ERR_INVALID_ARG (unknown scale_fmt, null pointers).
 * Device errors: EP_ERR_INVALID_EXPERT, EP_ERR_CAPACITY, EP_ERR_TIMEOUT. */
int ep_batched_prepare_fp8(const void *x, const int64_t *topk_idx, int64_t T, int K, int H,
                           int E, int E_local, int rank, int max_num_tokens,
                           uint8_t *b_q, void *b_scale, int scale_fmt, int round_scale,
                           int32_t *tokens_per_expert, int32_t *slot, int zero_pad,
                           void *ws, size_t ws_bytes, int32_t *err, ep_stream_t stream);

/* The expert-batched prepare with a per-expert capacity and a receive
 * alignment ([ND] TokenDispatcherConfig: moe_expert_capacity_factor, where
 * leaving it unset drops nothing, and moe_router_expert_pad_multiple; [UB]
 * Buffer.dispatch expert_alignment, which makes each local expert's received
 * count a multiple of it).  ep_batched_prepare and ep_batched_prepare_fp8 are
 * this call with capacity = 0, alignment = 1, dropped = NULL.
 *   capacity: 0 = max_num_tokens, with tokens past it dropped and reported as
 *     EP_ERR_CAPACITY (as ep_batched_prepare); 1 .. max_num_tokens = each local
 *     expert keeps the first `capacity` tokens naming it, in token order, and
 *     drops the later ones (slot -1, row not written) without an error: that
 *     is the capacity's purpose.  ep_expert_capacity gives it from a factor.
 *   alignment >= 1: tokens_per_expert[e] = min(round_up(kept_e, alignment),
 *     max_num_tokens) where kept_e is the number of tokens the expert kept;
 *     rows kept_e .. tokens_per_expert[e]-1 are zero rows (codes 0 and zero
 *     scale entries for fp8), so a grouped GEMM over the aligned counts reads
 *     zeros there.  Choose max_num_tokens a multiple of alignment.
 *   scale_fmt: -1 = bf16 rows (b_rows [E_local, M, H] bf16, b_scale NULL), or
 *     an EP_SCALE_* layout with round_scale as ep_batched_prepare_fp8 (b_rows
 *     holds e4m3 codes [E_local, M, H]).
 *   dropped: [E_local] int32 tokens dropped per expert, or NULL.
 *   zero_pad: also zero rows (and scale entries) past tokens_per_expert.
 *   ws: ep_workspace_size(T, K, E / E_local, E_local, 1) bytes.
 * Host errors: EP_ERR_INVALID_ARG (capacity outside 0..max_num_tokens,
 * alignment < 1, unknown scale_fmt), EP_ERR_UNSUPPORTED as for
 * ep_batched_prepare_fp8.  Device errors: EP_ERR_INVALID_EXPERT,
 * EP_ERR_CAPACITY (capacity = 0 only), EP_ERR_TIMEOUT. */
int ep_batched_prepare_ex(const void *x, const int64_t *topk_idx, int64_t T, int K, int H,
                          int E, int E_local, int rank, int max_num_tokens, int capacity, int alignment,
                          void *b_rows, void *b_scale, int scale_fmt, int round_scale,
                          int32_t *tokens_per_expert, int32_t *slot, int32_t *dropped, int zero_pad,
                          void *ws, size_t ws_bytes, int32_t *err, ep_stream_t stream);

/* Per-expert capacity from a capacity factor (host only): ceil(factor * T * K
 * / E), the expected tokens per expert scaled by the factor ([ND]
 * moe_expert_capacity_factor).  -1 for T < 0, K < 1, E < 1 or factor <= 0. */
int64_t ep_expert_capacity(int64_t T, int K, int E, double factor);

/* [VB] BatchedPrepareAndFinalize.finalize, [UB] Buffer.low_latency_combine
 * (a weighted reduction): this rank's partial
 *   out[t] = sum over k ascending with a local expert e_l = topk_idx[t,k] -
 *            rank*E_local and slot[t,k] >= 0 of topk_weights[t,k] * y[e_l, slot[t,k]]
 * with fp32 fused multiply-add from +0.0f, rounded once to bf16; tokens with
 * no local expert give +0.  Padding rows of y are never read.
 *   y [E_local, max_num_tokens, H] bf16, out [T,H] bf16.
 *   ws: optional scratch as for ep_combine.
 * Device errors: EP_ERR_CAPACITY (a slot >= max_num_tokens). */
int ep_batched_combine(const void *y, const int64_t *topk_idx, const float *topk_weights,
                       const int32_t *slot, int64_t T, int K, int H, int E_local, int rank,
                       int max_num_tokens, void *out, void *ws, size_t ws_bytes,
                       int32_t *err, ep_stream_t stream);

/* Synthetic local expert kernel for fp8 dispatch workloads (the local_kernel
 * argument of [AX] dispatch_chunked_forward; the local kernel "weights and
 * sums over K", [AX] module description).  Expert l maps a token to
 * dequant(x) * (1 + l/64) in bf16:
 *   d = e4m3(q) * scale,  y_k = bf16(d * (1 + l_k/64)) for send_idx[n,k] = l_k >= 0,
 *   out[n] = bf16(fma over k ascending of send_w[n,k] * y_k, from +0.0f).
 *   recv_q [N,H] e4m3, recv_scale [N,H/128] fp32, send_idx [N,K] int64,
 *   send_w [N,K] fp32, out [N,H] bf16.  H % 128 == 0. */
int ep_local_expert_fp8(const uint8_t *recv_q, const float *recv_scale, const int64_t *send_idx,
                        const float *send_w, int64_t N, int K, int H, void *out,
                        int32_t *err, ep_stream_t stream);

/* [AX] dispatch_chunked_forward on one GPU: dispatch -> local_kernel ->
 * combine over `chunks` contiguous token ranges ([AX] chunk_bounds).  The
 * split counts of every chunk come from ONE ep_compute_send_counts launch and
 * ONE device-to-host copy (into h_counts, pinned host memory of chunks*P
 * int32, after which the host waits once); then, per chunk in order on
 * `stream`: ep_build_send_layout, ep_dispatch (bf16, or fp8 when fp8 = 1),
 * local_kernel, ep_combine into the chunk's rows of out [T,H] bf16.  The
 * pages overlap the next chunk's all-to-alls with the current chunk's expert
 * compute; one GPU has no exchange to hide, so chunks run in order.
 *   local_kernel: called once per chunk with the chunk's received rows
 *     (recv_x, recv_scale, send_idx, send_w, n_rows of them) and must enqueue,
 *     on `stream`, the weighted sum over K of its experts into local_out
 *     [n_rows, H] bf16 ([AX] module description); it returns an ep_status.
 *     ep_local_expert_fp8_callback is the synthetic fp8 expert as a callback.
 *   b: device buffers sized by the caller; every chunk's rows must fit in
 *     max_rows (else EP_ERR_CAPACITY, returned before that chunk runs).
 * Returns the first non-OK status of the calls it makes. */
typedef int (*ep_local_kernel_fn)(void *user, int chunk, int64_t n_rows, int K, int H,
                                  const void *recv_x, const float *recv_scale,
                                  const int64_t *send_idx, const float *send_w, void *local_out,
                                  int32_t *err, ep_stream_t stream);

typedef struct ep_chunk_buffers {
    int32_t *dest;             /* [T,K] */
    uint8_t *is_in_rank;       /* [T,P] */
    int32_t *send_counts;      /* [chunks,P] */
    int32_t *rank_offsets;     /* [chunks,P+1] */
    int32_t *token_pos;        /* [T,P] */
    int64_t max_rows;          /* rows of the per-chunk buffers below */
    int32_t *send_token_idx;   /* [max_rows] */
    int32_t *send_rank;        /* [max_rows] */
    int64_t *send_idx;         /* [max_rows,K] */
    float *send_w;             /* [max_rows,K] */
    void *recv_x;              /* [max_rows,H] bf16, or e4m3 when fp8 */
    float *recv_scale;         /* [max_rows,H/128] when fp8, else NULL */
    void *local_out;           /* [max_rows,H] bf16 */
    void *ws;                  /* ep_workspace_size(T, K, P, E_local, chunks) bytes */
    size_t ws_bytes;
    void *combine_ws;          /* EP_COMBINE_WS_BYTES bytes, or NULL */
} ep_chunk_buffers;

int ep_dispatch_chunked_forward(const void *x, const int64_t *topk_idx, const float *topk_weights,
                                int64_t T, int K, int H, int P, int E_local, int chunks, int fp8,
                                ep_local_kernel_fn local_kernel, void *user, void *out,
                                const ep_chunk_buffers *b, int32_t *h_counts, int32_t *err,
                                ep_stream_t stream);

/* ep_local_expert_fp8 in the ep_local_kernel_fn shape (user and chunk unused). */
int ep_local_expert_fp8_callback(void *user, int chunk, int64_t n_rows, int K, int H,
                                 const void *recv_x, const float *recv_scale,
                                 const int64_t *send_idx, const float *send_w, void *local_out,
                                 int32_t *err, ep_stream_t stream);

/* [AX] dispatch_chunked_forward without a host round trip, pipelined over
 * two streams: the pages overlap chunk i+1's all-to-alls with chunk i's expert
 * compute, and [UB] Buffer.dispatch's "num_worst_tokens" mode sizes the
 * receive buffers for the worst case so that nothing waits on the CPU.  Per
 * chunk c (the token range of [AX] chunk_bounds):
 *   on aux_stream: ep_route_nosync (num_worst_rows = b->max_rows), ep_dispatch
 *     (bf16, or fp8 when fp8 = 1) into row set c % n_sets;
 *   on stream: local_kernel, then ep_combine into the chunk's rows of
 *     out [T,H] bf16.
 * With two row sets, chunk c+1's routing and dispatch run while chunk c's
 * local kernel and combine do; events order each set's reuse.  With one set
 * (aux_stream may then be NULL) everything runs in order on `stream`.  The
 * call never waits on the host, so it may be captured in a CUDA graph (stream
 * must be the capturing stream; aux_stream joins the capture through events)
 * and replayed on new inputs.  The results equal those of
 * ep_dispatch_chunked_forward with the same local kernel.
 *   local_kernel: as for ep_dispatch_chunked_forward, but it receives the row
 *     capacity max_rows and a DEVICE pointer n_rows to the chunk's row count
 *     (rank_offsets[c, P]); it must leave rows at or past *n_rows alone (they
 *     hold stale data) and enqueue only on `stream`.
 *     ep_local_expert_fp8_dev_callback is the synthetic fp8 expert in this form.
 *   b->max_rows: rows of every row set; (longest chunk) * min(K, P) never
 *     drops.  A chunk with more rows sets EP_ERR_CAPACITY on the device, and
 *     its rows past max_rows are neither dispatched nor combined.
 *   b->ws: ep_workspace_size(T, K, P, E_local, chunks) bytes; b->combine_ws:
 *     EP_COMBINE_WS_BYTES bytes or NULL.  Both are used by one stream each.
 * Returns the first non-OK status of the calls it makes; device errors go to
 * err as for the calls above. */
typedef int (*ep_local_kernel_dev_fn)(void *user, int chunk, int64_t max_rows, const int32_t *n_rows, int K,
                                      int H, const void *recv_x, const float *recv_scale,
                                      const int64_t *send_idx, const float *send_w, void *local_out,
                                      int32_t *err, ep_stream_t stream);

typedef struct ep_row_set {
    int32_t *send_token_idx;   /* [max_rows] */
    int32_t *send_rank;        /* [max_rows] */
    int64_t *send_idx;         /* [max_rows,K] */
    float *send_w;             /* [max_rows,K] */
    void *recv_x;              /* [max_rows,H] bf16, or e4m3 when fp8 */
    float *recv_scale;         /* [max_rows,H/128] when fp8, else NULL */
    void *local_out;           /* [max_rows,H] bf16 */
} ep_row_set;

typedef struct ep_pipeline_buffers {
    int32_t *dest;             /* [T,K] */
    uint8_t *is_in_rank;       /* [T,P] */
    int32_t *send_counts;      /* [chunks,P] */
    int32_t *rank_offsets;     /* [chunks,P+1] */
    int32_t *token_pos;        /* [T,P] */
    int64_t max_rows;
    int n_sets;                /* 1 or 2 */
    ep_row_set sets[2];        /* chunk c uses sets[c % n_sets] */
    void *ws;
    size_t ws_bytes;
    void *combine_ws;
} ep_pipeline_buffers;

int ep_dispatch_chunked_forward_nosync(const void *x, const int64_t *topk_idx, const float *topk_weights,
                                       int64_t T, int K, int H, int P, int E_local, int chunks, int fp8,
                                       ep_local_kernel_dev_fn local_kernel, void *user, void *out,
                                       const ep_pipeline_buffers *b, int32_t *err, ep_stream_t stream,
                                       ep_stream_t aux_stream);

/* ep_local_expert_fp8 in the ep_local_kernel_dev_fn shape: max_rows blocks,
 * rows at or past *n_rows skipped (user and chunk unused). */
int ep_local_expert_fp8_dev_callback(void *user, int chunk, int64_t max_rows, const int32_t *n_rows, int K,
                                     int H, const void *recv_x, const float *recv_scale,
                                     const int64_t *send_idx, const float *send_w, void *local_out,
                                     int32_t *err, ep_stream_t stream);

/* [ND] _DeepepManager._indices_to_multihot / _HybridEPManager.
 * _indices_to_multihot: top-k indices and probabilities to the multihot
 * routing map and the dense probabilities, a second metadata view of the
 * same topk_idx:
 *   routing_map[t,e] = 1 iff some slot k of token t names expert e, else 0;
 *   probs[t,e] = the sum of topk_probs[t,k] over the slots naming e, in fp32
 *     from +0.0f in ascending k (a single slot copies its probability),
 *     +0.0f where routing_map is 0.
 *   topk_idx [T,K] int64 (-1 masked), topk_probs [T,K] fp32 (may be NULL
 *   when probs is NULL), routing_map [T,E] uint8 or NULL, probs [T,E] fp32 or
 *   NULL (not both NULL).  One launch, no workspace, no host sync.
 * Device errors: EP_ERR_INVALID_EXPERT (an id outside [-1, E); the slot is
 * ignored). */
int ep_indices_to_multihot(const int64_t *topk_idx, const float *topk_probs, int64_t T, int K, int E,
                           uint8_t *routing_map, float *probs, int32_t *err, ep_stream_t stream);

/* Same as ep_compute_send_counts, but the caller passes no workspace: the
 * scratch lives in one fixed device array of EP_NOALLOC_SCRATCH_BYTES that the
 * library holds on every device that loads it, until the process exits.  The
 * pages have no counterpart of this call; it is for callers that cannot
 * allocate device memory themselves, such as engines that plan all device
 * memory up front and forbid allocation while they run (a plugin's enqueue
 * step, where the host thread must not call into an allocator).
 *   - Arguments are checked on the host first, as in ep_compute_send_counts
 *     (EP_ERR_INVALID_ARG), without touching a device.  Sizes whose workspace
 *     (ep_workspace_size) exceeds EP_NOALLOC_SCRATCH_BYTES are then rejected
 *     with EP_ERR_UNSUPPORTED before anything is launched (1 MiB covers e.g.
 *     T = 65536, P = 16, E = 256).
 *   - The first call on a device, with that device current, looks up the
 *     array's device address (cudaGetSymbolAddress) and caches it together
 *     with the id of the current context; make that first call before any
 *     stream capture begins.  A call under another context of the device
 *     (after a device reset, say) looks the address up again.
 *   - All calls on a device share the array and it keeps the last call's
 *     contents (nothing in it needs to start at zero).  Calls whose kernels
 *     overlap on the GPU -- on other streams or from other host threads --
 *     race on it; serialise them.
 *   - Allocates nothing: no cudaMalloc, cudaFree or allocating library call. */
#define EP_NOALLOC_SCRATCH_BYTES (1u << 20)

int ep_compute_send_counts_noalloc(const int64_t *topk_idx, int64_t T, int K, int P, int E_local,
                                   const int64_t *h_chunk_bounds, int chunks,
                                   int32_t *dest, uint8_t *is_in_rank, int32_t *send_counts,
                                   int32_t *rank_offsets, int32_t *tokens_per_expert,
                                   int32_t *err, ep_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* EP_GB300_H */
