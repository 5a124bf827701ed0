// Routing metadata kernels of libep_gb300:
//   counts  -- axolotl integrations.expert_parallel.torch_dispatch,
//              compute_send_counts; NeMo uccl_ep.buffer, get_dispatch_layout
//   layout  -- axolotl build_send_layout (rank-major, token-ascending order)
//   slots   -- vLLM BatchedPrepareAndFinalize.prepare (per-expert slots that
//              preserve token order)
//
// All three are the same pattern: one thread per token, a warp ballot per
// destination (rank or local expert) gives each warp's count and every lane's
// rank among the lanes before it, a shared-memory pass over the block's warps
// gives the block count, and a reduce-then-scan over blocks gives each
// block's starting offset.  The block partials go through the caller's
// workspace: either from one launch to the next, or, in the single-launch
// (cooperative) forms, across a bounded grid barrier inside one kernel.  No
// atomics decide any position, so every index is deterministic and the order
// is token-ascending by construction.
#include <algorithm>
#include <atomic>
#include <type_traits>

#include "ep_barrier.cuh"
#include "ep_device.cuh"
#include "ep_internal.h"
#include "ep_slots.cuh"

namespace ep {

constexpr int kWarps = kRouteThreads / 32;

// ----------------------------------------------------------------- counts --
__device__ __forceinline__ int chunk_of_block(const ChunkTable &ct, int b)
{
    int c = 0;
    while (c + 1 < ct.n && ct.first_block[c + 1] <= b)
        ++c;
    return c;
}

// One block of 256 tokens (never straddling a chunk): dest, is_in_rank, the
// block's per-rank token counts and, optionally, its per-expert token counts.
__global__ void __launch_bounds__(kRouteThreads)
count_kernel(const int64_t *__restrict__ idx, int K, int P, int E_local, ChunkTable ct,
             int32_t *__restrict__ dest, uint8_t *__restrict__ is_in_rank,
             int32_t *__restrict__ part_rank, int32_t *__restrict__ part_expert, int32_t *err)
{
    extern __shared__ int32_t smem[];
    int32_t *warp_cnt = smem;                 // [kWarps][P]
    int32_t *hist = smem + kWarps * P;        // [E], when part_expert != nullptr
    const int E = P * E_local;
    const int b = blockIdx.x;
    const int c = chunk_of_block(ct, b);
    const int64_t t = ct.start[c] + (int64_t)(b - ct.first_block[c]) * kRouteThreads + threadIdx.x;
    const bool valid = t < ct.start[c + 1];

    if (part_expert != nullptr) {
        for (int e = threadIdx.x; e < E; e += blockDim.x)
            hist[e] = 0;
        __syncthreads();
    }

    uint64_t mask = 0;
    int bad = 0;
    if (valid) {
        const int64_t *row = idx + t * K;
        int32_t *drow = dest + t * K;
        for (int k = 0; k < K; ++k) {
            const int64_t id = row[k];
            int d = -1;
            if (id >= 0 && id < E)
                d = (int)(id / E_local);
            else if (id != -1)
                bad = EP_ERR_INVALID_EXPERT;
            drow[k] = d;
            if (d >= 0) {
                mask |= 1ull << d;
                if (part_expert != nullptr) {
                    bool seen = false;          // count a token once per expert
                    for (int j = 0; j < k; ++j)
                        seen |= (row[j] == id);
                    if (!seen)
                        atomicAdd(&hist[id], 1);
                }
            }
        }
        uint8_t *irow = is_in_rank + t * P;
        for (int p = 0; p < P; ++p)
            irow[p] = (uint8_t)((mask >> p) & 1ull);
    }

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int p = 0; p < P; ++p) {
        const unsigned bal = __ballot_sync(kFull, (mask >> p) & 1ull);
        if (lane == 0)
            warp_cnt[warp * P + p] = __popc(bal);
    }
    __syncthreads();
    for (int p = threadIdx.x; p < P; p += blockDim.x) {
        int s = 0;
        for (int w = 0; w < kWarps; ++w)
            s += warp_cnt[w * P + p];
        part_rank[(int64_t)b * P + p] = s;
    }
    if (part_expert != nullptr)
        for (int e = threadIdx.x; e < E; e += blockDim.x)
            part_expert[(int64_t)b * E + e] = hist[e];
    raise(err, bad);
}

// Sum of `n` values strided by `stride`, with eight loads in flight at a time
// (a plain loop would wait for each L2 round trip in turn).
__device__ __forceinline__ int strided_sum(const int32_t *__restrict__ p, int n, int64_t stride)
{
    int s[8] = {0, 0, 0, 0, 0, 0, 0, 0};
    int i = 0;
    for (; i + 8 <= n; i += 8) {
#pragma unroll
        for (int u = 0; u < 8; ++u)
            s[u] += p[(int64_t)(i + u) * stride];
    }
    for (; i < n; ++i)
        s[0] += p[(int64_t)i * stride];
    return ((s[0] + s[1]) + (s[2] + s[3])) + ((s[4] + s[5]) + (s[6] + s[7]));
}

// Single block: per-chunk send_counts and rank_offsets, tokens_per_expert.
// Each column sum over the blocks' partials is split over `S` adjacent lanes
// (S = 1024 / columns, a power of two up to 32) and joined with shuffles.
__global__ void __launch_bounds__(1024)
count_finish_kernel(const int32_t *__restrict__ part_rank, const int32_t *__restrict__ part_expert,
                    int nb, int P, int E, ChunkTable ct, int32_t *__restrict__ send_counts,
                    int32_t *__restrict__ rank_offsets, int32_t *__restrict__ tokens_per_expert)
{
    __shared__ int32_t s_cnt[EP_MAX_CHUNKS * EP_MAX_RANKS];
    const int CP = ct.n * P;
    {
        int S = 1;
        while (S < 32 && CP * S * 2 <= (int)blockDim.x)
            S *= 2;
        for (int base = 0; base < CP * S; base += blockDim.x) {
            const int i = base + threadIdx.x;
            const int col = i / S, part = i % S;
            int v = 0;
            if (col < CP) {
                const int c = col / P, p = col % P;
                const int b0 = ct.first_block[c], nbc = ct.first_block[c + 1] - b0;
                const int per = (nbc + S - 1) / S;
                const int lo = min(nbc, part * per), hi = min(nbc, lo + per);
                v = strided_sum(part_rank + (int64_t)(b0 + lo) * P + p, hi - lo, P);
            }
            for (int off = S / 2; off > 0; off >>= 1)
                v += __shfl_down_sync(kFull, v, off, S);
            if (col < CP && part == 0) {
                send_counts[col] = v;
                s_cnt[col] = v;
            }
        }
    }
    if (tokens_per_expert != nullptr) {
        int S = 1;
        while (S < 32 && E * S * 2 <= (int)blockDim.x)
            S *= 2;
        const int per = (nb + S - 1) / S;
        for (int base = 0; base < E * S; base += blockDim.x) {
            const int i = base + threadIdx.x;
            const int e = i / S, part = i % S;
            int v = 0;
            if (e < E) {
                const int lo = min(nb, part * per), hi = min(nb, lo + per);
                v = strided_sum(part_expert + (int64_t)lo * E + e, hi - lo, E);
            }
            for (int off = S / 2; off > 0; off >>= 1)
                v += __shfl_down_sync(kFull, v, off, S);
            if (e < E && part == 0)
                tokens_per_expert[e] = v;
        }
    }
    if (rank_offsets != nullptr) {
        __syncthreads();
        for (int c = threadIdx.x; c < ct.n; c += blockDim.x) {
            int run = 0;
            for (int p = 0; p < P; ++p) {
                rank_offsets[c * (P + 1) + p] = run;
                run += s_cnt[c * P + p];
            }
            rank_offsets[c * (P + 1) + P] = run;
        }
    }
}

// ----------------------------------------------------------------- layout --
__device__ __forceinline__ uint64_t rank_mask(const uint8_t *__restrict__ is_in_rank, int64_t t, int P)
{
    uint64_t m = 0;
    const uint8_t *row = is_in_rank + t * P;
    for (int p = 0; p < P; ++p)
        m |= (uint64_t)(row[p] != 0) << p;
    return m;
}

__global__ void __launch_bounds__(kRouteThreads)
layout_count_kernel(const uint8_t *__restrict__ is_in_rank, int64_t T, int P,
                    int32_t *__restrict__ part_rank)
{
    __shared__ int32_t warp_cnt[kWarps][EP_MAX_RANKS];
    const int64_t t = (int64_t)blockIdx.x * kRouteThreads + threadIdx.x;
    const uint64_t mask = t < T ? rank_mask(is_in_rank, t, P) : 0;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int p = 0; p < P; ++p) {
        const unsigned bal = __ballot_sync(kFull, (mask >> p) & 1ull);
        if (lane == 0)
            warp_cnt[warp][p] = __popc(bal);
    }
    __syncthreads();
    for (int p = threadIdx.x; p < P; p += blockDim.x) {
        int s = 0;
        for (int w = 0; w < kWarps; ++w)
            s += warp_cnt[w][p];
        part_rank[(int64_t)blockIdx.x * P + p] = s;
    }
}

// Exclusive scan over the up-to-64 values held as (v0 for index lane,
// v1 for index lane+32) by one warp; returns the grand total.
__device__ __forceinline__ int warp_exclusive_scan64(int v0, int v1, int &e0, int &e1)
{
    const int lane = threadIdx.x & 31;
    int i0 = v0, i1 = v1;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int n0 = __shfl_up_sync(kFull, i0, off);
        const int n1 = __shfl_up_sync(kFull, i1, off);
        if (lane >= off) {
            i0 += n0;
            i1 += n1;
        }
    }
    const int s0 = __shfl_sync(kFull, i0, 31);
    const int s1 = __shfl_sync(kFull, i1, 31);
    e0 = i0 - v0;
    e1 = s0 + i1 - v1;
    return s0 + s1;
}

// Lane of the r-th (0-based) set bit of m; r < popc(m).  Binary search over
// halves, so the result is always a lane in [0, 32).
__device__ __forceinline__ int nth_set_bit(unsigned m, int r)
{
    int pos = 0;
#pragma unroll
    for (int width = 16; width > 0; width >>= 1) {
        const int c = __popc(m & ((1u << width) - 1u));
        if (r >= c) {
            r -= c;
            m >>= width;
            pos += width;
        }
    }
    return pos;
}

// s_tot[p] += sum over all blocks of part[bb*P + p]; s_before[p] += the same
// over blocks bb < b.  Thread i sums rank i % P over every (blockDim/P)-th
// block, eight loads in flight at a time, then adds into shared memory.
// The caller zeroes s_tot / s_before and synchronises before and after.
__device__ __forceinline__ int round_up(int v, int a) { return (v + a - 1) / a * a; }

// Pad rows of an aligned send layout (whole block; block b takes ranks b,
// b + gridDim, ...): rank p's segment holds its rows, then pad rows from
// pad_first[p] up to the next multiple of `align`; a pad row carries no token
// (token -1, rank p, no experts, zero weights).  Rows at or past num_rows are
// not written.
__device__ __forceinline__ void fill_pad_rows(const int32_t *pad_first, int P, int K, int align, int64_t num_rows,
                                              int32_t *send_token_idx, int32_t *send_rank, int64_t *send_idx,
                                              float *send_w)
{
    for (int p = blockIdx.x; p < P; p += gridDim.x) {   // ranks spread over the blocks
        const int64_t lo = pad_first[p], hi = round_up(pad_first[p], align);
        for (int64_t n = lo + threadIdx.x; n < hi && n < num_rows; n += blockDim.x) {
            send_token_idx[n] = -1;
            send_rank[n] = p;
            for (int k = 0; k < K; ++k) {
                send_idx[n * K + k] = -1;
                send_w[n * K + k] = 0.0f;
            }
        }
    }
}

// Which layout outputs are aligned for vector stores: the C ABI promises
// only natural alignment for them, so a wider store is taken only where the
// caller's pointer allows it (decided on the host, uniform over the launch).
struct VecOk {
    bool send_idx;     // 16 bytes: pairs of int64
    bool send_w;       // 16 bytes: four floats
    bool is_in_rank;   // 4 bytes: four flags
    bool token_pos;    // 16 bytes: four ints
};

static VecOk vec_ok(const int64_t *send_idx, const float *send_w, const uint8_t *is_in_rank,
                    const int32_t *token_pos = nullptr)
{
    return VecOk{aligned(send_idx, 16), aligned(send_w, 16), aligned(is_in_rank, 4), aligned(token_pos, 16)};
}

// Outputs and mode of layout_write_kernel.
struct LayoutArgs {
    const int64_t *idx;
    const float *w;
    const int32_t *dest;
    const uint8_t *is_in_rank;
    int64_t T;
    int K, P, E_local;
    int64_t num_rows;         // rows in the caller's send buffers
    int exact;                // 1: the routed count must equal num_rows; 0: num_rows is a worst-case capacity
    const int32_t *part_rank; // [nb][P] block partials
    int nb;
    const int32_t *part_expert;   // [nb][E] or null
    int32_t *send_counts;     // [P] or null (written by block 0)
    int32_t *rank_offsets;    // [P+1] or null (written by block 0)
    int32_t *tokens_per_expert;   // [E] or null (experts split over the blocks)
    int32_t *send_token_idx, *send_rank;
    int64_t *send_idx;
    float *send_w;
    int32_t *token_pos;
    int32_t *err;
    int align;                // rank segments start at multiples of it; tokens_per_expert rounded up
    VecOk vec;                // which outputs take vector stores
};

// One token's K-wide send_idx / send_w row for rank p, from the token's ids,
// weights and owning ranks held in registers (KC = K at compile time).
template <int KC>
__device__ __forceinline__ void write_send_row(int64_t *si, float *sw, const int64_t (&id)[KC],
                                               const float (&wt)[KC], const int8_t (&dr)[KC], int p,
                                               int64_t off, VecOk vec)
{
    if ((KC & 1) == 0 && vec.send_idx) {
#pragma unroll
        for (int k = 0; k < KC; k += 2)
            *reinterpret_cast<longlong2 *>(si + k) =
                make_longlong2(dr[k] == p ? id[k] - off : -1, dr[k + 1] == p ? id[k + 1] - off : -1);
    } else {
#pragma unroll
        for (int k = 0; k < KC; ++k)
            si[k] = dr[k] == p ? id[k] - off : -1;
    }
    if ((KC & 3) == 0 && vec.send_w) {
#pragma unroll
        for (int k = 0; k < KC; k += 4)
            *reinterpret_cast<float4 *>(sw + k) =
                make_float4(dr[k] == p ? wt[k] : 0.0f, dr[k + 1] == p ? wt[k + 1] : 0.0f,
                            dr[k + 2] == p ? wt[k + 2] : 0.0f, dr[k + 3] == p ? wt[k + 3] : 0.0f);
    } else {
#pragma unroll
        for (int k = 0; k < KC; ++k)
            sw[k] = dr[k] == p ? wt[k] : 0.0f;
    }
}

// One block of 256 tokens: the block's first row per rank from the partials,
// each lane's row from warp ballots, then the rows.  KC > 0 (K == KC at
// compile time): each thread loads its token's K ids, weights and owning
// ranks once into registers and writes its own rows (vector stores where the
// outputs are aligned for them).  KC == 0: a warp writes the K-wide send_idx /
// send_w rows of its tokens for one rank together (its rows for rank p are
// consecutive), reading each element where it writes it.
template <int KC>
__global__ void __launch_bounds__(kRouteThreads) layout_write_kernel(LayoutArgs a)
{
    allow_dependents();   // the dispatch after this kernel may start loading its input rows
    __shared__ int32_t s_base[EP_MAX_RANKS];
    __shared__ int32_t s_tot[EP_MAX_RANKS], s_before[EP_MAX_RANKS];
    __shared__ int32_t s_warp[kWarps][EP_MAX_RANKS];
    const int P = a.P, K = a.K;
    const int b = blockIdx.x;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x < P) {
        s_tot[threadIdx.x] = 0;
        s_before[threadIdx.x] = 0;
    }
    __syncthreads();
    block_rank_sums(a.part_rank, a.nb, P, b, s_tot, s_before);
    __syncthreads();
    if (warp == 0) {
        const int v0 = lane < P ? s_tot[lane] : 0;
        const int v1 = lane + 32 < P ? s_tot[lane + 32] : 0;
        int e0, e1;   // segment starts: exclusive scan of the aligned counts
        const int grand = warp_exclusive_scan64(round_up(v0, a.align), round_up(v1, a.align), e0, e1);
        if (lane < P)   // first pad row of each segment
            s_tot[lane] = e0 + v0;
        if (lane + 32 < P)
            s_tot[lane + 32] = e1 + v1;
        if (lane < P)
            s_base[lane] = e0 + s_before[lane];
        if (lane + 32 < P)
            s_base[lane + 32] = e1 + s_before[lane + 32];
        if (b == 0) {
            if (a.send_counts != nullptr) {
                if (lane < P)
                    a.send_counts[lane] = v0;
                if (lane + 32 < P)
                    a.send_counts[lane + 32] = v1;
            }
            if (a.rank_offsets != nullptr) {
                if (lane < P)
                    a.rank_offsets[lane] = e0;
                if (lane + 32 < P)
                    a.rank_offsets[lane + 32] = e1;
                if (lane == 0)
                    a.rank_offsets[P] = grand;
            }
            if (lane == 0) {
                if (a.exact && (int64_t)grand != a.num_rows)
                    raise(a.err, EP_ERR_COUNT_MISMATCH);
                if (!a.exact && (int64_t)grand > a.num_rows)
                    raise(a.err, EP_ERR_CAPACITY);
            }
        }
    }
    if (a.tokens_per_expert != nullptr) {
        // experts b, b + nb, ...: every thread adds one block partial at a time
        const int E = P * a.E_local;
        const int mine = (E - b + a.nb - 1) / a.nb;
        int32_t *s_tpe = &s_warp[0][0];   // reused before the ballots below
        constexpr int kRound = kWarps * EP_MAX_RANKS;
        for (int j0 = 0; j0 < mine; j0 += kRound) {
            const int m = min(kRound, mine - j0);
            for (int j = threadIdx.x; j < m; j += blockDim.x)
                s_tpe[j] = 0;
            __syncthreads();
            for (int i = threadIdx.x; i < m * a.nb; i += blockDim.x) {
                const int j = i / a.nb, bb = i % a.nb;
                atomicAdd(&s_tpe[j], a.part_expert[(int64_t)bb * E + b + (j0 + j) * a.nb]);
            }
            __syncthreads();
            for (int j = threadIdx.x; j < m; j += blockDim.x)
                a.tokens_per_expert[b + (j0 + j) * a.nb] = round_up(s_tpe[j], a.align);
            __syncthreads();
        }
    }
    __syncthreads();
    if (a.align > 1)
        fill_pad_rows(s_tot, P, K, a.align, a.num_rows, a.send_token_idx, a.send_rank, a.send_idx, a.send_w);

    const int64_t t0 = (int64_t)b * kRouteThreads + warp * 32;   // first token of this warp
    const int64_t t = t0 + lane;
    const bool valid = t < a.T;
    const uint64_t mask = valid ? rank_mask(a.is_in_rank, t, P) : 0;
    for (int p = 0; p < P; ++p) {
        const unsigned bal = __ballot_sync(kFull, (mask >> p) & 1ull);
        if (lane == 0)
            s_warp[warp][p] = __popc(bal);
    }
    __syncthreads();
    if (threadIdx.x < P) {
        int run = 0;
        for (int ww = 0; ww < kWarps; ++ww) {
            const int v = s_warp[ww][threadIdx.x];
            s_warp[ww][threadIdx.x] = run;
            run += v;
        }
    }
    __syncthreads();

    int bad = 0;
    if constexpr (KC > 0) {
        int64_t id[KC];
        float wt[KC];
        int8_t dr[KC];
        uint64_t dmask = 0;
#pragma unroll
        for (int k = 0; k < KC; ++k) {
            id[k] = -1;
            wt[k] = 0.0f;
            int d = -1;
            if (valid) {
                id[k] = a.idx[t * KC + k];
                wt[k] = a.w[t * KC + k];
                d = a.dest[t * KC + k];
            }
            dr[k] = (int8_t)(d >= 0 && d < P ? d : -1);
            if (dr[k] >= 0)
                dmask |= 1ull << d;
        }
        if (valid && dmask != mask)
            bad = EP_ERR_COUNT_MISMATCH;
        int32_t tpv[EP_MAX_RANKS];   // the token's token_pos row, written out at the end
        for (int p = 0; p < P; ++p) {
            const unsigned bal = __ballot_sync(kFull, (mask >> p) & 1ull);
            tpv[p] = -1;
            if (!valid)
                continue;
            if ((mask >> p) & 1ull) {
                const int64_t pos = (int64_t)s_base[p] + s_warp[warp][p] + __popc(bal & lanemask_lt());
                if (pos < a.num_rows) {
                    tpv[p] = (int32_t)pos;
                    a.send_token_idx[pos] = (int32_t)t;
                    a.send_rank[pos] = p;
                    write_send_row<KC>(a.send_idx + pos * KC, a.send_w + pos * KC, id, wt, dr, p,
                                       (int64_t)p * a.E_local, a.vec);
                } else {
                    bad = a.exact ? EP_ERR_COUNT_MISMATCH : EP_ERR_CAPACITY;
                }
            }
        }
        if (valid) {
            int32_t *tp = a.token_pos + t * P;
            if ((P & 3) == 0 && a.vec.token_pos) {
                for (int p = 0; p < P; p += 4)
                    *reinterpret_cast<int4 *>(tp + p) = make_int4(tpv[p], tpv[p + 1], tpv[p + 2], tpv[p + 3]);
            } else {
                for (int p = 0; p < P; ++p)
                    tp[p] = tpv[p];
            }
        }
        raise(a.err, bad);
        return;
    }
    if (valid) {
        uint64_t dmask = 0;
        for (int k = 0; k < K; ++k) {
            const int d = a.dest[t * K + k];
            if (d >= 0 && d < P)
                dmask |= 1ull << d;
        }
        if (dmask != mask)
            bad = EP_ERR_COUNT_MISMATCH;
    }
    for (int p = 0; p < P; ++p) {
        const unsigned bal = __ballot_sync(kFull, (mask >> p) & 1ull);
        if (bal == 0) {
            if (valid)
                a.token_pos[t * P + p] = -1;
            continue;
        }
        const int64_t n0 = (int64_t)s_base[p] + s_warp[warp][p];   // this warp's first row for rank p
        if (valid) {
            int32_t n = -1;
            if ((mask >> p) & 1ull) {
                const int64_t pos = n0 + __popc(bal & lanemask_lt());
                if (pos < a.num_rows) {
                    n = (int32_t)pos;
                    a.send_token_idx[n] = (int32_t)t;
                    a.send_rank[n] = p;
                } else {
                    bad = a.exact ? EP_ERR_COUNT_MISMATCH : EP_ERR_CAPACITY;
                }
            }
            a.token_pos[t * P + p] = n;
        }
        // K-wide rows n0 .. n0 + cnt - 1, written by the warp together
        const int cnt = __popc(bal);
        for (int e = lane; e < cnt * K; e += 32) {
            const int r = e / K, k = e - r * K;
            const int64_t n = n0 + r;
            if (n >= a.num_rows)
                break;
            const int src = nth_set_bit(bal, r);
            const int64_t ts = t0 + src;
            const bool own = a.dest[ts * K + k] == p;
            a.send_idx[n * K + k] = own ? a.idx[ts * K + k] - (int64_t)p * a.E_local : -1;
            a.send_w[n * K + k] = own ? a.w[ts * K + k] : 0.0f;
        }
    }
    raise(a.err, bad);
}

static void launch_layout_write(const LayoutArgs &a, int nb, cudaStream_t stream)
{
    switch (a.K) {
    case 2: layout_write_kernel<2><<<nb, kRouteThreads, 0, stream>>>(a); break;
    case 4: layout_write_kernel<4><<<nb, kRouteThreads, 0, stream>>>(a); break;
    case 6: layout_write_kernel<6><<<nb, kRouteThreads, 0, stream>>>(a); break;
    case 8: layout_write_kernel<8><<<nb, kRouteThreads, 0, stream>>>(a); break;
    default: layout_write_kernel<0><<<nb, kRouteThreads, 0, stream>>>(a); break;
    }
}

// ---------------------------------------------------- expert-batched slots --
constexpr bool kBatchedPrefetch = true;
// Local experts are handled 64 at a time (one ballot per expert of the group).
constexpr int kGroup = 64;

__device__ __forceinline__ uint64_t local_mask(const int64_t *__restrict__ row, int K, int64_t e_lo,
                                               int n_in_group)
{
    uint64_t m = 0;
    for (int k = 0; k < K; ++k) {
        const int64_t el = row[k] - e_lo;
        if (el >= 0 && el < n_in_group)
            m |= 1ull << el;
    }
    return m;
}

__global__ void __launch_bounds__(kRouteThreads)
batched_count_kernel(const int64_t *__restrict__ idx, int64_t T, int K, int E, int E_local,
                     int64_t e0, int32_t *__restrict__ part, int32_t *err)
{
    __shared__ int32_t warp_cnt[kWarps][kGroup];
    const int64_t t = (int64_t)blockIdx.x * kRouteThreads + threadIdx.x;
    const bool valid = t < T;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    int bad = 0;
    if (valid)
        for (int k = 0; k < K; ++k) {
            const int64_t id = idx[t * K + k];
            if (id < -1 || id >= E)
                bad = EP_ERR_INVALID_EXPERT;
        }
    for (int g0 = 0; g0 < E_local; g0 += kGroup) {
        const int ng = min(kGroup, E_local - g0);
        const uint64_t mask = valid ? local_mask(idx + t * K, K, e0 + g0, ng) : 0;
        for (int e = 0; e < ng; ++e) {
            const unsigned bal = __ballot_sync(kFull, (mask >> e) & 1ull);
            if (lane == 0)
                warp_cnt[warp][e] = __popc(bal);
        }
        __syncthreads();
        for (int e = threadIdx.x; e < ng; e += blockDim.x) {
            int s = 0;
            for (int ww = 0; ww < kWarps; ++ww)
                s += warp_cnt[ww][e];
            part[(int64_t)blockIdx.x * E_local + g0 + e] = s;
        }
        __syncthreads();
    }
    raise(err, bad);
}

__global__ void __launch_bounds__(kRouteThreads)
batched_slot_kernel(const int64_t *__restrict__ idx, int64_t T, int K, int E_local, int64_t e0, SlotLimits lim,
                    const int32_t *__restrict__ part, int nb, int32_t *__restrict__ tokens_per_expert,
                    int32_t *__restrict__ slot, int32_t *err)
{
    allow_dependents();   // the row scatter after this kernel may start loading its input rows
    __shared__ int32_t s_base[kGroup], s_tot[kGroup];
    __shared__ int32_t s_warp[kWarps][kGroup];
    const int64_t t = (int64_t)blockIdx.x * kRouteThreads + threadIdx.x;
    const bool valid = t < T;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    int bad = 0;
    if (valid)
        for (int k = 0; k < K; ++k)
            slot[t * K + k] = -1;

    for (int g0 = 0; g0 < E_local; g0 += kGroup) {
        const int ng = min(kGroup, E_local - g0);
        if (threadIdx.x < ng) {
            s_base[threadIdx.x] = 0;
            s_tot[threadIdx.x] = 0;
        }
        __syncthreads();
        for (int i = threadIdx.x; i < nb * ng; i += blockDim.x) {
            const int bb = i / ng, e = i % ng;
            const int v = part[(int64_t)bb * E_local + g0 + e];
            atomicAdd(&s_tot[e], v);
            if (bb < (int)blockIdx.x)
                atomicAdd(&s_base[e], v);
        }
        __syncthreads();
        if (blockIdx.x == 0 && threadIdx.x < ng)
            bad |= finish_expert_count(lim, g0 + threadIdx.x, s_tot[threadIdx.x], tokens_per_expert);
        const uint64_t mask = valid ? local_mask(idx + t * K, K, e0 + g0, ng) : 0;
        for (int e = 0; e < ng; ++e) {
            const unsigned bal = __ballot_sync(kFull, (mask >> e) & 1ull);
            if (lane == 0)
                s_warp[warp][e] = __popc(bal);
        }
        __syncthreads();
        if (threadIdx.x < ng) {
            int run = 0;
            for (int ww = 0; ww < kWarps; ++ww) {
                const int v = s_warp[ww][threadIdx.x];
                s_warp[ww][threadIdx.x] = run;
                run += v;
            }
        }
        __syncthreads();
        for (int e = 0; e < ng; ++e) {
            const unsigned bal = __ballot_sync(kFull, (mask >> e) & 1ull);
            if (!valid || !((mask >> e) & 1ull))
                continue;
            const int s = s_base[e] + s_warp[warp][e] + __popc(bal & lanemask_lt());
            const int32_t v = s < lim.cap ? s : -1;
            if (s >= lim.cap && !lim.silent)
                bad = EP_ERR_CAPACITY;
            for (int k = 0; k < K; ++k)
                if (idx[t * K + k] == e0 + g0 + e)
                    slot[t * K + k] = v;
        }
        __syncthreads();
    }
    raise(err, bad);
}

// ------------------------------------------------------- fused route kernel --
// Counts and send layout in one cooperative launch (all blocks resident at
// once).  Each thread owns one token and keeps its K expert ids, weights and
// owning ranks in registers from the counting phase to the layout phase;
// between the two, every block publishes its per-rank partial counts and an
// arrival flag, and waits (bounded) until every block's flag carries this
// launch's tag.
constexpr int kFusedThreads = 128;
constexpr int kFusedWarps = kFusedThreads / 32;
struct FusedArgs {
    const int64_t *idx;
    const float *w;
    int64_t T;
    int K, P, E_local;
    int64_t num_rows;
    int32_t *dest;
    uint8_t *is_in_rank;
    int32_t *send_counts, *rank_offsets, *tokens_per_expert;
    int32_t *send_token_idx, *send_rank;
    int64_t *send_idx;
    float *send_w;
    int32_t *token_pos;
    int32_t *part_rank;       // [gridDim][P]
    int32_t *part_expert;     // [gridDim][E] when tokens_per_expert is wanted
    GridBarrier bar;
    int align;                // rank segments start at multiples of it; tokens_per_expert rounded up
    int32_t *err;
    VecOk vec;                // which outputs take vector stores
};

// KC > 0: K == KC at compile time (vector row stores); KC == 0: any K <= 32.
template <int KC>
__global__ void __launch_bounds__(kFusedThreads) route_fused_kernel(FusedArgs a)
{
    allow_dependents();   // the dispatch after this kernel may start loading its input rows
    constexpr int KM = KC > 0 ? KC : EP_MAX_TOPK;
    extern __shared__ int32_t s_hist[];          // [E] when counting experts
    __shared__ int32_t s_warp[kFusedWarps][EP_MAX_RANKS];
    __shared__ int32_t s_tot[EP_MAX_RANKS], s_before[EP_MAX_RANKS], s_base[EP_MAX_RANKS];
    __shared__ int s_fail;
    __shared__ unsigned long long s_tag, s_epoch;
    const int K = KC > 0 ? KC : a.K;
    const int P = a.P, El = a.E_local, E = P * El;
    const int b = blockIdx.x, nb = gridDim.x;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t t = (int64_t)b * kFusedThreads + threadIdx.x;
    const bool valid = t < a.T;
    const bool want_tpe = a.tokens_per_expert != nullptr;

    // ------------------------------------------------------- counting phase
    if (want_tpe)
        for (int e = threadIdx.x; e < E; e += blockDim.x)
            s_hist[e] = 0;
    if (threadIdx.x == 0) {
        s_fail = 0;
        s_tag = barrier_tag(a.bar, &s_epoch);
    }
    int64_t id[KM];
    float wt[KM];
    int8_t dr[KM];
    uint64_t mask = 0;
    int bad = 0;
#pragma unroll
    for (int k = 0; k < KM; ++k) {
        id[k] = -1;
        wt[k] = 0.0f;
        dr[k] = -1;
        if (valid && k < K) {
            id[k] = a.idx[t * K + k];
            wt[k] = a.w[t * K + k];
        }
    }
    __syncthreads();   // s_hist zeroed
    if (valid) {
#pragma unroll
        for (int k = 0; k < KM; ++k) {
            if (k >= K)
                break;
            const int64_t e = id[k];
            int d = -1;
            if (e >= 0 && e < E)
                d = (int)(e / El);
            else if (e != -1)
                bad = EP_ERR_INVALID_EXPERT;
            dr[k] = (int8_t)d;
            if (d >= 0) {
                mask |= 1ull << d;
                if (want_tpe) {
                    bool seen = false;
#pragma unroll
                    for (int j = 0; j < KM; ++j)
                        seen |= (j < k && id[j] == e);
                    if (!seen)
                        atomicAdd(&s_hist[e], 1);
                }
            }
        }
    }
    for (int p = 0; p < P; ++p) {
        const unsigned bal = __ballot_sync(kFull, (mask >> p) & 1ull);
        if (lane == 0)
            s_warp[warp][p] = __popc(bal);
    }
    __syncthreads();
    if (threadIdx.x < P) {
        int run = 0;
        for (int ww = 0; ww < kFusedWarps; ++ww) {
            const int v = s_warp[ww][threadIdx.x];
            s_warp[ww][threadIdx.x] = run;          // exclusive prefix over this block's warps
            run += v;
        }
        a.part_rank[(int64_t)b * P + threadIdx.x] = run;
    }
    if (want_tpe)
        for (int e = threadIdx.x; e < E; e += blockDim.x)
            a.part_expert[(int64_t)b * E + e] = s_hist[e];
    __syncthreads();
    if (threadIdx.x == 0)
        barrier_arrive(a.bar, s_tag);
    // dest and is_in_rank are not read by other blocks: store them while the
    // other blocks arrive
    if (valid) {
#pragma unroll
        for (int k = 0; k < KM; ++k)
            if (k < K)
                a.dest[t * K + k] = dr[k];
        uint8_t *irow = a.is_in_rank + t * P;
        if ((P & 3) == 0 && a.vec.is_in_rank) {
            for (int p = 0; p < P; p += 4)
                *reinterpret_cast<uint32_t *>(irow + p) =
                    (uint32_t)((mask >> p) & 1ull) | (uint32_t)((mask >> (p + 1)) & 1ull) << 8 |
                    (uint32_t)((mask >> (p + 2)) & 1ull) << 16 | (uint32_t)((mask >> (p + 3)) & 1ull) << 24;
        } else {
            for (int p = 0; p < P; ++p)
                irow[p] = (uint8_t)((mask >> p) & 1ull);
        }
    }

    // -------------------------------------------------------- grid barrier
    if (!barrier_wait(a.bar, s_tag, s_epoch, &s_fail)) {
        if (threadIdx.x == 0)
            raise(a.err, EP_ERR_TIMEOUT);
        return;   // the whole block leaves together
    }

    // --------------------------------------------------------- layout phase
    if (threadIdx.x < P) {
        s_tot[threadIdx.x] = 0;
        s_before[threadIdx.x] = 0;
    }
    __syncthreads();
    block_rank_sums(a.part_rank, nb, P, b, s_tot, s_before);
    __syncthreads();
    if (warp == 0) {
        const int v0 = lane < P ? s_tot[lane] : 0;
        const int v1 = lane + 32 < P ? s_tot[lane + 32] : 0;
        int e0, e1;   // segment starts: exclusive scan of the aligned counts
        const int grand = warp_exclusive_scan64(round_up(v0, a.align), round_up(v1, a.align), e0, e1);
        if (lane < P)
            s_base[lane] = e0 + s_before[lane];
        if (lane + 32 < P)
            s_base[lane + 32] = e1 + s_before[lane + 32];
        if (lane < P)
            s_tot[lane] = e0 + v0;              // first pad row of the segment
        if (lane + 32 < P)
            s_tot[lane + 32] = e1 + v1;
        if (b == 0) {
            if (lane < P) {
                a.send_counts[lane] = v0;
                a.rank_offsets[lane] = e0;
            }
            if (lane + 32 < P) {
                a.send_counts[lane + 32] = v1;
                a.rank_offsets[lane + 32] = e1;
            }
            if (lane == 0) {
                a.rank_offsets[P] = grand;
                if ((int64_t)grand > a.num_rows)
                    raise(a.err, EP_ERR_CAPACITY);
            }
        }
    }
    if (want_tpe) {
        // experts b, b + nb, ...: one partial per thread and step
        const int mine = (E - b + nb - 1) / nb;
        for (int j0 = 0; j0 < mine; j0 += E) {
            for (int j = threadIdx.x; j < mine; j += blockDim.x)
                s_hist[j] = 0;
            __syncthreads();
            for (int i = threadIdx.x; i < mine * nb; i += blockDim.x) {
                const int j = i / nb, bb = i - j * nb;
                atomicAdd(&s_hist[j], a.part_expert[(int64_t)bb * E + b + j * nb]);
            }
            __syncthreads();
            for (int j = threadIdx.x; j < mine; j += blockDim.x)
                a.tokens_per_expert[b + j * nb] = round_up(s_hist[j], a.align);
        }
    }
    __syncthreads();
    if (a.align > 1)
        fill_pad_rows(s_tot, P, K, a.align, a.num_rows, a.send_token_idx, a.send_rank, a.send_idx, a.send_w);

    // the token's token_pos row is gathered here and written out at the end
    // with vector stores (one scattered 4-byte store per rank cost the layout
    // phase most of its store transactions)
    int32_t tpv[EP_MAX_RANKS];
    for (int p = 0; p < P; ++p)
        tpv[p] = -1;
    for (int p = 0; p < P; ++p) {
        const unsigned bal = __ballot_sync(kFull, (mask >> p) & 1ull);
        if (!((mask >> p) & 1ull))
            continue;
        const int64_t n = (int64_t)s_base[p] + s_warp[warp][p] + __popc(bal & lanemask_lt());
        if (n >= a.num_rows) {
            bad = EP_ERR_CAPACITY;
            continue;
        }
        tpv[p] = (int32_t)n;
        a.send_token_idx[n] = (int32_t)t;
        a.send_rank[n] = p;
        const int64_t off = (int64_t)p * El;
        int64_t *si = a.send_idx + n * K;
        float *sw = a.send_w + n * K;
        if constexpr (KC > 0) {
            write_send_row<KC>(si, sw, id, wt, dr, p, off, a.vec);
        } else {
#pragma unroll
            for (int k = 0; k < KM; ++k)
                if (k < K) {
                    si[k] = dr[k] == p ? id[k] - off : -1;
                    sw[k] = dr[k] == p ? wt[k] : 0.0f;
                }
        }
    }
    if (valid) {
        int32_t *tp = a.token_pos + t * P;
        if ((P & 3) == 0 && a.vec.token_pos) {
            for (int p = 0; p < P; p += 4)
                *reinterpret_cast<int4 *>(tp + p) = make_int4(tpv[p], tpv[p + 1], tpv[p + 2], tpv[p + 3]);
        } else {
            for (int p = 0; p < P; ++p)
                tp[p] = tpv[p];
        }
    }
    raise(a.err, bad);
}

template <int KC>
static int launch_route_fused(const FusedArgs &a, int nb, size_t smem, cudaStream_t stream, bool *launched)
{
    *launched = false;
    // blocks per SM, [counting experts?]; with dynamic shared memory the
    // count depends on smem, which a call with expert counts passes as E ints
    static PerDevice max_per_sm[2];
    const int slot = smem > 0 ? 1 : 0;
    const int dev = current_device();
    int per_sm = max_per_sm[slot].get(dev);
    if (per_sm < 0 || slot == 1) {
        int n = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, route_fused_kernel<KC>, kFusedThreads, smem) != cudaSuccess) {
            cudaGetLastError();
            n = 0;
        }
        per_sm = n;
        max_per_sm[slot].put(dev, n);
    }
    if ((int64_t)per_sm * device_sm_count() < nb)
        return EP_OK;   // cannot be co-resident: the caller falls back to two launches
    FusedArgs copy = a;
    void *args[] = {&copy};
    if (cudaLaunchCooperativeKernel((const void *)route_fused_kernel<KC>, dim3(nb), dim3(kFusedThreads), args, smem,
                                    stream) != cudaSuccess) {
        cudaGetLastError();
        return EP_ERR_CUDA;
    }
    *launched = true;
    return EP_OK;
}

static unsigned long long next_route_tag()
{
    static std::atomic<unsigned long long> epoch{0x9e3779b97f4a7c15ull};
    unsigned long long v;
    do {
        v = epoch.fetch_add(0x632be59bd9b4e019ull);
    } while (v == 0);
    return v;
}

// ------------------------------------------------ fused expert-batched slots --
// The slots of the expert-batched layout in one cooperative launch, like the
// fused route: each thread keeps its token's K expert ids in registers, warp
// ballots per local expert give block counts, every block publishes them with
// a tagged arrival flag, and after the bounded grid barrier each thread takes
// its slot from the block bases and its ballot prefix.  Needs E_local <= 64.
struct BatchedFusedArgs {
    const int64_t *idx;
    int64_t T;
    int K, E, E_local;
    int64_t e0;
    SlotLimits lim;
    int32_t *tokens_per_expert;
    int32_t *slot;
    int32_t *part;                    // [gridDim][E_local]
    GridBarrier bar;
    int32_t *err;
    RowPrefetch pf;                   // rows for the scatter after this kernel
};

template <int KC>
__global__ void __launch_bounds__(kFusedThreads) batched_fused_kernel(BatchedFusedArgs a)
{
    allow_dependents();   // the row scatter after this kernel may start loading its input rows
    constexpr int KM = KC > 0 ? KC : EP_MAX_TOPK;
    __shared__ int32_t s_warp[kFusedWarps][64];
    __shared__ int32_t s_tot[64], s_before[64];
    __shared__ int s_fail;
    __shared__ unsigned long long s_tag, s_epoch;
    const int K = KC > 0 ? KC : a.K;
    const int El = a.E_local;
    const int b = blockIdx.x, nb = gridDim.x;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t t = (int64_t)b * kFusedThreads + threadIdx.x;
    const bool valid = t < a.T;
    if (threadIdx.x == 0) {
        s_fail = 0;
        s_tag = barrier_tag(a.bar, &s_epoch);
    }

    int64_t id[KM];
    uint64_t mask = 0;
    int bad = 0;
#pragma unroll
    for (int k = 0; k < KM; ++k) {
        id[k] = -1;
        if (valid && k < K)
            id[k] = a.idx[t * K + k];
    }
#pragma unroll
    for (int k = 0; k < KM; ++k) {
        if (!valid || k >= K)
            continue;
        if (id[k] < -1 || id[k] >= a.E)
            bad = EP_ERR_INVALID_EXPERT;
        const int64_t el = id[k] - a.e0;
        if (el >= 0 && el < El)
            mask |= 1ull << el;
    }
    // The ballot of expert e is the warp's bit column for e: lane e & 31 keeps
    // it (word e < 32 in bal_lo, else bal_hi) for the slot phase.
    unsigned bal_lo = 0, bal_hi = 0;
    for (int e = 0; e < El; ++e) {
        const unsigned bal = __ballot_sync(kFull, (mask >> e) & 1ull);
        if (lane == (e & 31)) {
            if (e < 32)
                bal_lo = bal;
            else
                bal_hi = bal;
        }
    }
    if (lane < El)
        s_warp[warp][lane] = __popc(bal_lo);
    if (lane + 32 < El)
        s_warp[warp][lane + 32] = __popc(bal_hi);
    __syncthreads();
    if (threadIdx.x < El) {
        int run = 0;
        for (int ww = 0; ww < kFusedWarps; ++ww) {
            const int v = s_warp[ww][threadIdx.x];
            s_warp[ww][threadIdx.x] = run;
            run += v;
        }
        a.part[(int64_t)b * El + threadIdx.x] = run;
    }
    __syncthreads();
    if (threadIdx.x == 0)
        barrier_arrive(a.bar, s_tag);
    // HBM is otherwise idle while the blocks wait for one another: the rows
    // the scatter after this kernel reads (tokens with a local slot) are
    // fetched into the L2 now
    if (kBatchedPrefetch && a.pf.x != nullptr && mask != 0 && t < a.pf.tokens)
        prefetch_l2_bulk(static_cast<const uint8_t *>(a.pf.x) + t * a.pf.row_bytes, (uint32_t)a.pf.row_bytes);
    if (!barrier_wait(a.bar, s_tag, s_epoch, &s_fail)) {
        if (threadIdx.x == 0)
            raise(a.err, EP_ERR_TIMEOUT);
        return;
    }
    if (threadIdx.x < El) {
        s_tot[threadIdx.x] = 0;
        s_before[threadIdx.x] = 0;
    }
    __syncthreads();
    block_rank_sums(a.part, nb, El, b, s_tot, s_before);
    __syncthreads();
    if (b == 0 && threadIdx.x < El)
        bad |= finish_expert_count(a.lim, threadIdx.x, s_tot[threadIdx.x], a.tokens_per_expert);
    // slot of this token for expert e: the expert's block base, this warp's
    // base within the block, and the token's rank among the warp's lanes
    // naming e (lanes below it in e's ballot word); words and bases are held
    // by lane e & 31 and fetched by shuffle, so every lane takes the same path
    const int base_lo = lane < El ? s_before[lane] + s_warp[warp][lane] : 0;
    const int base_hi = lane + 32 < El ? s_before[lane + 32] + s_warp[warp][lane + 32] : 0;
    int32_t sl[KM];
#pragma unroll
    for (int k = 0; k < KM; ++k) {
        sl[k] = -1;
        if (k >= K)
            continue;
        const int64_t el = id[k] - a.e0;
        const bool local = el >= 0 && el < El;
        const int src = local ? (int)(el & 31) : 0;
        const unsigned w_lo = __shfl_sync(kFull, bal_lo, src), w_hi = __shfl_sync(kFull, bal_hi, src);
        const int b_lo = __shfl_sync(kFull, base_lo, src), b_hi = __shfl_sync(kFull, base_hi, src);
        if (!valid || !local)
            continue;
        const int s = (el < 32 ? b_lo : b_hi) + __popc((el < 32 ? w_lo : w_hi) & lanemask_lt());
        sl[k] = s < a.lim.cap ? s : -1;
        if (s >= a.lim.cap && !a.lim.silent)
            bad = EP_ERR_CAPACITY;
    }
    if (valid) {
#pragma unroll
        for (int k = 0; k < KM; ++k)
            if (k < K)
                a.slot[t * K + k] = sl[k];
    }
    raise(a.err, bad);
}

template <int KC>
static int launch_batched_fused(const BatchedFusedArgs &a, int nb, cudaStream_t stream, bool *launched)
{
    *launched = false;
    static PerDevice max_per_sm;
    const int dev = current_device();
    int per_sm = max_per_sm.get(dev);
    if (per_sm < 0) {
        int n = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, batched_fused_kernel<KC>, kFusedThreads, 0) != cudaSuccess) {
            cudaGetLastError();
            n = 0;
        }
        per_sm = n;
        max_per_sm.put(dev, n);
    }
    const int sms = device_sm_count();
    if ((int64_t)per_sm * sms < nb)
        return EP_OK;
    BatchedFusedArgs copy = a;
    void *args[] = {&copy};
    if (cudaLaunchCooperativeKernel((const void *)batched_fused_kernel<KC>, dim3(nb), dim3(kFusedThreads), args, 0,
                                    stream) != cudaSuccess) {
        cudaGetLastError();
        return EP_ERR_CUDA;
    }
    *launched = true;
    return EP_OK;
}

// ------------------------------------------- expert-batched slots, one cluster --
// The slots of the expert-batched layout for up to kClMaxCtas * kClTokens
// tokens, computed by ONE thread-block cluster.  CTA c of the cluster owns the
// contiguous tokens [c * per_cta, (c + 1) * per_cta) (per_cta <= kClTokens, a
// multiple of 32), so its ids and slots are the contiguous ranges
// [c * per_cta * K, ...) of topk_idx and slot:
//   1. ids are read in position order (consecutive threads, consecutive ids:
//      coalesced) into a byte table of local experts in shared memory, and
//      each token's local-expert mask is OR-ed together (by shuffles over its
//      K lanes when K divides 32, else from its table row);
//   2. one lane per token (rounds of kClThreads tokens, in token order): the
//      warp's 32 x 32 bit matrix of masks is transposed by shuffles, so lane e
//      holds expert e's ballot word (bit l: the warp's token l names e); its
//      population count is the (round, warp) count;
//   3. a warp scan turns the counts into bases within the CTA; each CTA writes
//      its totals into every CTA's shared memory (distributed shared memory,
//      after a barrier phase begun at the kernel's start shows that every CTA
//      has started) and one hardware cluster barrier makes them visible: no
//      flag in global memory is polled and no CTA touches another's memory
//      after the barrier;
//   4. slots are written in position order again (coalesced): slot of
//      position p (token p / K) for expert e = hits of the CTAs before + the
//      (round, warp) base + the lanes below the token's in e's ballot word.
// The launch is an ordinary one, so the row scatter after it waits only for
// this short chain.  Needs E_local <= 64.
constexpr int kClThreads = 1024;
constexpr int kClWarps = kClThreads / 32;
constexpr int kClRounds = 2;
constexpr int kClTokens = kClRounds * kClThreads;   // tokens per CTA at most
constexpr int kClMaxCtas = 16;

struct BatchedClusterArgs {
    const int64_t *idx;
    int64_t T;
    int K, E, E_local;
    int64_t e0;
    int per_cta;   // tokens owned by each CTA (the last CTAs may own fewer, or none)
    SlotLimits lim;
    int32_t *tokens_per_expert;
    int32_t *slot;
    int32_t *err;
};

// The 32-bit value v into the shared-memory address of *p in CTA `rank` of
// this cluster.
__device__ __forceinline__ void st_dsmem_s32(int32_t *p, uint32_t rank, int32_t v)
{
    uint32_t remote;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(smem_u32(p)), "r"(rank));
    asm volatile("st.shared::cluster.s32 [%0], %1;" ::"r"(remote), "r"(v) : "memory");
}

template <int KC>
__global__ void __launch_bounds__(kClThreads, 1) batched_cluster_kernel(BatchedClusterArgs a)
{
    allow_dependents();   // the row scatter after this kernel may start loading its input rows
    cluster_arrive_relaxed();   // waited for before the first write into another CTA's memory
    // dynamic: [per_cta] local-expert mask of each token, then [per_cta * K]
    // local expert of each slot (-1 if none)
    extern __shared__ __align__(16) uint64_t s_dyn[];
    uint64_t *s_mask = s_dyn;
    int8_t *s_el = reinterpret_cast<int8_t *>(s_dyn + a.per_cta);
    // [round][warp][expert] counts, then exclusive bases within the CTA; the
    // odd row length keeps the scan's column reads free of bank conflicts
    __shared__ int32_t s_cnt[kClRounds][kClWarps][65];
    __shared__ uint32_t s_bal[kClRounds][kClWarps][64];   // ballot word per (round, warp, expert)
    __shared__ int32_t s_tot[kClMaxCtas][64];             // per-expert totals of every CTA
    const int K = KC > 0 ? KC : a.K;
    const int El = a.E_local;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t c = cluster_ctarank(), nc = cluster_nctarank();
    const int64_t t0 = (int64_t)c * a.per_cta;
    const int64_t left = a.T - t0;
    const int nloc = left <= 0 ? 0 : (int)(left < a.per_cta ? left : (int64_t)a.per_cta);
    const int npos = nloc * K;
    const int64_t *ids = a.idx + t0 * K;
    constexpr bool kSeg = KC > 0 && 32 % (KC > 0 ? KC : 1) == 0;   // a token's K positions share one warp
    int bad = 0;

    // 1. ids in position order, four loads in flight per thread
    for (int base = 0; base < npos; base += 4 * kClThreads) {   // uniform over the CTA
        int64_t v[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int p = base + u * kClThreads + threadIdx.x;
            v[u] = p < npos ? ids[p] : -1;
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int p = base + u * kClThreads + threadIdx.x;
            int el = -1;
            if (p < npos) {
                if (v[u] < -1 || v[u] >= a.E)
                    bad = EP_ERR_INVALID_EXPERT;
                const int64_t d = v[u] - a.e0;
                el = d >= 0 && d < El ? (int)d : -1;
                s_el[p] = (int8_t)el;
            }
            if constexpr (kSeg) {
                // OR over the token's KC lanes (p = base + ... + lane, base a
                // multiple of 32): the lowest of them stores the mask
                uint64_t m = el >= 0 ? 1ull << el : 0;
#pragma unroll
                for (int o = 1; o < KC; o <<= 1)
                    m |= __shfl_xor_sync(kFull, m, o);
                if (p < npos && lane % KC == 0)
                    s_mask[p / KC] = m;
            }
        }
    }
    __syncthreads();
    // 2. per (round, warp): transposed masks give each expert's ballot word
    const int rounds = (nloc + kClThreads - 1) / kClThreads;
    for (int j = 0; j < rounds; ++j) {   // uniform over the CTA
        const int tl = j * kClThreads + threadIdx.x;
        uint64_t mask = 0;
        if (tl < nloc) {
            if constexpr (kSeg) {
                mask = s_mask[tl];
            } else {
                for (int k = 0; k < K; ++k) {
                    const int el = s_el[tl * K + k];
                    if (el >= 0)
                        mask |= 1ull << el;
                }
            }
        }
        const uint32_t w_lo = warp_transpose32((uint32_t)mask, lane);
        s_bal[j][warp][lane] = w_lo;
        s_cnt[j][warp][lane] = __popc(w_lo);
        if (El > 32) {   // uniform
            const uint32_t w_hi = warp_transpose32((uint32_t)(mask >> 32), lane);
            s_bal[j][warp][lane + 32] = w_hi;
            s_cnt[j][warp][lane + 32] = __popc(w_hi);
        }
    }
    __syncthreads();
    // 3. exclusive scan over (round, warp) of each expert's counts: warp w
    // scans experts w and w + 32, one lane per warp of the counted round; the
    // CTA's total goes to every CTA of the cluster, all of which have started
    // once the wait returns
    cluster_wait();
    for (int e = warp; e < El; e += kClWarps) {
        int run = 0;
        for (int j = 0; j < rounds; ++j) {
            const int v = s_cnt[j][lane][e];
            int incl = v;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int n = __shfl_up_sync(kFull, incl, o);
                if (lane >= o)
                    incl += n;
            }
            s_cnt[j][lane][e] = run + incl - v;
            run += __shfl_sync(kFull, incl, 31);
        }
        if (lane < (int)nc)
            st_dsmem_s32(&s_tot[c][e], (uint32_t)lane, run);
    }
    // every CTA's totals are in every CTA's s_tot, and the bases are visible
    // to the whole CTA; after this barrier no CTA touches another's memory
    cluster_sync();
    __shared__ int32_t s_pre[64];   // hits of the CTAs before this one
    if (threadIdx.x < El) {
        const int e = threadIdx.x;
        int pre = 0, tot = 0;
        for (int cc = 0; cc < (int)nc; ++cc) {
            const int v = s_tot[cc][e];
            pre += cc < (int)c ? v : 0;
            tot += v;
        }
        s_pre[e] = pre;
        if (c == 0)
            bad |= finish_expert_count(a.lim, e, tot, a.tokens_per_expert);
    }
    __syncthreads();
    // 4. slots in position order
    int32_t *out = a.slot + t0 * K;
    for (int p = threadIdx.x; p < npos; p += kClThreads) {
        const int el = s_el[p];
        int32_t sl = -1;
        if (el >= 0) {
            const int tl = p / K;
            const int j = tl / kClThreads, w = (tl / 32) % kClWarps, l = tl % 32;
            const int s = s_pre[el] + s_cnt[j][w][el] + __popc(s_bal[j][w][el] & ((1u << l) - 1u));
            sl = s < a.lim.cap ? s : -1;
            if (s >= a.lim.cap && !a.lim.silent)
                bad = EP_ERR_CAPACITY;
        }
        out[p] = sl;
    }
    raise(a.err, bad);
}

// Cluster size for the one-cluster slot kernel: 16 CTAs where the device
// schedules such clusters (a non-portable size), else 8; 0 if neither.
template <int KC>
static int batched_cluster_size()
{
    static PerDevice size;   // the attributes below are set per device
    const int dev = current_device();
    int n = size.get(dev);
    if (n >= 0)
        return n;
    n = 0;
    if (cudaFuncSetAttribute(batched_cluster_kernel<KC>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) !=
            cudaSuccess ||
        cudaFuncSetAttribute(batched_cluster_kernel<KC>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kClTokens * (8 + EP_MAX_TOPK)) != cudaSuccess)
        cudaGetLastError();
    for (int cs : {16, 8}) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(cs);
        cfg.blockDim = dim3(kClThreads);
        cfg.dynamicSmemBytes = kClTokens * (8 + EP_MAX_TOPK);
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = cs;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        int clusters = 0;
        if (cudaOccupancyMaxActiveClusters(&clusters, batched_cluster_kernel<KC>, &cfg) == cudaSuccess &&
            clusters >= 1) {
            n = cs;
            break;
        }
        cudaGetLastError();
    }
    size.put(dev, n);
    return n;
}

template <int KC>
static int launch_batched_cluster(const BatchedClusterArgs &a0, cudaStream_t stream, bool *launched)
{
    *launched = false;
    const int cs = batched_cluster_size<KC>();
    if (cs == 0 || a0.T > (int64_t)cs * kClTokens)
        return EP_OK;   // the caller takes the grid-wide form
    BatchedClusterArgs a = a0;
    a.per_cta = (int)align_up((size_t)ceil_div(a.T, cs), 32);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(cs);
    cfg.blockDim = dim3(kClThreads);
    cfg.dynamicSmemBytes = (size_t)a.per_cta * (8 + a.K);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = cs;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, batched_cluster_kernel<KC>, a) != cudaSuccess) {
        cudaGetLastError();
        return EP_ERR_CUDA;
    }
    *launched = true;
    return EP_OK;
}

int launch_batched_slots(const int64_t *topk_idx, int64_t T, int K, int E, int E_local, int rank,
                         const SlotLimits &lim, int32_t *tokens_per_expert, int32_t *slot,
                         void *ws, size_t ws_bytes, int32_t *err, cudaStream_t stream, const RowPrefetch &pf)
{
    const int64_t e0 = (int64_t)rank * E_local;
    if (T == 0) {   // every expert receives nothing
        for (int32_t *p : {tokens_per_expert, lim.dropped, lim.kept})
            if (p != nullptr && cudaMemsetAsync(p, 0, sizeof(int32_t) * E_local, stream) != cudaSuccess)
                return EP_ERR_CUDA;
        return EP_OK;
    }
    // one cluster when the local experts fit one mask word and the tokens fit
    // the cluster's rounds
    if (E_local <= 64) {
        BatchedClusterArgs ca{topk_idx, T, K, E, E_local, e0, 0, lim, tokens_per_expert, slot, err};
        bool launched = false;
        int rc;
        switch (K) {
        case 2: rc = launch_batched_cluster<2>(ca, stream, &launched); break;
        case 4: rc = launch_batched_cluster<4>(ca, stream, &launched); break;
        case 6: rc = launch_batched_cluster<6>(ca, stream, &launched); break;
        case 8: rc = launch_batched_cluster<8>(ca, stream, &launched); break;
        default: rc = launch_batched_cluster<0>(ca, stream, &launched); break;
        }
        if (rc != EP_OK || launched)
            return rc;
    }
    // else one cooperative launch when the blocks can be resident together and
    // the workspace holds partials + flags
    // workspace: [header: launch counter][partials][flags]
    char *wsb = static_cast<char *>(ws);
    const int nbf = (int)ceil_div(T, kFusedThreads);
    const size_t part_bytes = align_up((size_t)nbf * E_local * sizeof(int32_t), kWsAlign);
    if (E_local <= 64 && ws_bytes >= kWsAlign + part_bytes + (size_t)nbf * sizeof(unsigned long long)) {
        BatchedFusedArgs fa{topk_idx, T, K, E, E_local, e0, lim, tokens_per_expert, slot,
                            reinterpret_cast<int32_t *>(wsb + kWsAlign),
                            {reinterpret_cast<unsigned long long *>(wsb + kWsAlign + part_bytes),
                             reinterpret_cast<unsigned long long *>(wsb), next_route_tag()},
                            err, pf};
        bool launched = false;
        int rc;
        switch (K) {
        case 2: rc = launch_batched_fused<2>(fa, nbf, stream, &launched); break;
        case 4: rc = launch_batched_fused<4>(fa, nbf, stream, &launched); break;
        case 6: rc = launch_batched_fused<6>(fa, nbf, stream, &launched); break;
        case 8: rc = launch_batched_fused<8>(fa, nbf, stream, &launched); break;
        default: rc = launch_batched_fused<0>(fa, nbf, stream, &launched); break;
        }
        if (rc != EP_OK || launched)
            return rc;
    }
    const int nb = (int)ceil_div(T, kRouteThreads);
    int32_t *part = reinterpret_cast<int32_t *>(wsb + kWsAlign);
    batched_count_kernel<<<nb, kRouteThreads, 0, stream>>>(topk_idx, T, K, E, E_local, e0, part, err);
    if (launch_status() != EP_OK)
        return EP_ERR_CUDA;
    batched_slot_kernel<<<nb, kRouteThreads, 0, stream>>>(topk_idx, T, K, E_local, e0, lim, part, nb,
                                                          tokens_per_expert, slot, err);
    return launch_status();
}
}  // namespace ep

// ================================================================ C ABI ====
using namespace ep;

// Workspace regions shared by the routing calls (sized for routing blocks of
// 128 tokens, twice as many as the 256-token blocks most kernels use): a
// header holding the cooperative kernels' launch counter, per-block rank
// counts, per-block expert counts, per-block arrival flags.
struct WsLayout {
    unsigned long long *epoch;   // header: launch counter of the cooperative kernels
    int32_t *part_rank;
    int32_t *part_expert;
    unsigned long long *flags;
};

static size_t ws_blocks(int64_t T, int chunks) { return 2 * (size_t)route_blocks_max(T, chunks); }

static WsLayout ws_layout(void *ws, int64_t T, int chunks, int P, int E)
{
    const size_t nb = ws_blocks(T, chunks);
    char *base = static_cast<char *>(ws);
    WsLayout l;
    l.epoch = reinterpret_cast<unsigned long long *>(base);
    base += kWsAlign;
    l.part_rank = reinterpret_cast<int32_t *>(base);
    base += align_up(nb * P * sizeof(int32_t), kWsAlign);
    l.part_expert = reinterpret_cast<int32_t *>(base);
    base += align_up(nb * E * sizeof(int32_t), kWsAlign);
    l.flags = reinterpret_cast<unsigned long long *>(base);
    return l;
}

extern "C" size_t ep_workspace_size(int64_t T, int K, int P, int E_local, int chunks)
{
    (void)K;
    if (T < 0 || P < 1 || E_local < 1)
        return 0;
    const size_t nb = ws_blocks(T, chunks);
    const size_t E = (size_t)P * E_local;
    return kWsAlign + align_up(nb * P * sizeof(int32_t), kWsAlign) + align_up(nb * E * sizeof(int32_t), kWsAlign) +
           align_up(nb * sizeof(unsigned long long), kWsAlign) + align_up(E * sizeof(int32_t), kWsAlign);
}

extern "C" int ep_chunk_bounds(int64_t T, int chunks, int64_t *h_bounds)
{
    if (T < 0 || chunks < 1 || h_bounds == nullptr)
        return EP_ERR_INVALID_ARG;
    const int64_t size = T / chunks;
    for (int i = 0; i < chunks; ++i)
        h_bounds[i] = (int64_t)i * size;
    h_bounds[chunks] = T;
    return EP_OK;
}

static bool routing_shape_ok(int64_t T, int K, int P, int E_local)
{
    if (T < 0 || K < 1 || K > EP_MAX_TOPK || P < 1 || P > EP_MAX_RANKS || E_local < 1)
        return false;
    if ((int64_t)P * E_local > EP_MAX_EXPERTS)
        return false;
    return T * (int64_t)std::min(K, P) < ((int64_t)1 << 31) && T * (int64_t)K < ((int64_t)1 << 40);
}

extern "C" int ep_compute_send_counts(const int64_t *topk_idx, int64_t T, int K, int P, int E_local,
                                      const int64_t *h_chunk_bounds, int chunks, int32_t *dest,
                                      uint8_t *is_in_rank, int32_t *send_counts, int32_t *rank_offsets,
                                      int32_t *tokens_per_expert, void *ws, size_t ws_bytes,
                                      int32_t *err, ep_stream_t stream_)
{
    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
    if (!routing_shape_ok(T, K, P, E_local))
        return EP_ERR_INVALID_ARG;
    if (chunks > EP_MAX_CHUNKS)
        return EP_ERR_UNSUPPORTED;
    if (send_counts == nullptr || ws == nullptr || !aligned(ws, kWsAlign))
        return EP_ERR_INVALID_ARG;
    if (T > 0 && (topk_idx == nullptr || dest == nullptr || is_in_rank == nullptr))
        return EP_ERR_INVALID_ARG;
    if (ws_bytes < ep_workspace_size(T, K, P, E_local, chunks))
        return EP_ERR_INVALID_ARG;

    ChunkTable ct{};
    const int C = chunks > 1 ? chunks : 1;
    ct.n = C;
    if (C > 1) {
        if (h_chunk_bounds == nullptr || h_chunk_bounds[0] != 0 || h_chunk_bounds[C] != T)
            return EP_ERR_INVALID_ARG;
        for (int c = 0; c < C; ++c)
            if (h_chunk_bounds[c + 1] < h_chunk_bounds[c])
                return EP_ERR_INVALID_ARG;
    }
    int nb = 0;
    for (int c = 0; c < C; ++c) {
        ct.start[c] = C > 1 ? h_chunk_bounds[c] : 0;
        const int64_t end = C > 1 ? h_chunk_bounds[c + 1] : T;
        ct.first_block[c] = nb;
        nb += (int)ceil_div(end - ct.start[c], kRouteThreads);
    }
    ct.start[C] = T;
    ct.first_block[C] = nb;

    const int E = P * E_local;
    const WsLayout wl = ws_layout(ws, T, chunks, P, E);
    int32_t *part_rank = wl.part_rank;
    int32_t *pe = tokens_per_expert != nullptr ? wl.part_expert : nullptr;

    if (nb > 0) {
        const size_t smem = sizeof(int32_t) * (kWarps * P + (pe != nullptr ? E : 0));
        count_kernel<<<nb, kRouteThreads, smem, stream>>>(topk_idx, K, P, E_local, ct, dest, is_in_rank,
                                                          part_rank, pe, err);
        if (launch_status() != EP_OK)
            return EP_ERR_CUDA;
    }
    count_finish_kernel<<<1, 1024, 0, stream>>>(part_rank, pe, nb, P, E, ct, send_counts, rank_offsets,
                                                tokens_per_expert);
    return launch_status();
}

extern "C" int ep_build_send_layout(const int64_t *topk_idx, const float *topk_weights,
                                    const int32_t *dest, const uint8_t *is_in_rank, int64_t T, int K,
                                    int P, int E_local, int64_t num_send, int32_t *send_token_idx,
                                    int32_t *send_rank, int64_t *send_idx, float *send_w,
                                    int32_t *token_pos, void *ws, size_t ws_bytes, int32_t *err,
                                    ep_stream_t stream_)
{
    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
    if (!routing_shape_ok(T, K, P, E_local) || num_send < 0)
        return EP_ERR_INVALID_ARG;
    if (ws == nullptr || !aligned(ws, kWsAlign) || ws_bytes < ep_workspace_size(T, K, P, E_local, 1))
        return EP_ERR_INVALID_ARG;
    if (T > 0 && (topk_idx == nullptr || topk_weights == nullptr || dest == nullptr ||
                  is_in_rank == nullptr || token_pos == nullptr))
        return EP_ERR_INVALID_ARG;
    if (num_send > 0 && (send_token_idx == nullptr || send_rank == nullptr || send_idx == nullptr ||
                         send_w == nullptr))
        return EP_ERR_INVALID_ARG;
    if (T == 0)   // nothing is routed: the mismatch, if any, is known on the host
        return num_send == 0 ? EP_OK : EP_ERR_COUNT_MISMATCH;
    const int nb = (int)ceil_div(T, kRouteThreads);
    int32_t *part_rank = static_cast<int32_t *>(ws);
    layout_count_kernel<<<nb, kRouteThreads, 0, stream>>>(is_in_rank, T, P, part_rank);
    if (launch_status() != EP_OK)
        return EP_ERR_CUDA;
    LayoutArgs a{topk_idx, topk_weights, dest, is_in_rank, T, K, P, E_local, num_send, 1, part_rank, nb,
                 nullptr, nullptr, nullptr, nullptr, send_token_idx, send_rank, send_idx, send_w, token_pos, err, 1,
                 vec_ok(send_idx, send_w, is_in_rank, token_pos)};
    launch_layout_write(a, nb, stream);
    return launch_status();
}

static int route_nosync(const int64_t *topk_idx, const float *topk_weights, int64_t T, int K, int P, int E_local,
                        int64_t num_worst_rows, int align, int32_t *dest, uint8_t *is_in_rank, int32_t *send_counts,
                        int32_t *rank_offsets, int32_t *tokens_per_expert, int32_t *send_token_idx,
                        int32_t *send_rank, int64_t *send_idx, float *send_w, int32_t *token_pos, void *ws,
                        size_t ws_bytes, int32_t *err, ep_stream_t stream_)
{
    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
    if (!routing_shape_ok(T, K, P, E_local) || num_worst_rows < 0 || num_worst_rows >= ((int64_t)1 << 31))
        return EP_ERR_INVALID_ARG;
    if (align < 1 || align > (1 << 20))
        return EP_ERR_INVALID_ARG;
    if (ws == nullptr || !aligned(ws, kWsAlign) || ws_bytes < ep_workspace_size(T, K, P, E_local, 1))
        return EP_ERR_INVALID_ARG;
    if (send_counts == nullptr || rank_offsets == nullptr)
        return EP_ERR_INVALID_ARG;
    if (T > 0 && (topk_idx == nullptr || topk_weights == nullptr || dest == nullptr || is_in_rank == nullptr ||
                  token_pos == nullptr))
        return EP_ERR_INVALID_ARG;
    if (num_worst_rows > 0 && (send_token_idx == nullptr || send_rank == nullptr || send_idx == nullptr ||
                               send_w == nullptr))
        return EP_ERR_INVALID_ARG;
    const int E = P * E_local;
    const WsLayout wl = ws_layout(ws, T, 1, P, E);
    int32_t *pe = tokens_per_expert != nullptr ? wl.part_expert : nullptr;
    if (T == 0) {   // nothing routed: zero counts through the single-chunk finish
        ChunkTable ct{};
        ct.n = 1;
        count_finish_kernel<<<1, 1024, 0, stream>>>(wl.part_rank, nullptr, 0, P, E, ct, send_counts, rank_offsets,
                                                    tokens_per_expert);
        return launch_status();
    }

    // one cooperative launch when every block can be resident at once
    const int nbf = (int)ceil_div(T, kFusedThreads);
    const size_t smem_f = pe != nullptr ? sizeof(int32_t) * E : 0;
    FusedArgs fa{topk_idx, topk_weights, T, K, P, E_local, num_worst_rows, dest, is_in_rank, send_counts,
                 rank_offsets, tokens_per_expert, send_token_idx, send_rank, send_idx, send_w, token_pos,
                 wl.part_rank, pe, {wl.flags, wl.epoch, next_route_tag()}, align, err,
                 vec_ok(send_idx, send_w, is_in_rank, token_pos)};
    bool launched = false;
    int rc;
    switch (K) {
    case 2: rc = launch_route_fused<2>(fa, nbf, smem_f, stream, &launched); break;
    case 4: rc = launch_route_fused<4>(fa, nbf, smem_f, stream, &launched); break;
    case 6: rc = launch_route_fused<6>(fa, nbf, smem_f, stream, &launched); break;
    case 8: rc = launch_route_fused<8>(fa, nbf, smem_f, stream, &launched); break;
    default: rc = launch_route_fused<0>(fa, nbf, smem_f, stream, &launched); break;
    }
    if (rc != EP_OK || launched)
        return rc;

    // otherwise: count_kernel, then layout_write_kernel from its partials
    const int nb = (int)ceil_div(T, kRouteThreads);
    ChunkTable ct{};
    ct.n = 1;
    ct.start[0] = 0;
    ct.start[1] = T;
    ct.first_block[0] = 0;
    ct.first_block[1] = nb;
    const size_t smem = sizeof(int32_t) * (kWarps * P + (pe != nullptr ? E : 0));
    count_kernel<<<nb, kRouteThreads, smem, stream>>>(topk_idx, K, P, E_local, ct, dest, is_in_rank, wl.part_rank,
                                                      pe, err);
    if (launch_status() != EP_OK)
        return EP_ERR_CUDA;
    LayoutArgs a{topk_idx, topk_weights, dest, is_in_rank, T, K, P, E_local, num_worst_rows, 0, wl.part_rank, nb,
                 pe, send_counts, rank_offsets, tokens_per_expert, send_token_idx, send_rank, send_idx, send_w,
                 token_pos, err, align, vec_ok(send_idx, send_w, is_in_rank, token_pos)};
    launch_layout_write(a, nb, stream);
    return launch_status();
}

extern "C" int ep_route_nosync(const int64_t *topk_idx, const float *topk_weights, int64_t T, int K, int P,
                               int E_local, int64_t num_worst_rows, int32_t *dest, uint8_t *is_in_rank,
                               int32_t *send_counts, int32_t *rank_offsets, int32_t *tokens_per_expert,
                               int32_t *send_token_idx, int32_t *send_rank, int64_t *send_idx, float *send_w,
                               int32_t *token_pos, void *ws, size_t ws_bytes, int32_t *err, ep_stream_t stream)
{
    return route_nosync(topk_idx, topk_weights, T, K, P, E_local, num_worst_rows, 1, dest, is_in_rank, send_counts,
                        rank_offsets, tokens_per_expert, send_token_idx, send_rank, send_idx, send_w, token_pos, ws,
                        ws_bytes, err, stream);
}

extern "C" int ep_route_nosync_aligned(const int64_t *topk_idx, const float *topk_weights, int64_t T, int K, int P,
                                       int E_local, int64_t num_worst_rows, int alignment, int32_t *dest,
                                       uint8_t *is_in_rank, int32_t *send_counts, int32_t *rank_offsets,
                                       int32_t *tokens_per_expert, int32_t *send_token_idx, int32_t *send_rank,
                                       int64_t *send_idx, float *send_w, int32_t *token_pos, void *ws,
                                       size_t ws_bytes, int32_t *err, ep_stream_t stream)
{
    return route_nosync(topk_idx, topk_weights, T, K, P, E_local, num_worst_rows, alignment, dest, is_in_rank,
                        send_counts, rank_offsets, tokens_per_expert, send_token_idx, send_rank, send_idx, send_w,
                        token_pos, ws, ws_bytes, err, stream);
}

// ====================================================== no-allocation variant ==
// ep_compute_send_counts_noalloc: the same counts, with the per-block partial
// counts kept in a fixed device array that the library holds, so the caller
// passes no workspace.  It exists for callers that cannot allocate device
// memory themselves: engines that plan all device memory before they start
// and forbid allocation while they run (for example inside a plugin's enqueue
// step, where the host thread must not call into an allocator).
//
// The array below is set up once per device context: the first call on a
// device (with that device current) looks up its device address with
// cudaGetSymbolAddress and caches it with the id of the current context; a
// later call under another context (the device was reset, or its primary
// context released and created again) looks the address up again instead of
// reusing a stale one.  Every call on a device shares the one array, which
// keeps the last call's contents; the count kernels overwrite every partial
// they read, so nothing needs clearing between calls.  Calls whose kernels
// overlap on the GPU (other streams, other host threads) race on the array.
#include <cuda.h>

#include <mutex>

static __device__ __align__(256) unsigned char g_count_scratch[EP_NOALLOC_SCRATCH_BYTES];

namespace {
constexpr int kMaxDevices = 64;

// The driver API is reached through the runtime's entry-point query, so the
// library links no libcuda and still loads on a machine without a driver.
using CtxGetCurrentFn = CUresult (*)(CUcontext *);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long *);

struct ScratchSlot {
    void *addr = nullptr;
    unsigned long long ctx_id = 0;
};

std::mutex g_scratch_mutex;
ScratchSlot g_scratch[kMaxDevices];
CtxGetCurrentFn g_ctx_get_current = nullptr;
CtxGetIdFn g_ctx_get_id = nullptr;
bool g_ctx_fns_looked_up = false;

// Id of the context current on this thread, or 0 if none is current yet or
// the driver does not offer the query.  Called with g_scratch_mutex held.
unsigned long long current_context_id()
{
    if (!g_ctx_fns_looked_up) {
        g_ctx_fns_looked_up = true;
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_ctx_get_current = reinterpret_cast<CtxGetCurrentFn>(f);
        f = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_ctx_get_id = reinterpret_cast<CtxGetIdFn>(f);
        cudaGetLastError();
    }
    if (g_ctx_get_current == nullptr || g_ctx_get_id == nullptr)
        return 0;
    CUcontext ctx = nullptr;
    unsigned long long id = 0;
    if (g_ctx_get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr || g_ctx_get_id(ctx, &id) != CUDA_SUCCESS)
        return 0;
    return id;
}

// Device address of g_count_scratch on the current device.  Host code cannot
// use the symbol itself: on the host it names a stand-in, not device memory.
int count_scratch_address(void **out)
{
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return EP_ERR_CUDA;
    }
    if (dev < 0 || dev >= kMaxDevices)
        return EP_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    ScratchSlot &slot = g_scratch[dev];
    const unsigned long long id = current_context_id();
    // A cached address is used only under the context it was looked up in;
    // with no context id to compare (none current yet on this thread), it is
    // looked up again, which also makes the device's context current.
    if (slot.addr == nullptr || id == 0 || id != slot.ctx_id) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_count_scratch) != cudaSuccess || p == nullptr) {
            cudaGetLastError();
            slot = ScratchSlot{};
            return EP_ERR_CUDA;
        }
        slot.addr = p;
        slot.ctx_id = id != 0 ? id : current_context_id();
    }
    *out = slot.addr;
    return EP_OK;
}

// The host checks of ep_compute_send_counts that need no workspace, made
// before the device is touched (looking up the array's address can create
// the device's context).
int noalloc_args_status(const int64_t *topk_idx, int64_t T, int K, int P, int E_local,
                        const int64_t *h_chunk_bounds, int chunks, const int32_t *dest,
                        const uint8_t *is_in_rank, const int32_t *send_counts)
{
    if (!routing_shape_ok(T, K, P, E_local))
        return EP_ERR_INVALID_ARG;
    if (chunks > EP_MAX_CHUNKS)
        return EP_ERR_UNSUPPORTED;
    if (ep_workspace_size(T, K, P, E_local, chunks) > (size_t)EP_NOALLOC_SCRATCH_BYTES)
        return EP_ERR_UNSUPPORTED;
    if (send_counts == nullptr)
        return EP_ERR_INVALID_ARG;
    if (T > 0 && (topk_idx == nullptr || dest == nullptr || is_in_rank == nullptr))
        return EP_ERR_INVALID_ARG;
    if (chunks > 1) {
        if (h_chunk_bounds == nullptr || h_chunk_bounds[0] != 0 || h_chunk_bounds[chunks] != T)
            return EP_ERR_INVALID_ARG;
        for (int c = 0; c < chunks; ++c)
            if (h_chunk_bounds[c + 1] < h_chunk_bounds[c])
                return EP_ERR_INVALID_ARG;
    }
    return EP_OK;
}
}  // namespace

extern "C" int ep_compute_send_counts_noalloc(const int64_t *topk_idx, int64_t T, int K, int P, int E_local,
                                              const int64_t *h_chunk_bounds, int chunks, int32_t *dest,
                                              uint8_t *is_in_rank, int32_t *send_counts, int32_t *rank_offsets,
                                              int32_t *tokens_per_expert, int32_t *err, ep_stream_t stream)
{
    int rc = noalloc_args_status(topk_idx, T, K, P, E_local, h_chunk_bounds, chunks, dest, is_in_rank, send_counts);
    if (rc != EP_OK)
        return rc;
    void *scratch = nullptr;
    rc = count_scratch_address(&scratch);
    if (rc != EP_OK)
        return rc;
    return ep_compute_send_counts(topk_idx, T, K, P, E_local, h_chunk_bounds, chunks, dest, is_in_rank,
                                  send_counts, rank_offsets, tokens_per_expert, scratch,
                                  (size_t)EP_NOALLOC_SCRATCH_BYTES, err, stream);
}
