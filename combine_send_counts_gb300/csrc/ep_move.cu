// Row movement kernels of libep_gb300.
//
//   scatter  -- dispatch (axolotl integrations.expert_parallel.torch_dispatch,
//               dispatch; NeMo uccl_ep.buffer, Buffer.dispatch) and the
//               expert-batched prepare (vLLM BatchedPrepareAndFinalize.prepare):
//               every source row is read from HBM once and written to each of
//               its destination rows, as bf16 or quantised to fp8 (1x128).
//   zero     -- padding rows (and their scales) of the expert-batched layout.
//   expert   -- the synthetic fp8 local expert of the chunked forward.
//   (the combines live in ep_combine.cu)
//
// The bf16 scatter is an HBM-bound copy.  A group of G threads (a multiple of
// 32) owns one token; each thread moves U 16-byte vectors of the row, so a row
// is covered in one pass for H up to 8*G*U.  The destination row list of the
// block's tokens is resolved once into shared memory.  The fp8 scatter
// quantises each row once, in warps that also compute the group scales: one
// warp per token on the send layout, balanced runs of (token, 1024-column
// chunk) units per warp on the expert-batched layout.
#include <algorithm>
#include <atomic>
#include <type_traits>
#include <utility>
#include <climits>

#include <cuda_fp16.h>

#include "ep_device.cuh"
#include "ep_fp8.cuh"
#include "ep_internal.h"
#include "ep_rows.cuh"

namespace ep {

constexpr int kMoveThreads = 256;
constexpr int kMaxTokensPerBlock = kMoveThreads / 32;

struct Geometry {
    int nvec;   // 16-byte vectors per row (H / 8 for bf16)
    int G;      // threads per token
    int tpb;    // tokens per block
};

// Resolve the row lists of this block's tokens into shared memory; rows that
// fall outside [0, n_rows) are reported and dropped.
template <class Rows>
__device__ __forceinline__ void load_lists(const Rows &rows, int64_t T, int64_t t0, int tpb,
                                           int64_t n_rows, int err_bits, int32_t *s_rows,
                                           float *s_w, int32_t *err)
{
    const int D = rows.len();
    int bad = 0;
    for (int i = threadIdx.x; i < tpb * D; i += blockDim.x) {
        const int s = i / D, j = i % D;
        const int64_t t = t0 + s;
        int32_t r = -1;
        float wv = 0.0f;
        if (t < T) {
            r = rows.row(t, j);
            if (r >= n_rows) {
                bad = err_bits;
                r = -1;
            }
            if (r >= 0 && s_w != nullptr)
                wv = rows.weight(t, j);
        }
        s_rows[s * kMaxList + j] = r;
        if (s_w != nullptr)
            s_w[s * kMaxList + j] = wv;
    }
    raise(err, bad);
}

// ---------------------------------------------------------- bf16 scatter --
template <int U, class Rows>
__global__ void __launch_bounds__(kMoveThreads)
scatter_bf16_kernel(const uint4 *__restrict__ x, int64_t T, Geometry g, Rows rows, int64_t n_rows,
                    int err_bits, uint4 *__restrict__ out, int32_t *err)
{
    __shared__ int32_t s_rows[kMaxTokensPerBlock * kMaxList];
    const int64_t t0 = (int64_t)blockIdx.x * g.tpb;
    const int s = threadIdx.x / g.G, lt = threadIdx.x % g.G;
    const int64_t t = t0 + s;
    const bool active = s < g.tpb && t < T;
    const uint4 *src = x + t * g.nvec;
    // The rows are inputs, not outputs of the routing kernel before this one:
    // load the first batch while that kernel may still run (dependent launch).
    uint4 v[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
        const int i = lt + u * g.G;
        if (active && i < g.nvec)
            v[u] = ld_stream(src + i);
    }
    grid_dependency_wait();
    allow_dependents();   // a zero fill after this kernel reads only what the kernel before it wrote
    load_lists(rows, T, t0, g.tpb, n_rows, err_bits, s_rows, nullptr, err);
    __syncthreads();
    if (!active)
        return;
    const int D = rows.len();
    const int32_t *list = s_rows + s * kMaxList;
    for (int base = 0; base < g.nvec; base += g.G * U) {
        if (base > 0) {
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int i = base + lt + u * g.G;
                if (i < g.nvec)
                    v[u] = ld_stream(src + i);
            }
        }
        for (int j = 0; j < D; ++j) {
            const int32_t r = list[j];
            if (r < 0)
                continue;
            uint4 *dst = out + (int64_t)r * g.nvec;
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int i = base + lt + u * g.G;
                if (i < g.nvec)
                    st_stream(dst + i, v[u]);
            }
        }
    }
}

// ------------------------------------------------- fp8 (1x128) scatter --
// One warp per token (grid-stride loop over tokens).  Lanes j < D (and
// j + 32) resolve the token's rows; the warp quantises the row once, in
// chunks of U 16-byte vectors per lane (quantize_chunk), and writes each
// chunk's e4m3 codes and group scales to every row, taking the rows by
// shuffle; a destination row's scale base is computed once per token.  No
// shared memory and no block barrier.  SF is the scale layout (EP_SCALE_*),
// RS selects power-of-two scales.
template <int U, class Rows, int SF, bool RS, bool DB>
__global__ void __launch_bounds__(kMoveThreads, DB ? 3 : 4)
scatter_fp8_warp_kernel(const uint4 *__restrict__ x, int64_t T, int nvec, Rows rows, int64_t n_rows,
                        int err_bits, uint2 *__restrict__ out_q, ScaleSpec sp, int32_t *err)
{
    grid_dependency_wait();
    allow_dependents();   // a zero fill after this kernel reads only what the kernel before it wrote
    const int lane = threadIdx.x & 31;
    const int64_t nw = ((int64_t)gridDim.x * blockDim.x) >> 5;
    const int D = rows.len();
    const int groups = nvec / 16;
    int bad = 0;
    const int u_own = group_owner_u<U>(lane);                  // this lane's group in a chunk:
    const int i_own = 32 * u_own + (lane & 16);                 // its first vector from the chunk base
    const bool owner = (lane & (U == 4 ? 3 : 7)) == 0;          // one lane of the group's owners stores
    for (int64_t t = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; t < T; t += nw) {
        int32_t r_lo = -1, r_hi = -1;
        int64_t sb_lo = 0, sb_hi = 0;   // scale bases of the rows (column layouts)
        if (lane < D) {
            r_lo = rows.row(t, lane);
            if (r_lo >= n_rows) {
                bad = err_bits;
                r_lo = -1;
            }
            if (SF != EP_SCALE_ROW_F32 && r_lo >= 0)
                sb_lo = scale_row_base<SF>(sp, r_lo, groups);
        }
        if (lane + 32 < D) {
            r_hi = rows.row(t, lane + 32);
            if (r_hi >= n_rows) {
                bad = err_bits;
                r_hi = -1;
            }
            if (SF != EP_SCALE_ROW_F32 && r_hi >= 0)
                sb_hi = scale_row_base<SF>(sp, r_hi, groups);
        }
        const uint64_t valid =
            (uint64_t)__ballot_sync(kFull, r_lo >= 0) | ((uint64_t)__ballot_sync(kFull, r_hi >= 0) << 32);
        if (valid == 0)
            continue;   // warp-uniform: a token with no destination row is not read
        const uint4 *src = x + t * nvec;
        // DB: the next chunk is loaded while this one is quantised and stored
        uint4 nxt[U];
        if constexpr (DB) {
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int i = lane + 32 * u;
                nxt[u] = make_uint4(0, 0, 0, 0);
                if (i < nvec)
                    nxt[u] = ld_stream(src + i);
            }
        }
        for (int base = 0; base < nvec; base += 32 * U) {
            uint4 vin[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {   // all loads first: U vectors in flight
                if constexpr (DB) {
                    vin[u] = nxt[u];
                    const int i = base + 32 * U + lane + 32 * u;
                    nxt[u] = make_uint4(0, 0, 0, 0);
                    if (i < nvec)
                        nxt[u] = ld_stream(src + i);
                } else {
                    const int i = base + lane + 32 * u;
                    vin[u] = make_uint4(0, 0, 0, 0);
                    if (i < nvec)
                        vin[u] = ld_stream(src + i);
                }
            }
            uint2 q[U];
            float scale_own;
            uint32_t code_own;
            quantize_chunk<U, RS>(vin, lane, q, scale_own, code_own);
            const bool put = owner && base + i_own < nvec;
            for (uint64_t mm = valid; mm != 0; mm &= mm - 1) {   // warp-uniform
                const int j = __ffsll((long long)mm) - 1;
                const int32_t r = j < 32 ? __shfl_sync(kFull, r_lo, j) : __shfl_sync(kFull, r_hi, j - 32);
                int64_t sb;
                if (SF == EP_SCALE_ROW_F32)
                    sb = (int64_t)r * groups;
                else
                    sb = j < 32 ? __shfl_sync(kFull, sb_lo, j) : __shfl_sync(kFull, sb_hi, j - 32);
                uint2 *dq = out_q + (int64_t)r * nvec;
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const int i = base + lane + 32 * u;
                    if (i < nvec)
                        st_stream(dq + i, q[u]);
                }
                if (put)
                    put_scale<SF>(sp, sb, (base + i_own) >> 4, scale_own, code_own);
            }
        }
    }
    raise(err, bad);
}

// fp8 (1x128) scatter on the expert-batched layout, in balanced units.  A
// unit is one chunk (32 * U 16-byte vectors) of one token's row; warp w of
// the grid owns the contiguous units [w * units / nw, (w + 1) * units / nw),
// so every warp quantises the same number of chunks and the grid is one
// resident wave (no partial last wave of blocks: the per-token form, one
// token per warp in 1024 blocks of which 608 are resident, left the SMs idle
// for a quarter of its time).  A warp takes its units in order, resolving a
// token's rows (lanes j < K) once per token.
template <int U, int SF, bool RS>
__global__ void __launch_bounds__(kMoveThreads, 4)
scatter_fp8_units_kernel(const uint4 *__restrict__ x, int64_t T, int nvec, BatchedRows rows, int64_t n_rows,
                         int err_bits, uint2 *__restrict__ out_q, ScaleSpec sp, int32_t *err)
{
    const int lane = threadIdx.x & 31;
    constexpr int kChunk = 32 * U;   // vectors per unit
    const int nch = (nvec + kChunk - 1) / kChunk;
    const int64_t units = T * nch;
    const int64_t nw = ((int64_t)gridDim.x * blockDim.x) >> 5;
    const int64_t gw = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int64_t u_lo = gw * units / nw, u_hi = (gw + 1) * units / nw;
    grid_dependency_wait();
    allow_dependents();   // a zero fill after this kernel reads only what the kernel before it wrote
    const int groups = nvec / 16;
    const int u_own = group_owner_u<U>(lane);
    const int i_own = 32 * u_own + (lane & 16);
    const bool owner = (lane & (U == 4 ? 3 : 7)) == 0;
    int bad = 0;
    int64_t cur = -1;
    int32_t r = -1;       // lane j < K: the token's row for slot j, or -1
    int64_t sbase = 0;    // its scale base (column layouts)
    unsigned valid = 0;
    for (int64_t u = u_lo; u < u_hi; ++u) {
        const int64_t t = u / nch;
        if (t != cur) {
            cur = t;
            r = -1;
            sbase = 0;
            if (lane < rows.len()) {
                r = rows.row(t, lane);
                if (r >= n_rows) {
                    bad = err_bits;
                    r = -1;
                }
                if (SF != EP_SCALE_ROW_F32 && r >= 0)
                    sbase = scale_row_base<SF>(sp, r, groups);
            }
            valid = __ballot_sync(kFull, r >= 0);
        }
        if (valid == 0)
            continue;   // warp-uniform: a token with no row here is not read
        const int base = (int)(u - t * nch) * kChunk;
        const uint4 *src = x + t * nvec;
        uint4 vin[U];
#pragma unroll
        for (int u2 = 0; u2 < U; ++u2) {   // all loads first: U vectors in flight
            const int i = base + lane + 32 * u2;
            vin[u2] = make_uint4(0, 0, 0, 0);
            if (i < nvec)
                vin[u2] = ld_stream(src + i);
        }
        uint2 q[U];
        float scale_own;
        uint32_t code_own;
        quantize_chunk<U, RS>(vin, lane, q, scale_own, code_own);
        const bool put = owner && base + i_own < nvec;
        for (unsigned mm = valid; mm != 0; mm &= mm - 1) {   // warp-uniform
            const int j = __ffs(mm) - 1;
            const int32_t rj = __shfl_sync(kFull, r, j);
            const int64_t sb = SF == EP_SCALE_ROW_F32 ? (int64_t)rj * groups : __shfl_sync(kFull, sbase, j);
            uint2 *dq = out_q + (int64_t)rj * nvec;
#pragma unroll
            for (int u2 = 0; u2 < U; ++u2) {
                const int i = base + lane + 32 * u2;
                if (i < nvec)
                    st_stream(dq + i, q[u2]);
            }
            if (put)
                put_scale<SF>(sp, sb, (base + i_own) >> 4, scale_own, code_own);
        }
    }
    raise(err, bad);
}

// ------------------------------------------------------------- zero padding --
// The zero fills run after the row scatter as its programmatic dependents: the
// scatter lets them start once all its blocks have passed their own wait on the
// slot kernel, so the counts they read (kept and tokens_per_expert, written by
// the slot kernel) are final, and the rows they write (at or past an expert's
// kept count) are ones the scatter never writes.  Block (0, 0) of each waits
// for the kernel before it just before exiting, which is enough for the
// kernel's completion to imply that one's; the other blocks exit as soon as
// their rows are written instead of holding their SM slots.
//
// Zero rows [first[e], end) of every local expert, end = M when full, else
// tokens_per_expert[e] (the aligned count); 16-byte stores.
__global__ void zero_rows_kernel(uint4 *__restrict__ b_x, const int32_t *__restrict__ first,
                                 const int32_t *__restrict__ tokens_per_expert, int full, int M, int nvec)
{
    allow_dependents();   // the scale fill after this kernel is independent of it
    const int e = blockIdx.y;
    const int64_t lo = (int64_t)first[e] * nvec;
    const int64_t hi = (int64_t)(full ? M : tokens_per_expert[e]) * nvec;
    uint4 *base = b_x + (int64_t)e * M * nvec;
    const uint4 z = make_uint4(0, 0, 0, 0);
    for (int64_t i = lo + (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < hi; i += (int64_t)gridDim.x * blockDim.x)
        st_stream(base + i, z);
    if (blockIdx.x == 0 && blockIdx.y == 0)
        grid_dependency_wait();
}

// Zero the scale entries of slots [first[e], end) of every local expert (end
// as zero_rows_kernel), in any scale layout (4-byte entries; UE8M0 ints hold
// 4 groups of one slot).
__global__ void zero_scales_kernel(ScaleSpec sp, const int32_t *__restrict__ first,
                                   const int32_t *__restrict__ tokens_per_expert, int full, int groups)
{
    const int e = blockIdx.y;
    const int lo = first[e], hi = full ? sp.M : tokens_per_expert[e];
    const int per_row = sp.fmt == EP_SCALE_COL_UE8M0 ? groups / 4 : groups;
    uint32_t *base = static_cast<uint32_t *>(sp.out) + (int64_t)e * sp.M * per_row;
    const int64_t n = (int64_t)(hi - lo) * per_row;   // entries (slot s in [lo, hi), column c)
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t s = lo + i % (hi - lo), c = i / (hi - lo);
        base[sp.fmt == EP_SCALE_ROW_F32 ? s * per_row + c : c * sp.M + s] = 0u;
    }
    if (blockIdx.x == 0 && blockIdx.y == 0)
        grid_dependency_wait();
}

// -------------------------------------------------- synthetic fp8 expert --
// d = e4m3(q) * scale, y_k = bf16(d * (1 + l_k/64)),
// out = bf16(fma over k ascending of w_k * y_k from +0.0f).
// One warp per row, 8 rows per block: the lanes load the row's K expert ids
// and weights at once and compact the ones in use (ascending k, by ballot)
// into shared memory; each lane then issues kLocalU 16-byte code loads before
// it converts any, so that enough bytes are in flight to keep HBM busy, and
// applies the experts one at a time to all 16 values of a vector (16
// independent fma chains; each value's chain still runs over k ascending).
// The multiplies and fmas run as packed pairs (mul2_rn / fma2_rn) and the
// bf16 rounding of y converts two values per instruction, which cuts the
// kernel's instruction count by about a third.
constexpr int kLocalRowsPerBlock = 8;
constexpr int kLocalU = 4;

__global__ void __launch_bounds__(kLocalRowsPerBlock * 32, 4)
local_expert_fp8_kernel(const uint4 *__restrict__ q, const float *__restrict__ scale,
                        const int64_t *__restrict__ send_idx, const float *__restrict__ send_w, int64_t N,
                        const int32_t *__restrict__ n_rows, int K, int H, uint4 *__restrict__ out)
{
    __shared__ float s_fac[kLocalRowsPerBlock][EP_MAX_TOPK];
    __shared__ float s_w[kLocalRowsPerBlock][EP_MAX_TOPK];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t n = (int64_t)blockIdx.x * kLocalRowsPerBlock + warp;
    int64_t lim = N;
    if (n_rows != nullptr)   // rows past the device count are not in use
        lim = min(lim, (int64_t)*n_rows);
    if (n >= lim)
        return;   // the whole warp
    int64_t l = -1;
    float wk = 0.0f;
    if (lane < K) {
        l = send_idx[n * K + lane];
        wk = send_w[n * K + lane];
    }
    const bool use = lane < K && l >= 0;
    const unsigned used = __ballot_sync(kFull, use);
    if (use) {
        const int j = __popc(used & lanemask_lt());
        s_fac[warp][j] = __fadd_rn(1.0f, __fmul_rn((float)l, 0.015625f));
        s_w[warp][j] = wk;
    }
    __syncwarp();
    const int m = __popc(used);
    const float *fac = s_fac[warp], *wt = s_w[warp];
    const int V = H / 16;   // 16 codes per 16-byte vector
    const uint4 *qr = q + n * V;
    const float *sr = scale + n * (H / 128);
    uint4 *orow = out + n * V * 2;
    for (int base = 0; base < V; base += 32 * kLocalU) {
        uint4 v[kLocalU];
#pragma unroll
        for (int u = 0; u < kLocalU; ++u) {
            const int c = base + u * 32 + lane;
            if (c < V)
                v[u] = ld_stream(qr + c);
            else
                v[u] = make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int u = 0; u < kLocalU; ++u) {
            const int c = base + u * 32 + lane;
            if (c >= V)
                break;
            const float sc = __ldg(sr + c / 8);
            const float2 sc2 = make_float2(sc, sc);
            const uint32_t words[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
            float2 d[8], a[8];   // values 2i and 2i+1 of the vector
#pragma unroll
            for (int wi = 0; wi < 4; ++wi) {
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    const __nv_fp8x2_storage_t pair = (__nv_fp8x2_storage_t)(words[wi] >> (16 * hh));
                    const __half2_raw hr = __nv_cvt_fp8x2_to_halfraw2(pair, __NV_E4M3);
                    d[wi * 2 + hh] = mul2_rn(__half22float2(*reinterpret_cast<const __half2 *>(&hr)), sc2);
                }
            }
#pragma unroll
            for (int i = 0; i < 8; ++i)
                a[i] = make_float2(0.0f, 0.0f);
            // experts outermost: 16 independent accumulation chains per step
            for (int k = 0; k < m; ++k) {
                const float2 f = make_float2(fac[k], fac[k]), w = make_float2(wt[k], wt[k]);
#pragma unroll
                for (int i = 0; i < 8; ++i)
                    a[i] = fma2_rn(w, round_bf16x2(mul2_rn(d[i], f)), a[i]);
            }
            uint32_t packed[8];
#pragma unroll
            for (int i = 0; i < 8; ++i)
                packed[i] = pack_bf16x2(a[i].x, a[i].y);
            st_stream(orow + 2 * c, make_uint4(packed[0], packed[1], packed[2], packed[3]));
            st_stream(orow + 2 * c + 1, make_uint4(packed[4], packed[5], packed[6], packed[7]));
        }
    }
}

// ------------------------------------------------------------ launch policy --
static Geometry geometry_for(int nvec, int &U)
{
    U = nvec > 512 ? 8 : nvec > 256 ? 4 : nvec > 128 ? 2 : 1;
    int G = (int)ceil_div(ceil_div(nvec, U), 32) * 32;
    G = std::min(G, kMoveThreads);
    Geometry g;
    g.nvec = nvec;
    g.G = G;
    g.tpb = kMoveThreads / G;
    return g;
}

// Launch with programmatic stream serialisation when `dependent` (the kernel
// may start while the kernel before it runs; used only where the library
// launched that kernel itself and it writes nothing the early part reads).
template <typename... KArgs, typename... Args>
static cudaError_t launch_kernel(bool dependent, void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                                 cudaStream_t stream, Args &&...args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = dependent ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

int current_device()
{
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return -1;
    }
    return dev;
}

static int device_attribute(int dev, cudaDeviceAttr attr, int fallback)
{
    int v = 0;
    if (dev < 0 || cudaDeviceGetAttribute(&v, attr, dev) != cudaSuccess || v < 0) {
        cudaGetLastError();
        return fallback;
    }
    return v;
}

int device_sm_count()
{
    static PerDevice sms;
    const int dev = current_device();
    int v = sms.get(dev);
    if (v < 0) {
        v = device_attribute(dev, cudaDevAttrMultiProcessorCount, 152);
        sms.put(dev, v);
    }
    return v;
}

int64_t device_l2_bytes()
{
    static PerDevice bytes;
    const int dev = current_device();
    int v = bytes.get(dev);
    if (v < 0) {
        v = device_attribute(dev, cudaDevAttrL2CacheSize, 0);
        bytes.put(dev, v);
    }
    return v;
}

template <class Rows>
static int launch_scatter_bf16(const void *x, int64_t T, int H, const Rows &rows, int64_t n_rows,
                               int err_bits, void *out, int32_t *err, cudaStream_t stream, bool dependent)
{
    int U;
    const Geometry g = geometry_for(H / 8, U);
    const int64_t blocks = ceil_div(T, g.tpb);
    if (blocks == 0)
        return EP_OK;
    auto *xs = static_cast<const uint4 *>(x);
    auto *o = static_cast<uint4 *>(out);
    const dim3 grid((unsigned)blocks), block(g.G * g.tpb);
    cudaError_t e;
    switch (U) {
    case 8: e = launch_kernel(dependent, scatter_bf16_kernel<8, Rows>, grid, block, 0, stream, xs, T, g, rows, n_rows, err_bits, o, err); break;
    case 4: e = launch_kernel(dependent, scatter_bf16_kernel<4, Rows>, grid, block, 0, stream, xs, T, g, rows, n_rows, err_bits, o, err); break;
    case 2: e = launch_kernel(dependent, scatter_bf16_kernel<2, Rows>, grid, block, 0, stream, xs, T, g, rows, n_rows, err_bits, o, err); break;
    default: e = launch_kernel(dependent, scatter_bf16_kernel<1, Rows>, grid, block, 0, stream, xs, T, g, rows, n_rows, err_bits, o, err); break;
    }
    if (e != cudaSuccess) {
        cudaGetLastError();
        return EP_ERR_CUDA;
    }
    return EP_OK;
}


template <class Rows, int SF, bool RS>
static int launch_scatter_fp8_as(const void *x, int64_t T, int H, const Rows &rows, int64_t n_rows,
                                 int err_bits, void *out_q, const ScaleSpec &sp, int32_t *err,
                                 cudaStream_t stream, bool dependent)
{
    const int nvec = H / 8;
    const int64_t warps = kMoveThreads / 32;
    const int64_t blocks = std::min<int64_t>(ceil_div(T, warps), (int64_t)8 * device_sm_count());
    if (blocks == 0)
        return EP_OK;
    auto *xs = static_cast<const uint4 *>(x);
    auto *q = static_cast<uint2 *>(out_q);
    const dim3 grid((unsigned)blocks), block(kMoveThreads);
    // the next chunk in flight during this one's quantisation (3 CTAs per SM
    // instead of 4) pays on the send layout's longer rows (fp8 dispatch of 8192
    // tokens x 7168: 61.8 -> 60.2 us), not on the batched layout's (about 0.4 us
    // slower at H = 4096)
    constexpr bool DB = std::is_same<Rows, SendRows>::value;
    const cudaError_t e =
        nvec > 64 ? launch_kernel(dependent, scatter_fp8_warp_kernel<4, Rows, SF, RS, DB>, grid, block, 0, stream, xs,
                                  T, nvec, rows, n_rows, err_bits, q, sp, err)
                  : launch_kernel(dependent, scatter_fp8_warp_kernel<2, Rows, SF, RS, DB>, grid, block, 0, stream, xs,
                                  T, nvec, rows, n_rows, err_bits, q, sp, err);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return EP_ERR_CUDA;
    }
    return EP_OK;
}

// The send layout only takes row-major plain scales.
static int launch_scatter_fp8(const void *x, int64_t T, int H, const SendRows &rows, int64_t n_rows,
                              int err_bits, void *out_q, const ScaleSpec &sp, int32_t *err, cudaStream_t stream,
                              bool dependent)
{
    return launch_scatter_fp8_as<SendRows, EP_SCALE_ROW_F32, false>(x, T, H, rows, n_rows, err_bits, out_q, sp,
                                                                     err, stream, dependent);
}

template <int SF, bool RS>
static int launch_scatter_fp8_units(const void *x, int64_t T, int H, const BatchedRows &rows, int64_t n_rows,
                                    int err_bits, void *out_q, const ScaleSpec &sp, int32_t *err, cudaStream_t stream,
                                    bool dependent)
{
    const int nvec = H / 8;
    const bool u4 = nvec > 64;
    auto kernel = u4 ? scatter_fp8_units_kernel<4, SF, RS> : scatter_fp8_units_kernel<2, SF, RS>;
    static PerDevice per_sm_cache[2];
    const int dev = current_device();
    int per_sm = per_sm_cache[u4].get(dev);
    if (per_sm < 0) {
        int n = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel, kMoveThreads, 0) != cudaSuccess) {
            cudaGetLastError();
            n = 0;
        }
        per_sm = std::max(n, 1);
        per_sm_cache[u4].put(dev, per_sm);
    }
    const int chunk = 32 * (u4 ? 4 : 2);
    const int64_t units = T * ((nvec + chunk - 1) / chunk);
    // one resident wave, but at least about four units per warp
    const int64_t blocks = std::min<int64_t>((int64_t)per_sm * device_sm_count(),
                                             std::max<int64_t>(1, ceil_div(units, 4 * (kMoveThreads / 32))));
    if (T == 0)
        return EP_OK;
    const cudaError_t e = launch_kernel(dependent, kernel, dim3((unsigned)blocks), dim3(kMoveThreads), 0, stream,
                                        static_cast<const uint4 *>(x), T, nvec, rows, n_rows, err_bits,
                                        static_cast<uint2 *>(out_q), sp, err);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return EP_ERR_CUDA;
    }
    return EP_OK;
}

static int launch_scatter_fp8(const void *x, int64_t T, int H, const BatchedRows &rows, int64_t n_rows,
                              int err_bits, void *out_q, const ScaleSpec &sp, int32_t *err, cudaStream_t stream,
                              bool dependent)
{
    if (sp.fmt == EP_SCALE_COL_UE8M0)
        return launch_scatter_fp8_units<EP_SCALE_COL_UE8M0, true>(x, T, H, rows, n_rows, err_bits, out_q, sp, err,
                                                                  stream, dependent);
    if (sp.fmt == EP_SCALE_COL_F32)
        return sp.round ? launch_scatter_fp8_units<EP_SCALE_COL_F32, true>(x, T, H, rows, n_rows, err_bits, out_q,
                                                                           sp, err, stream, dependent)
                        : launch_scatter_fp8_units<EP_SCALE_COL_F32, false>(x, T, H, rows, n_rows, err_bits, out_q,
                                                                            sp, err, stream, dependent);
    return sp.round ? launch_scatter_fp8_units<EP_SCALE_ROW_F32, true>(x, T, H, rows, n_rows, err_bits, out_q, sp,
                                                                       err, stream, dependent)
                    : launch_scatter_fp8_units<EP_SCALE_ROW_F32, false>(x, T, H, rows, n_rows, err_bits, out_q, sp,
                                                                        err, stream, dependent);
}

static bool row_shape_ok(int64_t T, int H)
{
    return T >= 0 && H >= 8 && H % 8 == 0 && T < ((int64_t)1 << 31);
}

}  // namespace ep

// ================================================================ C ABI ====
using namespace ep;

extern "C" const char *ep_status_str(int status)
{
    switch (status) {
    case EP_OK: return "EP_OK";
    case EP_ERR_INVALID_ARG: return "EP_ERR_INVALID_ARG";
    case EP_ERR_INVALID_EXPERT: return "EP_ERR_INVALID_EXPERT";
    case EP_ERR_COUNT_MISMATCH: return "EP_ERR_COUNT_MISMATCH";
    case EP_ERR_CAPACITY: return "EP_ERR_CAPACITY";
    case EP_ERR_UNSUPPORTED: return "EP_ERR_UNSUPPORTED";
    case EP_ERR_CUDA: return "EP_ERR_CUDA";
    case EP_ERR_TIMEOUT: return "EP_ERR_TIMEOUT";
    default: return "EP_ERR_(combination)";
    }
}

namespace ep {
// ep_dispatch; `dependent` launches the scatter as a programmatic dependent of
// the routing kernel the library enqueued just before it.
int dispatch_rows(const void *x, int64_t T, int H, const int32_t *token_pos, int P, int64_t num_send,
                  void *recv_x, float *recv_scale, int fp8, int32_t *err, cudaStream_t stream, bool dependent)
{
    if (!row_shape_ok(T, H) || P < 1 || P > EP_MAX_RANKS || num_send < 0 || num_send >= ((int64_t)1 << 31))
        return EP_ERR_INVALID_ARG;
    if (fp8 != 0 && fp8 != 1)
        return EP_ERR_UNSUPPORTED;
    if (fp8 && H % 128 != 0)
        return EP_ERR_UNSUPPORTED;
    if (T > 0 && (x == nullptr || token_pos == nullptr || !aligned(x, 16)))
        return EP_ERR_INVALID_ARG;
    if (num_send > 0 && (recv_x == nullptr || !aligned(recv_x, 16)))
        return EP_ERR_INVALID_ARG;
    if (fp8 ? (num_send > 0 && recv_scale == nullptr) : recv_scale != nullptr)
        return EP_ERR_INVALID_ARG;
    if (T == 0)
        return EP_OK;
    const SendRows rows{token_pos, P};
    if (fp8)
        return launch_scatter_fp8(x, T, H, rows, num_send, EP_ERR_COUNT_MISMATCH, recv_x,
                                  ScaleSpec{recv_scale, EP_SCALE_ROW_F32, 0, 0}, err, stream, dependent);
    return launch_scatter_bf16(x, T, H, rows, num_send, EP_ERR_COUNT_MISMATCH, recv_x, err, stream, dependent);
}
}  // namespace ep

extern "C" int ep_dispatch(const void *x, int64_t T, int H, const int32_t *token_pos, int P,
                           int64_t num_send, void *recv_x, float *recv_scale, int fp8, int32_t *err,
                           ep_stream_t stream)
{
    return dispatch_rows(x, T, H, token_pos, P, num_send, recv_x, recv_scale, fp8, err,
                         reinterpret_cast<cudaStream_t>(stream), false);
}

// bf16 rows (sp == nullptr) or fp8 codes with scales as *sp; capacity 0
// means M with overflow reported, 1..M drops silently past it.
static int batched_prepare(const void *x, const int64_t *topk_idx, int64_t T, int K, int H, int E, int E_local,
                           int rank, int M, int capacity, int alignment, void *b_x, const ScaleSpec *sp,
                           int32_t *tokens_per_expert, int32_t *slot, int32_t *dropped, int zero_pad, void *ws,
                           size_t ws_bytes, int32_t *err, cudaStream_t stream)
{
    if (!row_shape_ok(T, H) || K < 1 || K > EP_MAX_TOPK || E_local < 1 || E < E_local || E % E_local != 0)
        return EP_ERR_INVALID_ARG;
    if (rank < 0 || (int64_t)(rank + 1) * E_local > E || M < 0)
        return EP_ERR_INVALID_ARG;
    if (capacity < 0 || capacity > M || alignment < 1)
        return EP_ERR_INVALID_ARG;
    if ((int64_t)E_local * M >= ((int64_t)1 << 31))
        return EP_ERR_UNSUPPORTED;
    if (tokens_per_expert == nullptr || ws == nullptr || !aligned(ws, kWsAlign))
        return EP_ERR_INVALID_ARG;
    if (T > 0 && (x == nullptr || topk_idx == nullptr || slot == nullptr || !aligned(x, 16)))
        return EP_ERR_INVALID_ARG;
    if ((int64_t)E_local * M > 0 &&
        (b_x == nullptr || !aligned(b_x, 16) || (sp != nullptr && (sp->out == nullptr || !aligned(sp->out, 4)))))
        return EP_ERR_INVALID_ARG;
    // the kept counts live at the end of the workspace; the slot launchers
    // take what is before them
    const size_t kept_bytes = align_up((size_t)E_local * sizeof(int32_t), kWsAlign);
    if (ws_bytes < kWsAlign + (size_t)ceil_div(T, kRouteThreads) * E_local * sizeof(int32_t) + kept_bytes)
        return EP_ERR_INVALID_ARG;
    const size_t slot_ws = (ws_bytes - kept_bytes) / kWsAlign * kWsAlign;
    int32_t *kept = reinterpret_cast<int32_t *>(static_cast<char *>(ws) + slot_ws);

    const SlotLimits lim{M, capacity > 0 ? capacity : M, capacity > 0, alignment, dropped, kept};
    // the slot kernel, then the row scatter as its dependent; where the slot
    // kernel has a grid-wide wait, its blocks ask the L2 for the rows the
    // bf16 scatter reads (up to three quarters of it) while they wait
    const int64_t row_bytes = (int64_t)H * 2;
    const RowPrefetch pf{sp == nullptr ? x : nullptr, row_bytes,
                         std::min<int64_t>(T, device_l2_bytes() / 4 * 3 / row_bytes)};
    int rc = launch_batched_slots(topk_idx, T, K, E, E_local, rank, lim, tokens_per_expert, slot, ws, slot_ws, err,
                                  stream, pf);
    if (rc != EP_OK)
        return rc;
    if (T > 0) {
        const BatchedRows rows{topk_idx, slot, nullptr, K, (int64_t)rank * E_local, E_local, M, true};
        const int64_t n_rows = (int64_t)E_local * M;
        // the slot kernel just enqueued writes nothing the scatter reads early
        rc = sp == nullptr ? launch_scatter_bf16(x, T, H, rows, n_rows, EP_ERR_CAPACITY, b_x, err, stream, true)
                           : launch_scatter_fp8(x, T, H, rows, n_rows, EP_ERR_CAPACITY, b_x, *sp, err, stream, true);
        if (rc != EP_OK)
            return rc;
    }
    // zero rows: the alignment rows [kept, aligned) always, the rest with zero_pad
    if ((zero_pad || alignment > 1) && M > 0) {
        const int nvec = sp == nullptr ? H / 8 : H / 16;   // 16-byte vectors per row
        // rows an expert may need zeroed: all of them with zero_pad, else
        // only the alignment rows (fewer than `alignment`)
        const int64_t zrows = zero_pad ? M : std::min<int64_t>(alignment - 1, M);
        dim3 grid((unsigned)std::max<int64_t>(1, std::min<int64_t>(ceil_div(zrows * nvec, 256), 1024)), E_local);
        // dependents of the scatter when there is one (see zero_rows_kernel)
        const bool dep = T > 0;
        if (launch_kernel(dep, zero_rows_kernel, grid, dim3(256), 0, stream, static_cast<uint4 *>(b_x),
                          (const int32_t *)kept, (const int32_t *)tokens_per_expert, zero_pad, M, nvec) != cudaSuccess) {
            cudaGetLastError();
            return EP_ERR_CUDA;
        }
        if (sp != nullptr) {
            dim3 sgrid((unsigned)std::max<int64_t>(1, std::min<int64_t>(ceil_div(zrows * (H / 128), 256), 256)),
                       E_local);
            if (launch_kernel(dep, zero_scales_kernel, sgrid, dim3(256), 0, stream, *sp, (const int32_t *)kept,
                              (const int32_t *)tokens_per_expert, zero_pad, H / 128) != cudaSuccess) {
                cudaGetLastError();
                return EP_ERR_CUDA;
            }
        }
    }
    return EP_OK;
}

static int scale_spec(int scale_fmt, int round_scale, int H, void *b_scale, int M, ScaleSpec *sp)
{
    if (scale_fmt != EP_SCALE_ROW_F32 && scale_fmt != EP_SCALE_COL_F32 && scale_fmt != EP_SCALE_COL_UE8M0)
        return EP_ERR_INVALID_ARG;
    if (round_scale != 0 && round_scale != 1)
        return EP_ERR_INVALID_ARG;
    if (H % 128 != 0 || (scale_fmt == EP_SCALE_COL_UE8M0 && (!round_scale || H % 512 != 0)))
        return EP_ERR_UNSUPPORTED;
    *sp = ScaleSpec{b_scale, scale_fmt, round_scale, M};
    return EP_OK;
}

extern "C" int ep_batched_prepare_ex(const void *x, const int64_t *topk_idx, int64_t T, int K, int H, int E,
                                     int E_local, int rank, int max_num_tokens, int capacity, int alignment,
                                     void *b_rows, void *b_scale, int scale_fmt, int round_scale,
                                     int32_t *tokens_per_expert, int32_t *slot, int32_t *dropped, int zero_pad,
                                     void *ws, size_t ws_bytes, int32_t *err, ep_stream_t stream)
{
    ScaleSpec sp{};
    if (scale_fmt >= 0) {
        const int rc = scale_spec(scale_fmt, round_scale, H, b_scale, max_num_tokens, &sp);
        if (rc != EP_OK)
            return rc;
    } else if (scale_fmt != -1) {
        return EP_ERR_INVALID_ARG;
    }
    return batched_prepare(x, topk_idx, T, K, H, E, E_local, rank, max_num_tokens, capacity, alignment, b_rows,
                           scale_fmt >= 0 ? &sp : nullptr, tokens_per_expert, slot, dropped, zero_pad, ws, ws_bytes,
                           err, reinterpret_cast<cudaStream_t>(stream));
}

extern "C" int64_t ep_expert_capacity(int64_t T, int K, int E, double factor)
{
    if (T < 0 || K < 1 || E < 1 || !(factor > 0.0))
        return -1;
    return (int64_t)ceil(factor * (double)T * (double)K / (double)E);
}

extern "C" int ep_batched_prepare(const void *x, const int64_t *topk_idx, int64_t T, int K, int H, int E,
                                  int E_local, int rank, int max_num_tokens, void *b_x,
                                  int32_t *tokens_per_expert, int32_t *slot, int zero_pad, void *ws,
                                  size_t ws_bytes, int32_t *err, ep_stream_t stream)
{
    return batched_prepare(x, topk_idx, T, K, H, E, E_local, rank, max_num_tokens, 0, 1, b_x, nullptr,
                           tokens_per_expert, slot, nullptr, zero_pad, ws, ws_bytes, err,
                           reinterpret_cast<cudaStream_t>(stream));
}

extern "C" int ep_batched_prepare_fp8(const void *x, const int64_t *topk_idx, int64_t T, int K, int H, int E,
                                      int E_local, int rank, int max_num_tokens, uint8_t *b_q, void *b_scale,
                                      int scale_fmt, int round_scale, int32_t *tokens_per_expert, int32_t *slot,
                                      int zero_pad, void *ws, size_t ws_bytes, int32_t *err, ep_stream_t stream)
{
    ScaleSpec sp{};
    const int rc = scale_spec(scale_fmt, round_scale, H, b_scale, max_num_tokens, &sp);
    if (rc != EP_OK)
        return rc;
    return batched_prepare(x, topk_idx, T, K, H, E, E_local, rank, max_num_tokens, 0, 1, b_q, &sp,
                           tokens_per_expert, slot, nullptr, zero_pad, ws, ws_bytes, err,
                           reinterpret_cast<cudaStream_t>(stream));
}

namespace ep {
int launch_local_expert_fp8(const uint8_t *recv_q, const float *recv_scale, const int64_t *send_idx,
                            const float *send_w, int64_t N, const int32_t *n_rows, int K, int H, void *out,
                            cudaStream_t stream)
{
    if (N < 0 || N >= ((int64_t)1 << 31) || K < 1 || K > EP_MAX_TOPK || H < 128 || H % 128 != 0)
        return EP_ERR_INVALID_ARG;
    if (N == 0)
        return EP_OK;
    if (recv_q == nullptr || recv_scale == nullptr || send_idx == nullptr || send_w == nullptr ||
        out == nullptr || !aligned(recv_q, 16) || !aligned(out, 16))
        return EP_ERR_INVALID_ARG;
    local_expert_fp8_kernel<<<(unsigned)ceil_div(N, kLocalRowsPerBlock), kLocalRowsPerBlock * 32, 0, stream>>>(
        reinterpret_cast<const uint4 *>(recv_q), recv_scale, send_idx, send_w, N, n_rows, K, H,
        static_cast<uint4 *>(out));
    return launch_status();
}
}  // namespace ep

extern "C" int ep_local_expert_fp8(const uint8_t *recv_q, const float *recv_scale, const int64_t *send_idx,
                                   const float *send_w, int64_t N, int K, int H, void *out, int32_t *err,
                                   ep_stream_t stream_)
{
    (void)err;
    return launch_local_expert_fp8(recv_q, recv_scale, send_idx, send_w, N, nullptr, K, H, out,
                                   reinterpret_cast<cudaStream_t>(stream_));
}
