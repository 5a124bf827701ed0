// Host-side helpers shared by the translation units of libep_gb300.
#pragma once

#include <atomic>
#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include "ep.h"

namespace ep {

constexpr int kRouteThreads = 256;   // = tokens per routing block
constexpr size_t kWsAlign = 256;

inline bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }
inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }
inline int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Launch status of the most recent kernel launch on this thread.
inline int launch_status()
{
    return cudaGetLastError() == cudaSuccess ? EP_OK : EP_ERR_CUDA;
}

// The current device (cudaGetDevice), or -1 if there is none.
int current_device();

// A non-negative value kept per device after its first lookup.  Function
// attributes belong to the context of the device that was current when they
// were set, and device attributes and occupancies may differ between
// devices, so the launch policies keep theirs per device.  Zero-initialised
// storage reads as "not yet known" (the value is stored plus one); devices
// past kMaxDevices are not cached.  Concurrent first calls may both look the
// value up and store the same result.
constexpr int kMaxDevices = 64;
class PerDevice {
public:
    int get(int dev) const   // -1 if not yet known
    {
        return dev >= 0 && dev < kMaxDevices ? v_[dev].load(std::memory_order_relaxed) - 1 : -1;
    }
    void put(int dev, int v)
    {
        if (dev >= 0 && dev < kMaxDevices)
            v_[dev].store(v + 1, std::memory_order_relaxed);
    }

private:
    std::atomic<int> v_[kMaxDevices];
};

// Attributes of the current device, read on its first use and kept.
int device_sm_count();        // streaming multiprocessors (152 if unreadable)
int64_t device_l2_bytes();    // L2 cache size in bytes (0 if unreadable)

// Upper bound on routing blocks for T tokens split into `chunks` ranges.
inline int64_t route_blocks_max(int64_t T, int chunks)
{
    return ceil_div(T, kRouteThreads) + (chunks > 1 ? chunks : 1);
}

// Per-chunk block decomposition for the routing kernels: block b belongs to
// the chunk c with first_block[c] <= b < first_block[c+1] and covers tokens
// start[c] + (b - first_block[c]) * 256 ... (clipped to start[c+1]).
struct ChunkTable {
    int n;
    int first_block[EP_MAX_CHUNKS + 1];
    int64_t start[EP_MAX_CHUNKS + 1];
};

// Per-expert slot limits of the expert-batched layout.
struct SlotLimits {
    int M;              // rows per expert in the layout
    int cap;            // slots kept per expert (<= M); later tokens are dropped
    int silent;         // drops past cap are the capacity's purpose (no error bit)
    int align;          // tokens_per_expert = min(round_up(kept, align), M)
    int32_t *dropped;   // [E_local] tokens dropped per expert, or null
    int32_t *kept;      // [E_local] tokens kept per expert, or null
};

// Rows that a routing kernel asks the L2 to fetch while its blocks wait for
// one another, for the kernel that moves them next: the rows t < tokens of
// x (row_bytes each, 16-byte aligned) that have a destination.  x == nullptr:
// none.
struct RowPrefetch {
    const void *x;
    int64_t row_bytes;
    int64_t tokens;
};

// Launchers implemented in ep_route.cu and used by the batched entry points.
// The workspace [ws, ws + ws_bytes) is theirs.
int launch_batched_slots(const int64_t *topk_idx, int64_t T, int K, int E, int E_local, int rank,
                         const SlotLimits &lim, int32_t *tokens_per_expert, int32_t *slot,
                         void *ws, size_t ws_bytes, int32_t *err, cudaStream_t stream,
                         const RowPrefetch &pf = RowPrefetch{});

// ep_dispatch (ep_move.cu); dependent = launch the scatter as a programmatic
// dependent of the kernel the library enqueued just before it.
int dispatch_rows(const void *x, int64_t T, int H, const int32_t *token_pos, int P, int64_t num_send,
                  void *recv_x, float *recv_scale, int fp8, int32_t *err, cudaStream_t stream, bool dependent);

// The synthetic fp8 expert over N rows (ep_move.cu); with n_rows non-NULL,
// rows at or past the device value *n_rows are skipped.
int launch_local_expert_fp8(const uint8_t *recv_q, const float *recv_scale, const int64_t *send_idx,
                            const float *send_w, int64_t N, const int32_t *n_rows, int K, int H, void *out,
                            cudaStream_t stream);

}  // namespace ep
