// Row lists of the two layouts (internal to libep_gb300): for a token t, the
// rows it is sent to (scatter) or gathered from (combine), in the order the
// reduction uses.
#pragma once

#include <climits>
#include <cstdint>

namespace ep {

constexpr int kMaxList = 64;   // >= max(P, K)

// Send layout: the rows of token t are token_pos[t, p] (p ascending), -1 = none.
struct SendRows {
    const int32_t *token_pos;
    int P;
    __host__ __device__ __forceinline__ int len() const { return P; }
    __device__ __forceinline__ int32_t row(int64_t t, int j) const { return token_pos[t * P + j]; }
    __device__ __forceinline__ float weight(int64_t, int) const { return 1.0f; }
    // Split lookup for prefetching: load() only issues loads, decode() uses them.
    struct Raw {
        int32_t pos;
    };
    __device__ __forceinline__ Raw load(int64_t t, int j) const { return Raw{token_pos[t * P + j]}; }
    __device__ __forceinline__ int32_t decode(const Raw &r) const { return r.pos; }
    __device__ __forceinline__ float weight(const Raw &) const { return 1.0f; }
};

// Expert-batched layout: slot k of token t names local expert e_l and slot s:
// row e_l * M + s.  `dedup` drops a slot naming the same expert as an earlier
// slot of the token (the scatter writes each (expert, token) row once; the
// weighted combine keeps every slot's term).
struct BatchedRows {
    const int64_t *idx;
    const int32_t *slot;
    const float *w;
    int K;
    int64_t e0;
    int E_local;
    int M;
    bool dedup;
    __host__ __device__ __forceinline__ int len() const { return K; }
    __device__ __forceinline__ int32_t row(int64_t t, int j) const
    {
        const int32_t s = slot[t * K + j];
        const int64_t id = idx[t * K + j];
        const int64_t el = id - e0;
        if (s < 0 || el < 0 || el >= E_local)
            return -1;
        if (s >= M)                     // not a slot of this layout: reported by the caller
            return INT32_MAX;
        if (dedup)
            for (int i = 0; i < j; ++i)
                if (idx[t * K + i] == id)
                    return -1;
        return (int32_t)(el * M + s);
    }
    __device__ __forceinline__ float weight(int64_t t, int j) const { return w ? w[t * K + j] : 1.0f; }
    // Split lookup for prefetching (no dedup: the combine keeps every slot).
    struct Raw {
        int32_t s;
        int64_t id;
        float w;
    };
    __device__ __forceinline__ Raw load(int64_t t, int j) const
    {
        return Raw{slot[t * K + j], idx[t * K + j], w ? w[t * K + j] : 1.0f};
    }
    __device__ __forceinline__ int32_t decode(const Raw &r) const
    {
        const int64_t el = r.id - e0;
        if (r.s < 0 || el < 0 || el >= E_local)
            return -1;
        if (r.s >= M)
            return INT32_MAX;
        return (int32_t)(el * M + r.s);
    }
    __device__ __forceinline__ float weight(const Raw &r) const { return r.w; }
};

}  // namespace ep
