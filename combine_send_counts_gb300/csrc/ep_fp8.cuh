// fp8 (1x128) group quantisation of libep_gb300 (internal, not part of the C
// ABI): where the group scales go, and the quantisation of one chunk of a
// bf16 row by one warp.  NeMo uccl_ep.buffer, Buffer.dispatch (fp8 payload:
// e4m3 codes with one fp32 scale per 128 columns) and Buffer.low_latency_dispatch
// (column-major scales, power-of-two scales, UE8M0 codes).
#pragma once

#include <cstdint>

#include "ep_device.cuh"

namespace ep {

// Where and how the group scales go: the layout (EP_SCALE_*) and whether the
// scales are powers of two.  Column-major layouts index destination row
// r = e * M + s as (e, s).
struct ScaleSpec {
    void *out;
    int fmt;
    int round;
    int M;
};

// Index of group 0's scale of destination row r (4-byte entries; bytes for
// UE8M0), computed once per row; put_scale adds the group's offset.
template <int SF>
__device__ __forceinline__ int64_t scale_row_base(const ScaleSpec &sp, int32_t r, int groups)
{
    if (SF == EP_SCALE_ROW_F32)
        return (int64_t)r * groups;
    const int e = r / sp.M, s = r - e * sp.M;
    if (SF == EP_SCALE_COL_F32)
        return (int64_t)e * groups * sp.M + s;
    return ((int64_t)e * (groups >> 2) * sp.M + s) * 4;
}

template <int SF>
__device__ __forceinline__ void put_scale(const ScaleSpec &sp, int64_t base, int gi, float sc, uint32_t code)
{
    if (SF == EP_SCALE_ROW_F32)
        static_cast<float *>(sp.out)[base + gi] = sc;
    else if (SF == EP_SCALE_COL_F32)
        static_cast<float *>(sp.out)[base + (int64_t)gi * sp.M] = sc;
    else
        static_cast<uint8_t *>(sp.out)[base + (int64_t)(gi >> 2) * sp.M * 4 + (gi & 3)] = (uint8_t)code;
}

// Group maxima of one chunk.  m[u] is a lane's own maximum over the 8 values
// of its vector u; a group is vector u of the 16 lanes of one half-warp.  The
// first log2(U) butterfly steps each hand half of a lane's values to its
// partner, so that lane l ends with the whole maximum of group
// u = (l >> 2) & 3 (U = 4) or (l >> 3) & 1 (U = 2) of its half-warp after
// U + 3 shuffles (instead of 4U).  max is exact, so the order of the steps
// does not change the value.
template <int U>
__device__ __forceinline__ float half_warp_group_max(const float (&m)[U], int lane)
{
    static_assert(U == 2 || U == 4, "two or four vectors per lane");
    float k;
    if constexpr (U == 4) {
        const bool b3 = lane & 8, b2 = lane & 4;
        const float k0 = fmaxf(b3 ? m[2] : m[0], __shfl_xor_sync(kFull, b3 ? m[0] : m[2], 8));
        const float k1 = fmaxf(b3 ? m[3] : m[1], __shfl_xor_sync(kFull, b3 ? m[1] : m[3], 8));
        k = fmaxf(b2 ? k1 : k0, __shfl_xor_sync(kFull, b2 ? k0 : k1, 4));
    } else {
        const bool b3 = lane & 8;
        k = fmaxf(b3 ? m[1] : m[0], __shfl_xor_sync(kFull, b3 ? m[0] : m[1], 8));
        k = fmaxf(k, __shfl_xor_sync(kFull, k, 4));
    }
    k = fmaxf(k, __shfl_xor_sync(kFull, k, 2));
    return fmaxf(k, __shfl_xor_sync(kFull, k, 1));
}

// the vector u whose group maximum lane l holds after half_warp_group_max
template <int U>
__device__ __forceinline__ int group_owner_u(int lane)
{
    return U == 4 ? (lane >> 2) & 3 : (lane >> 3) & 1;
}

// One chunk of a row, quantised by one warp: lane l holds vectors l, l + 32,
// ..., l + 32 (U - 1) of the chunk (eight bf16 values each; vectors past the
// row are zeros, whole half-warps of them); lanes 0-15 and 16-31 each hold
// one 128-element group per u.  q[u] receives the lane's eight e4m3 codes of
// vector u.  The 2U group maxima end up one per lane quad (U = 4) or octet
// (U = 2) (half_warp_group_max); the lane holding group u_own's maximum
// (group_owner_u) gets its scale (and UE8M0 code) in scale_own / code_own,
// and each group's reciprocal reaches its lanes by one shuffle per vector.
// With a = max(max|x|, 1e-4):
//   plain (RS = false): q = e4m3_rn_satfinite(x * (448 / a)), scale = a / 448;
//   power of two:       scale = 2^e, the smallest power of two >= a / 448 (from
//                       the bits of the fp32 quotient), q = e4m3_rn_satfinite(x * 2^-e),
//                       UE8M0 code e + 127.
// NaN elements do not enter the maximum (fmaxf).  A group holding +-inf has
// a = inf: scale +inf and reciprocal +0 in both forms (UE8M0 code 255), so
// its finite elements give +-0 and its infinities NaN codes.
template <int U, bool RS>
__device__ __forceinline__ void quantize_chunk(const uint4 (&vin)[U], int lane, uint2 (&q)[U], float &scale_own,
                                               uint32_t &code_own)
{
    float m[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {   // vectors past the row are whole half-warps of zeros
        const uint32_t w[4] = {vin[u].x, vin[u].y, vin[u].z, vin[u].w};
        m[u] = 0.0f;
#pragma unroll
        for (int e = 0; e < 4; ++e)
            m[u] = fmaxf(m[u], fmaxf(fabsf(bf16_lo(w[e])), fabsf(bf16_hi(w[e]))));
    }
    // this lane's group: its scale (and UE8M0 code) and the reciprocal
    const float a = fmaxf(half_warp_group_max<U>(m, lane), 1e-4f);
    float inv_own;
    code_own = 0;
    if (RS) {
        const uint32_t b = __float_as_uint(__fdiv_rn(a, 448.0f));
        const uint32_t eb = (b >> 23) + ((b & 0x7fffffu) != 0u);
        scale_own = __uint_as_float(eb << 23);
        inv_own = eb < 255u ? __uint_as_float((254u - eb) << 23) : 0.0f;   // a = inf: 1 / inf
        code_own = eb;
    } else {
        inv_own = __fdiv_rn(448.0f, a);
        scale_own = __fdiv_rn(a, 448.0f);
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
        const float inv = __shfl_sync(kFull, inv_own, (lane & 16) | (U == 4 ? u << 2 : u << 3));
        const float2 inv2 = make_float2(inv, inv);
        const uint32_t w[4] = {vin[u].x, vin[u].y, vin[u].z, vin[u].w};
        uint32_t packed[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float2 pr = mul2_rn(make_float2(bf16_lo(w[e]), bf16_hi(w[e])), inv2);
            packed[e] = (uint32_t)__nv_cvt_float2_to_fp8x2(pr, __NV_SATFINITE, __NV_E4M3);
        }
        q[u] = make_uint2(packed[0] | (packed[1] << 16), packed[2] | (packed[3] << 16));
    }
}

}  // namespace ep
