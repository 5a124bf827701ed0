// Test harness, not part of the library: CUDA's own fp32 -> fp8 e4m3
// conversion (round to nearest even, saturating to +-448; OCP OFP8 E4M3, the
// fp8 payload of NeMo uccl_ep.buffer, Buffer.dispatch) applied to a range of
// fp32 bit patterns, so that a test can compare the oracle's encoder with the
// device's conversion over every pattern.
//   cvt_e4m3_range: out_pair[i] = the pair conversion (the form the library's
//   quantising kernels use) of the pattern start + i, taken two at a time;
//   out_single[i] = the single-value conversion of the same pattern.  n must
//   be even; both outputs hold n bytes on the device.
#include <cstdint>

#include <cuda_fp8.h>
#include <cuda_runtime.h>

namespace {

__global__ void cvt_e4m3_kernel(uint32_t start, uint64_t n, uint8_t *out_pair, uint8_t *out_single)
{
    const uint64_t pairs = n / 2;
    const uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
    for (uint64_t p = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; p < pairs; p += stride) {
        const uint32_t b0 = start + (uint32_t)(2 * p);
        const float2 v = make_float2(__uint_as_float(b0), __uint_as_float(b0 + 1u));
        const __nv_fp8x2_storage_t q = __nv_cvt_float2_to_fp8x2(v, __NV_SATFINITE, __NV_E4M3);
        reinterpret_cast<uint16_t *>(out_pair)[p] = (uint16_t)q;   // .x in the low byte
        out_single[2 * p] = (uint8_t)__nv_cvt_float_to_fp8(v.x, __NV_SATFINITE, __NV_E4M3);
        out_single[2 * p + 1] = (uint8_t)__nv_cvt_float_to_fp8(v.y, __NV_SATFINITE, __NV_E4M3);
    }
}

}  // namespace

// Returns the CUDA error of the launch (0 on success); asynchronous on stream.
extern "C" int cvt_e4m3_range(uint32_t start, uint64_t n, void *out_pair, void *out_single, void *stream)
{
    if (n % 2 != 0 || out_pair == nullptr || out_single == nullptr)
        return (int)cudaErrorInvalidValue;
    if (n == 0)
        return 0;
    const uint64_t pairs = n / 2;
    const unsigned threads = 256;
    const uint64_t want = (pairs + threads - 1) / threads;
    const unsigned blocks = (unsigned)(want < 4096 ? want : 4096);
    cvt_e4m3_kernel<<<blocks, threads, 0, static_cast<cudaStream_t>(stream)>>>(
        start, n, static_cast<uint8_t *>(out_pair), static_cast<uint8_t *>(out_single));
    return (int)cudaGetLastError();
}
