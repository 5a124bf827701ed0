// Test harness, not part of the library: runs the library's bounded mbarrier
// wait (the one the combine's bulk-copy ring uses) on a barrier phase that
// nothing completes, or on one that completes, so that a test can check that
// the time limit ends the wait with a status the host reads, without a fault
// or a hang.  One block, thread 0 only; it completes the phase itself before
// exiting, so no barrier is left pending.
#include "ep_device.cuh"

namespace {

__global__ void wait_probe_kernel(unsigned long long limit_ns, int complete_first, int32_t *status,
                                  unsigned long long *elapsed_ns)
{
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x == 0) {
        ep::mbar_init(&bar, 1);
        ep::fence_mbar_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        if (complete_first)
            ep::mbar_arrive(&bar);
        const uint64_t t0 = ep::global_timer_ns();
        const bool ok = ep::mbar_wait(&bar, 0, limit_ns);
        *elapsed_ns = ep::global_timer_ns() - t0;
        *status = ok ? EP_OK : EP_ERR_TIMEOUT;
        if (!ok)
            ep::mbar_arrive(&bar);
    }
}

}  // namespace

// Returns the CUDA error of the launch and synchronisation (0 on success);
// *status is EP_OK or EP_ERR_TIMEOUT, *elapsed_ns the wait's duration.
extern "C" int wait_probe(unsigned long long limit_ns, int complete_first, int32_t *status,
                          unsigned long long *elapsed_ns)
{
    int32_t *d_status = nullptr;
    unsigned long long *d_elapsed = nullptr;
    cudaError_t e = cudaMalloc(&d_status, sizeof(int32_t));
    if (e == cudaSuccess)
        e = cudaMalloc(&d_elapsed, sizeof(unsigned long long));
    if (e == cudaSuccess) {
        wait_probe_kernel<<<1, 32>>>(limit_ns, complete_first, d_status, d_elapsed);
        e = cudaGetLastError();
    }
    if (e == cudaSuccess)
        e = cudaDeviceSynchronize();
    if (e == cudaSuccess)
        e = cudaMemcpy(status, d_status, sizeof(int32_t), cudaMemcpyDeviceToHost);
    if (e == cudaSuccess)
        e = cudaMemcpy(elapsed_ns, d_elapsed, sizeof(unsigned long long), cudaMemcpyDeviceToHost);
    cudaFree(d_status);
    cudaFree(d_elapsed);
    return (int)e;
}
