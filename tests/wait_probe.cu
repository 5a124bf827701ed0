// Test harness, not part of the library: runs the library's bounded waits on
// something that never happens, so that a test can check that the time limit
// ends the wait with a status the host reads, without a fault or a hang.
//   wait_probe:    the mbarrier wait of the combine's bulk-copy ring, on a
//                  phase that nothing completes (or on a completed one).  One
//                  block, thread 0 only; it completes the phase itself before
//                  exiting, so no barrier is left pending.
//   barrier_probe: the grid barrier of the cooperative routing kernels, in a
//                  cooperative launch of two blocks of which one may leave
//                  without arriving.
#include "ep_barrier.cuh"
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

__global__ void barrier_probe_kernel(ep::GridBarrier bar, int absent_block, int32_t *status)
{
    __shared__ int s_fail;
    __shared__ unsigned long long s_tag, s_epoch;
    if (threadIdx.x == 0) {
        s_fail = 0;
        s_tag = ep::barrier_tag(bar, &s_epoch);
    }
    __syncthreads();
    if ((int)blockIdx.x == absent_block)
        return;   // this block never arrives
    if (threadIdx.x == 0)
        ep::barrier_arrive(bar, s_tag);
    const bool ok = ep::barrier_wait(bar, s_tag, s_epoch, &s_fail);
    if (threadIdx.x == 0)
        status[blockIdx.x] = ok ? EP_OK : EP_ERR_TIMEOUT;
}

}  // namespace

// Two blocks of 32 threads in one cooperative launch; block absent_block (or
// none, -1) leaves before arriving.  status[2] receives each waiting block's
// EP_OK / EP_ERR_TIMEOUT (-1 for a block that left).  Returns the CUDA error
// of the launch and synchronisation (0 on success).
extern "C" int barrier_probe(int absent_block, unsigned long long host_tag, int32_t *status)
{
    unsigned long long *d_words = nullptr;   // [flag 0, flag 1, launch counter]
    int32_t *d_status = nullptr;
    cudaError_t e = cudaMalloc(&d_words, 3 * sizeof(unsigned long long));
    if (e == cudaSuccess)
        e = cudaMemset(d_words, 0, 3 * sizeof(unsigned long long));
    if (e == cudaSuccess)
        e = cudaMalloc(&d_status, 2 * sizeof(int32_t));
    if (e == cudaSuccess)
        e = cudaMemset(d_status, 0xff, 2 * sizeof(int32_t));
    if (e == cudaSuccess) {
        ep::GridBarrier bar{d_words, d_words + 2, host_tag};
        void *args[] = {&bar, &absent_block, &d_status};
        e = cudaLaunchCooperativeKernel((const void *)barrier_probe_kernel, dim3(2), dim3(32), args, 0, 0);
    }
    if (e == cudaSuccess)
        e = cudaDeviceSynchronize();
    if (e == cudaSuccess)
        e = cudaMemcpy(status, d_status, 2 * sizeof(int32_t), cudaMemcpyDeviceToHost);
    cudaFree(d_words);
    cudaFree(d_status);
    return (int)e;
}

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
