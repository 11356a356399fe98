// Self-test of the device-side failure path: a kernel whose wait can never
// be satisfied must give up after its time limit, record
// MDN_ERR_DEVICE_TIMEOUT in the device status word, release what it holds
// and return, leaving the context usable.
//
// One CTA of two warps, shaped like the pipelined kernels: warp 1 owns a
// tensor-memory allocation, both warps wait on an mbarrier that nothing
// arrives at, using the same bounded wait as every other kernel of the
// library.  The first warp to time out sets the CTA's abort flag, the other
// sees it and stops waiting; warp 1 frees the tensor memory, thread 0
// reports the status.
#include "mdn_internal.cuh"
#include "mdn_sm100.cuh"

namespace mdn {
namespace {

using namespace sm100;

__global__ void __launch_bounds__(64, 1)
wait_selftest_kernel(uint64_t limit_ns, int *status) {
    __shared__ uint64_t bar;
    __shared__ uint32_t tmem_base;
    __shared__ int abort_flag;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);          // one arrival expected; none will come
        abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(&tmem_base, 32);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    volatile int *abort = &abort_flag;
    const bool ok = mbar_wait(&bar, 0, abort, limit_ns);
    __syncwarp();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem_base, 32);
    if (threadIdx.x == 0 && status && (!ok || *abort))
        atomicExch(status, (int)MDN_ERR_DEVICE_TIMEOUT);
    (void)lane;
}

}  // namespace

cudaError_t launch_wait_selftest(uint64_t limit_ns, int *status, cudaStream_t st) {
    wait_selftest_kernel<<<1, 64, 0, st>>>(limit_ns, status);
    return cudaGetLastError();
}

}  // namespace mdn
