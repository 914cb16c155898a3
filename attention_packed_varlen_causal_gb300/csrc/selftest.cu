// selftest.cu -- diagnostic kernel for the failure path of the pipeline waits.
//
// Every pipeline wait of the attention kernels goes through bg::mbar_wait, which gives up
// after kWaitTimeoutNs instead of spinning forever.  This kernel makes exactly such a wait
// run out -- an mbarrier that nothing ever arrives on -- so that a test can check, on a real
// GPU and without faulting or hanging it, that the wait ends, that BG_DEVSTAT_TIMEOUT reaches
// the host, and that the context stays usable afterwards.
#include "bg_internal.h"
#include "bg_ptx.cuh"

namespace bg {

namespace {
__global__ void wait_timeout_kernel(int32_t *dev_status, unsigned long long *waited_ns)
{
    __shared__ uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);      // phase 0 needs one arrive; none ever comes
        abort_flag = 0;
        fence_barrier_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        const uint64_t t0 = globaltimer_ns();
        const bool completed = mbar_wait(&bar, 0, &abort_flag);
        const uint64_t t1 = globaltimer_ns();
        if (!completed && dev_status) atomicOr(dev_status, BG_DEVSTAT_TIMEOUT);
        if (waited_ns) *waited_ns = static_cast<unsigned long long>(t1 - t0);
    }
}
}  // namespace

cudaError_t launch_wait_timeout_selftest(int32_t *dev_status, unsigned long long *waited_ns, cudaStream_t stream)
{
    wait_timeout_kernel<<<1, 32, 0, stream>>>(dev_status, waited_ns);
    return cudaGetLastError();
}

}  // namespace bg
