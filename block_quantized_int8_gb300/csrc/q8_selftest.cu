// q8_selftest.cu -- a check of the kernels' failure path that needs no fault.
//
// Every wait in the kernels of this library is an mbarrier wait bounded by
// the global timer; on expiry the kernel ORs Q8_DEV_TIMEOUT into the caller's
// status word and returns, so the context stays usable.  This kernel runs
// that same bounded wait on an mbarrier that nothing ever arrives on, with a
// caller-chosen limit, and reports the status bit and the time it waited.
#include "q8_dev.cuh"
#include "q8_internal.h"

namespace q8 {

namespace {

__global__ void wait_timeout_kernel(uint64_t limit_ns, uint32_t *status, uint64_t *elapsed_ns) {
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        fence_mbar_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        const uint64_t t0 = globaltimer_ns();
        const bool ok = mbar_wait_bounded(&bar, 0, limit_ns);  // nobody arrives
        const uint64_t t1 = globaltimer_ns();
        if (!ok && status) atomicOr(status, Q8_DEV_TIMEOUT);
        if (elapsed_ns) *elapsed_ns = t1 - t0;
    }
}

}  // namespace

q8_status launch_selftest_wait_timeout(uint64_t limit_ns, uint32_t *status, uint64_t *elapsed_ns,
                                       cudaStream_t stream) {
    wait_timeout_kernel<<<1, 32, 0, stream>>>(limit_ns, status, elapsed_ns);
    return cudaGetLastError() == cudaSuccess ? Q8_OK : Q8_ERR_CUDA;
}

}  // namespace q8
