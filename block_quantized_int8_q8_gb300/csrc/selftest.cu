// selftest.cu -- device self-test of the bounded waits every pipeline in this library relies on.
//
// CTA 0 waits with mbar_wait, CTA 1 with mbar_wait_relaxed, each on a shared-memory mbarrier that
// nothing ever arrives at.  Both waits must give up after the library's time limit, raise their CTA's
// abort flag, record MMQ_DEVERR_TIMEOUT in the device error word and return; the kernel then exits
// normally, so the context stays usable.  No fault and no unbounded wait is involved.
#include <cstdint>
#include "internal.h"
#include "mmq_device.cuh"

namespace mmq {

__global__ void wait_timeout_selftest_kernel(int* result) {
    __shared__ __align__(8) uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&bar), 1);
        abort_flag = 0;
        fence_barrier_init();
    }
    __syncthreads();
    bool completed = true;
    if (threadIdx.x == 0) {
        volatile int* flag = &abort_flag;
        completed = blockIdx.x == 0 ? mbar_wait(smem_u32(&bar), 0, flag) : mbar_wait_relaxed(smem_u32(&bar), 0, flag);
        result[2 * blockIdx.x] = completed ? 1 : 0;
        result[2 * blockIdx.x + 1] = *flag;
    }
}

cudaError_t run_wait_timeout_selftest(int* result, cudaStream_t s) {
    wait_timeout_selftest_kernel<<<2, 32, 0, s>>>(result);
    return cudaGetLastError();
}

MMQ_DEFINE_ERROR_READER(selftest)

}  // namespace mmq
