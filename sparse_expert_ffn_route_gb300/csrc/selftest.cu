// selftest.cu -- exercises the error path of the library's bounded device-side waits without
// faulting or hanging the GPU: one CTA waits, a bounded number of polls, on an mbarrier that
// nothing arrives at, gives up and records kErrTimeout in the workspace error word, the same
// way the tensor-core pipeline's waits do.  The host reads the word with moe_check_errors.
#include "device_util.cuh"
#include "launch.cuh"
#include "moe_internal.cuh"

namespace moe {

namespace {

__global__ void selftest_wait_kernel(int32_t *err, int polls)
{
    __shared__ uint64_t bar;
    pdl_wait();
    pdl_launch_dependents();
    if (threadIdx.x != 0) return;
    mbar_init(&bar, 1);
    fence_mbar_init();
    // nothing arrives: the phase never completes and every poll fails
    bool done = false;
    for (int n = 0; n < polls && !done; ++n) done = mbar_try_wait(&bar, 0);
    if (!done) atomicOr(err, kErrTimeout);
}

}  // namespace

cudaError_t launch_selftest_wait(int32_t *err, int polls, cudaStream_t st)
{
    return launch_kernel(selftest_wait_kernel, dim3(1), dim3(32), 0, st, 1, err, polls);
}

}  // namespace moe
