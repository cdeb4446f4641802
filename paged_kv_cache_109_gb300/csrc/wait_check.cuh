// wait_check.cuh -- a one-CTA kernel that exercises the bounded pipeline wait.
//
// Every kernel here synchronises its roles through mbarriers and never waits
// without a bound: after kWaitLimitCycles a wait gives up, the kernel raises
// PA_DEVERR_TIMEOUT and returns, so a copy that never lands cannot hang the
// GPU.  This kernel runs the same helpers on a barrier that may be left
// short of its arrivals, with a caller-chosen (short) bound, so the timeout
// path can be checked on a live GPU: the wait gives up, the bit is raised and
// the context stays usable.
#pragma once

#include "common.cuh"
#include "ptx.cuh"

namespace pa {

// `expected` arrivals complete the barrier's first phase; threads 0 ..
// arrivals - 1 arrive once each (arrivals <= expected <= blockDim.x), then
// every thread waits for the phase with the given bound.
__global__ void wait_check_kernel(int32_t expected, int32_t arrivals, long long limit_cycles) {
    __shared__ uint64_t bar;
    const uint32_t b = smem_u32(&bar);
    if (threadIdx.x == 0) {
        mbar_init(b, (uint32_t)expected);
        mbar_fence_init();
    }
    __syncthreads();
    if ((int32_t)threadIdx.x < arrivals) mbar_arrive(b);
    const bool done = mbar_wait_bounded(b, 0, limit_cycles);
    if (!done && threadIdx.x == 0) raise_error(PA_DEVERR_TIMEOUT);
}

}  // namespace pa
