// Check of the timeout path every tensor-core kernel takes when one of its
// mbarrier waits gives up: a one-thread kernel waits on a barrier that
// nothing completes, with a short limit, and so sets the abort flag and the
// timeout bit of the status word exactly as a stuck copy or MMA would.  The
// host then sees the step fail through dp_step_status and the gradient
// kernels skip their writes.  The wait is bounded, nothing faults.
#include "../../include/dp_clip.h"
#include "internal.h"
#include "tc_common.cuh"

namespace {

__global__ void k_wait_expires(unsigned* status, uint64_t limit_ns) {
    __shared__ uint64_t bar;
    __shared__ int abort_flag;
    tc::mbar_init(&bar, 1);
    abort_flag = 0;
    tc::fence_barrier_init();
    // phase 0 of a fresh barrier whose one arrival never comes
    tc::mbar_wait_for(&bar, 0, &abort_flag, status, limit_ns);
}

}  // namespace

cudaError_t launch_wait_expiry(unsigned* status, uint64_t limit_ns, cudaStream_t s) {
    k_wait_expires<<<1, 1, 0, s>>>(status, limit_ns);
    count_launch(KL_WAIT_EXPIRES);
    return cudaGetLastError();
}
