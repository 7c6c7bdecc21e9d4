// A self-test of the library's bounded waits.
//
// Every wait inside the library's kernels gives up after a time limit, raises
// the device status word and lets the kernel return, so that a stuck pipeline
// surfaces as SLA_ERR_DEVICE_TIMEOUT instead of a hung GPU.  This kernel runs
// that path on purpose in the smallest setting: one thread initialises an
// mbarrier that expects one arrival, never arrives, and waits on it with the
// library's own mbar_wait and a short limit.  Nothing else is in flight, so
// the give-up leaves the device as it was.
#include "launch.h"
#include "tc_ptx.cuh"

namespace sla {
namespace {

__global__ void __launch_bounds__(32) wait_selftest_kernel(unsigned long long limit_ns,
                                                           unsigned* status) {
    __shared__ __align__(8) uint64_t bar;
    __shared__ int abort_word;
    if (threadIdx.x != 0) return;
    volatile int* abort_flag = &abort_word;
    *abort_flag = 0;
    ptx::mbar_init(&bar, 1);
    ptx::fence_mbar_init();
    // phase 0 never completes: the wait runs out, raises kStatusTimeout, and
    // sets the abort word as it would for the other roles of a real kernel
    if (ptx::mbar_wait(&bar, 0, abort_flag, status, limit_ns)) raise_status(status, kStatusLayout);
}

}  // namespace

cudaError_t launch_wait_selftest(unsigned long long limit_ns, unsigned* status,
                                 cudaStream_t stream) {
    wait_selftest_kernel<<<1, 32, 0, stream>>>(limit_ns, status);
    return cudaGetLastError();
}

}  // namespace sla
