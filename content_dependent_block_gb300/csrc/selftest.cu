// Failure-path self-test of the bounded waits (not a step of the method).
//
// Every hand-off in the tensor-core kernels is an mbarrier wait or a wait on
// a counter in global memory, and each gives up after a time limit, records
// BSA_ERR_TIMEOUT in the device status word and lets the kernel return.  This
// kernel runs those same wait functions (tc::mbar_wait, tc::wait_counter) on
// a barrier that no thread arrives on and a counter that no thread raises,
// with a short limit, so that a test can watch the limit run out and the
// kernel come back with the error recorded -- without a fault, a trap or a
// wait that never ends.
#include "bsa_device.cuh"
#include "bsa_internal.h"
#include "tc.cuh"

namespace bsa {
namespace {

// A counter nothing in the library ever writes: it stays 0.
__device__ int32_t g_never_raised = 0;

// One warp.  kind 0: a wait on an mbarrier initialised for one arrival that
// never comes; kind 1: a wait for g_never_raised >= 1.
__global__ void __launch_bounds__(32) wait_selftest_kernel(int32_t kind, uint64_t limit_ns,
                                                           int32_t *status) {
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x == 0) {
        tc::mbar_init(&bar, 1);
        tc::fence_barrier_init();
    }
    __syncwarp();
    if (kind == 0) {
        tc::mbar_wait(&bar, 0, status, limit_ns);
    } else if (threadIdx.x == 0) {
        tc::wait_counter(&g_never_raised, 1, status, limit_ns);
    }
    __syncwarp();
}

}  // namespace

cudaError_t launch_wait_selftest(int32_t kind, uint64_t limit_ns, int32_t *status,
                                 cudaStream_t st) {
    wait_selftest_kernel<<<1, 32, 0, st>>>(kind, limit_ns, status);
    return cudaGetLastError();
}

}  // namespace bsa
