// Self-test of the bounded waits that every TMA and tensor-core kernel of this library uses.
//
// Each mbarrier wait in those kernels gives up after a time limit, records
// kDevErrMbarTimeout in the device error word and lets the kernel return, so that a copy or
// an MMA that never completes cannot hang the GPU. This kernel exercises that path on its
// own: one thread waits on an mbarrier that nothing arrives on (no copy, TMA load or MMA is
// in flight), with a short limit, and must come back with the error recorded.
#include "common.cuh"
#include "internal.h"

namespace spops {
namespace {

__global__ void __launch_bounds__(32) wait_selftest_kernel(uint64_t limit_ns, int* err,
                                                           unsigned long long* waited_ns) {
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&bar), 1);  // one arrival completes a phase; none ever comes
        fence_mbar_init();
    }
    __syncwarp();
    if (threadIdx.x == 0) {
        const uint64_t t0 = global_timer_ns();
        const bool done = mbar_wait_for(smem_u32(&bar), 0, err, limit_ns);
        const uint64_t t1 = global_timer_ns();
        if (waited_ns) *waited_ns = done ? 0ull : (unsigned long long)(t1 - t0);
    }
}

}  // namespace

cudaError_t launch_wait_selftest(uint64_t limit_ns, unsigned long long* waited_ns, cudaStream_t s) {
    int* err = device_error_word();
    if (!err) return cudaErrorInvalidDevice;
    wait_selftest_kernel<<<1, 32, 0, s>>>(limit_ns, err, waited_ns);
    count_launches(1);
    return cudaGetLastError();
}

}  // namespace spops
