// Self-test of the failure path every kernel of the library shares: a bounded
// mbarrier wait that runs out sets the device error word (TT_ERR_TIMEOUT) and the
// kernel returns, leaving the context usable.
//
// The kernel initialises one mbarrier in shared memory that nothing ever arrives on
// (no TMA copy, no tensor-core operation and no other thread is involved), waits on
// it through the same helper the other kernels use, with the caller's limit, and
// reports the timeout.  It is there so that a test can make a wait run out on
// purpose without any fault, trap or endless loop.
#include "tt_device.cuh"
#include "tt_internal.h"

namespace tti {
namespace {

__global__ void __launch_bounds__(32) wait_timeout_kernel(int* err, unsigned long long limit_ns,
                                                          int* waited_out) {
    __shared__ __align__(8) unsigned long long bar;
    const uint32_t a = ttk::smem_u32(&bar);
    if (threadIdx.x == 0) {
        ttk::mbar_init(a, 1);
        ttk::fence_mbar_init();
    }
    __syncwarp();
    if (threadIdx.x == 0) {
        const bool ok = ttk::mbar_wait_for(a, 0u, limit_ns);
        if (!ok) ttk::report_error(err, ttk::kErrTimeout);
        if (waited_out != nullptr) *waited_out = ok ? 0 : 1;
    }
}

}  // namespace

cudaError_t launch_wait_timeout(int* err, unsigned long long limit_ns, int* waited_out,
                                cudaStream_t stream) {
    wait_timeout_kernel<<<1, 32, 0, stream>>>(err, limit_ns, waited_out);
    return cudaGetLastError();
}

}  // namespace tti
