// qk_watchdog.cu -- exercises the bounded-wait path that every kernel with
// an mbarrier wait uses: one thread waits on a barrier nothing arrives on,
// the wait runs out after limit_ns, the timeout lands in the device status
// word and the kernel returns (no trap, no fault, the context stays usable).
#include "qk_internal.h"
#include "qk_ptx.cuh"

namespace qk {
namespace {
__global__ void stalled_wait_kernel(unsigned* status, uint64_t limit_ns) {
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);   // phase 0 completes after one arrival, which never comes
        fence_barrier_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) mbar_wait_bounded(&bar, 0, status, limit_ns);
}
}  // namespace

cudaError_t launch_stalled_wait(unsigned* status, uint64_t limit_ns, cudaStream_t s) {
    stalled_wait_kernel<<<1, 32, 0, s>>>(status, limit_ns);
    return cudaGetLastError();
}
}  // namespace qk
