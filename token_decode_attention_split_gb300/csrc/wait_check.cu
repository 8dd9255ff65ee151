// A check of the kernels' failure path: one thread waits, with the same bounded mbarrier wait
// the decode pipelines use, on a barrier that nothing ever completes.  The wait gives up after
// the limit, the thread records kErrWaitCheck in the device error word and the kernel returns,
// so a caller sees a timed-out wait as an error code while the context stays usable.
#include "launch.h"

namespace da {

__global__ void wait_check_kernel(unsigned* err, uint64_t limit_ns) {
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        fence_mbarrier_init();
    }
    __syncthreads();
    // No thread arrives on `bar`, so its phase 0 never completes.
    if (threadIdx.x == 0 && !mbar_wait(&bar, 0u, nullptr, limit_ns)) record_error(err, kErrWaitCheck);
}

cudaError_t launch_wait_check(unsigned* err, uint64_t limit_ns, cudaStream_t stream) {
    wait_check_kernel<<<1, 32, 0, stream>>>(err, limit_ns);
    return cudaGetLastError();
}

}  // namespace da
