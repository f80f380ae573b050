// wait_limit.cu -- test-only diagnostic (libgdr_diag.so): the bounded
// mbarrier wait the library's kernels use, run against a barrier nothing
// ever arrives on, so that a test can see a wait give up after its limit,
// set the error word and leave the kernel and the context usable -- the
// failure path of every wait in the library, exercised without a fault.
#include <cuda_runtime.h>

#include "sm100_ptx.cuh"

namespace gdr {
namespace {

using namespace sm100;

// One CTA of 32 threads: thread 0 initialises an mbarrier expecting one
// arrival, which never comes; every thread waits on its first phase with
// the given limit, and each one that gives up adds one to *gave_up.
__global__ void __launch_bounds__(32, 1)
    gdr_selftest_wait_kernel(unsigned long long limit_ns, int *gave_up) {
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        fence_mbar_init();
    }
    __syncthreads();
    if (!mbar_wait_bounded(&bar, 0, limit_ns)) atomicAdd(gave_up, 1);
}

}  // namespace
}  // namespace gdr

// Launches the wait on `stream` with a limit of limit_ns nanoseconds
// (1 ms .. 1 s); `gave_up` a device int the kernel adds one to per thread
// whose wait ran out.  Returns 0, -1 for bad arguments, or the cudaError_t
// of the launch.
extern "C" __attribute__((visibility("default"))) int gdr_diag_wait_limit(
    unsigned long long limit_ns, int *gave_up, void *stream) {
    if (!gave_up || limit_ns < 1000000ull || limit_ns > 1000000000ull) return -1;
    gdr::gdr_selftest_wait_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(limit_ns,
                                                                                gave_up);
    return (int)cudaGetLastError();
}
