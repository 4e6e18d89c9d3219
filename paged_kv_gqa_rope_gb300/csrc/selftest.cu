// Self-test of the bounded wait every kernel of the library uses: a wait on
// an mbarrier phase that nothing completes gives up after the wait limit
// (about a second) and reports PA_DEV_TIMEOUT, and the context stays usable.
#include "common.cuh"
#include "internal.h"

namespace pa {
namespace {

__global__ void wait_timeout_kernel(int32_t *status) {
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        fence_barrier_init();
    }
    __syncthreads();
    // Nothing arrives on `bar`: its phase 0 never completes.
    if (threadIdx.x == 0 && !mbar_wait(&bar, 0)) report(status, PA_DEV_TIMEOUT);
}

}  // namespace
}  // namespace pa

extern "C" int pa_selftest_wait_timeout(int32_t *dev_status, pa_stream_t stream) {
    if (!dev_status) return PA_ERR_INVALID;
    pa::wait_timeout_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(dev_status);
    return pa::launch_status();
}
