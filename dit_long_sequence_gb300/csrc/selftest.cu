// selftest.cu -- exercises the bounded-wait (watchdog) path on the GPU without
// a fault: one CTA waits on an mbarrier that nothing ever arrives on, gives up
// after the limit, records DIT_ERR_TIMEOUT in the device status word (wait
// site kSiteSelfTest) and returns normally, so the context stays usable.
#include <cuda_runtime.h>

#include <cstdint>

#include "internal.h"
#include "ptx.cuh"

namespace dit {
namespace {

constexpr uint32_t kRoleSelfTest = 9;
constexpr uint32_t kSiteSelfTest = 99;

__global__ void watchdog_selftest_kernel(unsigned int* status, unsigned long long limit_ns) {
    __shared__ uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&bar), 1);
        abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();
    const Watchdog wd{status, limit_ns, &abort_flag};
    // Phase 0 never completes: every thread gives up after limit_ns (or when
    // the first one to give up raises the abort flag).
    wait_bounded(smem_u32(&bar), 0, wd, kRoleSelfTest, kSiteSelfTest);
    __syncthreads();
}

}  // namespace

cudaError_t launch_watchdog_selftest(unsigned int* status, unsigned long long limit_ns, cudaStream_t stream) {
    watchdog_selftest_kernel<<<1, 64, 0, stream>>>(status, limit_ns);
    return cudaGetLastError();
}

}  // namespace dit
