// selftest.cu -- csa2_selftest_bounded_wait: the failure-detection check of the library's
// device waits.
//
// Every wait in these kernels (an mbarrier phase that a TMA copy, an MMA commit or another
// warp completes) is bounded: after its poll limit it gives up, the kernel sets
// CSA2_DEV_TIMEOUT in the caller's status word and returns, so a lost arrival ends the
// kernel instead of hanging the GPU, and the context stays usable.  This kernel makes that
// happen on purpose, without any fault: its threads wait, through the same routine the
// kernels use, on an mbarrier that nothing ever arrives on.
#include "common.cuh"
#include "internal.h"
#include "tc_util.cuh"

namespace csa2 {
namespace {

__global__ void __launch_bounds__(32) bounded_wait_selftest_kernel(uint32_t polls, uint32_t *d_status)
{
    __shared__ uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        tc::mbar_init(&bar, 1);           // one arrival would complete phase 0; none comes
        tc::fence_mbar_init();
        abort_flag = 0;
    }
    __syncthreads();
    const bool done = tc::mbar_wait_limit(&bar, 0u, &abort_flag, polls);
    if (!__any_sync(0xffffffffu, done) && threadIdx.x == 0) dev_flag(d_status, CSA2_DEV_TIMEOUT);
}

} // namespace

cudaError_t launch_bounded_wait_selftest(uint32_t polls, uint32_t *d_status, cudaStream_t s)
{
    bounded_wait_selftest_kernel<<<1, 32, 0, s>>>(polls, d_status);
    return cudaGetLastError();
}

} // namespace csa2
