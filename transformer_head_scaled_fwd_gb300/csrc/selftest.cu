// selftest.cu -- a kernel whose pipeline wait is made to run out, so the failure
// path every tensor-core kernel relies on (bounded mbarrier wait -> status code in
// the device status word -> the kernel ends) can be exercised on a GPU without
// faulting, trapping or hanging it.
//
// One thread initialises an mbarrier that expects one arrival, never arrives on
// it, and waits on its first phase through the same bounded wait the pipelines
// use, with a budget of 1024 try_wait rounds instead of the pipelines' 2^24. The
// wait gives up, records `code` and the kernel returns. Nothing else is in
// flight: no TMA copy, no MMA, no tensor memory.
#include "mha_internal.h"
#include "ptx.cuh"

namespace mha {
namespace {

constexpr uint32_t kSelftestWaitLimit = 1024;

__global__ void __launch_bounds__(32) wait_timeout_kernel(int* status, int code) {
    __shared__ uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        abort_flag = 0;
        fence_barrier_init();
    }
    __syncwarp();
    if (threadIdx.x == 0) mbar_wait_limit<kSelftestWaitLimit>(&bar, 0, &abort_flag, status, code);
}

}  // namespace

cudaError_t launch_wait_timeout_selftest(int* status, int code, cudaStream_t s) {
    wait_timeout_kernel<<<1, 32, 0, s>>>(status, code);
    return cudaGetLastError();
}

}  // namespace mha
