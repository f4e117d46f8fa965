// Test hook for the bounded device waits that every pipelined kernel of the
// library uses: one thread waits on an mbarrier phase that nothing completes, so
// the wait runs out at its deadline, records where it gave up, sets
// MOE_ERR_TIMEOUT in the status word and returns; the kernel then exits and the
// context stays usable.  This is how a lost producer shows up on this path
// without faulting or hanging the GPU.
#include "ptx.cuh"

namespace moe {
namespace {

__global__ void wait_timeout_kernel(int* status, int* diag) {
    __shared__ uint64_t bar;
    __shared__ volatile int abort_flag;
    if (threadIdx.x != 0) return;
    abort_flag = 0;
    mbar_init(&bar, 1);  // one arrival completes phase 0; none comes
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    if (mbar_wait(&bar, 0u, &abort_flag, status, diag, 1, 0, 0, 0)) {
        // the phase cannot complete: reaching this would mean the wait is broken
        set_status(status, MOE_ERR_CUDA);
    }
}

}  // namespace
}  // namespace moe

extern "C" int moe_debug_wait_timeout(int* status_dev, int32_t* diag_dev, void* stream) {
    if (!status_dev || !diag_dev) return MOE_ERR_INVALID_ARG;
    moe::wait_timeout_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(status_dev, diag_dev);
    return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
