// selftest.cu -- a kernel whose bounded waits cannot be met, so that the
// failure path of the device error word can be exercised without faulting or
// hanging the GPU: the waits give up after a few thousand polls and set the
// same bits the library's kernels set when a TMA/MMA completion or a
// look-back flag never arrives.
#include "la_launch.h"
#include "tc_common.cuh"

namespace la {
namespace {

using namespace la::tcf;

__global__ void expired_waits_kernel(unsigned* status, const unsigned* flag, uint32_t limit) {
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x != 0) return;
    mbar_init(&bar, 1);
    fence_mbar_init();
    // the barrier's first phase needs one arrival and gets none
    if (!mbar_wait(&bar, 0u, limit)) atomicOr(status, kErrWait);
    // a flag that nothing sets
    uint32_t n = 0;
    while (ld_acquire(flag) == 0u) {
        if (++n > limit) {
            atomicOr(status, kErrLookback);
            break;
        }
        __nanosleep(256);
    }
}

}  // namespace

cudaError_t selftest_expired_waits(const LaunchCtx& c) {
    unsigned* flag = nullptr;
    cudaError_t e = scratch_alloc(c, reinterpret_cast<void**>(&flag), sizeof(unsigned));
    if (e != cudaSuccess) return e;
    if ((e = cudaMemsetAsync(flag, 0, sizeof(unsigned), c.stream)) == cudaSuccess) {
        expired_waits_kernel<<<1, 32, 0, c.stream>>>(c.status_word, flag, 4096u);
        note_launch();
        e = cudaGetLastError();
    }
    scratch_free(c, flag);
    return e;
}

}  // namespace la
