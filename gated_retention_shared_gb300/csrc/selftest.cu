// selftest.cu -- checks the library's failure path on the device without faulting
// it: one thread waits on an mbarrier that nothing ever completes, with the same
// bounded wait the tensor-core kernels use, gives up after `limit_ns` and records
// the status word in the workspace exactly as a stalled kernel would.
#include "common.cuh"
#include "kernels.h"
#include "tc.cuh"

namespace yoco {

__global__ void selftest_wait_kernel(int *err, uint64_t limit_ns) {
    __shared__ uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x != 0) return;
    abort_flag = 0;
    tc::mbar_init(&bar, 1);
    tc::fence_mbar_init();
    // nothing arrives on `bar`: phase 0 never completes
    if (!tc::mbar_wait(&bar, 0, &abort_flag, limit_ns)) atomicExch(err, (int)(kErrMagic | 0xEEu));
}

}  // namespace yoco

namespace yoco_host {

cudaError_t selftest_wait(void *ws, uint64_t limit_ns, cudaStream_t st) {
    count_launches(1);
    yoco::selftest_wait_kernel<<<1, 32, 0, st>>>((int *)ws, limit_ns);
    return cudaGetLastError();
}

}  // namespace yoco_host
