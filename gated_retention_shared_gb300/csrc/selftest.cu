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

// Occupies SMs for a while, to run the library's calls on a device shared with
// other work: each CTA claims most of an SM's shared memory (so no CTA of another
// kernel that needs much of it fits beside it) and sleeps until `ns` of wall time
// have passed since it started.  It reads and writes no global memory.
constexpr int kOccupySmem = 200 * 1024;

__global__ void selftest_occupy_kernel(uint64_t ns) {
    extern __shared__ uint8_t claim[];
    uint64_t t0, t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t0));
    do {
        __nanosleep(20000);
        asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    } while (t - t0 < ns);
    if (threadIdx.x == 0 && t == 0) claim[0] = 0;  // keeps the claim: never true
}

}  // namespace yoco

namespace yoco_host {

cudaError_t selftest_occupy(int ctas, uint64_t ns, cudaStream_t st) {
    cudaError_t e = cudaFuncSetAttribute(yoco::selftest_occupy_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         yoco::kOccupySmem);
    if (e != cudaSuccess) return e;
    count_launches(1);
    yoco::selftest_occupy_kernel<<<ctas, 32, yoco::kOccupySmem, st>>>(ns);
    return cudaGetLastError();
}

cudaError_t selftest_wait(void *ws, uint64_t limit_ns, cudaStream_t st) {
    count_launches(1);
    yoco::selftest_wait_kernel<<<1, 32, 0, st>>>((int *)ws, limit_ns);
    return cudaGetLastError();
}

}  // namespace yoco_host
