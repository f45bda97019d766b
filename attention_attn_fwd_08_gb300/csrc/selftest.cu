// selftest.cu -- exercises the bounded-wait path without faulting the GPU.
//
// One thread waits on an mbarrier that nothing will ever complete, gives up
// after `timeout_us`, records ST_SELFTEST in the status word and returns, so
// the context stays usable and the host reads the timeout as a status code.
#include "kernels.h"

namespace attn {
namespace {

__global__ void selftest_wait_kernel(unsigned int* status, unsigned long long limit_ns) {
    __shared__ uint64_t bar;
    if (threadIdx.x != 0) return;
    const uint32_t b = smem_u32(&bar);
    mbar_init(b, 1);
    fence_barrier_init();
    const unsigned long long t0 = globaltimer();
    bool done = false;
    while (!done) {
        done = mbar_try_wait(b, 0);  // phase 0 never completes: nobody arrives
        if (!done && globaltimer() - t0 > limit_ns) {
            atomicOr(status, (unsigned int)ST_SELFTEST);
            break;
        }
    }
}

}  // namespace

cudaError_t launch_selftest_wait(unsigned int* status, unsigned int timeout_us, cudaStream_t s) {
    selftest_wait_kernel<<<1, 32, 0, s>>>(status, (unsigned long long)timeout_us * 1000ull);
    return cudaGetLastError();
}

}  // namespace attn
